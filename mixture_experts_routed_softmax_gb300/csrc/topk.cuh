// topk.cuh — top-k with renormalised softmax weights for one token, one warp.
//
// Routing over many experts with top-k selection is the setting of PocketLLM
// "Qwen4-Exp Heterogeneous TP4 Performance", §Runtime architecture. Each lane
// keeps the logits of experts lane, lane+32, ... in registers; k rounds of a
// warp arg-max pick the slots in descending order (equal values: lower index
// first). Slot j's lane then computes exp(l_j - l_0) and the warp sums them.
// The whole warp must call it (it shuffles).
#pragma once
#include "common.cuh"

namespace moe {

__device__ __forceinline__ bool ranks_above(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// lrow: the token's E logits; forced: its k caller-chosen experts or NULL;
// writes idx_out[0..k) and w_out[0..k)
template <int NV>   // logits per lane: 32 * NV >= E
__device__ __forceinline__ void topk_warp(const float* __restrict__ lrow,
                                          const int32_t* __restrict__ forced, int E, int k,
                                          int lane, int32_t* __restrict__ idx_out,
                                          float* __restrict__ w_out, int* status) {
  float my_v = -INFINITY;  // slot `lane`'s logit (lanes < k)
  int my_i = 0;
  bool valid = true;
  if (forced) {
    if (lane < k) {
      my_i = forced[lane];
      valid = (my_i >= 0 && my_i < E);
      if (valid) my_v = lrow[my_i];
      else raise_status(status, MOE_ERR_DEVICE_INDEX);
    }
  } else {
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? lrow[e] : -INFINITY;
    }
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && ranks_above(v[i], e, bv, bi)) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
        if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
      }
      if (bi != 0x7FFFFFFF && (bi & 31) == lane) taken |= 1u << (bi >> 5);
      if (lane == j) { my_v = bv; my_i = (bi == 0x7FFFFFFF) ? 0 : bi; }
    }
  }
  // renormalised softmax over the k slots
  float m = (lane < k && valid) ? my_v : -INFINITY;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
  float ex = (lane < k && valid) ? expf(my_v - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
  if (lane < k) {
    idx_out[lane] = my_i;
    w_out[lane] = sum > 0.f ? ex / sum : 0.f;
  }
}

}  // namespace moe
