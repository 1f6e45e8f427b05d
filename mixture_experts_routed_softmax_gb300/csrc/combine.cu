// combine.cu — the fp32 score-weighted gather-sum back to token order, and
// its transpose for the backward.
//
// prime-rl PR #3885 (DeepSeek-V4.1 Flash perf work), §Changes, "Single-pass
// DeepEP local layout": one fp32 score-weighted gather-sum back from the
// padded expert-grouped layout, with gathers (not scatters) in backward. Both
// kernels read rows by index and write each output exactly once: no atomics,
// fixed summation order.
#include "common.cuh"
#include "internal.h"

namespace moe {

// out[t] = sum_j w[t, j] * rows[dst_row[t*k + j]]  (slot order, fp32); one warp
// per (token, 256 columns), so a handful of tokens still spreads over many warps
__global__ void __launch_bounds__(256) combine_kernel(const moe_bf16* __restrict__ rows,
                                                      const int32_t* __restrict__ dst_row,
                                                      const float* __restrict__ topk_w,
                                                      int64_t T, int k, int d,
                                                      moe_bf16* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int nv = d / 8;
  const int nchunk = (nv + 31) / 32;
  const int64_t w = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (w >= T * nchunk) return;
  const int64_t t = w / nchunk;
  const int v = (int)(w - t * nchunk) * 32 + lane;
  int32_t my_r = -1;
  float my_w = 0.f;
  if (lane < k) {
    my_r = dst_row[t * k + lane];
    my_w = topk_w ? topk_w[t * k + lane] : 1.f;
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // the rows of up to four slots are loaded together, then summed in slot order
  for (int j0 = 0; j0 < k; j0 += 4) {
    uint4 rv[4];
    float wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q;
      const int32_t r = __shfl_sync(0xFFFFFFFFu, my_r, j & 31);
      wv[q] = __shfl_sync(0xFFFFFFFFu, my_w, j & 31);
      const bool ok = j < k && r >= 0 && v < nv;
      rv[q] = ok ? reinterpret_cast<const uint4*>(rows + (int64_t)r * d)[v]
                 : make_uint4(0u, 0u, 0u, 0u);
      if (!ok) wv[q] = 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float f[8];
      unpack8(rv[q], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wv[q], f[i], acc[i]);
    }
  }
  if (v < nv) reinterpret_cast<uint4*>(out + t * d)[v] = pack8(acc);
}

cudaError_t launch_combine(const moe_bf16* rows, const int32_t* dst_row, const float* topk_w,
                           int64_t T, int k, int d, moe_bf16* out, cudaStream_t s) {
  timer_before(MOE_KERNEL_COMBINE, s);
  const int64_t warps = T * (((int64_t)d / 8 + 31) / 32);
  combine_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(rows, dst_row, topk_w, T, k, d, out);
  note_launches(1);
  timer_after(MOE_KERNEL_COMBINE, s);
  return cudaGetLastError();
}

// Transpose of the weighted combine, one warp per row r of the layout:
//   dyp[r] = w(p) * dy[t(p)],  d_topk_w[p] = <dy[t(p)], yp[r]>  (fp32)
// with p = src_pair[r]; padding rows get dyp = 0. Rows >= offsets[E] are
// not touched.
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const moe_bf16* __restrict__ dy, const moe_bf16* __restrict__ yp,
    const int32_t* __restrict__ src_pair, const float* __restrict__ topk_w,
    const int64_t* __restrict__ offsets, int k, int E, int d, int64_t R_cap,
    moe_bf16* __restrict__ dyp, float* __restrict__ d_topk_w) {
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= R_cap || r >= offsets[E]) return;
  const int nv = d / 8;
  uint4* out = reinterpret_cast<uint4*>(dyp + r * d);
  const int32_t p = src_pair[r];
  if (p < 0) {
    for (int v = lane; v < nv; v += 32) out[v] = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const int64_t t = p / k;
  const float w = topk_w[p];
  const uint4* g = reinterpret_cast<const uint4*>(dy + t * d);
  const uint4* y = reinterpret_cast<const uint4*>(yp + r * d);
  float dot = 0.f;
  // four 16-byte pieces of each row in flight per lane, then used in order
  for (int v0 = lane; v0 < nv; v0 += 128) {
    uint4 gv[4], yv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + 32 * u;
      if (v < nv) { gv[u] = g[v]; yv[u] = y[v]; }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nv) break;
      float a[8], b[8], o[8];
      unpack8(gv[u], a);
      unpack8(yv[u], b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dot = fmaf(a[i], b[i], dot);
        o[i] = w * a[i];
      }
      out[v] = pack8(o);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
  if (lane == 0) d_topk_w[p] = dot;
}

cudaError_t launch_combine_bwd(const moe_bf16* dy, const moe_bf16* yp, const int32_t* src_pair,
                               const float* topk_w, const int64_t* offsets, int64_t T, int k,
                               int E, int d, int64_t R_cap, moe_bf16* dyp, float* d_topk_w,
                               cudaStream_t s) {
  (void)T;
  timer_before(MOE_KERNEL_COMBINE_BWD, s);
  combine_bwd_kernel<<<(unsigned)((R_cap + 7) / 8), 256, 0, s>>>(dy, yp, src_pair, topk_w,
                                                                 offsets, k, E, d, R_cap, dyp,
                                                                 d_topk_w);
  note_launches(1);
  timer_after(MOE_KERNEL_COMBINE_BWD, s);
  return cudaGetLastError();
}

}  // namespace moe
