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

// out[t] = sum_j w[t, j] * rows[dst_row[t*k + j]] + sum_s rows[dst_row[T*k + s*T + t]]
// (fp32 rows, slot order, the S shared experts' rows last with weight 1, fp32
// sum, rounded to bf16 once); one warp per (token, 256 columns), so a handful
// of tokens still spreads over many warps
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ rows,
                                                      const int32_t* __restrict__ dst_row,
                                                      const float* __restrict__ topk_w,
                                                      int64_t T, int k, int S, int d,
                                                      moe_bf16* __restrict__ out) {
  pdl_enter();
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
  } else if (lane < k + S) {
    my_r = dst_row[T * k + (int64_t)(lane - k) * T + t];
    my_w = 1.f;
  }
  const int slots = k + S;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  // the 8-column pieces of up to four slots' rows are loaded together, then
  // summed in slot order
  for (int j0 = 0; j0 < slots; j0 += 4) {
    float4 rv[4][2];
    float wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + q;
      const int32_t r = __shfl_sync(0xFFFFFFFFu, my_r, j & 31);
      wv[q] = __shfl_sync(0xFFFFFFFFu, my_w, j & 31);
      const bool ok = j < slots && r >= 0 && v < nv;
      if (ok) {
        const float4* src = reinterpret_cast<const float4*>(rows + (int64_t)r * d) + 2 * v;
        rv[q][0] = src[0];
        rv[q][1] = src[1];
      } else {
        rv[q][0] = rv[q][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        wv[q] = 0.f;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[0] = fmaf(wv[q], rv[q][0].x, acc[0]); acc[1] = fmaf(wv[q], rv[q][0].y, acc[1]);
      acc[2] = fmaf(wv[q], rv[q][0].z, acc[2]); acc[3] = fmaf(wv[q], rv[q][0].w, acc[3]);
      acc[4] = fmaf(wv[q], rv[q][1].x, acc[4]); acc[5] = fmaf(wv[q], rv[q][1].y, acc[5]);
      acc[6] = fmaf(wv[q], rv[q][1].z, acc[6]); acc[7] = fmaf(wv[q], rv[q][1].w, acc[7]);
    }
  }
  if (v < nv) reinterpret_cast<uint4*>(out + t * d)[v] = pack8(acc);
}

cudaError_t launch_combine(const float* rows, const int32_t* dst_row, const float* topk_w,
                           int64_t T, int k, int S, int d, moe_bf16* out, cudaStream_t s) {
  timer_before(MOE_KERNEL_COMBINE, s);
  const int64_t warps = T * (((int64_t)d / 8 + 31) / 32);
  launch_pdl(pdl_for_tokens(T), combine_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s,
             rows, dst_row, topk_w, T, k, S, d, out);
  note_launches(1);
  timer_after(MOE_KERNEL_COMBINE, s);
  return cudaGetLastError();
}

// Transpose of the weighted combine, one warp per row r of the layout, with
// p = src_pair[r] and t its token (a routed pair p < T*k: t = p / k, weight
// w(p); a shared expert's pair T*k + s*T + t: weight 1):
//   dyg[r] = dy[t]                 (the gathered upstream gradient, unscaled:
//                                   the down dgrad's operand; the score is
//                                   applied there to the fp32 accumulator)
//   dyp[r] = w(p) * dy[t]          (bf16: the weight gradient's operand)
// Padding rows get dyg = dyp = 0. Rows >= offsets[E] are not touched. The
// gradient of the top-k weights, <dy[t], Yu>, is taken in the down dgrad's
// epilogue instead, where dy . W_down^T and the unrounded A meet.
__global__ void __launch_bounds__(256) combine_bwd_kernel(
    const moe_bf16* __restrict__ dy, const int32_t* __restrict__ src_pair,
    const float* __restrict__ topk_w, const int64_t* __restrict__ offsets, int64_t T, int k,
    int E, int d, int64_t R_cap, moe_bf16* __restrict__ dyg, moe_bf16* __restrict__ dyp) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= R_cap || r >= offsets[E]) return;
  const int nv = d / 8;
  uint4* outg = reinterpret_cast<uint4*>(dyg + r * d);
  uint4* outp = reinterpret_cast<uint4*>(dyp + r * d);
  const int32_t p = src_pair[r];
  if (p < 0) {
    for (int v = lane; v < nv; v += 32) {
      outg[v] = make_uint4(0u, 0u, 0u, 0u);
      outp[v] = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }
  const int64_t Pr = T * k;
  const int64_t t = p < Pr ? p / k : (p - Pr) % T;
  const float w = p < Pr ? topk_w[p] : 1.f;
  const uint4* g = reinterpret_cast<const uint4*>(dy + t * d);
  // four 8-column pieces of the row in flight per lane
  for (int v0 = lane; v0 < nv; v0 += 128) {
    uint4 gv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + 32 * u;
      if (v < nv) gv[u] = g[v];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nv) break;
      float a[8], o[8];
      unpack8(gv[u], a);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = w * a[i];
      outg[v] = gv[u];
      outp[v] = pack8(o);
    }
  }
}

cudaError_t launch_combine_bwd(const moe_bf16* dy, const int32_t* src_pair, const float* topk_w,
                               const int64_t* offsets, int64_t T, int k, int E, int d,
                               int64_t R_cap, moe_bf16* dyg, moe_bf16* dyp, cudaStream_t s) {
  timer_before(MOE_KERNEL_COMBINE_BWD, s);
  launch_pdl(pdl_for_tokens(T), combine_bwd_kernel, dim3((unsigned)((R_cap + 7) / 8)), dim3(256), 0,
             s, dy, src_pair, topk_w, offsets, T, k, E, d, R_cap, dyg, dyp);
  note_launches(1);
  timer_after(MOE_KERNEL_COMBINE_BWD, s);
  return cudaGetLastError();
}

// d_topk_w[p] = sum_{s < slots} part[dst_row[p]][s], in slot order (the down
// dgrad's per-tile partials of <dy . W_down^T, A>); pairs dropped from the
// layout (dst_row = -1) are left untouched.
__global__ void __launch_bounds__(256) dtw_finalize_kernel(const float* __restrict__ part,
                                                           int slots,
                                                           const int32_t* __restrict__ dst_row,
                                                           int64_t P, float* __restrict__ d_topk_w) {
  pdl_enter();
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= P) return;
  const int32_t r = dst_row[p];
  if (r < 0) return;
  const float* q = part + (int64_t)r * slots;
  float a = 0.f;
  for (int s = 0; s < slots; ++s) a += q[s];
  d_topk_w[p] = a;
}

cudaError_t launch_dtw_finalize(const float* part, int slots, const int32_t* dst_row, int64_t P,
                                float* d_topk_w, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  launch_pdl(pdl_for_pairs(P), dtw_finalize_kernel, dim3((unsigned)((P + 255) / 256)), dim3(256), 0,
             s, part, slots, dst_row, P, d_topk_w);
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
