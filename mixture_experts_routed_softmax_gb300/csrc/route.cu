// route.cu — router: logits, top-k with renormalised softmax weights, and the
// router backward.
//
// Routing over many experts with top-k selection is the setting of PocketLLM
// "Qwen4-Exp Heterogeneous TP4 Performance", §Runtime architecture (512
// routed experts, top-10), where the router is its own per-layer phase
// (§Remaining prefill attribution). The formula (softmax over the experts,
// keep the k largest, renormalise over them) is the plainest reading: the
// full softmax denominator cancels, so selecting on the logits and taking
// the softmax over the selected ones gives the same weights without ties
// created by rounding of exp.
#include "common.cuh"
#include "internal.h"

namespace moe {

// ---------------------------------------------------------------------------
// logits[T, E] = x[T, d] (bf16) . W_r[d, E] (fp32) + b on the tensor cores.
// W_r is split exactly into three bf16 parts, W_hi + W_mid + W_lo (8 + 8 + 8
// significant bits: the fp32 value to within its last bit); a bf16 x bf16
// product is exact in fp32, so x . W_r accumulates in fp32 from exact
// products, as a CUDA-core fp32 dot product would. The parts are stacked
// along K in the workspace, [3d, E8] with E8 = E rounded up to 8 (16-byte
// rows for TMA), and one grouped-GEMM launch reduces over all 3d rows.
// ---------------------------------------------------------------------------
static inline int round8(int v) { return (v + 7) & ~7; }

static inline size_t al256r(size_t b) { return (b + 255) & ~(size_t)255; }

// workspace: the split weight [3d, E8] bf16, then (split K) fp32 partials [ksplit, T, E]
size_t route_ws_bytes(int64_t T, int d, int E) {
  const int sp = router_ksplit(T, d, E);
  return al256r((size_t)3 * d * round8(E) * 2) + (sp > 1 ? al256r((size_t)sp * T * E * 4) : 0);
}

// logits = sum of the split-K partials in split order, plus the bias
__global__ void router_reduce_kernel(const float* __restrict__ part, int ksplit, int64_t n, int E,
                                     const float* __restrict__ bias, float* __restrict__ logits) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float acc = 0.f;
  for (int sp = 0; sp < ksplit; ++sp) acc += part[(int64_t)sp * n + i];
  logits[i] = acc + (bias ? bias[i % E] : 0.f);
}

__global__ void split_router_weight_kernel(const float* __restrict__ wr, int d, int E, int E8,
                                           moe_bf16* __restrict__ w_split) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)d * E8) return;
  const int row = (int)(i / E8), e = (int)(i % E8);
  const float w = (e < E) ? wr[(int64_t)row * E + e] : 0.f;
  const __nv_bfloat16 hi = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(mid);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
  const int64_t plane = (int64_t)d * E8;
  w_split[i] = __bfloat16_as_ushort(hi);
  w_split[plane + i] = __bfloat16_as_ushort(mid);
  w_split[2 * plane + i] = __bfloat16_as_ushort(lo);
}

cudaError_t launch_router_logits(const moe_bf16* x, const float* w_router, const float* bias,
                                 int64_t T, int d, int E, float* logits, void* ws, int* status,
                                 cudaStream_t s) {
  const int E8 = round8(E);
  moe_bf16* w_split = static_cast<moe_bf16*>(ws);
  const int64_t n = (int64_t)d * E8;
  timer_before(MOE_KERNEL_ROUTER_LOGITS, s);
  split_router_weight_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(w_router, d, E, E8,
                                                                        w_split);
  note_launches(1);
  cudaError_t e = cudaGetLastError();
  const int sp = router_ksplit(T, d, E);
  if (sp == 1) {
    if (e == cudaSuccess) e = launch_router_gemm(x, w_split, bias, T, d, E, E8, 1, logits, status, s);
  } else {
    float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) +
                                           al256r((size_t)3 * d * E8 * 2));
    if (e == cudaSuccess) e = launch_router_gemm(x, w_split, bias, T, d, E, E8, sp, part, status, s);
    if (e == cudaSuccess) {
      const int64_t nel = T * E;
      router_reduce_kernel<<<(unsigned)((nel + 255) / 256), 256, 0, s>>>(part, sp, nel, E, bias,
                                                                         logits);
      note_launches(1);
      e = cudaGetLastError();
    }
  }
  timer_after(MOE_KERNEL_ROUTER_LOGITS, s);
  return e;
}

// ---------------------------------------------------------------------------
// Top-k and weights: one warp per token. Each lane keeps the logits of
// experts lane, lane+32, ... in registers; k rounds of a warp arg-max pick the
// slots in descending order (equal values: lower index first). Slot j's lane
// then computes exp(l_j - l_0) and the warp sums them.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool ranks_above(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   const int32_t* __restrict__ forced, int64_t T,
                                                   int E, int k, int32_t* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w, int* status) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  const float* lrow = logits + t * E;
  float my_v = -INFINITY;  // slot `lane`'s logit (lanes < k)
  int my_i = 0;
  bool valid = true;
  if (forced) {
    if (lane < k) {
      my_i = forced[t * k + lane];
      valid = (my_i >= 0 && my_i < E);
      if (valid) my_v = lrow[my_i];
      else raise_status(status, MOE_ERR_DEVICE_INDEX);
    }
  } else {
    float v[kMaxExperts / 32];
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < E) ? lrow[e] : -INFINITY;
    }
    uint32_t taken = 0;
    for (int j = 0; j < k; ++j) {
      float bv = -INFINITY;
      int bi = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; ++i) {
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
    topk_idx[t * k + lane] = my_i;
    topk_w[t * k + lane] = sum > 0.f ? ex / sum : 0.f;
  }
}

cudaError_t launch_topk(const float* logits, const int32_t* forced_idx, int64_t T, int E, int k,
                        int32_t* topk_idx, float* topk_w, int* status, cudaStream_t s) {
  const int warps = 8;
  dim3 grid((unsigned)((T + warps - 1) / warps));
  timer_before(MOE_KERNEL_TOPK, s);
  topk_kernel<<<grid, warps * 32, 0, s>>>(logits, forced_idx, T, E, k, topk_idx, topk_w, status);
  note_launches(1);
  timer_after(MOE_KERNEL_TOPK, s);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Router backward.
//   dl_t,j = w_j (dw_j - sum_j' w_j' dw_j')  on the selected slots
//   dx[t] += sum_j dl_t,j W_r[:, e_j]
//   dW_r[:, e] = sum over e's rows of dl * xp[row];  db[e] = sum of dl
// The last two are fixed-order two-phase sums: phase 1 sums each (128-row
// block) n (expert group) segment of the padded layout into a partial row,
// phase 2 adds each expert's partial rows in row order. No atomics.
// ---------------------------------------------------------------------------
constexpr int kRbRows = 128;   // rows of the padded layout per phase-1 CTA
constexpr int kRbCols = 1024;  // columns of d per phase-1 CTA (128 threads x 8)

static inline int seg_unit(int align) { return align < kRbRows ? align : kRbRows; }

static inline size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

size_t route_bwd_ws_bytes(int64_t T, int d, int E, int k, int align) {
  const int64_t R_cap = T * k + (int64_t)E * (align - 1);
  const int64_t slots = (R_cap + seg_unit(align) - 1) / seg_unit(align);
  return al256((size_t)E * d * 4) + al256((size_t)T * k * 4) + al256((size_t)slots * d * 4) +
         al256((size_t)slots * 4);
}

__global__ void transpose_f32_kernel(const float* __restrict__ in, int rows, int cols,
                                     float* __restrict__ out) {
  __shared__ float tile[32][33];
  const int c = blockIdx.x * 32 + threadIdx.x;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int r = blockIdx.y * 32 + i;
    tile[i][threadIdx.x] = (r < rows && c < cols) ? in[(int64_t)r * cols + c] : 0.f;
  }
  __syncthreads();
  const int r2 = blockIdx.y * 32 + threadIdx.x;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int c2 = blockIdx.x * 32 + i;
    if (c2 < cols && r2 < rows) out[(int64_t)c2 * rows + r2] = tile[threadIdx.x][i];
  }
}

// one warp per token: dl for its k slots, then dx[t]. With dxp given, dx[t] =
// sum_j dxp[dst_row[t, j]] + sum_j dl_j W_r[:, e_j] in fp32, written once (the
// permute transpose fused in); without it, dx[t] += sum_j dl_j W_r[:, e_j].
__global__ void __launch_bounds__(256) route_bwd_token_kernel(
    const float* __restrict__ d_topk_w, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ wrT, int64_t T, int d, int E,
    int k, float* __restrict__ dl_pair, moe_bf16* __restrict__ dx,
    const moe_bf16* __restrict__ dxp, const int32_t* __restrict__ dst_row) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  float w = 0.f, dw = 0.f;
  int e = -1, r = -1;
  if (lane < k) {
    w = topk_w[t * k + lane];
    dw = d_topk_w[t * k + lane];
    e = topk_idx[t * k + lane];
    if (e < 0 || e >= E) { e = -1; w = 0.f; dw = 0.f; }
    if (dxp) r = dst_row[t * k + lane];
  }
  float inner = w * dw;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) inner += __shfl_xor_sync(0xFFFFFFFFu, inner, off);
  const float dl = w * (dw - inner);
  if (lane < k) dl_pair[t * k + lane] = dl;
  moe_bf16* dxr = dx + t * d;
  // every lane runs the same number of iterations: the shuffles need the whole warp
  for (int c0 = 0; c0 < d; c0 += 256) {
    const int c = c0 + lane * 8;
    const bool in = c < d;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (in && !dxp) unpack8(*reinterpret_cast<const uint4*>(dxr + c), acc);
    for (int j = 0; j < k; ++j) {
      const int rj = __shfl_sync(0xFFFFFFFFu, r, j);
      if (!in || rj < 0) continue;
      float f[8];
      unpack8(*reinterpret_cast<const uint4*>(dxp + (int64_t)rj * d + c), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    float add[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int j = 0; j < k; ++j) {
      const float dlj = __shfl_sync(0xFFFFFFFFu, dl, j);
      const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
      if (ej < 0 || !in) continue;
      const float4 a = *reinterpret_cast<const float4*>(wrT + (int64_t)ej * d + c);
      const float4 b = *reinterpret_cast<const float4*>(wrT + (int64_t)ej * d + c + 4);
      add[0] = fmaf(dlj, a.x, add[0]); add[1] = fmaf(dlj, a.y, add[1]);
      add[2] = fmaf(dlj, a.z, add[2]); add[3] = fmaf(dlj, a.w, add[3]);
      add[4] = fmaf(dlj, b.x, add[4]); add[5] = fmaf(dlj, b.y, add[5]);
      add[6] = fmaf(dlj, b.z, add[6]); add[7] = fmaf(dlj, b.w, add[7]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += add[i];
    if (in) *reinterpret_cast<uint4*>(dxr + c) = pack8(acc);
  }
}

__device__ __forceinline__ int expert_of_row(const int64_t* offsets, int E, int64_t r) {
  // largest e with offsets[e] <= r (offsets non-decreasing, offsets[0] = 0)
  int lo = 0, hi = E;  // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// phase 1: CTA (b, cb) sums rows [b*128, b*128+128) for columns [cb*1024, +1024)
// (8 per thread, 16-byte loads), one partial row per expert segment it meets;
// slot = segment start / unit.
__global__ void __launch_bounds__(128) route_bwd_partial_kernel(
    const int64_t* __restrict__ offsets, const int32_t* __restrict__ src_pair,
    const moe_bf16* __restrict__ xp, const float* __restrict__ dl_pair, int E, int d, int unit,
    float* __restrict__ part, float* __restrict__ part_db) {
  __shared__ float s_dl[kRbRows];     // dl of each row's pair, 0 for padding rows
  __shared__ int s_real[kRbRows];
  const int64_t r_begin = (int64_t)blockIdx.x * kRbRows;
  const int64_t R_pad = offsets[E];
  if (r_begin >= R_pad) return;
  const int64_t r_end = min(r_begin + kRbRows, R_pad);
  {
    const int64_t q = r_begin + threadIdx.x;
    const int pr = (q < r_end) ? src_pair[q] : -1;
    s_real[threadIdx.x] = pr >= 0;
    s_dl[threadIdx.x] = pr >= 0 ? dl_pair[pr] : 0.f;
  }
  __syncthreads();
  const int c = blockIdx.y * kRbCols + threadIdx.x * 8;
  int64_t r = r_begin;
  while (r < r_end) {
    const int e = expert_of_row(offsets, E, r);
    const int64_t seg_end = min(r_end, offsets[e + 1]);
    const int64_t slot = r / unit;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float adb = 0.f;
#pragma unroll 4
    for (int64_t q = r; q < seg_end; ++q) {
      const int i = (int)(q - r_begin);
      if (!s_real[i]) continue;
      const float dl = s_dl[i];
      adb += dl;
      if (c < d) {
        float f[8];
        unpack8(*reinterpret_cast<const uint4*>(xp + q * d + c), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = fmaf(dl, f[j], a[j]);
      }
    }
    if (c < d) {
      float4* o = reinterpret_cast<float4*>(part + slot * d + c);
      o[0] = make_float4(a[0], a[1], a[2], a[3]);
      o[1] = make_float4(a[4], a[5], a[6], a[7]);
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) part_db[slot] = adb;
    r = seg_end;
  }
}

// phase 2: per expert, add its partial rows in row order (2 columns per thread).
constexpr int kRdCols = 256;
__global__ void __launch_bounds__(128) route_bwd_reduce_kernel(
    const int64_t* __restrict__ offsets, const float* __restrict__ part,
    const float* __restrict__ part_db, int E, int d, int unit, float* __restrict__ dw_router,
    float* __restrict__ dbias) {
  const int e = blockIdx.x;
  const int c = blockIdx.y * kRdCols + threadIdx.x * 2;
  const int64_t g0 = offsets[e], g1 = offsets[e + 1];
  float a0 = 0.f, a1 = 0.f, adb = 0.f;
  int64_t r = g0;
  while (r < g1) {
    const int64_t slot = r / unit;
    if (c < d) {
      a0 += part[slot * d + c];
      a1 += part[slot * d + c + 1];
    }
    adb += part_db[slot];
    r = min(g1, (r / kRbRows + 1) * kRbRows);  // next 128-row block boundary
  }
  if (c < d) {
    dw_router[(int64_t)c * E + e] = a0;
    dw_router[(int64_t)(c + 1) * E + e] = a1;
  }
  if (dbias && blockIdx.y == 0 && threadIdx.x == 0) dbias[e] = adb;
}

cudaError_t launch_route_bwd(const float* d_topk_w, const float* topk_w, const int32_t* topk_idx,
                             const float* w_router, const int64_t* offsets,
                             const int32_t* src_pair, const moe_bf16* xp, int64_t T, int d, int E,
                             int k, int align, moe_bf16* dx_inout, const moe_bf16* dxp,
                             const int32_t* dst_row, float* dw_router, float* dbias, void* ws,
                             cudaStream_t s) {
  const int64_t R_cap = T * k + (int64_t)E * (align - 1);
  const int unit = seg_unit(align);
  char* p = static_cast<char*>(ws);
  float* wrT = reinterpret_cast<float*>(p);
  p += al256((size_t)E * d * 4);
  float* dl_pair = reinterpret_cast<float*>(p);
  p += al256((size_t)T * k * 4);
  const int64_t slots = (R_cap + unit - 1) / unit;
  float* part = reinterpret_cast<float*>(p);
  p += al256((size_t)slots * d * 4);
  float* part_db = reinterpret_cast<float*>(p);

  timer_before(MOE_KERNEL_ROUTE_BWD, s);
  transpose_f32_kernel<<<dim3((E + 31) / 32, (d + 31) / 32), dim3(32, 8), 0, s>>>(w_router, d, E,
                                                                                  wrT);
  if (T > 0)
    route_bwd_token_kernel<<<(unsigned)((T + 7) / 8), 256, 0, s>>>(d_topk_w, topk_w, topk_idx,
                                                                   wrT, T, d, E, k, dl_pair,
                                                                   dx_inout, dxp, dst_row);
  const int cblocks = (d + kRbCols - 1) / kRbCols;
  route_bwd_partial_kernel<<<dim3((unsigned)((R_cap + kRbRows - 1) / kRbRows), cblocks), 128, 0,
                             s>>>(offsets, src_pair, xp, dl_pair, E, d, unit, part, part_db);
  route_bwd_reduce_kernel<<<dim3(E, (d + kRdCols - 1) / kRdCols), 128, 0, s>>>(
      offsets, part, part_db, E, d, unit, dw_router, dbias);
  note_launches(T > 0 ? 4 : 3);
  timer_after(MOE_KERNEL_ROUTE_BWD, s);
  return cudaGetLastError();
}

}  // namespace moe
