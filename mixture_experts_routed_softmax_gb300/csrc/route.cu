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
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

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

// A few tokens (decode) take the CUDA cores in two launches: row-slice partial
// dot products, then one CTA per token that adds them, writes the logits and
// takes the top-k. The slices: at most kSmallSlices per 128 experts.
constexpr int kRouterSmallMaxT = 32;   // route_is_small
constexpr int kSmallTok = 8;        // tokens a CTA of the partial kernel multiplies
constexpr int kSmallCols = 128;     // experts a CTA covers: 4 per lane
constexpr int kSmallSlices = 32;
constexpr int kSmallWarps = 8;

static inline int small_slice_rows(int d) {
  const int n = (d + 63) / 64 < kSmallSlices ? (d + 63) / 64 : kSmallSlices;
  const int rs = (d + n - 1) / n;
  return (rs + kSmallWarps - 1) / kSmallWarps * kSmallWarps;   // whole rows per warp
}

// workspace: the split weight [3d, E8] bf16, then (split K) fp32 partials
// [ksplit, T, E]; a few tokens use it for their row-slice partials instead
size_t route_ws_bytes(int64_t T, int d, int E) {
  const int sp = router_ksplit(T, d, E);
  const size_t big = al256r((size_t)3 * d * round8(E) * 2) + (sp > 1 ? al256r((size_t)sp * T * E * 4) : 0);
  if (T > kRouterSmallMaxT) return big;
  const int rs = small_slice_rows(d), ns = (d + rs - 1) / rs;
  const size_t small = al256r((size_t)ns * T * E * 4);
  return big > small ? big : small;
}

// logits = sum of the split-K partials in split order, plus the bias
__global__ void router_reduce_kernel(const float* __restrict__ part, int ksplit, int64_t n, int E,
                                     const float* __restrict__ bias, float* __restrict__ logits) {
  pdl_enter();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  float acc = 0.f;
  for (int sp = 0; sp < ksplit; ++sp) acc += part[(int64_t)sp * n + i];
  logits[i] = acc + (bias ? bias[i % E] : 0.f);
}

__global__ void split_router_weight_kernel(const float* __restrict__ wr, int d, int E, int E8,
                                           moe_bf16* __restrict__ w_split) {
  pdl_enter();
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

// Partial logits of a few tokens: CTA (chunk, slice, token group) multiplies
// rows [slice * rs, slice * rs + rs) of W_r[:, chunk * 128 : + 128] with up to
// eight tokens. Each warp takes rs / 8 consecutive rows, a lane four experts
// (16-byte loads, eight rows' loads in flight), in fp32 from exact products of
// bf16 and fp32 values; the warps' sums meet in shared memory in warp order.
// part: [ns, T, E].
__global__ void __launch_bounds__(kSmallWarps * 32) router_small_partial_kernel(
    const moe_bf16* __restrict__ x, const float* __restrict__ w_router, int64_t T, int d, int E,
    int rs, float* __restrict__ part) {
  pdl_enter();
  __shared__ float4 red[kSmallWarps][kSmallTok][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e0 = blockIdx.x * kSmallCols + 4 * lane;
  const int slice = blockIdx.y, t0 = blockIdx.z * kSmallTok;
  const int nt = (int)(T - t0 < kSmallTok ? T - t0 : kSmallTok);
  const int rpw = rs / kSmallWarps;
  const int r0 = slice * rs + warp * rpw;
  const bool vec = (E % 4) == 0 && (reinterpret_cast<uintptr_t>(w_router) & 15u) == 0;
  float acc[kSmallTok][4];
#pragma unroll
  for (int t = 0; t < kSmallTok; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  for (int rb = 0; rb < rpw; rb += 8) {
    float4 wv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = r0 + rb + u;
      wv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rb + u < rpw && i < d) {
        const float* src = w_router + (int64_t)i * E + e0;
        if (vec && e0 + 3 < E) {
          wv[u] = __ldg(reinterpret_cast<const float4*>(src));
        } else {
          if (e0 < E) wv[u].x = __ldg(src);
          if (e0 + 1 < E) wv[u].y = __ldg(src + 1);
          if (e0 + 2 < E) wv[u].z = __ldg(src + 2);
          if (e0 + 3 < E) wv[u].w = __ldg(src + 3);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = r0 + rb + u;
      if (rb + u >= rpw || i >= d) break;
#pragma unroll
      for (int t = 0; t < kSmallTok; ++t) {
        if (t < nt) {
          const float xv = __bfloat162float(__ushort_as_bfloat16(x[(t0 + t) * (int64_t)d + i]));
          acc[t][0] = fmaf(xv, wv[u].x, acc[t][0]);
          acc[t][1] = fmaf(xv, wv[u].y, acc[t][1]);
          acc[t][2] = fmaf(xv, wv[u].z, acc[t][2]);
          acc[t][3] = fmaf(xv, wv[u].w, acc[t][3]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kSmallTok; ++t)
    red[warp][t][lane] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
  __syncthreads();
  for (int o = threadIdx.x; o < nt * kSmallCols; o += blockDim.x) {
    const int t = o / kSmallCols, col = o % kSmallCols, e = blockIdx.x * kSmallCols + col;
    if (e >= E) continue;
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kSmallWarps; ++w) sum += reinterpret_cast<const float*>(&red[w][t][0])[col];
    part[((int64_t)slice * T + t0 + t) * E + e] = sum;
  }
}

// One CTA per token: logits = the slices' partials in slice order + bias, then
// the top-k with renormalised weights (topk.cuh) on them.
template <int NV>
__global__ void __launch_bounds__(256) router_small_topk_kernel(
    const float* __restrict__ part, int ns, int64_t T, int E, int k,
    const float* __restrict__ bias, const int32_t* __restrict__ forced,
    float* __restrict__ logits, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int* status) {
  pdl_enter();
  __shared__ float lrow[kMaxExperts];
  const int64_t t = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float sum = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = s0 + u < ns ? __ldg(part + ((int64_t)(s0 + u) * T + t) * E + e) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) sum += v[u];
    }
    sum += bias ? bias[e] : 0.f;
    lrow[e] = sum;
    logits[t * E + e] = sum;
  }
  __syncthreads();
  if (threadIdx.x < 32)
    topk_warp<NV>(lrow, forced ? forced + t * k : nullptr, E, k, threadIdx.x, topk_idx + t * k,
                  topk_w + t * k, status);
}

template <int NV>
static void launch_small_topk(const float* part, int ns, int64_t T, int E, int k,
                              const float* bias, const int32_t* forced, float* logits,
                              int32_t* topk_idx, float* topk_w, int* status, cudaStream_t s) {
  launch_pdl(pdl_for_tokens(T), router_small_topk_kernel<NV>, dim3((unsigned)T), dim3(256), 0, s,
             part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status);
}

// The whole routing of a few tokens: two launches (partials; logits + top-k).
cudaError_t launch_route_small(const moe_bf16* x, const float* w_router, const float* bias,
                               const int32_t* forced, int64_t T, int d, int E, int k,
                               float* logits, int32_t* topk_idx, float* topk_w, void* ws,
                               int* status, cudaStream_t s) {
  const int rs = small_slice_rows(d), ns = (d + rs - 1) / rs;
  float* part = static_cast<float*>(ws);
  const dim3 grid((unsigned)((E + kSmallCols - 1) / kSmallCols), (unsigned)ns,
                  (unsigned)((T + kSmallTok - 1) / kSmallTok));
  timer_before(MOE_KERNEL_ROUTER_LOGITS, s);
  launch_pdl(pdl_for_tokens(T), router_small_partial_kernel, dim3(grid), dim3(kSmallWarps * 32), 0,
             s, x, w_router, T, d, E, rs, part);
  note_launches(1);
  timer_after(MOE_KERNEL_ROUTER_LOGITS, s);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  timer_before(MOE_KERNEL_TOPK, s);
  const int nv = (E + 31) / 32;
  if (nv <= 1) launch_small_topk<1>(part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status, s);
  else if (nv <= 2) launch_small_topk<2>(part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status, s);
  else if (nv <= 4) launch_small_topk<4>(part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status, s);
  else if (nv <= 8) launch_small_topk<8>(part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status, s);
  else if (nv <= 16) launch_small_topk<16>(part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status, s);
  else launch_small_topk<kMaxExperts / 32>(part, ns, T, E, k, bias, forced, logits, topk_idx, topk_w, status, s);
  note_launches(1);
  timer_after(MOE_KERNEL_TOPK, s);
  return cudaGetLastError();
}

// Many tokens: logits on the tensor cores (the top-k is its own launch).
cudaError_t launch_router_logits(const moe_bf16* x, const float* w_router, const float* bias,
                                 int64_t T, int d, int E, float* logits, void* ws, int* status,
                                 cudaStream_t s) {
  const int E8 = round8(E);
  moe_bf16* w_split = static_cast<moe_bf16*>(ws);
  const int64_t n = (int64_t)d * E8;
  timer_before(MOE_KERNEL_ROUTER_LOGITS, s);
  launch_pdl(pdl_for_tokens(T), split_router_weight_kernel, dim3((unsigned)((n + 255) / 256)),
             dim3(256), 0, s, w_router, d, E, E8, w_split);
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
      launch_pdl(pdl_for_tokens(T), router_reduce_kernel, dim3((unsigned)((nel + 255) / 256)),
                 dim3(256), 0, s, part, sp, nel, E, bias, logits);
      note_launches(1);
      e = cudaGetLastError();
    }
  }
  timer_after(MOE_KERNEL_ROUTER_LOGITS, s);
  return e;
}

// ---------------------------------------------------------------------------
// Top-k and weights: one warp per token (topk.cuh).
// ---------------------------------------------------------------------------
template <int NV>   // logits per lane: 32 * NV >= E
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits,
                                                   const int32_t* __restrict__ forced, int64_t T,
                                                   int E, int k, int32_t* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w, int* status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (t >= T) return;
  topk_warp<NV>(logits + t * E, forced ? forced + t * k : nullptr, E, k, lane, topk_idx + t * k,
                topk_w + t * k, status);
}

cudaError_t launch_topk(const float* logits, const int32_t* forced_idx, int64_t T, int E, int k,
                        int32_t* topk_idx, float* topk_w, int* status, cudaStream_t s) {
  const int warps = 8;
  dim3 grid((unsigned)((T + warps - 1) / warps));
  timer_before(MOE_KERNEL_TOPK, s);
  const int nv = (E + 31) / 32;
  if (nv <= 1)
    launch_pdl(pdl_for_tokens(T), topk_kernel<1>, dim3(grid), dim3(warps * 32), 0, s, logits,
               forced_idx, T, E, k, topk_idx, topk_w, status);
  else if (nv <= 2)
    launch_pdl(pdl_for_tokens(T), topk_kernel<2>, dim3(grid), dim3(warps * 32), 0, s, logits,
               forced_idx, T, E, k, topk_idx, topk_w, status);
  else if (nv <= 4)
    launch_pdl(pdl_for_tokens(T), topk_kernel<4>, dim3(grid), dim3(warps * 32), 0, s, logits,
               forced_idx, T, E, k, topk_idx, topk_w, status);
  else if (nv <= 8)
    launch_pdl(pdl_for_tokens(T), topk_kernel<8>, dim3(grid), dim3(warps * 32), 0, s, logits,
               forced_idx, T, E, k, topk_idx, topk_w, status);
  else if (nv <= 16)
    launch_pdl(pdl_for_tokens(T), topk_kernel<16>, dim3(grid), dim3(warps * 32), 0, s, logits,
               forced_idx, T, E, k, topk_idx, topk_w, status);
  else
    launch_pdl(pdl_for_tokens(T), topk_kernel<kMaxExperts / 32>, dim3(grid), dim3(warps * 32), 0, s,
               logits, forced_idx, T, E, k, topk_idx, topk_w, status);
  note_launches(1);
  timer_after(MOE_KERNEL_TOPK, s);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Router backward.
//   dl_t,j = w_j (dw_j - sum_j' w_j' dw_j')  on the selected slots (0 elsewhere)
//   dx[t] += sum_j dl_t,j W_r[:, e_j]
//   dW_r = x^T . dl  (dl as a dense [T, E] matrix)   db = column sums of dl
// dW_r runs on the tensor cores like the forward logits: dl is split exactly
// into three bf16 parts, laid side by side in a dense [T, 3 E8] matrix, and one
// grouped-GEMM launch (split K, fixed-order reduce) forms x^T . [hi | mid | lo];
// a bf16 x bf16 product is exact in fp32, so this is an fp32 accumulation of
// exact products. db sums dl over each expert's rows of the padded layout in
// row order. No atomics.
// ---------------------------------------------------------------------------
static inline size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }
static inline int n3_of(int E) { return 3 * round8(E); }

// workspace: W_r^T [E, d] fp32 | dl per pair [T*k] fp32 | dl3 [T, 3 E8] bf16 |
// the GEMM's split-K partials [ksplit, d, 3 E8] fp32
size_t route_bwd_ws_bytes(int64_t T, int d, int E, int k, int align) {
  (void)align;
  const int N3 = n3_of(E);
  const int sp = router_wgrad_ksplit(T, d, N3);
  return al256((size_t)E * d * 4) + al256((size_t)T * k * 4) + al256((size_t)T * N3 * 2) +
         al256((size_t)sp * d * N3 * 4);
}

__global__ void transpose_f32_kernel(const float* __restrict__ in, int rows, int cols,
                                     float* __restrict__ out) {
  pdl_enter();
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

// one warp per token: dl for its k slots (to dl_pair, and as three bf16 parts
// into the token's dense row of dl3), then dx[t]. With dxp (fp32 rows) given,
// dx[t] = sum_j dxp[dst_row[t, j]] + sum_s dxp[dst_row[T*k + s*T + t]] +
// sum_j dl_j W_r[:, e_j] in fp32, rounded to bf16 once (the permute transpose,
// shared experts' rows included, fused in); without it, dx[t] += sum_j dl_j
// W_r[:, e_j]. The dxp rows of up to four slots are loaded together; few
// registers, so that many warps per SM keep enough loads in flight.
__global__ void __launch_bounds__(256, 4) route_bwd_token_kernel(
    const float* __restrict__ d_topk_w, const float* __restrict__ topk_w,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ wrT, int64_t T, int d, int E,
    int E8, int k, int S, float* __restrict__ dl_pair, moe_bf16* __restrict__ dl3,
    moe_bf16* __restrict__ dx, const float* __restrict__ dxp,
    const int32_t* __restrict__ dst_row) {
  pdl_enter();
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
  } else if (lane < k + S && dxp) {
    r = dst_row[T * k + (int64_t)(lane - k) * T + t];
  }
  const int slots = k + S;
  float inner = w * dw;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) inner += __shfl_xor_sync(0xFFFFFFFFu, inner, off);
  const float dl = w * (dw - inner);
  if (lane < k) dl_pair[t * k + lane] = dl;

  // dense dl row: zeros, then the three parts of each slot at columns p E8 + e
  const int N3 = 3 * E8;
  moe_bf16* drow = dl3 + t * N3;
  for (int c = lane * 8; c < N3; c += 256)
    *reinterpret_cast<uint4*>(drow + c) = make_uint4(0u, 0u, 0u, 0u);
  __syncwarp();
  if (lane < k && e >= 0) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(dl);
    const float r1 = dl - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    drow[e] = __bfloat16_as_ushort(hi);
    drow[E8 + e] = __bfloat16_as_ushort(mid);
    drow[2 * E8 + e] = __bfloat16_as_ushort(lo);
  }

  moe_bf16* dxr = dx + t * d;
  // every lane runs the same number of iterations: the shuffles need the whole warp
  for (int c0 = 0; c0 < d; c0 += 256) {
    const int c = c0 + lane * 8;
    const bool in = c < d;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (in && !dxp) unpack8(*reinterpret_cast<const uint4*>(dxr + c), acc);
    if (dxp) {
      for (int j0 = 0; j0 < slots; j0 += 4) {
        float4 v[4][2];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = j0 + q;
          const int rj = __shfl_sync(0xFFFFFFFFu, r, j & 31);
          if (in && j < slots && rj >= 0) {
            const float4* src = reinterpret_cast<const float4*>(dxp + (int64_t)rj * d + c);
            v[q][0] = src[0];
            v[q][1] = src[1];
          } else {
            v[q][0] = v[q][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[0] += v[q][0].x; acc[1] += v[q][0].y; acc[2] += v[q][0].z; acc[3] += v[q][0].w;
          acc[4] += v[q][1].x; acc[5] += v[q][1].y; acc[6] += v[q][1].z; acc[7] += v[q][1].w;
        }
      }
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

// blockIdx.y == 0: dW_r[i, e] = sum over the K chunks s, in order, of
// part[s][i][e] + part[s][i][E8 + e] + part[s][i][2 E8 + e];
// blockIdx.y == 1: one warp per expert, db[e] = sum of dl over e's rows of the
// padded layout (lane-strided in row order, then a fixed shuffle tree).
__global__ void __launch_bounds__(256) route_bwd_reduce_kernel(
    const float* __restrict__ part, int ksplit, int d, int E, int E8,
    const int64_t* __restrict__ offsets, const int32_t* __restrict__ src_pair,
    const float* __restrict__ dl_pair, float* __restrict__ dw_router, float* __restrict__ dbias) {
  pdl_enter();
  if (blockIdx.y == 0) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)d * E) return;
    const int i = (int)(idx / E), e = (int)(idx % E);
    const int N3 = 3 * E8;
    float a = 0.f;
    for (int s = 0; s < ksplit; ++s) {
      const float* q = part + ((int64_t)s * d + i) * N3 + e;
      a += q[0] + q[E8] + q[2 * E8];
    }
    dw_router[idx] = a;
  } else {
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    if (e >= E) return;
    const int64_t g0 = offsets[e], g1 = offsets[e + 1];
    float a = 0.f;
    for (int64_t r = g0 + lane; r < g1; r += 32) {
      const int p = src_pair[r];
      if (p >= 0) a += dl_pair[p];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, off);
    if (lane == 0) dbias[e] = a;
  }
}

cudaError_t launch_route_bwd(const float* d_topk_w, const float* topk_w, const int32_t* topk_idx,
                             const float* w_router, const int64_t* offsets,
                             const int32_t* src_pair, const moe_bf16* x, int64_t T, int d, int E,
                             int k, int S, int align, moe_bf16* dx_inout, const float* dxp,
                             const int32_t* dst_row, float* dw_router, float* dbias, void* ws,
                             int* status, cudaStream_t s) {
  (void)align;
  const int E8 = round8(E);
  const int N3 = n3_of(E);
  const int sp = router_wgrad_ksplit(T, d, N3);
  char* p = static_cast<char*>(ws);
  float* wrT = reinterpret_cast<float*>(p);
  p += al256((size_t)E * d * 4);
  float* dl_pair = reinterpret_cast<float*>(p);
  p += al256((size_t)T * k * 4);
  moe_bf16* dl3 = reinterpret_cast<moe_bf16*>(p);
  p += al256((size_t)T * N3 * 2);
  float* part = reinterpret_cast<float*>(p);

  timer_before(MOE_KERNEL_ROUTE_BWD, s);
  launch_pdl(pdl_for_tokens(T), transpose_f32_kernel, dim3((E + 31) / 32, (d + 31) / 32),
             dim3(32, 8), 0, s, w_router, d, E, wrT);
  note_launches(1);
  if (T > 0) {
    launch_pdl(pdl_for_tokens(T), route_bwd_token_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256),
               0, s, d_topk_w, topk_w, topk_idx, wrT, T, d, E, E8, k, S, dl_pair, dl3, dx_inout,
               dxp, dst_row);
    note_launches(1);
  }
  cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) err = launch_router_wgrad_gemm(x, dl3, T, d, N3, sp, part, status, s);
  if (err == cudaSuccess) {
    const int64_t n = (int64_t)d * E;
    const unsigned gx = (unsigned)std::max<int64_t>((n + 255) / 256, (E + 7) / 8);
    launch_pdl(pdl_for_tokens(T), route_bwd_reduce_kernel, dim3(gx, dbias ? 2 : 1), dim3(256), 0, s,
               part, sp, d, E, E8, offsets, src_pair, dl_pair, dw_router, dbias);
    note_launches(1);
    err = cudaGetLastError();
  }
  timer_after(MOE_KERNEL_ROUTE_BWD, s);
  return err;
}

}  // namespace moe
