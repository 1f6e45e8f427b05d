// decode.cu — the layer's forward for a handful of tokens (decode), in one
// cooperative kernel.
//
// With T <= 8 tokens the layer is bound by reading the selected experts'
// weights once (Halo "Performance", §Levers that do not help here: small-M
// experts are bound by weight bandwidth); launching the general path's seven
// kernels costs more than the work. One persistent kernel, one CTA per SM, runs
// five phases separated by grid barriers:
//   A  router logits: (token, 8 experts) units, fp32 dot products
//   B  CTA 0: top-k and renormalised weights per token (topk.cuh), then the
//      selected experts in ascending id with their pairs in ascending pair id,
//      cut into segments of at most kDecMaxT pairs
//   C  gate/up: (selected expert, 64 columns of f) units; every token routed
//      to the expert multiplies the same weight stream; A = silu(G) * U (fp32)
//   D  down: (selected expert, 64 columns of d) units; Yp per pair (fp32)
//   E  combine: y[t] = sum_j w[t, j] * Yp[t*k + j] in slot order, rounded once
// Each unit's partial sums (16 warps, each a 1/16 share of the rows) are added
// in a fixed order, so results are deterministic. The grid barriers are a
// counter in the workspace (zeroed by the host before the launch) with a
// bounded wait: on expiry the kernel records MOE_ERR_DEVICE_TIMEOUT and every
// CTA skips the remaining phases.
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace moe {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMaxT = 8;
constexpr int kDecMaxPairs = kDecMaxT * kMaxTopK;
constexpr int kDecCols = 64;          // output columns per unit: two per lane
constexpr int kDecRouterCols = 8;     // experts per router unit
constexpr int kDecUnroll = 8;         // rows whose weight loads are in flight together

struct DecodeCtl {
  int n_sel;
  int seg_begin[kDecMaxPairs + 1];
  int seg_e[kDecMaxPairs];
  int sorted_pair[kDecMaxPairs];
};

__host__ __device__ static inline size_t al256d(size_t b) { return (b + 255) & ~(size_t)255; }

// workspace: barrier counter | control table | A [P, f] fp32 | Yp [P, d] fp32
size_t decode_ws_bytes(int64_t T, int d, int f, int k) {
  const int64_t P = T * k;
  return 256 + al256d(sizeof(DecodeCtl)) + al256d((size_t)P * f * 4) + al256d((size_t)P * d * 4);
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// all CTAs of the grid reach this point before any goes on (bounded wait)
__device__ bool grid_sync(unsigned* ctr, unsigned& target, volatile int* s_abort, int* status) {
  target += gridDim.x;
  __syncthreads();
  if (threadIdx.x == 0 && !*s_abort) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
      if (ld_acquire_u32(ctr) >= target) break;
      if ((i & 63u) == 63u && global_ns() - t0 > (uint64_t)kWaitLimitNs) {
        *s_abort = 1;
        raise_status(status, MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return *s_abort == 0;
}

__device__ __forceinline__ float bf16_at(const moe_bf16* p) {
  return __bfloat162float(__ushort_as_bfloat16(*p));
}

// red: [kDecWarps][kDecMaxT][kDecCols] partial sums; the warps' shares of
// entry (q, col), added in warp order
__device__ __forceinline__ float red_sum(const float* red, int q, int col) {
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) s += red[(w * kDecMaxT + q) * kDecCols + col];
  return s;
}
__device__ __forceinline__ void red_put(float* red, int warp, int q, int lane, float a,
                                        float b) {
  float* r = red + (warp * kDecMaxT + q) * kDecCols + 2 * lane;
  r[0] = a;
  r[1] = b;
}

template <int NV>
__global__ void __launch_bounds__(kDecThreads, 1) decode_fwd_kernel(
    const moe_bf16* __restrict__ x, const float* __restrict__ w_router,
    const float* __restrict__ bias, const int32_t* __restrict__ forced, int T, int d, int f,
    int E, int k, const moe_bf16* __restrict__ w_gate, const moe_bf16* __restrict__ w_up,
    const moe_bf16* __restrict__ w_down, float* __restrict__ logits,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, moe_bf16* __restrict__ y,
    char* __restrict__ ws, int* status) {
  // Data that other CTAs wrote in an earlier phase is read with ld.global.cg
  // (from L2, never from this SM's L1).
  extern __shared__ float red[];   // kDecWarps * kDecMaxT * kDecCols floats
  __shared__ volatile int s_abort;
  __shared__ int s_e[kDecMaxPairs];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_abort = 0;
  __syncthreads();
  unsigned* ctr = reinterpret_cast<unsigned*>(ws);
  DecodeCtl* ctl = reinterpret_cast<DecodeCtl*>(ws + 256);
  const int P = T * k;
  float* Abuf = reinterpret_cast<float*>(ws + 256 + al256d(sizeof(DecodeCtl)));
  float* Ybuf = Abuf + al256d((size_t)P * f * 4) / 4;
  unsigned target = 0;

  // ---------------------------------------------------------------- A --
  const int nEc = (E + kDecRouterCols - 1) / kDecRouterCols;
  for (int u = blockIdx.x; u < T * nEc; u += gridDim.x) {
    const int t = u / nEc, e0 = (u % nEc) * kDecRouterCols;
    const int ne = min(kDecRouterCols, E - e0);
    float acc[kDecRouterCols];
#pragma unroll
    for (int j = 0; j < kDecRouterCols; ++j) acc[j] = 0.f;
    for (int i = tid; i < d; i += kDecThreads) {
      const float xv = bf16_at(x + (int64_t)t * d + i);
      const float* wr = w_router + (int64_t)i * E + e0;
#pragma unroll
      for (int j = 0; j < kDecRouterCols; ++j)
        if (j < ne) acc[j] = fmaf(xv, wr[j], acc[j]);
    }
#pragma unroll
    for (int j = 0; j < kDecRouterCols; ++j) red[j * kDecThreads + tid] = acc[j];
    __syncthreads();
    for (int w = kDecThreads / 2; w > 0; w >>= 1) {
      if (tid < w) {
#pragma unroll
        for (int j = 0; j < kDecRouterCols; ++j)
          red[j * kDecThreads + tid] += red[j * kDecThreads + tid + w];
      }
      __syncthreads();
    }
    if (tid < ne)
      logits[(int64_t)t * E + e0 + tid] = red[tid * kDecThreads] + (bias ? bias[e0 + tid] : 0.f);
    __syncthreads();
  }
  if (!grid_sync(ctr, target, &s_abort, status)) return;

  // ---------------------------------------------------------------- B --
  if (blockIdx.x == 0) {
    // the logits (T x E, at most 32 KiB) to shared memory, then top-k per warp
    for (int o = tid; o < T * E; o += kDecThreads) red[o] = __ldcg(logits + o);
    __syncthreads();
    if (warp < T)
      topk_warp<NV>(red + warp * E, forced ? forced + warp * k : nullptr, E, k, lane,
                    topk_idx + warp * k, topk_w + warp * k, status);
    __syncthreads();
    for (int p = tid; p < P; p += kDecThreads) {
      const int e = topk_idx[p];   // an invalid forced id is kept here: dropped below
      s_e[p] = (e >= 0 && e < E) ? e : E;
    }
    __syncthreads();
    // sort the pairs by (expert, pair); invalid ones (key E) last
    for (int p = tid; p < P; p += kDecThreads) {
      int rank = 0;
      for (int q = 0; q < P; ++q)
        rank += (s_e[q] < s_e[p]) || (s_e[q] == s_e[p] && q < p);
      ctl->sorted_pair[rank] = p;
    }
    __syncthreads();
    if (tid == 0) {
      int n = 0;
      int prev = -1;
      int pos = 0;
      for (; pos < P; ++pos) {
        const int e = s_e[ctl->sorted_pair[pos]];
        if (e >= E) break;
        // a new segment per expert, and every kDecMaxT pairs within one (caller-
        // chosen ids may repeat an expert for a token)
        if (e != prev || pos - ctl->seg_begin[n - 1] == kDecMaxT) {
          ctl->seg_e[n] = e;
          ctl->seg_begin[n] = pos;
          ++n;
          prev = e;
        }
      }
      ctl->seg_begin[n] = pos;
      ctl->n_sel = n;
    }
  }
  if (!grid_sync(ctr, target, &s_abort, status)) return;

  const int n_sel = __ldcg(&ctl->n_sel);
  // ---------------------------------------------------------------- C --
  const int nfc = f / kDecCols;
  for (int u = blockIdx.x; u < n_sel * nfc; u += gridDim.x) {
    const int s = u / nfc, c0 = (u % nfc) * kDecCols;
    const int e = __ldcg(&ctl->seg_e[s]);
    const int pb = __ldcg(&ctl->seg_begin[s]), np = __ldcg(&ctl->seg_begin[s + 1]) - pb;
    int tok[kDecMaxT], pr[kDecMaxT];
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) {
      pr[q] = q < np ? __ldcg(&ctl->sorted_pair[pb + q]) : 0;
      tok[q] = pr[q] / k;
    }
    float ga[kDecMaxT][2], ua[kDecMaxT][2];
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) ga[q][0] = ga[q][1] = ua[q][0] = ua[q][1] = 0.f;
    const moe_bf16* wg = w_gate + (int64_t)e * d * f + c0 + 2 * lane;
    const moe_bf16* wu = w_up + (int64_t)e * d * f + c0 + 2 * lane;
    for (int i0 = warp; i0 < d; i0 += kDecWarps * kDecUnroll) {
      uint32_t gv[kDecUnroll], uv[kDecUnroll];
#pragma unroll
      for (int r = 0; r < kDecUnroll; ++r) {
        const int i = i0 + kDecWarps * r;
        gv[r] = i < d ? *reinterpret_cast<const uint32_t*>(wg + (int64_t)i * f) : 0u;
        uv[r] = i < d ? *reinterpret_cast<const uint32_t*>(wu + (int64_t)i * f) : 0u;
      }
#pragma unroll
      for (int r = 0; r < kDecUnroll; ++r) {
        const int i = i0 + kDecWarps * r;
        if (i >= d) break;
        const float g0 = __uint_as_float(gv[r] << 16), g1 = __uint_as_float(gv[r] & 0xFFFF0000u);
        const float u0 = __uint_as_float(uv[r] << 16), u1 = __uint_as_float(uv[r] & 0xFFFF0000u);
#pragma unroll
        for (int q = 0; q < kDecMaxT; ++q) {
          if (q < np) {
            const float xv = bf16_at(x + (int64_t)tok[q] * d + i);
            ga[q][0] = fmaf(xv, g0, ga[q][0]);
            ga[q][1] = fmaf(xv, g1, ga[q][1]);
            ua[q][0] = fmaf(xv, u0, ua[q][0]);
            ua[q][1] = fmaf(xv, u1, ua[q][1]);
          }
        }
      }
    }
    // G through the reduction buffer into registers, then U, then A = silu(G) * U
    float gsum[2] = {0.f, 0.f};   // entries tid and tid + 512 of the (pair, column) grid
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) red_put(red, warp, q, lane, ga[q][0], ga[q][1]);
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = tid + h * kDecThreads;
      if (o < np * kDecCols) gsum[h] = red_sum(red, o / kDecCols, o % kDecCols);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) red_put(red, warp, q, lane, ua[q][0], ua[q][1]);
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = tid + h * kDecThreads;
      if (o < np * kDecCols) {
        const int q = o / kDecCols, col = o % kDecCols;
        const float g = gsum[h], uu = red_sum(red, q, col);
        Abuf[(int64_t)pr[q] * f + c0 + col] = __fdividef(g, 1.0f + __expf(-g)) * uu;
      }
    }
    __syncthreads();
  }
  if (!grid_sync(ctr, target, &s_abort, status)) return;

  // ---------------------------------------------------------------- D --
  const int ndc = d / kDecCols;
  for (int u = blockIdx.x; u < n_sel * ndc; u += gridDim.x) {
    const int s = u / ndc, c0 = (u % ndc) * kDecCols;
    const int e = __ldcg(&ctl->seg_e[s]);
    const int pb = __ldcg(&ctl->seg_begin[s]), np = __ldcg(&ctl->seg_begin[s + 1]) - pb;
    int pr[kDecMaxT];
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) pr[q] = q < np ? __ldcg(&ctl->sorted_pair[pb + q]) : 0;
    float ya[kDecMaxT][2];
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) ya[q][0] = ya[q][1] = 0.f;
    const moe_bf16* wd = w_down + (int64_t)e * f * d + c0 + 2 * lane;
    for (int i0 = warp; i0 < f; i0 += kDecWarps * kDecUnroll) {
      uint32_t dv[kDecUnroll];
#pragma unroll
      for (int r = 0; r < kDecUnroll; ++r) {
        const int i = i0 + kDecWarps * r;
        dv[r] = i < f ? *reinterpret_cast<const uint32_t*>(wd + (int64_t)i * d) : 0u;
      }
#pragma unroll
      for (int r = 0; r < kDecUnroll; ++r) {
        const int i = i0 + kDecWarps * r;
        if (i >= f) break;
        const float w0 = __uint_as_float(dv[r] << 16), w1 = __uint_as_float(dv[r] & 0xFFFF0000u);
#pragma unroll
        for (int q = 0; q < kDecMaxT; ++q) {
          if (q < np) {
            const float av = __ldcg(Abuf + (int64_t)pr[q] * f + i);
            ya[q][0] = fmaf(av, w0, ya[q][0]);
            ya[q][1] = fmaf(av, w1, ya[q][1]);
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kDecMaxT; ++q) red_put(red, warp, q, lane, ya[q][0], ya[q][1]);
    __syncthreads();
    for (int o = tid; o < np * kDecCols; o += kDecThreads) {
      const int q = o / kDecCols, col = o % kDecCols;
      Ybuf[(int64_t)pr[q] * d + c0 + col] = red_sum(red, q, col);
    }
    __syncthreads();
  }
  if (!grid_sync(ctr, target, &s_abort, status)) return;

  // ---------------------------------------------------------------- E --
  for (int64_t o = (int64_t)blockIdx.x * kDecThreads + tid; o < (int64_t)T * d;
       o += (int64_t)gridDim.x * kDecThreads) {
    const int t = (int)(o / d), c = (int)(o % d);
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const int p = t * k + j;
      const int e = __ldcg(topk_idx + p);
      if (e < 0 || e >= E) continue;
      acc = fmaf(__ldcg(topk_w + p), __ldcg(Ybuf + (int64_t)p * d + c), acc);
    }
    y[o] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  }
}

cudaError_t launch_decode_fwd(const moe_bf16* x, const float* w_router, const float* bias,
                              const int32_t* forced, int T, int d, int f, int E, int k,
                              const moe_bf16* w_gate, const moe_bf16* w_up,
                              const moe_bf16* w_down, float* logits, int32_t* topk_idx,
                              float* topk_w, moe_bf16* y, void* ws, int* status,
                              cudaStream_t s) {
  constexpr int kRed = kDecWarps * kDecMaxT * kDecCols * 4;   // 32 KiB
  static_assert(kRed >= kDecRouterCols * kDecThreads * 4, "router reduction fits");
  static_assert(kRed >= kDecMaxT * kMaxExperts * 4, "the logits fit");
  const int nv = (E + 31) / 32;
  const int variant = nv <= 1 ? 0 : nv <= 2 ? 1 : nv <= 4 ? 2 : nv <= 8 ? 3 : nv <= 16 ? 4 : 5;
  void (*const kerns[6])(const moe_bf16*, const float*, const float*, const int32_t*, int, int,
                         int, int, int, const moe_bf16*, const moe_bf16*, const moe_bf16*,
                         float*, int32_t*, float*, moe_bf16*, char*, int*) = {
      decode_fwd_kernel<1>, decode_fwd_kernel<2>, decode_fwd_kernel<4>,
      decode_fwd_kernel<8>, decode_fwd_kernel<16>, decode_fwd_kernel<kMaxExperts / 32>};
  auto kern = kerns[variant];
  // shared-memory opt-in and the residency check, once per variant and device
  constexpr int kDevices = 64;
  static int ready[6][kDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  if (!ready[variant][dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRed);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, kRed);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ready[variant][dev] = 1;
  }
  const int grid = num_sms();   // one CTA per SM: all resident, as the barriers need
  err = cudaMemsetAsync(ws, 0, 256, s);   // the barrier counter
  if (err != cudaSuccess) return err;
  char* wsb = static_cast<char*>(ws);
  void* args[] = {(void*)&x,      (void*)&w_router, (void*)&bias,  (void*)&forced, (void*)&T,
                  (void*)&d,      (void*)&f,        (void*)&E,     (void*)&k,      (void*)&w_gate,
                  (void*)&w_up,   (void*)&w_down,   (void*)&logits, (void*)&topk_idx,
                  (void*)&topk_w, (void*)&y,        (void*)&wsb,   (void*)&status};
  timer_before(MOE_KERNEL_DECODE, s);
  err = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kDecThreads), args, kRed,
                                    s);
  note_launches(1);
  timer_after(MOE_KERNEL_DECODE, s);
  return err;
}

}  // namespace moe
