// permute.cu — the padded expert-grouped layout, built without atomics, and
// the single gather of token copies into it.
//
// Halo "Performance", §Levers that help: the atomic-free expert permute.
// prime-rl PR #3885 (DeepSeek-V4.1 Flash perf work), §Changes, "Single-pass
// DeepEP local layout": one gather into the padded expert-grouped layout
// instead of several full copies of the routed activations.
//
// Four kernels, all deterministic:
//   hist    per block of 4096 pairs: per-warp expert histograms built with
//           warp match (__match_any_sync) — the leader lane of each expert
//           group adds the group's size, so no two lanes ever write the same
//           counter; warp-local ranks are kept per pair.
//   scan    one CTA: exclusive scan over blocks for each expert (n_e and each
//           block's base), the padded sizes ceil(n_e/align)*align and their
//           exclusive scan over experts (the 64-bit offsets).
//   scatter dst_row[p] = offsets[e] + block base + rank; src_pair[dst] = p.
//   gather  xp[r] = x[src_pair[r] / k] for real rows, zeros for padding rows.
// Pair p's rank inside its expert is therefore its rank in ascending p.
// Shared experts (S of them, every token's copy with weight 1: prime-rl PR
// #3885, §Changes, "Fused FP8 shared expert") follow the routed groups: group
// E + s holds the T pairs T*k + s*T + t in token order (padded to `align`);
// the scan writes their counts and offsets, the gather their rows and maps.
#include "common.cuh"
#include "internal.h"

namespace moe {

constexpr int kHistWarps = 16;
constexpr int kHistSteps = 8;
constexpr int kHistChunk = kHistWarps * 32 * kHistSteps;   // pairs per block

static inline size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

static inline int64_t hist_blocks(int64_t P) { return (P + kHistChunk - 1) / kHistChunk; }

size_t permute_ws_bytes(int64_t T, int k, int E) {
  const int64_t P = T * k;
  return al256((size_t)hist_blocks(P) * E * 4) + al256((size_t)P * 4);
}

__device__ __forceinline__ int valid_expert(const int32_t* idx, int64_t p, int64_t P, int E,
                                            int* status) {
  if (p >= P) return -1;
  const int e = idx[p];
  if (e < 0 || e >= E) {
    raise_status(status, MOE_ERR_DEVICE_INDEX);
    return -1;
  }
  return e;
}

__global__ void __launch_bounds__(kHistWarps * 32) permute_hist_kernel(
    const int32_t* __restrict__ idx, int64_t P, int E, int32_t* __restrict__ blk_count,
    int32_t* __restrict__ rank_in_blk, int* status) {
  pdl_enter();
  extern __shared__ int32_t hist[];   // [kHistWarps][E]
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kHistWarps * E; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int64_t base = (int64_t)blockIdx.x * kHistChunk + (int64_t)w * 32 * kHistSteps;
  int32_t* wh = hist + w * E;
  const uint32_t lt_mask = (1u << lane) - 1u;
#pragma unroll
  for (int step = 0; step < kHistSteps; ++step) {
    const int64_t p = base + step * 32 + lane;
    const int e = valid_expert(idx, p, P, E, status);
    const uint32_t same = __match_any_sync(0xFFFFFFFFu, e);
    const int before = __popc(same & lt_mask);
    const int cur = (e >= 0) ? wh[e] : 0;
    __syncwarp();
    if (e >= 0 && before == 0) wh[e] = cur + __popc(same);
    __syncwarp();
    if (p < P) rank_in_blk[p] = (e >= 0) ? cur + before : -1;
  }
  __syncthreads();
  // each expert: exclusive scan over the warps, block total to global
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int ww = 0; ww < kHistWarps; ++ww) {
      const int c = hist[ww * E + e];
      hist[ww * E + e] = run;
      run += c;
    }
    blk_count[(int64_t)blockIdx.x * E + e] = run;
  }
  __syncthreads();
  // warp-local rank -> rank inside the block
#pragma unroll
  for (int step = 0; step < kHistSteps; ++step) {
    const int64_t p = base + step * 32 + lane;
    if (p >= P) continue;
    const int e = idx[p];
    if (e < 0 || e >= E) continue;
    rank_in_blk[p] += wh[e];
  }
}

// One CTA of 1024 threads; thread e owns expert e.
// counts and offsets of the S shared groups after the routed total
__device__ __forceinline__ void shared_groups(int E, int S, int64_t T, int align,
                                              int64_t routed_end, int32_t* counts,
                                              int64_t* offsets) {
  const int64_t Tp = ((T + align - 1) / align) * align;
  for (int s = 0; s < S; ++s) {
    counts[E + s] = (int32_t)T;
    offsets[E + 1 + s] = routed_end + (int64_t)(s + 1) * Tp;
  }
}

__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t* __restrict__ blk_count,
                                                            int64_t nblk, int E, int S, int64_t T,
                                                            int align,
                                                            int32_t* __restrict__ counts,
                                                            int64_t* __restrict__ offsets) {
  pdl_enter();
  __shared__ int64_t warp_tot[32];
  const int e = threadIdx.x;
  const int lane = e & 31, w = e >> 5;
  int64_t n = 0;
  if (e < E) {
    for (int64_t b = 0; b < nblk; ++b) {
      const int32_t c = blk_count[b * E + e];
      blk_count[b * E + e] = (int32_t)n;
      n += c;
    }
  }
  const int64_t padded = (e < E) ? ((n + align - 1) / align) * align : 0;
  // block-wide exclusive scan of `padded`
  int64_t incl = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int64_t v = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t o = __shfl_up_sync(0xFFFFFFFFu, v, off);
      if (lane >= off) v += o;
    }
    warp_tot[lane] = v;   // inclusive over warps
  }
  __syncthreads();
  const int64_t excl = incl - padded + (w > 0 ? warp_tot[w - 1] : 0);
  if (e < E) {
    counts[e] = (int32_t)n;
    offsets[e] = excl;
    for (int64_t b = 0; b < nblk; ++b) blk_count[b * E + e] += (int32_t)excl;
  }
  if (e == E - 1) {
    offsets[E] = excl + padded;
    shared_groups(E, S, T, align, excl + padded, counts, offsets);
  }
}

__global__ void permute_scatter_kernel(const int32_t* __restrict__ idx, int64_t P, int E,
                                       const int32_t* __restrict__ blk_base,
                                       const int32_t* __restrict__ rank_in_blk,
                                       int32_t* __restrict__ dst_row,
                                       int32_t* __restrict__ src_pair) {
  pdl_enter();
  const int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= P) return;
  const int e = idx[p];
  if (e < 0 || e >= E) {
    dst_row[p] = -1;
    return;
  }
  const int32_t dst = blk_base[(p / kHistChunk) * E + e] + rank_in_blk[p];
  dst_row[p] = dst;
  src_pair[dst] = (int32_t)p;
}

// A few pairs (decode): hist, scan and scatter in one CTA of 1024 threads.
// Thread e counts expert e's pairs, the padded sizes are scanned as above,
// and pair p's rank is the number of earlier pairs with its expert — the same
// layout as the four-kernel path.
constexpr int kSmallPairs = 256;
__global__ void __launch_bounds__(1024) permute_small_kernel(
    const int32_t* __restrict__ idx, int64_t P, int E, int S, int64_t T, int align,
    int32_t* __restrict__ counts,
    int64_t* __restrict__ offsets, int32_t* __restrict__ dst_row,
    int32_t* __restrict__ src_pair, int* status) {
  pdl_enter();
  __shared__ int32_t s_idx[kSmallPairs];
  __shared__ int64_t warp_tot[32];
  __shared__ int64_t s_off[1024];
  const int tid = threadIdx.x;
  const int lane = tid & 31, w = tid >> 5;
  for (int p = tid; p < P; p += blockDim.x) s_idx[p] = valid_expert(idx, p, P, E, status);
  __syncthreads();
  int64_t n = 0;
  if (tid < E)
    for (int p = 0; p < P; ++p) n += (s_idx[p] == tid);
  const int64_t padded = (tid < E) ? ((n + align - 1) / align) * align : 0;
  int64_t incl = padded;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int64_t v = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t o = __shfl_up_sync(0xFFFFFFFFu, v, off);
      if (lane >= off) v += o;
    }
    warp_tot[lane] = v;
  }
  __syncthreads();
  const int64_t excl = incl - padded + (w > 0 ? warp_tot[w - 1] : 0);
  s_off[tid] = excl;
  if (tid < E) {
    counts[tid] = (int32_t)n;
    offsets[tid] = excl;
  }
  if (tid == E - 1) {
    offsets[E] = excl + padded;
    shared_groups(E, S, T, align, excl + padded, counts, offsets);
  }
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = s_idx[p];
    if (e < 0) {
      dst_row[p] = -1;
      continue;
    }
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (s_idx[q] == e);
    const int32_t dst = (int32_t)(s_off[e] + rank);
    dst_row[p] = dst;
    src_pair[dst] = (int32_t)p;
  }
}

__device__ __forceinline__ int expert_of_row_p(const int64_t* offsets, int E, int64_t r) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// one warp per row; a shared expert's row also writes its pair's maps
__global__ void __launch_bounds__(256) permute_gather_kernel(
    const moe_bf16* __restrict__ x, int d, int k, int64_t T, const int64_t* __restrict__ offsets,
    const int32_t* __restrict__ counts, int E, int S, int64_t R_cap,
    int32_t* __restrict__ src_pair, int32_t* __restrict__ dst_row, moe_bf16* __restrict__ xp) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  if (r >= R_cap) return;
  const int64_t R_pad = offsets[E + S];
  if (r >= R_pad) {
    if (lane == 0) src_pair[r] = -1;
    return;
  }
  const int e = expert_of_row_p(offsets, E + S, r);
  const int64_t i = r - offsets[e];
  const bool real = i < (int64_t)counts[e];
  const int nv = d / 8;
  if (real) {
    int64_t t;
    if (e < E) {
      t = src_pair[r] / k;
    } else {
      t = i;
      const int64_t p = T * k + (int64_t)(e - E) * T + i;
      if (lane == 0) {
        src_pair[r] = (int32_t)p;
        dst_row[p] = (int32_t)r;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(xp + r * d);
    const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
    // four 16-byte pieces in flight per lane
    for (int v0 = lane; v0 < nv; v0 += 128) {
      uint4 c[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nv) c[u] = src[v0 + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nv) dst[v0 + 32 * u] = c[u];
    }
  } else {
    if (lane == 0) src_pair[r] = -1;
    uint4* dst = reinterpret_cast<uint4*>(xp + r * d);
    for (int v = lane; v < nv; v += 32) dst[v] = make_uint4(0u, 0u, 0u, 0u);
  }
}

cudaError_t launch_permute(const int32_t* topk_idx, int64_t T, int k, int E, int S, int align,
                           const moe_bf16* x, int d, int64_t R_cap, int32_t* counts,
                           int64_t* offsets, int32_t* dst_row, int32_t* src_pair, moe_bf16* xp,
                           void* ws, int* status, cudaStream_t s) {
  const int64_t P = T * k;
  const int64_t nblk = hist_blocks(P);
  int32_t* blk_count = static_cast<int32_t*>(ws);
  int32_t* rank_in_blk =
      reinterpret_cast<int32_t*>(static_cast<char*>(ws) + al256((size_t)nblk * E * 4));
  const size_t hist_smem = (size_t)kHistWarps * E * 4;
  cudaError_t err = cudaFuncSetAttribute(permute_hist_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)hist_smem);
  if (err != cudaSuccess) return err;
  timer_before(MOE_KERNEL_PERMUTE, s);
  int launches = 2;
  if (P > 0 && P <= kSmallPairs) {
    launch_pdl(pdl_for_tokens(T), permute_small_kernel, dim3(1), dim3(1024), 0, s, topk_idx, P, E,
               S, T, align, counts, offsets, dst_row, src_pair, status);
  } else {
    if (P > 0)
      launch_pdl(pdl_for_tokens(T), permute_hist_kernel, dim3((unsigned)nblk),
                 dim3(kHistWarps * 32), hist_smem, s, topk_idx, P, E, blk_count, rank_in_blk,
                 status);
    launch_pdl(pdl_for_tokens(T), permute_scan_kernel, dim3(1), dim3(1024), 0, s, blk_count, nblk,
               E, S, T, align, counts, offsets);
    if (P > 0)
      launch_pdl(pdl_for_tokens(T), permute_scatter_kernel, dim3((unsigned)((P + 255) / 256)),
                 dim3(256), 0, s, topk_idx, P, E, blk_count, rank_in_blk, dst_row, src_pair);
    launches = P > 0 ? 4 : 2;
  }
  launch_pdl(pdl_for_tokens(T), permute_gather_kernel, dim3((unsigned)((R_cap + 7) / 8)), dim3(256),
             0, s, x, d, k, T, offsets, counts, E, S, R_cap, src_pair, dst_row, xp);
  note_launches(launches);
  timer_after(MOE_KERNEL_PERMUTE, s);
  return cudaGetLastError();
}

}  // namespace moe
