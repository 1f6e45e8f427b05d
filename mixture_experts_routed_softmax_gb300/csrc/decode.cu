// decode.cu — the layer's forward for a handful of tokens (decode), in one
// cooperative kernel.
//
// With T <= 8 tokens the layer is bound by reading the selected experts'
// weights once (Halo "Performance", §Levers that do not help here: small-M
// experts are bound by weight bandwidth); launching the general path's seven
// kernels costs more than the work. One persistent kernel, one CTA per SM,
// runs these phases, separated by grid barriers (|):
//   A   router partial dot products: (128-row slice of W_r, 128 experts) units
//   |
//   B   every CTA sums the partials into the logits, takes the top-k with
//       renormalised weights (topk.cuh) and cuts the kept pairs, sorted by
//       (expert, pair id), into segments of at most 4 pairs of one expert
//       (an expert with more pairs has its weights read once per segment);
//       CTA 0 writes logits, topk_idx and topk_w
//   C   gate/up products (stream-K): the selected experts' W_gate and W_up
//       rows, grouped by (segment, matrix, 64 columns), are cut into equal
//       contiguous ranges of 4-row quads, one range per warp of the grid;
//       a warp keeps fp32 sums for every pair of the segment and writes one
//       partial per group it touched
//   |
//   C2  G and U = the partials of each group added in warp order;
//       A = silu(G) * U (fp32), stored [f, pairs]
//   |
//   D   down products (stream-K) over W_down rows grouped by (segment,
//       64 columns of d), A as the left operand, partials as in C
//   |
//   E   y[t] = sum_j w[t, j] * (partials of pair (t, j) in warp order); the
//       k terms are added in a fixed butterfly over lanes, rounded to bf16 once
// Weights move with 16-byte loads, eight lanes per 128-byte row segment, and
// each warp keeps eight quads' loads in flight while it multiplies. Every sum has a fixed order, so two runs on
// one GPU are bitwise equal. The grid barriers are a counter in the
// workspace (zeroed by the host before the launch) with a bounded wait: on
// expiry the kernel records MOE_ERR_DEVICE_TIMEOUT and every CTA skips the
// remaining phases.
#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace moe {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMaxT = kDecodeMaxT;
constexpr int kDecMaxPairs = kDecMaxT * kMaxTopK;
constexpr int kDecMaxD = kDecodeMaxD;   // x is kept in shared memory: d * 16 bytes
constexpr int kDecCols = 64;          // columns of a weight group: 8 lanes x 8 bf16
constexpr int kDecSeg = 4;            // pairs of one expert whose sums one warp keeps
constexpr int kDecGroupFloats = kDecSeg * kDecCols;   // one partial: [pair][column]
constexpr int kDecBatch = 8;          // quads per warp whose loads are in flight together
constexpr int kDecRCols = 128;        // router: experts per unit (4 per lane)
constexpr int kDecRedFloats = kDecWarps * kDecMaxT * kDecRCols;   // 64 KiB
constexpr int kDecRouterPartialFloats = 16384;   // partial logits each CTA sums in phase B

static_assert(kDecRedFloats >= kDecMaxT * kMaxExperts, "the logits fit the reduction buffer");

__host__ __device__ static inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ static inline size_t al256d(size_t b) { return (b + 255) & ~(size_t)255; }

// Sizes shared by the host (workspace size, launch) and the kernel.
struct DecGeom {
  int nw;        // warps in the grid
  int maxg;      // partial slots per warp (groups one warp's range can touch)
  int nslice;    // router row slices
  int rs;        // router rows per slice (a multiple of kDecWarps)
  size_t off_part_a, off_part, off_ai, total;
};

static DecGeom decode_geom(int64_t T, int d, int f, int E, int k, int grid) {
  DecGeom g{};
  const int64_t P = T * k;
  g.nw = grid * kDecWarps;
  // stream-K bound: a range of L quads touches at most ceil(L / QG) + 1 groups
  const int64_t nqc = P * 2 * (f / kDecCols) * (d / 4), qgc = d / 4;
  const int64_t nqd = P * (d / kDecCols) * (f / 4), qgd = f / 4;
  const int64_t mc = cdiv64(cdiv64(nqc, g.nw), qgc) + 1;
  const int64_t md = cdiv64(cdiv64(nqd, g.nw), qgd) + 1;
  g.maxg = (int)(mc > md ? mc : md);
  int64_t ns = kDecRouterPartialFloats / (T * E > 0 ? T * E : 1);
  ns = ns < 1 ? 1 : ns;
  const int64_t ns_max = cdiv64(d, 128);
  g.nslice = (int)(ns < ns_max ? ns : ns_max);
  g.rs = (int)(cdiv64(cdiv64(d, g.nslice), kDecWarps) * kDecWarps);
  g.nslice = (int)cdiv64(d, g.rs);
  g.off_part_a = 256;
  g.off_part = g.off_part_a + al256d((size_t)g.nslice * T * E * 4);
  g.off_ai = g.off_part + al256d((size_t)g.nw * g.maxg * kDecGroupFloats * 4);
  g.total = g.off_ai + al256d((size_t)f * P * 4);
  return g;
}

size_t decode_ws_bytes(int64_t T, int d, int f, int E, int k) {
  return decode_geom(T, d, f, E, k, num_sms()).total;
}

struct DecArgs {
  const moe_bf16* x;
  const float* w_router;
  const float* bias;
  const int32_t* forced;
  const moe_bf16* w_gate;
  const moe_bf16* w_up;
  const moe_bf16* w_down;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  moe_bf16* y;
  char* ws;
  int* status;
  int T, d, f, E, k, maxg, nslice, rs;
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// weights stream through once: skip L1
__device__ __forceinline__ uint4 ld_stream16(const moe_bf16* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
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
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
  return *s_abort == 0;
}

// Stream-K partition: warp w of nw owns quads [w*nq/nw, (w+1)*nq/nw).
__device__ __forceinline__ uint32_t range_begin(uint32_t w, uint32_t nq, uint32_t nw) {
  return (uint32_t)(((uint64_t)w * nq) / nw);
}

// Sum of group g's partials at (pair slot qq, column col), in warp order.
// part: [nw][maxg][kDecSeg][kDecCols]; a group holds quads [g*qg, (g+1)*qg).
// The contributing warps' range starts follow from one division (w*nq = qb*nw
// + r, stepped by nq = qs*nw + rs), and their loads are issued eight at a
// time before any is added.
__device__ float sum_partials(const float* part, uint32_t g, int qq, int col, uint32_t qg,
                              uint32_t nq, uint32_t nw, int maxg) {
  const uint64_t a = (uint64_t)g * qg, b = a + qg;
  // the last warp whose range starts at or before quad a, and the one for quad b - 1
  const uint32_t w0 = (uint32_t)(((a + 1) * nw + nq - 1) / nq - 1);
  const uint32_t w1 = (uint32_t)((b * nw + nq - 1) / nq - 1);
  const uint32_t qs = nq / nw, rs = nq - qs * nw;
  const uint64_t t0 = (uint64_t)w0 * nq;
  uint32_t qb = (uint32_t)(t0 / nw), r = (uint32_t)(t0 - (uint64_t)qb * nw);
  const float* src = part + qq * kDecCols + col;
  float s = 0.f;
  for (uint32_t w = w0; w <= w1; w += 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      // range of warp w + u: [qb, qe)
      uint32_t qe = qb + qs, r2 = r + rs;
      if (r2 >= nw) { r2 -= nw; ++qe; }
      v[u] = 0.f;
      if (w + u <= w1 && qb < qe) {
        const int j = (int)(g - qb / qg);
        if (j >= 0 && j < maxg)
          v[u] = __ldcg(src + ((size_t)(w + u) * maxg + j) * kDecGroupFloats);
      }
      qb = qe;
      r = r2;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) s += v[u];
  }
  return s;
}

// Adds the four row-lanes' sums (lanes l, l^8, l^16, l^24 share columns) and
// stores the warp's partial of group g for the np pairs of its segment.
__device__ __forceinline__ void flush_partial(float (&acc)[kDecSeg][8], int np, float* part,
                                              uint32_t gw, int maxg, int j, int lane) {
#pragma unroll
  for (int qq = 0; qq < kDecSeg; ++qq) {
    if (qq < np) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        float v = acc[qq][c];
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 8);
        v += __shfl_xor_sync(0xFFFFFFFFu, v, 16);
        acc[qq][c] = v;
      }
    }
  }
  if (lane < 8) {
    if (j >= 0 && j < maxg) {
      float* dst = part + ((size_t)gw * maxg + j) * kDecGroupFloats + lane * 8;
#pragma unroll
      for (int qq = 0; qq < kDecSeg; ++qq) {
        if (qq < np) {
          reinterpret_cast<float4*>(dst + qq * kDecCols)[0] =
              make_float4(acc[qq][0], acc[qq][1], acc[qq][2], acc[qq][3]);
          reinterpret_cast<float4*>(dst + qq * kDecCols)[1] =
              make_float4(acc[qq][4], acc[qq][5], acc[qq][6], acc[qq][7]);
        }
      }
    }   // j is always in range: maxg bounds the groups any warp's range touches
  }
#pragma unroll
  for (int qq = 0; qq < kDecSeg; ++qq)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[qq][c] = 0.f;
}

__device__ __forceinline__ float bf16_bits_to_f(unsigned short b) {
  return __uint_as_float((uint32_t)b << 16);
}

template <int NV>
__global__ void __launch_bounds__(kDecThreads, 1) decode_fwd_kernel(const DecArgs a) {
  extern __shared__ __align__(16) float red[];   // kDecRedFloats, then x as [d][8] bf16
  unsigned short* xs = reinterpret_cast<unsigned short*>(red + kDecRedFloats);
  __shared__ volatile int s_abort;
  __shared__ int s_idx[kDecMaxPairs];
  __shared__ float s_w[kDecMaxPairs];
  __shared__ int s_key[kDecMaxPairs];        // expert of the pair, E if dropped
  __shared__ int s_pair[kDecMaxPairs];       // pairs sorted by (expert, pair id)
  __shared__ int s_tok[kDecMaxPairs];        // token of the pair at a position
  __shared__ int s_pos[kDecMaxPairs];        // position of a pair in that order
  __shared__ int s_posseg[kDecMaxPairs];     // segment of a position
  __shared__ int s_segb[kDecMaxPairs + 1];   // first position of a segment
  __shared__ int s_sege[kDecMaxPairs];       // expert of a segment
  __shared__ int s_nsel, s_nvalid;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, d = a.d, f = a.f, E = a.E, k = a.k, maxg = a.maxg;
  const int P = T * k;
  if (tid == 0) s_abort = 0;
  unsigned* ctr = reinterpret_cast<unsigned*>(a.ws);
  float* part_a = reinterpret_cast<float*>(a.ws + 256);
  const size_t off_part = 256 + al256d((size_t)a.nslice * T * E * 4);
  float* part = reinterpret_cast<float*>(a.ws + off_part);
  const uint32_t nw = gridDim.x * kDecWarps, gw = blockIdx.x * kDecWarps + warp;
  unsigned target = 0;

  // x to shared memory, [row][token]
  for (int o = tid; o < T * d; o += kDecThreads) {
    const int t = o / d, i = o - t * d;
    xs[i * kDecMaxT + t] = a.x[o];
  }
  __syncthreads();

  // ---------------------------------------------------------------- A --
  {
    const int nchunk = (E + kDecRCols - 1) / kDecRCols;
    const int rpw = a.rs / kDecWarps;   // rows per warp
    const bool vec = (E % 4) == 0 && (reinterpret_cast<uintptr_t>(a.w_router) & 15u) == 0;
    for (int u = blockIdx.x; u < nchunk * a.nslice; u += gridDim.x) {
      const int chunk = u % nchunk, slice = u / nchunk;
      const int e0 = chunk * kDecRCols + 4 * lane;
      float acc[kDecMaxT][4];
#pragma unroll
      for (int t = 0; t < kDecMaxT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      for (int r0 = 0; r0 < rpw; r0 += 8) {
        float4 wv[8];
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int i = slice * a.rs + warp * rpw + r0 + rr;
          wv[rr] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r0 + rr < rpw && i < d) {
            const float* src = a.w_router + (int64_t)i * E + e0;
            if (vec && e0 + 3 < E) {
              wv[rr] = __ldg(reinterpret_cast<const float4*>(src));
            } else {
              if (e0 < E) wv[rr].x = __ldg(src);
              if (e0 + 1 < E) wv[rr].y = __ldg(src + 1);
              if (e0 + 2 < E) wv[rr].z = __ldg(src + 2);
              if (e0 + 3 < E) wv[rr].w = __ldg(src + 3);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < 8; ++rr) {
          const int i = slice * a.rs + warp * rpw + r0 + rr;
          if (r0 + rr >= rpw || i >= d) break;
#pragma unroll
          for (int t = 0; t < kDecMaxT; ++t) {
            if (t < T) {
              const float xv = bf16_bits_to_f(xs[i * kDecMaxT + t]);
              acc[t][0] = fmaf(xv, wv[rr].x, acc[t][0]);
              acc[t][1] = fmaf(xv, wv[rr].y, acc[t][1]);
              acc[t][2] = fmaf(xv, wv[rr].z, acc[t][2]);
              acc[t][3] = fmaf(xv, wv[rr].w, acc[t][3]);
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kDecMaxT; ++t)
        if (t < T)
          reinterpret_cast<float4*>(red + (warp * kDecMaxT + t) * kDecRCols)[lane] =
              make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
      __syncthreads();
      for (int o = tid; o < T * kDecRCols; o += kDecThreads) {
        const int t = o / kDecRCols, col = o % kDecRCols, e = chunk * kDecRCols + col;
        if (e >= E) continue;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) s += red[(w * kDecMaxT + t) * kDecRCols + col];
        part_a[((size_t)slice * T + t) * E + e] = s;
      }
      __syncthreads();
    }
  }
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // ---------------------------------------------------------------- B --
  for (int o = tid; o < T * E; o += kDecThreads) {
    float s = 0.f;
    for (int sl0 = 0; sl0 < a.nslice; sl0 += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = sl0 + u < a.nslice ? __ldcg(part_a + (size_t)(sl0 + u) * T * E + o) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    s += a.bias ? a.bias[o % E] : 0.f;
    red[o] = s;
    if (blockIdx.x == 0) a.logits[o] = s;
  }
  __syncthreads();
  if (warp < T)
    topk_warp<NV>(red + warp * E, a.forced ? a.forced + warp * k : nullptr, E, k, lane,
                  s_idx + warp * k, s_w + warp * k, a.status);
  __syncthreads();
  for (int p = tid; p < P; p += kDecThreads) {
    const int e = s_idx[p];   // an invalid caller-chosen id is kept in topk_idx, dropped here
    s_key[p] = (e >= 0 && e < E) ? e : E;
    if (blockIdx.x == 0) {
      a.topk_idx[p] = e;
      a.topk_w[p] = s_w[p];
    }
  }
  __syncthreads();
  for (int p = tid; p < P; p += kDecThreads) {
    int rank = 0;
    for (int q = 0; q < P; ++q) rank += (s_key[q] < s_key[p]) || (s_key[q] == s_key[p] && q < p);
    s_pair[rank] = p;
    s_tok[rank] = p / k;
    s_pos[p] = rank;
  }
  __syncthreads();
  if (tid == 0) {
    int n = 0, prev = -1, pos = 0;
    for (; pos < P; ++pos) {
      const int e = s_key[s_pair[pos]];
      if (e >= E) break;
      // a new segment per expert, and every kDecSeg pairs within one
      if (e != prev || pos - s_segb[n - 1] == kDecSeg) {
        s_sege[n] = e;
        s_segb[n] = pos;
        ++n;
        prev = e;
      }
      s_posseg[pos] = n - 1;
    }
    s_segb[n] = pos;
    s_nsel = n;
    s_nvalid = pos;
  }
  __syncthreads();
  const int n_sel = s_nsel, n_valid = s_nvalid;
  const int rq = lane >> 3, cq = (lane & 7) * 8;

  // ---------------------------------------------------------------- C --
  // Each warp walks its quads with a ring of kDecBatch loads in flight: a
  // slot's quad is multiplied, then the slot is refilled kDecBatch quads ahead.
  const uint32_t nfc = f / kDecCols, qgc = d / 4;
  const uint32_t ngc = (uint32_t)n_sel * 2 * nfc, nqc = ngc * qgc;
  {
    const uint32_t qb = range_begin(gw, nqc, nw), qe = range_begin(gw + 1, nqc, nw);
    auto group_row0 = [&](uint32_t g) {   // row rq, column cq of group g
      const uint32_t sg = g / (2 * nfc), m = (g / nfc) & 1u, c = g % nfc;
      const int e = sg < (uint32_t)n_sel ? s_sege[sg] : 0;
      return (m ? a.w_up : a.w_gate) + ((int64_t)e * d + rq) * f + c * kDecCols + cq;
    };
    uint32_t lq = qb, lg = qb / qgc, lr = qb - (qb / qgc) * qgc;
    const moe_bf16* lrow = group_row0(lg);
    auto issue = [&](uint4& slot) {
      if (lq < qe) slot = ld_stream16(lrow + (int64_t)lr * 4 * f);
      ++lq;
      if (++lr == qgc) {
        lr = 0;
        ++lg;
        if (lg < ngc) lrow = group_row0(lg);
      }
    };
    uint4 v[kDecBatch];
#pragma unroll
    for (int b = 0; b < kDecBatch; ++b) issue(v[b]);
    float acc[kDecSeg][8];
#pragma unroll
    for (int qq = 0; qq < kDecSeg; ++qq)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[qq][c] = 0.f;
    const int g_first = (int)(qb / qgc);
    int cur_g = -1, np = 0, pb = 0;
    uint32_t pq = qb, pg = g_first, pr = qb - g_first * qgc;
    while (pq < qe) {
#pragma unroll
      for (int b = 0; b < kDecBatch; ++b) {
        if (pq >= qe) break;
        if ((int)pg != cur_g) {
          if (cur_g >= 0) flush_partial(acc, np, part, gw, maxg, cur_g - g_first, lane);
          cur_g = (int)pg;
          const int sg = (int)(pg / (2 * nfc));
          pb = s_segb[sg];
          np = s_segb[sg + 1] - pb;
        }
        const int i = (int)pr * 4 + rq;
        float wv[8];
        unpack8(v[b], wv);
        issue(v[b]);
#pragma unroll
        for (int qq = 0; qq < kDecSeg; ++qq) {
          if (qq < np) {
            const float xv = bf16_bits_to_f(xs[i * kDecMaxT + s_tok[pb + qq]]);
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[qq][c] = fmaf(xv, wv[c], acc[qq][c]);
          }
        }
        ++pq;
        if (++pr == qgc) {
          pr = 0;
          ++pg;
        }
      }
    }
    if (cur_g >= 0) flush_partial(acc, np, part, gw, maxg, cur_g - g_first, lane);
  }
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // --------------------------------------------------------------- C2 --
  float* ai = reinterpret_cast<float*>(a.ws + off_part +
                                       al256d((size_t)nw * maxg * kDecGroupFloats * 4));
  for (int64_t o = (int64_t)blockIdx.x * kDecThreads + tid; o < (int64_t)n_valid * f;
       o += (int64_t)gridDim.x * kDecThreads) {
    const int pos = (int)(o / f), i = (int)(o - (int64_t)pos * f);
    const int sg = s_posseg[pos], qq = pos - s_segb[sg];
    const uint32_t gg = (uint32_t)sg * 2 * nfc + i / kDecCols;
    const float g = sum_partials(part, gg, qq, i % kDecCols, qgc, nqc, nw, maxg);
    const float u = sum_partials(part, gg + nfc, qq, i % kDecCols, qgc, nqc, nw, maxg);
    ai[(int64_t)i * P + pos] = __fdividef(g, 1.0f + __expf(-g)) * u;
  }
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // ---------------------------------------------------------------- D --
  // As C. A for the rows of slot b's quad is fetched at refill time by lanes
  // 4b .. 4b+3 (one row each, every pair of the segment) and handed to the
  // multiplying lanes by shuffle.
  const uint32_t ndc = d / kDecCols, qgd = f / 4;
  const uint32_t ngd = (uint32_t)n_sel * ndc, nqd = ngd * qgd;
  {
    const uint32_t qb = range_begin(gw, nqd, nw), qe = range_begin(gw + 1, nqd, nw);
    int lpb = 0, lnp = 0;
    auto group_row0 = [&](uint32_t g) {
      const uint32_t sg = g / ndc, c = g % ndc;
      const int e = sg < (uint32_t)n_sel ? s_sege[sg] : 0;
      if (sg < (uint32_t)n_sel) {
        lpb = s_segb[sg];
        lnp = s_segb[sg + 1] - lpb;
      }
      return a.w_down + ((int64_t)e * f + rq) * d + c * kDecCols + cq;
    };
    uint32_t lq = qb, lg = qb / qgd, lr = qb - (qb / qgd) * qgd;
    const moe_bf16* lrow = group_row0(lg);
    float av[kDecSeg];
#pragma unroll
    for (int qq = 0; qq < kDecSeg; ++qq) av[qq] = 0.f;
    auto issue = [&](uint4& slot, int b) {
      if (lq < qe) {
        slot = ld_stream16(lrow + (int64_t)lr * 4 * d);
        if ((lane >> 2) == b) {
          const float* src = ai + (int64_t)(lr * 4 + (lane & 3)) * P + lpb;
#pragma unroll
          for (int qq = 0; qq < kDecSeg; ++qq) av[qq] = qq < lnp ? __ldcg(src + qq) : 0.f;
        }
      }
      ++lq;
      if (++lr == qgd) {
        lr = 0;
        ++lg;
        if (lg < ngd) lrow = group_row0(lg);
      }
    };
    uint4 v[kDecBatch];
#pragma unroll
    for (int b = 0; b < kDecBatch; ++b) issue(v[b], b);
    float acc[kDecSeg][8];
#pragma unroll
    for (int qq = 0; qq < kDecSeg; ++qq)
#pragma unroll
      for (int c = 0; c < 8; ++c) acc[qq][c] = 0.f;
    const int g_first = (int)(qb / qgd);
    int cur_g = -1, np = 0;
    uint32_t pq = qb, pg = g_first, pr = qb - g_first * qgd;
    while (pq < qe) {
#pragma unroll
      for (int b = 0; b < kDecBatch; ++b) {
        if (pq >= qe) break;
        if ((int)pg != cur_g) {
          if (cur_g >= 0) flush_partial(acc, np, part, gw, maxg, cur_g - g_first, lane);
          cur_g = (int)pg;
          const int sg = (int)(pg / ndc);
          np = s_segb[sg + 1] - s_segb[sg];
        }
        float wv[8], xv[kDecSeg];
        unpack8(v[b], wv);
#pragma unroll
        for (int qq = 0; qq < kDecSeg; ++qq)
          xv[qq] = __shfl_sync(0xFFFFFFFFu, av[qq], b * 4 + rq);
        issue(v[b], b);
#pragma unroll
        for (int qq = 0; qq < kDecSeg; ++qq) {
          if (qq < np) {
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[qq][c] = fmaf(xv[qq], wv[c], acc[qq][c]);
          }
        }
        ++pq;
        if (++pr == qgd) {
          pr = 0;
          ++pg;
        }
      }
    }
    if (cur_g >= 0) flush_partial(acc, np, part, gw, maxg, cur_g - g_first, lane);
  }
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // ---------------------------------------------------------------- E --
  // kp = k rounded up to a power of two lanes per output element: lane j
  // forms w[t, j] * (expert output of pair (t, j)), the kp lanes add theirs
  // in a fixed butterfly, the first writes y.
  {
    int kp = 1;
    while (kp < k) kp <<= 1;
    const int64_t total = (int64_t)T * d * kp;   // a multiple of 64: whole warps
    for (int64_t o = (int64_t)blockIdx.x * kDecThreads + tid; o < total;
         o += (int64_t)gridDim.x * kDecThreads) {
      const int j = (int)(o % kp);
      const int64_t el = o / kp;
      const int t = (int)(el / d), col = (int)(el - (int64_t)t * d);
      float v = 0.f;
      const int p = t * k + j;
      if (j < k && s_key[p] < E) {
        const int pos = s_pos[p], sg = s_posseg[pos];
        const uint32_t g = (uint32_t)sg * ndc + col / kDecCols;
        v = s_w[p] * sum_partials(part, g, pos - s_segb[sg], col % kDecCols, qgd, nqd, nw, maxg);
      }
      for (int off = kp >> 1; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
      if (j == 0) a.y[el] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  }
}

cudaError_t launch_decode_fwd(const moe_bf16* x, const float* w_router, const float* bias,
                              const int32_t* forced, int T, int d, int f, int E, int k,
                              const moe_bf16* w_gate, const moe_bf16* w_up,
                              const moe_bf16* w_down, float* logits, int32_t* topk_idx,
                              float* topk_w, moe_bf16* y, void* ws, int* status,
                              cudaStream_t s) {
  const int nv = (E + 31) / 32;
  const int variant = nv <= 1 ? 0 : nv <= 2 ? 1 : nv <= 4 ? 2 : nv <= 8 ? 3 : nv <= 16 ? 4 : 5;
  void (*const kerns[6])(const DecArgs) = {
      decode_fwd_kernel<1>, decode_fwd_kernel<2>, decode_fwd_kernel<4>,
      decode_fwd_kernel<8>, decode_fwd_kernel<16>, decode_fwd_kernel<kMaxExperts / 32>};
  auto kern = kerns[variant];
  const int smem_max = kDecRedFloats * 4 + kDecMaxD * kDecMaxT * 2;   // 192 KiB
  const int smem = kDecRedFloats * 4 + d * kDecMaxT * 2;
  // shared-memory opt-in and the residency check, once per variant and device
  constexpr int kDevices = 64;
  static int ready[6][kDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  if (!ready[variant][dev]) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecThreads, smem_max);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    ready[variant][dev] = 1;
  }
  const int grid = num_sms();   // one CTA per SM: all resident, as the barriers need
  const DecGeom g = decode_geom(T, d, f, E, k, grid);
  DecArgs args{x,      w_router, bias,   forced,      w_gate, w_up,     w_down,
               logits, topk_idx, topk_w, y,           static_cast<char*>(ws), status,
               T,      d,        f,      E,           k,      g.maxg,   g.nslice, g.rs};
  err = cudaMemsetAsync(ws, 0, 256, s);   // the barrier counter
  if (err != cudaSuccess) return err;
  void* kargs[] = {(void*)&args};
  timer_before(MOE_KERNEL_DECODE, s);
  err = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kDecThreads), kargs, smem,
                                    s);
  note_launches(1);
  timer_after(MOE_KERNEL_DECODE, s);
  return err;
}

}  // namespace moe
