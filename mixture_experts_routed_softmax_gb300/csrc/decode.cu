// decode.cu — the layer's forward for a handful of tokens (decode), in one
// cooperative kernel.
//
// With T <= 8 tokens the layer is bound by reading the selected experts'
// weights once (Halo "Performance", §Levers that do not help here: small-M
// experts are bound by weight bandwidth); launching the general path's seven
// kernels costs more than the work. One persistent kernel, one CTA per SM,
// runs these phases, separated by grid barriers (|):
//   A   router partial dot products: (row slice of W_r, 128 experts) units
//   |
//   B   every CTA sums the partials into the logits, takes the top-k with
//       renormalised weights (topk.cuh) and cuts the kept pairs, sorted by
//       (expert, pair id), into segments of at most 4 pairs of one expert
//       (an expert with more pairs has its weights read once per segment);
//       CTA 0 writes logits, topk_idx and topk_w
//   C   gate/up products: the selected experts' W_gate and W_up are read in
//       stages of R whole rows (contiguous memory; rows wider than 4096
//       columns are cut into equal column blocks), each stage a few TMA boxes
//       landing in a ring of shared-memory stages. Groups are (segment,
//       matrix, column block); their stages are cut into equal contiguous
//       ranges, one per CTA (stream-K). A thread owns 8 columns of a block
//       and a lane of rows, and multiplies them with every pair of the
//       segment; at the end of a group the CTA adds its lanes' sums (fixed
//       order) and writes one partial
//   |
//   C2  G and U = the partials of each group added in a fixed order (a few
//       lanes, each over every n-th contributing CTA, then a butterfly);
//       A = silu(G) * U (fp32), stored per segment as [f][4]
//   |
//   D   down products over W_down in the same way (groups: segment, column
//       block of d); each stage's copy also brings its rows of A
//   |
//   E1  the expert output of every pair = its group's partials (fixed order)
//   |
//   E   y[t] = sum_j w[t, j] * (expert output of pair (t, j)) in slot order,
//       rounded to bf16 once
// A seventeenth warp of each CTA issues the TMA copies in the streaming phases
// while the other sixteen multiply; it computes nothing in the other phases.
// Every sum has a fixed order, so two runs on one GPU are bitwise equal. Every
// wait is bounded: a grid barrier (a counter in the workspace, zeroed by the
// host before the launch) or a ring barrier that times out records
// MOE_ERR_DEVICE_TIMEOUT; the CTA then stops computing, lets the copies it
// issued land, and skips the remaining phases.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "topk.cuh"

namespace moe {

constexpr int kDecThreads = 512;              // the threads that compute, in every phase
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecProducer = kDecWarps;       // one more warp: it issues the TMA copies
constexpr int kDecConsumers = kDecWarps;
constexpr int kDecBlock = kDecThreads + 32;   // threads of a CTA
constexpr int kDecMaxT = kDecodeMaxT;
constexpr int kDecMaxPairs = kDecMaxT * kMaxTopK;
constexpr int kDecMaxBlockCols = kDecThreads * 8;   // a thread owns 8 columns of a block
constexpr int kDecMaxStages = 16;
constexpr int kDecSeg = 4;            // pairs of one expert a segment holds
constexpr int kDecRCols = 128;        // router: experts per unit (4 per lane)
constexpr int kDecRedFloats = kDecWarps * kDecMaxT * kDecRCols;   // 64 KiB
constexpr int kDecRouterPartialFloats = 16384;   // partial logits each CTA sums in phase B
constexpr int kDecFlushFloats = 4096;            // 16 KiB: warp groups' sums at a group's end
constexpr int kDecMaxGrid = 256;                 // CTAs (SMs) the range tables hold

static_assert(kDecRedFloats >= kDecMaxT * kMaxExperts, "the logits fit the reduction buffer");

__host__ __device__ static inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ static inline size_t al256d(size_t b) { return (b + 255) & ~(size_t)255; }

// How one streaming phase cuts a weight matrix of `rows` x `cols` (per expert)
// and maps it to threads. A thread owns 8 columns (an octet) of a block and a
// row lane; the L row lanes of an octet sit in one warp (lanes o + l * opw),
// so their sums meet by shuffles; wg groups of warps split the rows further.
struct PhaseGeom {
  int nblk;         // column blocks
  int cb;           // columns of a block (a multiple of 8, at most 4096)
  int no;           // 8-column octets of a block
  int L;            // row lanes inside a warp
  int opw;          // octets per warp: 32 / L
  int nwo;          // warps that cover the octets of one row lane set
  int wg;           // warp groups (row lanes L * wg in all)
  int R;            // rows of a stage: a power of two <= 64, so it divides rows
  int bw;           // columns of a TMA box
  int nbox;         // boxes of a stage
  int box_stride;   // shared-memory bytes between the boxes of a stage
  int stage_bytes;  // nbox * box_stride
  int slot_bytes;   // a ring slot: the boxes (then, in D, the A values), 1 KiB aligned
  int tx_bytes;     // bytes the boxes of a stage deliver
  int spg;          // stages per group: rows / R
};

// Bytes of one ring stage, about. A CTA's ring completes stages at a roughly
// fixed rate whatever its depth, so stages are made large (up to 48 KiB),
// leaving room for three of them next to x (d * 16 bytes) and the 16 KiB
// flush buffer.
__host__ __device__ static inline int stage_target(int d) {
  const int ring = 220000 - 1024 - 16384 - 16 * d;
  const int t = ring / 3;
  return t > 49152 ? 49152 : (t < 8192 ? 8192 : t);
}

// down: a slot also carries the stage's A values (R rows x kDecSeg floats)
__host__ __device__ static inline PhaseGeom phase_geom(int cols, int rows, bool down, int target) {
  PhaseGeom p;
  p.nblk = (cols + kDecMaxBlockCols - 1) / kDecMaxBlockCols;
  p.cb = cols / p.nblk;
  p.no = p.cb / 8;
  p.L = 1;
  for (int l = 32; l >= 1; --l) {
    const int opw = 32 / l;
    if ((p.no + opw - 1) / opw <= kDecConsumers) {
      p.L = l;
      break;
    }
  }
  p.opw = 32 / p.L;
  p.nwo = (p.no + p.opw - 1) / p.opw;
  p.wg = kDecConsumers / p.nwo;
  if (p.wg * p.no > 128) p.wg = p.no >= 128 ? 1 : 128 / p.no;   // the flush buffer's 16 KiB
  int r = target / (2 * p.cb);
  r = r < 1 ? 1 : (r > 64 ? 64 : r);
  p.R = 1;
  while (2 * p.R <= r) p.R *= 2;
  p.bw = p.cb < 256 ? p.cb : 256;
  p.nbox = (p.cb + p.bw - 1) / p.bw;
  p.box_stride = (p.R * p.bw * 2 + 127) & ~127;
  p.stage_bytes = p.nbox * p.box_stride;
  p.slot_bytes = (p.stage_bytes + (down ? 64 * kDecSeg * 4 : 0) + 1023) & ~1023;
  p.tx_bytes = p.nbox * p.bw * p.R * 2;
  p.spg = rows / p.R;
  return p;
}

// the shapes phase_geom takes: equal column blocks of whole octets
static bool phase_ok(int cols) {
  const int nblk = (cols + kDecMaxBlockCols - 1) / kDecMaxBlockCols;
  return cols % nblk == 0 && (cols / nblk) % 8 == 0;
}

// Workspace layout and partition sizes, shared by the host (size, launch)
// and the kernel.
struct DecGeom {
  int maxg;      // partial slots per CTA (groups one CTA's range of stages can touch)
  int slotf;     // floats of one partial slot: kDecSeg x the wider block
  int nslice;    // router row slices
  int rs;        // router rows per slice (a multiple of kDecWarps)
  size_t off_part, off_ai, off_yp, total;
};

static DecGeom decode_geom(int64_t T, int d, int f, int E, int k, int grid) {
  DecGeom g{};
  const int64_t P = T * k;
  const PhaseGeom pc = phase_geom(f, d, false, stage_target(d));
  const PhaseGeom pd = phase_geom(d, f, true, stage_target(d));
  // a range of L stages touches at most ceil(L / stages per group) + 1 groups
  const int64_t nqc = P * 2 * pc.nblk * pc.spg, nqd = P * pd.nblk * pd.spg;
  const int64_t mc = cdiv64(cdiv64(nqc, grid), pc.spg) + 1;
  const int64_t md = cdiv64(cdiv64(nqd, grid), pd.spg) + 1;
  g.maxg = (int)(mc > md ? mc : md);
  g.slotf = kDecSeg * (pc.cb > pd.cb ? pc.cb : pd.cb);
  int64_t ns = kDecRouterPartialFloats / (T * E > 0 ? T * E : 1);
  ns = ns < 1 ? 1 : ns;
  const int64_t ns_max = cdiv64(d, 128);
  g.nslice = (int)(ns < ns_max ? ns : ns_max);
  g.rs = (int)(cdiv64(cdiv64(d, g.nslice), kDecWarps) * kDecWarps);
  g.nslice = (int)cdiv64(d, g.rs);
  g.off_part = 256 + al256d((size_t)g.nslice * T * E * 4);
  g.off_ai = g.off_part + al256d((size_t)grid * g.maxg * g.slotf * 4);
  g.off_yp = g.off_ai + al256d((size_t)P * f * kDecSeg * 4);
  g.total = g.off_yp + al256d((size_t)P * d * 4);
  return g;
}

bool decode_shape_ok(int d, int f) { return phase_ok(d) && phase_ok(f); }

size_t decode_ws_bytes(int64_t T, int d, int f, int E, int k) {
  return decode_geom(T, d, f, E, k, num_sms()).total;
}

struct DecArgs {
  const moe_bf16* x;
  const float* w_router;
  const float* bias;
  const int32_t* forced;
  float* logits;
  int32_t* topk_idx;
  float* topk_w;
  moe_bf16* y;
  char* ws;
  int* status;
  int T, d, f, E, k, maxg, slotf, nslice, rs, stages, stage_slot;
  size_t off_part, off_ai, off_yp;
};

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ float bf16_bits_to_f(unsigned short b) {
  return __uint_as_float((uint32_t)b << 16);
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

// Stream-K partition: unit w of nw owns items [w*nq/nw, (w+1)*nq/nw).
__device__ __forceinline__ uint32_t range_begin(uint32_t w, uint32_t nq, uint32_t nw) {
  return (uint32_t)(((uint64_t)w * nq) / nw);
}

// The first item of each CTA's stream-K range, tq[w] = w*nq/nw for w in
// [0, nw], and the group it falls in, tg[w] = tq[w] / qg: built once per
// phase in shared memory so that reductions divide nothing.
__device__ void build_ranges(uint32_t* tq, uint32_t* tg, uint32_t nq, uint32_t qg) {
  for (uint32_t w = threadIdx.x; w <= gridDim.x; w += blockDim.x) {
    tq[w] = range_begin(w, nq, gridDim.x);
    tg[w] = tq[w] / qg;
  }
}

// Lanes per reduced element: enough that each adds at most four partials in
// one round. A group of qg items meets at most qg / L + 2 CTA ranges of L.
__device__ __forceinline__ int reduce_lanes(uint32_t nq, uint32_t qg) {
  const uint32_t L = nq / gridDim.x > 0 ? nq / gridDim.x : 1;
  const uint32_t c = qg / L + 2;
  return c <= 4 ? 1 : c <= 8 ? 2 : c <= 16 ? 4 : 8;
}

// The partials of group g at (pair slot qq, column col of the block), summed
// by nsub consecutive lanes of a warp (sub = lane % nsub, the whole warp taking
// part): lane s adds those of contributing CTAs w0 + s, w0 + s + nsub, ... in
// order, then the nsub lanes meet in a fixed butterfly; every lane returns
// the sum as lane s = 0 forms it. Two groups (g0, g1) are reduced together so
// that their loads are in flight at once. part: [nw][maxg][slotf], a slot laid
// out [pair][cb]; group g holds items [g*qg, (g+1)*qg).
template <int NG>
__device__ void sum_partials(const float* part, const uint32_t* tq, const uint32_t* tg,
                             const uint32_t (&g)[NG], int qq, int col, int cb, uint32_t qg,
                             int maxg, int slotf, int sub, int nsub, float (&out)[NG]) {
  const uint32_t nw = gridDim.x;
  const float* src = part + qq * cb + col;
  uint32_t w[NG], b[NG];
#pragma unroll
  for (int h = 0; h < NG; ++h) {
    const uint32_t a = g[h] * qg;
    b[h] = a + qg;
    uint32_t lo = 0, hi = nw;   // tq[lo] <= a < tq[hi]: the last CTA starting at or before a
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (tq[mid] <= a) lo = mid;
      else hi = mid;
    }
    w[h] = lo + sub;
    out[h] = 0.f;
  }
  for (;;) {
    float v[NG][4];
    bool more = false;
#pragma unroll
    for (int h = 0; h < NG; ++h) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t wu = w[h] + nsub * u;
        v[h][u] = 0.f;
        if (wu < nw && tq[wu] < b[h] && tq[wu] < tq[wu + 1]) {
          const int j = (int)(g[h] - tg[wu]);
          if (j >= 0 && j < maxg) v[h][u] = __ldcg(src + ((size_t)wu * maxg + j) * slotf);
        }
      }
      w[h] += 4 * nsub;
      more = more || (w[h] < nw && tq[w[h]] < b[h]);
    }
#pragma unroll
    for (int h = 0; h < NG; ++h)
#pragma unroll
      for (int u = 0; u < 4; ++u) out[h] += v[h][u];
    if (!more) break;
  }
#pragma unroll
  for (int h = 0; h < NG; ++h) {
    for (int m = nsub >> 1; m > 0; m >>= 1) out[h] += __shfl_xor_sync(0xFFFFFFFFu, out[h], m);
    out[h] = __shfl_sync(0xFFFFFFFFu, out[h], (threadIdx.x & 31) & ~(nsub - 1));
  }
}

// 1-D bulk copy global -> shared, counted on an mbarrier (16-byte aligned,
// size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// orders this thread's view of global memory written by other CTAs (seen
// through the grid barrier) before its later asynchronous-proxy reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// barrier of the computing warps only (named barrier 1)
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"r"(kDecThreads) : "memory");
}

// bounded wait used on the way out: ignores the abort flag, still time-limited
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  volatile int never = 0;
  mbar_wait_bounded(bar, parity, &never, status);
}

// The shared-memory ring of TMA stages. Stages are numbered by `seq` across
// the phases of one launch; stage m uses slot m % slots in its
// (m / slots)-th use.
struct Ring {
  unsigned char* base;   // slot 0
  uint32_t buf;     // shared address of slot 0
  uint32_t full;    // shared address of full barrier 0 (8 bytes apart)
  uint32_t empty;   // empty barrier 0: one arrival per warp
  int slots;
  int slot_bytes;
  uint32_t seq;     // stages of earlier phases
};

// One streaming phase (C: DOWN = false, D: DOWN = true) over this CTA's range
// of stages. Groups of C: g = (segment * 2 + matrix) * nblk + block, matrix 0
// gate, 1 up, rows of d; groups of D: g = segment * nblk + block, rows of f.
// The loop runs the same iterations and barriers in every thread whatever the
// waits return; after a failed wait it only stops computing and issuing.
template <bool DOWN>
__device__ void stream_phase(Ring& ring, const PhaseGeom pg, const CUtensorMap* map0,
                             const CUtensorMap* map1, uint32_t ngroups,
                             const unsigned short* xs, const float* ai, int P,
                             const int* s_segb, const int* s_sege, const int* s_tok,
                             float* part, int maxg, int slotf, float* flush,
                             volatile int* s_abort, int* status) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wgi = warp / pg.nwo, wo = warp - wgi * pg.nwo;
  const int l = lane / pg.opw, o = lane - l * pg.opw;
  const int c8 = wo * pg.opw + o;                     // octet of the block
  const bool active = warp < kDecConsumers && wgi < pg.wg && l < pg.L && c8 < pg.no;
  const int lrow = wgi * pg.L + l, nlanes = pg.L * pg.wg;   // row lane, row lanes
  const int bo = pg.bw / 8;                                  // octets of a box
  const uint32_t col_off = (uint32_t)((c8 / bo) * pg.box_stride + (c8 % bo) * 16);
  const uint32_t spg = (uint32_t)pg.spg;
  const uint32_t nq = ngroups * spg;
  const uint32_t qb = range_begin(blockIdx.x, nq, gridDim.x);
  const uint32_t qe = range_begin(blockIdx.x + 1, nq, gridDim.x);
  const uint32_t nst = qe - qb;
  const uint32_t S = (uint32_t)ring.slots;
  const uint32_t seq0 = ring.seq;
  const uint32_t per_seg = (DOWN ? 1u : 2u) * pg.nblk;   // groups per segment

  // ---- producer (lane 0 of the producer warp): runs up to S stages ahead.
  // In D a stage also carries its rows' A values: R rows of the segment's
  // [f][4] block, one bulk copy counted on the same barrier.
  if (warp == kDecProducer) {
    if (lane == 0) {
      if (DOWN) fence_proxy_async_global();
      uint32_t issued = 0, p_g = 0, p_sr = 0;
      if (nst > 0) {
        p_g = qb / spg;
        p_sr = qb - p_g * spg;
      }
      const int f = pg.spg * pg.R;   // rows of a D group
      while (issued < nst && !*s_abort) {
        const uint32_t m = seq0 + issued;
        const uint32_t sl = m % S, use = m / S;
        if (use > 0 && !mbar_wait_bounded(ring.empty + 8 * sl, (use - 1) & 1u, s_abort, status))
          break;
        const uint32_t sg = p_g / per_seg, blk = p_g % pg.nblk;
        const bool up = !DOWN && ((p_g / pg.nblk) & 1u);
        const int e = s_sege[sg];
        const uint32_t bar = ring.full + 8 * sl, dst = ring.buf + sl * ring.slot_bytes;
        mbar_arrive_expect_tx(bar, pg.tx_bytes + (DOWN ? pg.R * kDecSeg * 4 : 0));
        for (int b = 0; b < pg.nbox; ++b)
          tma_load_3d(dst + b * pg.box_stride, up ? map1 : map0, bar,
                      (int)blk * pg.cb + b * pg.bw, (int)(p_sr * pg.R), e);
        if (DOWN)
          bulk_load(dst + pg.stage_bytes, ai + ((int64_t)sg * f + p_sr * pg.R) * kDecSeg,
                    pg.R * kDecSeg * 4, bar);
        ++issued;
        if (++p_sr == spg) {
          p_sr = 0;
          ++p_g;
        }
      }
      if (*s_abort) {
        // let the copies already issued land before the shared memory goes away
        const uint32_t lo = issued > S ? issued - S : 0;
        for (uint32_t n = lo; n < issued; ++n) {
          const uint32_t m = seq0 + n;
          drain_wait(ring.full + 8 * (m % S), (m / S) & 1u, status);
        }
      }
    }
    __syncwarp();
    ring.seq = seq0 + nst;
    return;
  }

  // ---- consumers (the other warps): cursor over the stages, the same in every one
  float acc[kDecSeg][8];
#pragma unroll
  for (int qq = 0; qq < kDecSeg; ++qq)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[qq][c] = 0.f;
  uint32_t g = 0, sr = 0;
  if (nst > 0) {
    g = qb / spg;
    sr = qb - g * spg;
  }
  const uint32_t g_first = g;
  int pb = 0, np = 0;
  if (nst > 0) {
    const uint32_t sg = g / per_seg;
    pb = s_segb[sg];
    np = s_segb[sg + 1] - pb;
  }
  for (uint32_t n = 0; n < nst; ++n) {
    const uint32_t m = seq0 + n, sl = m % S, use = m / S;
    uint32_t g2 = g, sr2 = sr + 1;   // the next stage
    if (sr2 == spg) {
      sr2 = 0;
      ++g2;
    }
    const bool ok = mbar_wait_bounded(ring.full + 8 * sl, use & 1u, s_abort, status);
    if (ok) {
      if (active) {
        const uint32_t base = ring.buf + sl * ring.slot_bytes + col_off;
        const float* as = reinterpret_cast<const float*>(ring.base + (size_t)sl * ring.slot_bytes +
                                                         pg.stage_bytes);
        for (int rr = lrow; rr < pg.R; rr += nlanes) {
          const uint4 v = lds128(base + rr * (pg.bw * 2));
          float wv[8];
          unpack8(v, wv);
          const int row = (int)(sr * pg.R) + rr;
#pragma unroll
          for (int qq = 0; qq < kDecSeg; ++qq) {
            if (qq < np) {
              const float xv = DOWN ? as[rr * kDecSeg + qq]
                                    : bf16_bits_to_f(xs[row * kDecMaxT + s_tok[pb + qq]]);
#pragma unroll
              for (int c = 0; c < 8; ++c) acc[qq][c] = fmaf(xv, wv[c], acc[qq][c]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(ring.empty + 8 * sl);
    }
    if (g2 != g || n + 1 == nst) {
      // end of a group in this range: the row lanes of a warp add theirs in
      // lane order by shuffles; with several warp groups their sums meet in
      // shared memory, in group order
      const int j = (int)(g - g_first);   // < maxg by the slot bound
#pragma unroll
      for (int qq = 0; qq < kDecSeg; ++qq) {
        if (qq < np) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            float t = __shfl_sync(0xFFFFFFFFu, acc[qq][c], o);
            for (int l2 = 1; l2 < pg.L; ++l2)
              t += __shfl_sync(0xFFFFFFFFu, acc[qq][c], o + l2 * pg.opw);
            acc[qq][c] = t;
          }
        }
      }
      if (pg.wg == 1) {
        if (active && l == 0 && j < maxg) {
          float* dst = part + ((size_t)blockIdx.x * maxg + j) * slotf + c8 * 8;
#pragma unroll
          for (int qq = 0; qq < kDecSeg; ++qq) {
            if (qq < np) {
              reinterpret_cast<float4*>(dst + qq * pg.cb)[0] =
                  make_float4(acc[qq][0], acc[qq][1], acc[qq][2], acc[qq][3]);
              reinterpret_cast<float4*>(dst + qq * pg.cb)[1] =
                  make_float4(acc[qq][4], acc[qq][5], acc[qq][6], acc[qq][7]);
            }
          }
        }
      } else {
        if (active && l == 0) {
#pragma unroll
          for (int qq = 0; qq < kDecSeg; ++qq) {
            if (qq < np) {
              float4* dst = reinterpret_cast<float4*>(flush + (wgi * kDecSeg + qq) * pg.cb + c8 * 8);
              dst[0] = make_float4(acc[qq][0], acc[qq][1], acc[qq][2], acc[qq][3]);
              dst[1] = make_float4(acc[qq][4], acc[qq][5], acc[qq][6], acc[qq][7]);
            }
          }
        }
        consumers_sync();
        if (j < maxg) {
          float* out = part + ((size_t)blockIdx.x * maxg + j) * slotf;
          for (int oo = tid; oo < np * pg.cb; oo += kDecThreads) {
            const int qq = oo / pg.cb, col = oo - qq * pg.cb;
            float t = 0.f;
            for (int w = 0; w < pg.wg; ++w) t += flush[(w * kDecSeg + qq) * pg.cb + col];
            out[oo] = t;
          }
        }
        consumers_sync();
      }
#pragma unroll
      for (int qq = 0; qq < kDecSeg; ++qq)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[qq][c] = 0.f;
      if (n + 1 < nst) {
        const uint32_t sg = g2 / per_seg;
        pb = s_segb[sg];
        np = s_segb[sg + 1] - pb;
      }
    }
    g = g2;
    sr = sr2;
  }
  ring.seq = seq0 + nst;
}

template <int NV>
__global__ void __launch_bounds__(kDecBlock, 1)
    decode_fwd_kernel(const __grid_constant__ CUtensorMap map_gate,
                      const __grid_constant__ CUtensorMap map_up,
                      const __grid_constant__ CUtensorMap map_down, const DecArgs a) {
  // dynamic shared memory: ring slots (the first 64 KiB doubling as the
  // router's reduction buffer before any copy is issued) | flush buffer
  // (16 KiB) | x as [d][8] bf16
  extern __shared__ __align__(16) unsigned char dsm[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dsm) + 1023) & ~(uintptr_t)1023);
  float* red = reinterpret_cast<float*>(base);
  const size_t ring_bytes = (size_t)a.stages * a.stage_slot;
  float* flush = reinterpret_cast<float*>(
      base + (ring_bytes > kDecRedFloats * 4 ? ring_bytes : (size_t)kDecRedFloats * 4));
  unsigned short* xs = reinterpret_cast<unsigned short*>(flush + kDecFlushFloats);
  __shared__ __align__(8) uint64_t s_bar[2 * kDecMaxStages];
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
  __shared__ uint32_t s_tq[kDecMaxGrid + 1], s_tg[kDecMaxGrid + 1];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, d = a.d, f = a.f, E = a.E, k = a.k, maxg = a.maxg;
  const int P = T * k;
  Ring ring{base,     smem_u32(base),  smem_u32(&s_bar[0]), smem_u32(&s_bar[kDecMaxStages]),
            a.stages, a.stage_slot,    0u};
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(ring.full + 8 * i, 1);
      mbar_init(ring.empty + 8 * i, kDecConsumers);
    }
    fence_mbar_init();
    tma_prefetch_desc(&map_gate);
    tma_prefetch_desc(&map_up);
    tma_prefetch_desc(&map_down);
  }
  unsigned* ctr = reinterpret_cast<unsigned*>(a.ws);
  float* part_a = reinterpret_cast<float*>(a.ws + 256);
  float* part = reinterpret_cast<float*>(a.ws + a.off_part);
  float* ai = reinterpret_cast<float*>(a.ws + a.off_ai);
  unsigned target = 0;

  // x to shared memory as [row][token]: one row's T tokens per thread, one
  // 16-byte store
  for (int i = tid; i < d && tid < kDecThreads; i += kDecThreads) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int t = 0; t < kDecMaxT; ++t)
      if (t < T) w[t >> 1] |= (uint32_t)a.x[(int64_t)t * d + i] << ((t & 1) * 16);
    reinterpret_cast<uint4*>(xs)[i] = make_uint4(w[0], w[1], w[2], w[3]);
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
          if (warp < kDecWarps && r0 + rr < rpw && i < d) {
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
          if (warp >= kDecWarps || r0 + rr >= rpw || i >= d) break;
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
      if (warp < kDecWarps) {
#pragma unroll
        for (int t = 0; t < kDecMaxT; ++t)
          if (t < T)
            reinterpret_cast<float4*>(red + (warp * kDecMaxT + t) * kDecRCols)[lane] =
                make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
      }
      __syncthreads();
      for (int o = tid; o < T * kDecRCols && tid < kDecThreads; o += kDecThreads) {
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
  for (int o = tid; o < T * E && tid < kDecThreads; o += kDecThreads) {
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

  // ---------------------------------------------------------------- C --
  const PhaseGeom pc = phase_geom(f, d, false, stage_target(d));
  const uint32_t ngc = (uint32_t)n_sel * 2 * pc.nblk;
  stream_phase<false>(ring, pc, &map_gate, &map_up, ngc, xs, ai, P, s_segb, s_sege, s_tok, part,
                      maxg, a.slotf, flush, &s_abort, a.status);
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // --------------------------------------------------------------- C2 --
  // a few lanes per element of A (see sum_partials); A is stored per
  // segment as [f][4] (16-byte rows: the down phase's stages copy it in bulk)
  const uint32_t nqc = ngc * (uint32_t)pc.spg;
  build_ranges(s_tq, s_tg, nqc, pc.spg);
  __syncthreads();
  {
    const int nsub = reduce_lanes(nqc, pc.spg), lg = __ffs(nsub) - 1;
    for (int64_t o = (int64_t)blockIdx.x * kDecThreads + tid;
         warp < kDecWarps && o < ((int64_t)n_valid * f << lg);
         o += (int64_t)gridDim.x * kDecThreads) {   // a multiple of 64: whole warps
      const int64_t el = o >> lg;
      const int pos = (int)(el / f), i = (int)(el - (int64_t)pos * f);
      const int sg = s_posseg[pos], qq = pos - s_segb[sg];
      const int blk = i / pc.cb, col = i - blk * pc.cb;
      const uint32_t gg[2] = {(uint32_t)(sg * 2) * pc.nblk + blk,
                              (uint32_t)(sg * 2 + 1) * pc.nblk + blk};
      const int sub = (int)(o & (nsub - 1));
      float gu[2];
      sum_partials<2>(part, s_tq, s_tg, gg, qq, col, pc.cb, pc.spg, maxg, a.slotf, sub, nsub, gu);
      if (sub == 0)
        ai[((int64_t)sg * f + i) * kDecSeg + qq] = __fdividef(gu[0], 1.0f + __expf(-gu[0])) * gu[1];
    }
  }
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // ---------------------------------------------------------------- D --
  const PhaseGeom pd = phase_geom(d, f, true, stage_target(d));
  const uint32_t ngd = (uint32_t)n_sel * pd.nblk;
  stream_phase<true>(ring, pd, &map_down, &map_down, ngd, xs, ai, P, s_segb, s_sege, s_tok, part,
                     maxg, a.slotf, flush, &s_abort, a.status);
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // --------------------------------------------------------------- E1 --
  // the expert output of every kept pair, Yp [P, d] fp32
  float* yp = reinterpret_cast<float*>(a.ws + a.off_yp);
  {
    const uint32_t nqd = ngd * (uint32_t)pd.spg;
    build_ranges(s_tq, s_tg, nqd, pd.spg);
    __syncthreads();
    const int nsub = reduce_lanes(nqd, pd.spg), lg = __ffs(nsub) - 1;
    for (int64_t o = (int64_t)blockIdx.x * kDecThreads + tid;
         warp < kDecWarps && o < ((int64_t)n_valid * d << lg);
         o += (int64_t)gridDim.x * kDecThreads) {   // a multiple of 64: whole warps
      const int64_t el = o >> lg;
      const int pos = (int)(el / d), cold = (int)(el - (int64_t)pos * d);
      const int sg = s_posseg[pos];
      const int blk = cold / pd.cb, col = cold - blk * pd.cb;
      const uint32_t g1[1] = {(uint32_t)sg * pd.nblk + blk};
      const int sub = (int)(o & (nsub - 1));
      float v[1];
      sum_partials<1>(part, s_tq, s_tg, g1, pos - s_segb[sg], col, pd.cb, pd.spg, maxg, a.slotf,
                      sub, nsub, v);
      if (sub == 0) yp[el] = v[0];
    }
  }
  if (!grid_sync(ctr, target, &s_abort, a.status)) return;

  // ---------------------------------------------------------------- E --
  // y[t] = sum_j w[t, j] * Yp[pair (t, j)], in slot order, rounded once
  for (int64_t o = (int64_t)blockIdx.x * kDecThreads + tid; tid < kDecThreads && o < (int64_t)T * d;
       o += (int64_t)gridDim.x * kDecThreads) {
    const int t = (int)(o / d), col = (int)(o - (int64_t)t * d);
    float acc = 0.f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      float v[8], w[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u, p = t * k + j;
        const bool kept = j < k && s_key[p] < E;
        v[u] = kept ? __ldcg(yp + (int64_t)s_pos[p] * d + col) : 0.f;
        w[u] = kept ? s_w[p] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (j0 + u < k) acc = fmaf(w[u], v[u], acc);
    }
    a.y[o] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
  }
}

// ------------------------------------------------------------------ host --

typedef CUresult (*DecEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static DecEncodeFn dec_encode_fn() {
  static DecEncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<DecEncodeFn>(p);
  });
  return fn;
}

// 3-D bf16 map over [E, rows, cols] (cols innermost), box [1, R, bw], no
// swizzle; boxes past the last column are zero-filled
static bool dec_map(CUtensorMap* m, const void* ptr, uint64_t cols, uint64_t rows, uint64_t E,
                    const PhaseGeom& pg) {
  DecEncodeFn fn = dec_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {cols, rows, E};
  cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
  cuuint32_t box[3] = {(cuuint32_t)pg.bw, (cuuint32_t)pg.R, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_decode_fwd(const moe_bf16* x, const float* w_router, const float* bias,
                              const int32_t* forced, int T, int d, int f, int E, int k,
                              const moe_bf16* w_gate, const moe_bf16* w_up,
                              const moe_bf16* w_down, float* logits, int32_t* topk_idx,
                              float* topk_w, moe_bf16* y, void* ws, int* status,
                              cudaStream_t s) {
  if (!decode_shape_ok(d, f)) return cudaErrorInvalidValue;
  const int nv = (E + 31) / 32;
  const int variant = nv <= 1 ? 0 : nv <= 2 ? 1 : nv <= 4 ? 2 : nv <= 8 ? 3 : nv <= 16 ? 4 : 5;
  void (*const kerns[6])(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                         const DecArgs) = {
      decode_fwd_kernel<1>, decode_fwd_kernel<2>, decode_fwd_kernel<4>,
      decode_fwd_kernel<8>, decode_fwd_kernel<16>, decode_fwd_kernel<kMaxExperts / 32>};
  auto kern = kerns[variant];
  // dynamic shared memory the kernel may use, once per variant and device
  constexpr int kDevices = 64;
  static int dyn_max[6][kDevices] = {};
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kDevices) return cudaErrorInvalidDevice;
  if (!dyn_max[variant][dev]) {
    int optin = 0;
    err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    cudaFuncAttributes fa{};
    err = cudaFuncGetAttributes(&fa, kern);
    if (err != cudaSuccess) return err;
    const int avail = optin - (int)fa.sharedSizeBytes;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, avail);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDecBlock, avail);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    dyn_max[variant][dev] = avail;
  }
  const PhaseGeom pc = phase_geom(f, d, false, stage_target(d));
  const PhaseGeom pd = phase_geom(d, f, true, stage_target(d));
  // ring: what is left after the 1 KiB alignment slack, the flush buffer and x
  // (at least the 64 KiB the router's reduction borrows)
  const int slot = pc.slot_bytes > pd.slot_bytes ? pc.slot_bytes : pd.slot_bytes;
  const int fixed = 1024 + kDecFlushFloats * 4 + d * kDecMaxT * 2;
  int stages = (dyn_max[variant][dev] - fixed) / slot;
  stages = stages > kDecMaxStages ? kDecMaxStages : stages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const int ring = stages * slot > kDecRedFloats * 4 ? stages * slot : kDecRedFloats * 4;
  if (fixed + ring > dyn_max[variant][dev]) return cudaErrorInvalidConfiguration;
  const int smem = fixed + ring;

  CUtensorMap mg, mu, md;
  if (!dec_map(&mg, w_gate, f, d, E, pc) || !dec_map(&mu, w_up, f, d, E, pc) ||
      !dec_map(&md, w_down, d, f, E, pd))
    return cudaErrorInvalidValue;
  const int grid = num_sms();   // one CTA per SM: all resident, as the barriers need
  if (grid > kDecMaxGrid) return cudaErrorInvalidConfiguration;
  const DecGeom g = decode_geom(T, d, f, E, k, grid);
  DecArgs args{x,       w_router, bias,     forced, logits, topk_idx, topk_w, y,
               static_cast<char*>(ws),      status, T,      d,        f,      E,
               k,       g.maxg,   g.slotf,  g.nslice, g.rs, stages,   slot,   g.off_part,
               g.off_ai, g.off_yp};
  err = cudaMemsetAsync(ws, 0, 256, s);   // the barrier counter
  if (err != cudaSuccess) return err;
  void* kargs[] = {(void*)&mg, (void*)&mu, (void*)&md, (void*)&args};
  timer_before(MOE_KERNEL_DECODE, s);
  err = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kDecBlock), kargs, smem,
                                    s);
  note_launches(1);
  timer_after(MOE_KERNEL_DECODE, s);
  return err;
}

}  // namespace moe
