// gemm.cu — grouped expert GEMMs on the 5th-generation tensor cores.
//
// Halo "Performance", §Levers that help: one grouped expert matmul instead of
// a per-expert loop, with the GLU fused. prime-rl PR #3885 (DeepSeek-V4.1
// Flash perf work), §Changes: grouped forward, dgrad and wgrad GEMMs ("FP8
// routed experts"), the weight gradient as a K-grouped GEMM and the bf16
// gate/up output kept for backward ("FP8 Mega MoE").
//
// One persistent, warp-specialised kernel template serves the six GEMMs of the
// layer, the router's two and the fused forward:
//   warp 0      TMA producer: tiles of A and B into a shared-memory ring of
//               as many stages as fit 192 KiB (4 of 48 KiB, 6 of 32 KiB; the
//               down dgrad of a CTA pair keeps 5 and gives 32 KiB to its
//               epilogue's G/U loads)
//   warp 1      MMA issuer: tcgen05.mma 128 x N x 16 (bf16 in, fp32 in tensor
//               memory), two accumulator buffers so the epilogue of one tile
//               overlaps the main loop of the next
//   warp 2      tensor-memory allocator
//   warps 4-11  epilogue, two warpgroups (each half of the tile's columns):
//               tcgen05.ld of the accumulator (one row per thread), the fused
//               element-wise step, TMA stores staged through a 3-slot ring
//               (per warpgroup, or per warp for the down dgrad)
// Kinds:
//   GateUpFwd    [G | U] = Xp . [W_gate[e] | W_up[e]]  (two accumulators),
//                epilogue A = act(G, U) (the SwiGLU, clamped or plain:
//                swiglu() below); stores G, U (fp32, for the backward's
//                activation gradient) and A (bf16)            (M-grouped)
//   DownFwd      Yp = A . W_down[e]  (optionally * row_w), fp32  (M-grouped)
//   DownDgrad    dAu = dY[t(r)] . W_down[e]^T from the unscaled gathered rows
//                of dY; epilogue dA = w(r) * dAu (the pair's score on the
//                fp32 accumulator; 1 for a shared expert's row),
//                dG = dA * dact/dG, dU = dA * dact/dU, and the row's share of
//                the top-k weight gradient <dAu, act(G, U)> (= <dY, A.W_down>
//                with A unrounded), one fp32 partial per (n-tile, column
//                half)                                          (M-grouped)
//   GateUpDgrad  dXp = dG . W_gate[e]^T + dU . W_up[e]^T (two K segments), fp32
//   WgradDown    dW_down[e] = A_e^T . dYp_e                     (K-grouped)
//   WgradGateUp  dW_gate[e] = Xp_e^T . dG_e, dW_up[e] = Xp_e^T . dU_e
//   FusedFwd     GateUpFwd's tiles (A only) and then DownFwd's (Yp scaled by
//                the pair's score) in one launch, each down tile waiting for
//                the gate/up tiles of its rows (prime-rl PR #3885, §Changes,
//                "FP8 Mega MoE": the expert layer as one op)
//   RouterLogits, RouterWgrad: the router's GEMMs (route.cu); GateUpFwdNarrow
//   and DownFwdNarrow: 64- and 128-wide tiles for few rows per expert
// "M-grouped": expert e's output rows are its rows [offsets[e], offsets[e+1])
// of the padded layout, cut into 128-row tiles (a tile may run past the group
// end; those rows are computed and not stored). "K-grouped": the reduction
// runs over expert e's rows, in 64-row steps; the last step issues only the
// 16-row MMA slices inside the group (groups are multiples of 16 rows), and
// an expert with no rows gets a zero tile.
#include "common.cuh"
#include "internal.h"

#include <mutex>

namespace moe {

enum class Kind {
  GateUpFwd, DownFwd, DownDgrad, GateUpDgrad, WgradDown, WgradGateUp, RouterLogits,
  RouterWgrad,      // dW_r partials = x^T . dl (dl's three bf16 parts side by side in N)
  GateUpFwdNarrow,  // GateUpFwd with 64-column tiles, for experts of at most ~128 rows
  FusedFwd,         // the fused expert forward: gate/up + act, then down (below)
  DownFwdNarrow     // DownFwd with 128-column tiles, for experts of at most ~128 rows
};

constexpr int BM = 128;            // tile rows (TMEM lanes)
constexpr int BK = 64;             // k per stage: one 128-byte swizzle atom of bf16
constexpr int kABytes = BM * BK * 2;                      // 16 KiB
constexpr int kRingBytes = 192 * 1024;                    // the TMA ring: 4 x 48 KiB, 6 x 32 KiB
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 8;       // epilogue warps: two warpgroups, each half the columns

template <Kind K>
struct Tr {
  static constexpr bool gateup_fwd = (K == Kind::GateUpFwd || K == Kind::GateUpFwdNarrow);
  static constexpr bool fused = (K == Kind::FusedFwd);
  // dual: two B tiles side by side, one N = 256 MMA (the fused forward's down
  // tiles use the same stage layout with one 256-column B tile)
  static constexpr bool dual = (gateup_fwd || K == Kind::WgradGateUp || fused);
  static constexpr bool two_seg = (K == Kind::GateUpDgrad);
  static constexpr bool kgrouped = (K == Kind::WgradDown || K == Kind::WgradGateUp);
  // one group of M rows, fp32 output (split K: one partial per chunk)
  static constexpr bool dense = (K == Kind::RouterLogits || K == Kind::RouterWgrad);
  static constexpr bool a_mn = kgrouped || K == Kind::RouterWgrad;         // A is M-contiguous
  static constexpr bool down_fwd = (K == Kind::DownFwd || K == Kind::DownFwdNarrow);
  static constexpr bool narrow = (K == Kind::GateUpFwdNarrow);
  static constexpr bool down_narrow = (K == Kind::DownFwdNarrow);
  static constexpr bool b_mn = (gateup_fwd || down_fwd || kgrouped || dense || fused);
  static constexpr int BN = narrow ? 64 : (dual || down_narrow) ? 128 : 256;   // per accumulator
  // tile width chosen per launch (at most BN): the K-major-B kinds, whose B box
  // is exactly the tile's rows, and the router, whose N is the expert count
  static constexpr bool var_bn = (K == Kind::DownDgrad || K == Kind::GateUpDgrad || dense);
  // each epilogue warp stages and stores its own 32 rows, so warps never wait
  // for each other at a slice: the down dgrad, whose threads wait on their
  // rows' G and U loads, and the weight gradients, bound by their stores when
  // experts hold few rows (the others store 128-row boxes per warpgroup,
  // fewer and larger TMA stores)
  static constexpr bool warp_stage = (K == Kind::DownDgrad || kgrouped);
  // bytes TMA lands per stage (A tile + one or two B tiles), and as many stages as fit
  static constexpr int tx_bytes = kABytes + (dual ? 2 : 1) * BN * BK * 2;
  static constexpr int stages = kRingBytes / tx_bytes > kMaxStages ? kMaxStages
                                                                   : kRingBytes / tx_bytes;
  static constexpr int kernel_id =
      fused ? MOE_KERNEL_FUSED_FWD
      : gateup_fwd ? MOE_KERNEL_GATEUP_FWD
      : down_fwd ? MOE_KERNEL_DOWN_FWD
      : K == Kind::DownDgrad ? MOE_KERNEL_DOWN_DGRAD
      : K == Kind::GateUpDgrad ? MOE_KERNEL_GATEUP_DGRAD
      : K == Kind::WgradDown ? MOE_KERNEL_WGRAD_DOWN
      : K == Kind::WgradGateUp ? MOE_KERNEL_WGRAD_GATEUP
      : K == Kind::RouterWgrad ? MOE_KERNEL_ROUTE_BWD
                               : MOE_KERNEL_ROUTER_LOGITS;
};

// Shared-memory ring per CTA: one A tile and all of B's tile (or, in a CTA
// pair, this CTA's half of B's columns) per stage, as many stages as fit.
// The down dgrad of a CTA pair (half the B bytes per stage) gives the ring's
// tail to its epilogue: gu_slots slots per epilogue warp, each 8 fp32 columns
// of the warp's 32 rows of G and of U ([32 rows x 32 bytes] x 2, loaded by
// TMA), so the saved activations arrive ahead of use without holding
// registers (two slots and five 32 KiB stages measured faster than four and
// four, or none and six). A single CTA keeps its four 48 KiB stages and loads
// G and U into registers.
template <Kind K, bool PAIR>
struct Geo {
  using T = Tr<K>;
  static constexpr int b_bytes = (T::dual ? 2 : 1) * T::BN * BK * 2 / (PAIR ? 2 : 1);
  static constexpr int stage_bytes = kABytes + b_bytes;
  static constexpr int gu_slots = (K == Kind::DownDgrad && PAIR) ? 2 : 0;
  static constexpr int gu_slot_bytes = 2 * 32 * 32;
  static constexpr int gu_bytes = gu_slots * kEpiWarps * gu_slot_bytes;
  static constexpr int ring = kRingBytes - gu_bytes;
  static constexpr int stages = ring / stage_bytes > kMaxStages ? kMaxStages : ring / stage_bytes;
};

constexpr int kTmemCols = 512;                            // 2 accumulator buffers x 256 columns
constexpr int kThreads = 128 + 32 * kEpiWarps;
// Epilogues stage their outputs through shared memory for TMA stores: a ring
// of kStgSlots slots per epilogue warpgroup, each [128 rows x 32 bytes] (16
// bf16 or 8 fp32 columns of one output), or, for the kinds that stage per
// warp (Tr::warp_stage), the same bytes as a ring per warp of [32 rows x 32
// bytes] slots
constexpr int kStgSlots = 3;
constexpr int kStagePerGroup = kStgSlots * 128 * 32;
constexpr int kStageOutBytes = (kEpiWarps / 4) * kStagePerGroup;
// the tile table, rounded up so the staging slots after it sit on 1 KiB
// boundaries (the 32-byte swizzle pattern is taken from address bits 4-7)
constexpr int kTstartBytes = (4 * (kMaxExperts + 1) + 1023) & ~1023;
constexpr int kSmemBytes = kRingBytes + 1024 /*bars*/ + kTstartBytes + kStageOutBytes + 1024;

// The experts' gated activation, A = h(min(G, L)) * (clamp(U, -L, L) + c) with
// h(g) = g * sigmoid(alpha g): the clamped SwiGLU of GPT-OSS-style layers
// (prime-rl PR #3885, §Changes, "FP8 routed experts"), and with L = inf,
// alpha = 1, c = 0 the plain SwiGLU silu(G) * U (Halo "Performance", §Levers
// that help, fused GLU).
struct Act {
  float limit, alpha, c;
};
__device__ __forceinline__ float swiglu(float g, float u, const Act& a) {
  const float gc = fminf(g, a.limit);
  const float uc = fminf(fmaxf(u, -a.limit), a.limit);
  return __fdividef(gc, 1.0f + __expf(-a.alpha * gc)) * (uc + a.c);
}

struct GemmArgs {
  const int64_t* offsets;
  int E;
  int M, N;        // K-grouped: per-expert output is M x N. M-grouped: N output columns
  int nk_seg;      // M-grouped: k-steps per K segment
  int64_t R_cap;
  void* out0;      // bf16, or fp32 (G, U of GateUpFwd; DownFwd; GateUpDgrad)
  void* out1;
  void* out2;
  const float* row_w;
  const float* in0;          // DownDgrad in one CTA: the saved G, U (fp32; a pair reads them by TMA)
  const float* in1;
  const float* pair_w;       // DownDgrad: the score of each routed pair ([T*k], via src_pair)
  int64_t p_routed;          // DownDgrad: pairs below this are routed; the rest shared (weight 1)
  Act act;                   // GateUpFwd, DownDgrad: the activation
  float* dtw_part;           // DownDgrad: [R_cap][dtw_slots] partials of the top-k weight grad
  int dtw_slots;             // 2 per n-tile (one per epilogue warpgroup)
  // RouterLogits: fp32 output, bias, number of K segments and the K offset of each in B
  float* outf;
  const float* bias;
  int nseg;
  int seg_koff;
  int ksplit;         // RouterLogits: K split into this many chunks (1: write logits + bias)
  int ksteps_split;   // k-steps per chunk
  int bn;             // single-accumulator kinds: tile width (multiple of 16, <= 256)
  const int32_t* src_pair;   // pair of each layout row (-1: padding): K-grouped (or NULL), DownDgrad, FusedFwd
  int* status;
  // FusedFwd: N = f (gate/up tiles, nk_seg k-steps over d), N2 = d (down
  // tiles, nk2 k-steps over f); out2 = A (bf16), out3 = Yp (fp32, scaled by
  // each row's score via src_pair / pair_w); ready[m-tile] counts the
  // gate/up tiles done
  int N2;
  int nk2;
  void* out3;
  int* ready;
};

struct TileInfo {
  int e;
  int ph;           // FusedFwd: 0 gate/up tile, 1 down tile
  int mt;           // FusedFwd: the m-tile's index in the tile table
  int64_t m0;       // first output row (M-grouped: row of the layout; K-grouped: row of dW[e])
  int n0;
  int nk;           // k-steps
  int64_t row_end;  // M-grouped: end of the expert's group; K-grouped: group length (rows)
  int64_t kbeg;     // K-grouped: first row of the group
};

// tile width: BN, or for the var_bn kinds the width the launch chose so that
// N splits into equal tiles (N = 2880: twelve of 240)
template <Kind K>
__device__ __forceinline__ int tile_bn(const GemmArgs& a) {
  return Tr<K>::var_bn ? a.bn : Tr<K>::BN;
}

// A CTA pair (PAIR) takes 256-row tiles: rank 0 the first 128 rows, rank 1
// the next 128 (past the group's end: computed, not stored).
template <Kind K, bool PAIR>
__device__ __forceinline__ void decode_tile(int tile, const GemmArgs& a, const int* tstart,
                                            int nN, int rank, TileInfo& ti) {
  using T = Tr<K>;
  constexpr int TM = PAIR ? 2 * BM : BM;
  const int bn = tile_bn<K>(a);
  int nt = tile % nN;
  int mt = tile / nN;
  ti.n0 = nt * bn;
  ti.ph = 0;
  if constexpr (T::fused) {
    // gate/up tiles (128 + 128 columns of f) of every m-tile first, then the
    // down tiles (256 columns of d); both in the tile table's expert order
    const int nN1 = (a.N + 127) / 128, nN2 = (a.N2 + 255) / 256;
    const int tiles1 = tstart[a.E] * nN1;
    if (tile < tiles1) {
      mt = tile / nN1;
      ti.n0 = (tile % nN1) * 128;
      ti.nk = a.nk_seg;
    } else {
      const int t2 = tile - tiles1;
      ti.ph = 1;
      mt = t2 / nN2;
      ti.n0 = (t2 % nN2) * 256;
      ti.nk = a.nk2;
    }
    ti.mt = mt;
  }
  if constexpr (T::dense) {
    // tile = (m-tile * nN + n-tile) * ksplit + split; e holds the split
    const int sp = tile % a.ksplit;
    const int mn = tile / a.ksplit;
    ti.e = sp;
    ti.n0 = (mn % nN) * bn;
    ti.m0 = (int64_t)(mn / nN) * BM;
    ti.row_end = a.M;
    ti.kbeg = (int64_t)sp * a.ksteps_split;
    const int total_steps = a.nk_seg * a.nseg;
    ti.nk = (int)min((int64_t)a.ksteps_split, (int64_t)total_steps - ti.kbeg);
  } else if constexpr (T::kgrouped) {
    const int nM = (a.M + TM - 1) / TM;
    ti.e = mt / nM;
    ti.m0 = (int64_t)(mt % nM) * TM + rank * BM;
    ti.kbeg = a.offsets[ti.e];
    // the reduction stops after the expert's real rows (rounded up to the MMA's
    // 16-row step; the padding rows are zero in both operands)
    ti.row_end = tstart[ti.e];
    ti.nk = (int)((ti.row_end + BK - 1) / BK);
  } else {
    int lo = 0, hi = a.E;  // largest e with tstart[e] <= mt
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tstart[mid] <= mt) lo = mid; else hi = mid;
    }
    ti.e = lo;
    ti.m0 = a.offsets[lo] + (int64_t)(mt - tstart[lo]) * TM + rank * BM;
    ti.row_end = a.offsets[lo + 1];
    ti.kbeg = 0;
    if constexpr (!T::fused) ti.nk = a.nk_seg * (T::two_seg ? 2 : 1);
  }
}

// The group's named barrier, returning whether every thread of the group passed `ok`:
// the group decides together whether to go on, so no warp is left waiting at
// a group barrier that another warp has abandoned.
__device__ __forceinline__ bool group_all(int group, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "bar.red.and.pred pout, %2, 128, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(group + 1)
      : "memory");
  return r != 0;
}

// Named barrier over one epilogue warpgroup (ids 1 and 2; id 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, 128;" ::"r"(group + 1) : "memory");
}

// Writes one 32-byte slice (16 bf16 or 8 fp32 columns, v[o][0..1]) of each of
// NOUT outputs for this thread's row. When the rows of the staging unit all
// belong to the group (stage_tma) — the warpgroup's 128 rows, or with WARP the
// warp's 32 — the unit stages the slices in its shared memory, one slot of
// [rows x 32 bytes] per output, and one thread (the warpgroup's first, or the
// warp's lane 0) issues one TMA store per slot (coordinates {col, r0} or
// {col, r0, e}, r0 the unit's first row; the maps clip at the tensor edge),
// each its own bulk group. The slots rotate through the unit's ring of
// kStgSlots, advancing only with stores issued, so a slot is written again as
// soon as the store that last used it has read it, while the later stores are
// still in flight. Rows are stored with the maps' 32-byte swizzle (the two
// 16-byte halves of rows 4-7 of every 8 swapped), so the warp's shared-memory
// writes hit distinct banks. Otherwise every thread stores its own row with
// masks. Columns from lim on (the tile's end, or N) are not written; N is the
// row stride; esz[o] the element size of output o (every output's slice
// starts at column col); rloc the thread's row within the unit.
template <int NOUT, bool K3D, bool WARP>
__device__ __forceinline__ void put_slice(const uint4 (&v)[NOUT][2], uint8_t* stg, int& slot,
                                          const CUtensorMap* const* maps, uint8_t* const* outs,
                                          const int* esz, bool stage_tma, bool row_ok,
                                          int64_t row, int rloc, int col, int N, int lim, int r0,
                                          int e, int group, bool leader, uint64_t policy) {
  static_assert(NOUT <= kStgSlots, "one slot per output");
  constexpr int kSlot = (WARP ? 32 : 128) * 32;
  if (stage_tma) {
    // the stores that last used these NOUT slots have read them
    if (leader) bulk_wait_read_n<kStgSlots - NOUT>();
    if constexpr (WARP) __syncwarp(); else group_sync(group);
    const int sw = ((rloc >> 2) & 1) * 16;
#pragma unroll
    for (int o = 0; o < NOUT; ++o) {
      int so = slot + o;
      so = so >= kStgSlots ? so - kStgSlots : so;
      uint8_t* d = stg + so * kSlot + rloc * 32;
      *reinterpret_cast<uint4*>(d + sw) = v[o][0];
      *reinterpret_cast<uint4*>(d + (16 - sw)) = v[o][1];
    }
    fence_async_smem();
    if constexpr (WARP) __syncwarp(); else group_sync(group);
    if (leader && col < lim) {
#pragma unroll
      for (int o = 0; o < NOUT; ++o) {
        int so = slot + o;
        so = so >= kStgSlots ? so - kStgSlots : so;
        const uint32_t src = smem_u32(stg + so * kSlot);
        if constexpr (K3D)
          tma_store_3d(maps[o], src, col, r0, e, policy);
        else
          tma_store_2d(maps[o], src, col, r0, policy);
        bulk_commit();
      }
    }
    // col and lim are the same in every thread of the unit
    if (col < lim) {
      slot += NOUT;
      slot = slot >= kStgSlots ? slot - kStgSlots : slot;
    }
  } else if (row_ok) {
#pragma unroll
    for (int o = 0; o < NOUT; ++o) {
      const int per16 = 16 / esz[o];   // columns per 16-byte piece
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = col + per16 * h;
        if (c < lim) *reinterpret_cast<uint4*>(outs[o] + (row * N + c) * esz[o]) = v[o][h];
      }
    }
  }
}

// the 16-byte halves of a 32-byte slice of packed bf16 pairs pk[8 * h .. 8 * h + 7]
template <int NOUT, int W>
__device__ __forceinline__ void slice_of(const uint32_t (&pk)[NOUT][W], int h,
                                         uint4 (&v)[NOUT][2]) {
#pragma unroll
  for (int o = 0; o < NOUT; ++o) {
    v[o][0] = make_uint4(pk[o][8 * h + 0], pk[o][8 * h + 1], pk[o][8 * h + 2], pk[o][8 * h + 3]);
    v[o][1] = make_uint4(pk[o][8 * h + 4], pk[o][8 * h + 5], pk[o][8 * h + 6], pk[o][8 * h + 7]);
  }
}

// bounded wait used on the way out: ignores the abort flag, still time-limited
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  volatile int never = 0;
  mbar_wait_bounded(bar, parity, &never, status);
}

// Waits until the count at `cnt` (bumped with release by other CTAs) reaches
// `target`, then orders the async proxy's later reads after it. Gives up like
// mbar_wait_bounded: false on the CTA's abort flag, or after kWaitLimitNs
// (then it sets the flag and raises MOE_ERR_DEVICE_TIMEOUT).
__device__ __noinline__ bool wait_count(const int* cnt, int target, volatile int* abort_flag,
                                        int* status) {
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0;; ++i) {
    if (ld_acquire_gpu(cnt) >= target) {
      fence_async_global();
      return true;
    }
    if ((i & 15u) == 15u) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > (uint64_t)kWaitLimitNs) {
        *abort_flag = 1;
        raise_status(status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
    __nanosleep(128);
  }
}

// The barrier over all eight epilogue warps (id 3), returning whether every
// thread passed `ok`: the fused forward's epilogue decides together, because
// its gate/up tiles end at a barrier of both warpgroups.
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "bar.red.and.pred pout, 3, %2, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(32 * kEpiWarps)
      : "memory");
  return r != 0;
}

template <Kind K, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA0,
                        const __grid_constant__ CUtensorMap mapA1,
                        const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB1,
                        const __grid_constant__ CUtensorMap mapO0,
                        const __grid_constant__ CUtensorMap mapO1,
                        const __grid_constant__ CUtensorMap mapO2,
                        const __grid_constant__ CUtensorMap mapB2,
                        const __grid_constant__ CUtensorMap mapO3, const GemmArgs args) {
  if constexpr (Tr<K>::fused)
    pdl_wait();   // CTAs wait on one another: no dependent kernel is scheduled before the end
  else
    pdl_enter();
  using T = Tr<K>;
  using G = Geo<K, PAIR>;
  static_assert(!PAIR || (!T::dense && !T::narrow && !T::down_narrow), "pairs: grouped kinds");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t s_base = smem_u32(smem);
  constexpr int kStages = G::stages;
  constexpr int kStageBytes = G::stage_bytes;           // a multiple of 8 KiB: atoms stay aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingBytes);
  // bars: full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2], drain
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kMaxStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kMaxStages + 4);
  // the down dgrad's G/U slots: one barrier per slot of each epilogue warp
  auto gu_bar = [&](int ew, int s) { return bar0 + 256u + 8u * (ew * 4 + s); };
  static_assert(G::gu_slots <= 4, "G/U slot barriers");
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 5);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int* tstart = reinterpret_cast<int*>(smem + kRingBytes + 1024);
  uint8_t* stage_out = smem + kRingBytes + 1024 + kTstartBytes;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pair: rank 0 issues the MMAs and owns the barriers both CTAs' loads
  // and epilogues report to
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const bool rank0 = rank == 0;
  // this CTA's (or pair's) first tile and the tile stride, read where used
  // (no register held across the kernel)
#define GEMM_CID (PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x)
#define GEMM_NCL (PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(drain_bar, 1);
    for (int ew = 0; ew < kEpiWarps; ++ew)
      for (int b = 0; b < G::gu_slots; ++b) mbar_init(gu_bar(ew, b), 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA0);
    tma_prefetch_desc(&mapB0);
    if (T::two_seg) tma_prefetch_desc(&mapA1);
    if (T::dual || T::two_seg) tma_prefetch_desc(&mapB1);
  }
  if (warp == 2) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(s_tmem), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(s_tmem), kTmemCols);
      tmem_relinquish();
    }
  }
  // K-grouped: tstart[e] = the rows of expert e the reduction runs over: its
  // real rows rounded up to 16 (the real rows come first in the group, then
  // the padding, whose src_pair is -1), or the whole group without src_pair
  if constexpr (T::kgrouped) {
    for (int e = threadIdx.x; e < args.E; e += kThreads) {
      const int64_t g0 = args.offsets[e], g1 = args.offsets[e + 1];
      int64_t n = g1 - g0;
      if (args.src_pair) {
        int64_t lo = g0, hi = g1;   // the first padding row is in [lo, hi]
        while (lo < hi) {
          const int64_t mid = (lo + hi) >> 1;
          if (args.src_pair[mid] >= 0) lo = mid + 1; else hi = mid;
        }
        n = ((lo - g0) + 15) & ~(int64_t)15;
        if (n > g1 - g0) n = g1 - g0;
      }
      tstart[e] = (int)n;
    }
  }
  // M-grouped tile table: tstart[e] = sum_{e'<e} ceil(L_e' / tile rows)
  constexpr int TM = PAIR ? 2 * BM : BM;
  if constexpr (!T::kgrouped && !T::dense) {
    for (int e = threadIdx.x; e < args.E; e += kThreads) {
      const int64_t L = args.offsets[e + 1] - args.offsets[e];
      tstart[e + 1] = (int)((L + TM - 1) / TM);
    }
    __syncthreads();
    if (warp == 3) {
      int run = 0;
      for (int b = 0; b < args.E; b += 32) {
        const int e = b + lane;
        int v = (e < args.E) ? tstart[e + 1] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xFFFFFFFFu, v, off);
          if (lane >= off) v += o;
        }
        if (e < args.E) tstart[e + 1] = run + v;
        run += __shfl_sync(0xFFFFFFFFu, v, 31);
      }
      if (lane == 0) tstart[0] = 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // the peer's barriers are initialised
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;

  const int bn = tile_bn<K>(args);
  const int nN = (args.N + bn - 1) / bn;
  int total;
  if constexpr (T::kgrouped) {
    total = args.E * ((args.M + TM - 1) / TM) * nN;
  } else if constexpr (T::dense) {
    total = ((args.M + BM - 1) / BM) * nN * args.ksplit;
  } else if constexpr (T::fused) {
    total = tstart[args.E] * (nN + (args.N2 + 255) / 256);
  } else {
    total = tstart[args.E] * nN;
  }
  // dual kinds: the two B tiles sit side by side in shared memory ([B0 | B1],
  // 64-column chunks at a fixed stride), so one N = 256 MMA fills both
  // accumulators (columns 0-127 and 128-255) and the A tile is read once
  // (a pair: one M = 256 MMA, B's columns split between the two CTAs; for the
  // dual kinds rank 0 holds B0 and rank 1 B1)
  constexpr uint32_t kIdesc =
      idesc_bf16(TM, T::dual ? 2 * T::BN : T::BN, T::a_mn ? 1 : 0, T::b_mn ? 1 : 0);
  constexpr uint32_t kBBytes = (uint32_t)T::BN * BK * 2;
  // B of a var_bn kind: bn rows (K-major) or ceil(bn / 64) 64-column boxes (N-major);
  // in a pair each CTA loads bn / 2 rows (K-major) or two boxes (N-major)
  const int nbox = (bn + 63) / 64;
  uint32_t b_bytes;
  if constexpr (PAIR)
    b_bytes = (T::dual || T::b_mn) ? 2u * (BK * 128) : (uint32_t)(bn / 2) * (BK * 2);
  else
    b_bytes = T::b_mn ? (uint32_t)nbox * (BK * 128) : (uint32_t)bn * (BK * 2);
  const uint32_t tx_bytes =
      (PAIR || T::var_bn) ? (uint32_t)kABytes + b_bytes : (uint32_t)G::stage_bytes;
  static_assert(kStages * kStageBytes <= G::ring && kStageBytes % 8192 == 0, "ring layout");

  if (warp == 0 && T::fused) {
    if (lane == 0) {
      // ----------------------------------------- producer (fused forward) --
      // Gate/up tiles: A from the gathered rows xp, B = W_gate and W_up
      // (in a pair: rank 0 W_gate, rank 1 W_up). Down tiles: A from the
      // activations buffer once every gate/up tile of their rows has
      // published it (a bounded wait on the m-tile's count), B = W_down (in
      // a pair each CTA half of the 256 columns). All by TMA; in a pair each
      // CTA loads its own 128 rows and its half of B for rank 0's barrier.
      const uint64_t pol_w = l2_evict_last();
      const int nN1 = nN;
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0;
      bool ok = true;
      for (int tile = GEMM_CID; tile < total && ok; tile += GEMM_NCL) {
        TileInfo ti;
        decode_tile<K, PAIR>(tile, args, tstart, nN, rank, ti);
        if (ti.ph == 1 &&
            !wait_count(args.ready + ti.mt, nN1 * (PAIR ? 2 : 1), s_abort, args.status))
          break;
        // rank 1's half of a group's last pair tile may lie past the group:
        // its rows then come from past the buffer (zeros, no traffic)
        const int arow = (PAIR && ti.m0 >= ti.row_end) ? (int)args.R_cap : (int)ti.m0;
        const void* mA = ti.ph ? (const void*)&mapA1 : (const void*)&mapA0;
        for (int ks = 0; ks < ti.nk; ++ks) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.status)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          const uint32_t sA = s_base + stage * kStageBytes;
          const uint32_t sB0 = sA + kABytes;
          const int kk = ks * BK;
          if constexpr (PAIR) {
            const uint32_t fbl = rank0 ? fb : mapa_shared(fb, 0);
            if (rank0) mbar_arrive_expect_tx(fb, 2u * tx_bytes);
            tma_load_2d_pair(sA, mA, fbl, kk, arow);
            const void* mB = ti.ph ? (const void*)&mapB2
                                   : (rank ? (const void*)&mapB1 : (const void*)&mapB0);
            const int bcol = ti.ph ? ti.n0 + 128 * rank : ti.n0;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              tma_load_3d_pair(sB0 + j * (BK * 128), mB, fbl, bcol + 64 * j, kk, ti.e, pol_w);
          } else {
            mbar_arrive_expect_tx(fb, tx_bytes);
            tma_load_2d(sA, mA, fb, kk, arow);
            if (ti.ph == 0) {
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                tma_load_3d_hint(sB0 + j * (BK * 128), &mapB0, fb, ti.n0 + 64 * j, kk, ti.e,
                                 pol_w);
                tma_load_3d_hint(sB0 + kBBytes + j * (BK * 128), &mapB1, fb, ti.n0 + 64 * j, kk,
                                 ti.e, pol_w);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                tma_load_3d_hint(sB0 + j * (BK * 128), &mapB2, fb, ti.n0 + 64 * j, kk, ti.e,
                                 pol_w);
            }
          }
          ++fills;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (*s_abort) {
        // let the copies already issued land before the CTA's shared memory goes away
        if (!PAIR || rank0) {
          const int outstanding = fills < kStages ? fills : kStages;
          int st = stage;
          uint32_t ph = phase;
          for (int i = 0; i < outstanding; ++i) {
            if (--st < 0) { st = kStages - 1; ph ^= 1u; }
            drain_wait(full_bar(st), ph, args.status);
          }
        } else {
          const uint64_t t0 = global_ns();
          while (global_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ producer --
      const uint64_t pol_w = l2_evict_last();   // expert weights: re-read by every m-tile
      int stage = 0;
      uint32_t phase = 0;
      int fills = 0;
      bool ok = true;
      if constexpr (PAIR) {
        // each CTA loads its A rows and its share of B's columns into its own
        // ring; the bytes are counted on rank 0's full barrier, which rank 0
        // arms for both
        for (int tile = GEMM_CID; tile < total && ok; tile += GEMM_NCL) {
          TileInfo ti;
          decode_tile<K, PAIR>(tile, args, tstart, nN, rank, ti);
          int nv = (args.N - ti.n0 + 15) & ~15;   // the columns the pair multiplies
          nv = nv < bn ? nv : bn;
          const int bcol = T::dual ? ti.n0 : ti.n0 + rank * (nv >> 1);
          // rank 1's half of a group's last 256-row tile may lie wholly past the
          // group: its A rows then come from past the tensor's end (zero-filled,
          // no memory traffic) instead of from the next group
          const int arow = (!T::kgrouped && ti.m0 >= ti.row_end) ? (int)args.R_cap : (int)ti.m0;
          const void* mBd = (T::dual && rank) ? (const void*)&mapB1 : (const void*)&mapB0;
          for (int ks = 0; ks < ti.nk; ++ks) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = full_bar(stage);
            const uint32_t fbl = rank0 ? fb : mapa_shared(fb, 0);
            const uint32_t sA = s_base + stage * kStageBytes;
            const uint32_t sB = sA + kABytes;
            if (rank0) mbar_arrive_expect_tx(fb, 2u * tx_bytes);
            if constexpr (T::kgrouped) {
              const int row0 = (int)(ti.kbeg + (int64_t)ks * BK);
#pragma unroll
              for (int i = 0; i < BM / 64; ++i)
                tma_load_2d_pair(sA + i * (BK * 128), &mapA0, fbl, (int)ti.m0 + 64 * i, row0);
#pragma unroll
              for (int j = 0; j < 2; ++j)
                tma_load_2d_pair(sB + j * (BK * 128), mBd, fbl, bcol + 64 * j, row0);
            } else {
              const int seg = (T::two_seg && ks >= args.nk_seg) ? 1 : 0;
              const int kk = (ks - seg * args.nk_seg) * BK;
              const void* mA = seg ? (const void*)&mapA1 : (const void*)&mapA0;
              const void* mB = seg ? (const void*)&mapB1 : (const void*)&mapB0;
              tma_load_2d_pair(sA, mA, fbl, kk, arow);
              if constexpr (T::b_mn) {
#pragma unroll
                for (int j = 0; j < 2; ++j)
                  tma_load_3d_pair(sB + j * (BK * 128), mBd, fbl, bcol + 64 * j, kk, ti.e, pol_w);
              } else {
                tma_load_3d_pair(sB, mB, fbl, kk, bcol, ti.e, pol_w);
              }
            }
            ++fills;
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          }
        }
      } else {
        for (int tile = GEMM_CID; tile < total && ok; tile += GEMM_NCL) {
          TileInfo ti;
          decode_tile<K, PAIR>(tile, args, tstart, nN, 0, ti);
          for (int ks = 0; ks < ti.nk; ++ks) {
            if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, s_abort, args.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = full_bar(stage);
            const uint32_t sA = s_base + stage * kStageBytes;
            const uint32_t sB0 = sA + kABytes;
            const uint32_t sB1 = sB0 + kBBytes;
            mbar_arrive_expect_tx(fb, tx_bytes);
            if constexpr (T::kgrouped) {
              const int row0 = (int)(ti.kbeg + (int64_t)ks * BK);
#pragma unroll
              for (int i = 0; i < BM / 64; ++i)
                tma_load_2d(sA + i * (BK * 128), &mapA0, fb, (int)ti.m0 + 64 * i, row0);
#pragma unroll
              for (int j = 0; j < T::BN / 64; ++j) {
                tma_load_2d(sB0 + j * (BK * 128), &mapB0, fb, ti.n0 + 64 * j, row0);
                if constexpr (T::dual)
                  tma_load_2d(sB1 + j * (BK * 128), &mapB1, fb, ti.n0 + 64 * j, row0);
              }
            } else if constexpr (T::dense) {
              // K segment s of B starts at row s * seg_koff; A is the same in every segment
              const int kg = (int)ti.kbeg + ks;
              const int seg = kg / args.nk_seg;
              const int kk = (kg - seg * args.nk_seg) * BK;
              if constexpr (T::a_mn) {
#pragma unroll
                for (int i = 0; i < BM / 64; ++i)
                  tma_load_2d(sA + i * (BK * 128), &mapA0, fb, (int)ti.m0 + 64 * i, kk);
              } else {
                tma_load_2d(sA, &mapA0, fb, kk, (int)ti.m0);
              }
#pragma unroll
              for (int j = 0; j < T::BN / 64; ++j)
                if (j < nbox)
                  tma_load_2d_hint(sB0 + j * (BK * 128), &mapB0, fb, ti.n0 + 64 * j,
                                 seg * args.seg_koff + kk, pol_w);
            } else {
              const int seg = (T::two_seg && ks >= args.nk_seg) ? 1 : 0;
              const int kk = (ks - seg * args.nk_seg) * BK;
              const void* mA = seg ? (const void*)&mapA1 : (const void*)&mapA0;
              const void* mB = seg ? (const void*)&mapB1 : (const void*)&mapB0;
              tma_load_2d(sA, mA, fb, kk, (int)ti.m0);
              if constexpr (T::b_mn) {
#pragma unroll
                for (int j = 0; j < T::BN / 64; ++j) {
                  tma_load_3d_hint(sB0 + j * (BK * 128), &mapB0, fb, ti.n0 + 64 * j, kk, ti.e,
                                   pol_w);
                  if constexpr (T::dual)
                    tma_load_3d_hint(sB1 + j * (BK * 128), &mapB1, fb, ti.n0 + 64 * j, kk, ti.e,
                                     pol_w);
                }
              } else {
                tma_load_3d_hint(sB0, mB, fb, kk, ti.n0, ti.e, pol_w);
              }
            }
            ++fills;
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          }
        }
      }
      if (*s_abort) {
        // let the copies already issued land before the CTA's shared memory goes away
        if (!PAIR || rank0) {
          const int outstanding = fills < kStages ? fills : kStages;
          int st = stage;
          uint32_t ph = phase;
          for (int i = 0; i < outstanding; ++i) {
            if (--st < 0) { st = kStages - 1; ph ^= 1u; }
            drain_wait(full_bar(st), ph, args.status);
          }
        } else {
          // rank 1's copies report to rank 0's barriers: give them a fixed,
          // generous time to land instead
          const uint64_t t0 = global_ns();
          while (global_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank0) {
      // ---------------------------------------------------------- MMA --
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = GEMM_CID; tile < total && ok; tile += GEMM_NCL) {
        TileInfo ti;
        decode_tile<K, PAIR>(tile, args, tstart, nN, 0, ti);
        if (ti.nk == 0) continue;
        if (!mbar_wait_bounded(tempty_bar(acc), acc_phase ^ 1u, s_abort, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)acc * 256u;
        // a tile at the right edge multiplies only the columns that exist
        // (rounded up to the MMA's 16-column step; B rows past N are zero-filled)
        uint32_t idesc = kIdesc;
        if constexpr (!T::dual) {
          int nv = (args.N - ti.n0 + 15) & ~15;
          nv = nv < bn ? nv : bn;
          if (nv != T::BN) idesc = idesc_bf16(TM, nv, T::a_mn ? 1 : 0, T::b_mn ? 1 : 0);
        }
        for (int ks = 0; ks < ti.nk; ++ks) {
          if (!mbar_wait_bounded(full_bar(stage), phase, s_abort, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = s_base + stage * kStageBytes;
          const uint32_t sB0 = sA + kABytes;
          int nsub = BK / 16;
          if constexpr (T::kgrouped) {
            const int64_t left = ti.row_end - (int64_t)ks * BK;
            if (left < BK) nsub = (int)(left / 16);
          }
          for (int kk = 0; kk < nsub; ++kk) {
            const uint64_t ad = T::a_mn ? sdesc_sw128(sA + kk * 2048, BK * 128, 1024)
                                        : sdesc_sw128(sA + kk * 32, 16, 1024);
            const uint64_t bd0 = T::b_mn ? sdesc_sw128(sB0 + kk * 2048, BK * 128, 1024)
                                         : sdesc_sw128(sB0 + kk * 32, 16, 1024);
            const uint32_t accum = (ks > 0 || kk > 0) ? 1u : 0u;
            if constexpr (PAIR)
              umma_bf16_pair(d_tmem, ad, bd0, idesc, accum);
            else
              umma_bf16(d_tmem, ad, bd0, idesc, accum);
          }
          if constexpr (PAIR)
            umma_commit_pair(empty_bar(stage), 3);   // the slot is free in both CTAs
          else
            umma_commit(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(tfull_bar(acc), 3);
        else
          umma_commit(tfull_bar(acc));
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      // every MMA issued by this thread has finished before tensor memory is freed
      if constexpr (PAIR)
        umma_commit_pair(drain_bar, 3);
      else
        umma_commit(drain_bar);
      drain_wait(drain_bar, 0, args.status);
    } else if (PAIR && lane == 0) {
      // rank 1: rank 0's MMAs write this CTA's tensor memory; they finish first
      drain_wait(drain_bar, 0, args.status);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue --
    const uint64_t pol_out = l2_evict_first();   // outputs stream through L2
    const int wq = (warp - 4) & 3;             // TMEM lane quarter of this warp
    const int rloc = wq * 32 + lane;           // accumulator row of this thread
    // the two epilogue warpgroups split each accumulator's columns in halves
    constexpr int kHalf = T::BN / 2;
    const int c_lo = ((warp - 4) >> 2) * kHalf;
    const int c_hi = c_lo + kHalf < bn ? c_lo + kHalf : bn;
    const int group = (warp - 4) >> 2;
    constexpr bool WS = T::warp_stage;
    // this thread's staging unit: its warp (32 rows) or its warpgroup (128)
    uint8_t* stg = stage_out + group * kStagePerGroup + (WS ? wq * (kStagePerGroup / 4) : 0);
    const int srow = WS ? lane : rloc;                  // row within the unit
    const bool leader = WS ? lane == 0 : (wq == 0 && lane == 0);
    int slot = 0;   // next staging slot of the unit's ring (the same in all its threads)
    const CUtensorMap* maps[3] = {&mapO0, &mapO1, &mapO2};
    uint8_t* outs[3] = {static_cast<uint8_t*>(args.out0), static_cast<uint8_t*>(args.out1),
                        static_cast<uint8_t*>(args.out2)};
    int acc = 0;
    uint32_t acc_phase = 0;
    // DownDgrad: the saved G and U of this warp's rows come by TMA into its
    // slots, 8 columns per chunk, in the order the epilogue reads them. A
    // cursor walks this warp's chunks over the CTA's tiles and keeps the
    // slots filled (up to gu_slots chunks ahead of the one being read, across
    // tile boundaries); lane 0 issues, every lane keeps the same counters.
    constexpr int NS = G::gu_slots > 0 ? G::gu_slots : 1;
    const int ew = warp - 4;
    const uint8_t* gu_mem = smem + kStages * kStageBytes + ew * NS * G::gu_slot_bytes;
    int gu_issue = 0, gu_use = 0, gu_done = 0;   // chunks issued, read, seen complete
    int cur_tile = GEMM_CID, cur_j = 0, cur_n = 0, cur_row0 = 0, cur_col0 = 0;
    // (no evict_first hint on these loads: each brings a whole 128-byte line
    // whose other three chunks the warp asks for next; with the hint the line
    // was often gone by then — Qwen3-30B-A3B shape 0.283 -> 0.260 ms)
    // the cursor's tile: this warp's rows and chunk count (none when the
    // warp's rows all lie past the group: nothing of them is stored)
    auto gu_tile = [&]() {
      TileInfo tt;
      decode_tile<K, PAIR>(cur_tile, args, tstart, nN, rank, tt);
      const int ce = min(c_hi, args.N - tt.n0);
      cur_row0 = (int)tt.m0 + wq * 32;
      cur_n = (ce > c_lo && cur_row0 < tt.row_end) ? (ce - c_lo + 7) >> 3 : 0;
      cur_col0 = tt.n0 + c_lo;
    };
    auto gu_fill = [&]() {   // issue chunks while a slot is free (warp-uniform)
      if (__shfl_sync(0xFFFFFFFFu, *s_abort, 0)) return;
      while (gu_issue < gu_done + NS && gu_issue < gu_use + NS && cur_tile < total) {
        if (cur_j < cur_n) {
          if (lane == 0) {
            const int sl = gu_issue % NS;
            const uint32_t bar = gu_bar(ew, sl);
            const uint32_t dst = smem_u32(gu_mem + sl * G::gu_slot_bytes);
            const int x = cur_col0 + 8 * cur_j;
            mbar_arrive_expect_tx(bar, (uint32_t)G::gu_slot_bytes);
            tma_load_2d(dst, &mapA1, bar, x, cur_row0);
            tma_load_2d(dst + G::gu_slot_bytes / 2, &mapB1, bar, x, cur_row0);
          }
          ++gu_issue;
          ++cur_j;
        } else {
          cur_tile += GEMM_NCL;
          cur_j = 0;
          if (cur_tile < total) gu_tile();
        }
      }
    };
    // 8 columns of G and U of this thread's row from the next chunk's slot
    // (the slot's two boxes carry the 32-byte swizzle: halves of rows 4-7 swapped)
    auto gu_get = [&](float* gf, float* uf) {
      const int sl = gu_use % NS;
      const bool ok = mbar_wait_bounded(gu_bar(ew, sl), (uint32_t)((gu_use / NS) & 1), s_abort,
                                        args.status);
      const uint8_t* p = gu_mem + sl * G::gu_slot_bytes + lane * 32;
      const int sw = ((lane >> 2) & 1) * 16;
      const float4 g0 = *reinterpret_cast<const float4*>(p + sw);
      const float4 g1 = *reinterpret_cast<const float4*>(p + (16 - sw));
      const float4 u0 = *reinterpret_cast<const float4*>(p + G::gu_slot_bytes / 2 + sw);
      const float4 u1 = *reinterpret_cast<const float4*>(p + G::gu_slot_bytes / 2 + (16 - sw));
      gf[0] = g0.x; gf[1] = g0.y; gf[2] = g0.z; gf[3] = g0.w;
      gf[4] = g1.x; gf[5] = g1.y; gf[6] = g1.z; gf[7] = g1.w;
      uf[0] = u0.x; uf[1] = u0.y; uf[2] = u0.z; uf[3] = u0.w;
      uf[4] = u1.x; uf[5] = u1.y; uf[6] = u1.z; uf[7] = u1.w;
      if (ok && gu_done == gu_use) ++gu_done;
      ++gu_use;
    };
    if constexpr (G::gu_slots > 0) {
      if (cur_tile < total) gu_tile();
      gu_fill();
    }
    for (int tile = GEMM_CID; tile < total; tile += GEMM_NCL) {
      TileInfo ti;
      decode_tile<K, PAIR>(tile, args, tstart, nN, rank, ti);
      const int64_t row = ti.m0 + rloc;
      if constexpr (T::kgrouped) {
        const bool row_ok = row < args.M;
        const int64_t estride = (int64_t)args.M * args.N;
        if (ti.nk == 0) {
          if (row_ok) {
            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
            for (int c = c_lo; c < c_hi; c += 8) {
              const int col = ti.n0 + c;
              if (col >= args.N) break;
              const int64_t o = ti.e * estride + row * args.N + col;
              reinterpret_cast<uint4*>(static_cast<moe_bf16*>(args.out0) + o)[0] = z;
              if constexpr (T::dual)
                reinterpret_cast<uint4*>(static_cast<moe_bf16*>(args.out1) + o)[0] = z;
            }
          }
          continue;
        }
      }
      const bool row_ok = T::kgrouped ? false : (row < ti.row_end);
      const int c_end = min(c_hi, args.N - ti.n0);   // columns of this half that exist
      const int col_lim = ti.n0 + c_end;
      // DownDgrad in one CTA: the saved G, U of the next 16 columns are loaded
      // while the current ones are computed; the first loads and the row's
      // score go out before the accumulator is ready
      const int64_t gu_base = row * args.N;
      float4 gc[4], uc[4];
      auto load_gu = [&](int c, float4* g, float4* u) {   // 16 fp32 columns of G and U
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int col = ti.n0 + c + 4 * v;
          if (row_ok && col < col_lim) {
            g[v] = *reinterpret_cast<const float4*>(args.in0 + gu_base + col);
            u[v] = *reinterpret_cast<const float4*>(args.in1 + gu_base + col);
          } else {
            g[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            u[v] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      };
      float rscale = 1.0f;
      if constexpr (K == Kind::DownDgrad) {
        rscale = 0.0f;
        if (row_ok) {
          const int32_t p = args.src_pair[row];
          if (p >= 0) rscale = p < args.p_routed ? args.pair_w[p] : 1.0f;
        }
        if constexpr (G::gu_slots == 0)
          if (c_lo < c_end) load_gu(c_lo, gc, uc);
      } else if constexpr (T::down_fwd) {
        if (args.row_w && row_ok) rscale = args.row_w[row];
      }
      const bool got = mbar_wait_bounded(tfull_bar(acc), acc_phase, s_abort, args.status);
      if (!(T::fused ? epi_all(got) : group_all(group, got))) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)acc * 256u;

      // the staging unit's rows inside its group (dW tiles: TMA clips at M) ->
      // staged TMA stores; else masked row stores
      const int64_t r0 = ti.m0 + (WS ? wq * 32 : 0);
      const int urows = WS ? 32 : BM;
      const bool tile_tma = T::kgrouped ? r0 < args.M : r0 + urows <= ti.row_end;
      if constexpr (T::gateup_fwd) {
        // G, U fp32 in 8-column slices, A bf16 in 16-column slices (each
        // with the first of every two G / U slices)
        constexpr int es[3] = {4, 4, 2};
#pragma unroll 1
        for (int c = c_lo; c < c_end; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(t_row + c, g);
          tmem_ld32(t_row + T::BN + c, u);
          tmem_ld_wait();
          uint32_t pa[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            pa[i] = pack_bf16(swiglu(g0, u0, args.act), swiglu(g1, u1, args.act));
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v[3][2];
            v[0][0] = make_uint4(g[8 * q + 0], g[8 * q + 1], g[8 * q + 2], g[8 * q + 3]);
            v[0][1] = make_uint4(g[8 * q + 4], g[8 * q + 5], g[8 * q + 6], g[8 * q + 7]);
            v[1][0] = make_uint4(u[8 * q + 0], u[8 * q + 1], u[8 * q + 2], u[8 * q + 3]);
            v[1][1] = make_uint4(u[8 * q + 4], u[8 * q + 5], u[8 * q + 6], u[8 * q + 7]);
            const int col = ti.n0 + c + 8 * q;
            if ((q & 1) == 0) {
              const int h = q >> 1;
              v[2][0] = make_uint4(pa[8 * h + 0], pa[8 * h + 1], pa[8 * h + 2], pa[8 * h + 3]);
              v[2][1] = make_uint4(pa[8 * h + 4], pa[8 * h + 5], pa[8 * h + 6], pa[8 * h + 7]);
              put_slice<3, false, WS>(v, stg, slot, maps, outs, es, tile_tma, row_ok, row, srow, col,
                                  args.N, col_lim, (int)r0, 0, group, leader, pol_out);
            } else {
              uint4 w2[2][2] = {{v[0][0], v[0][1]}, {v[1][0], v[1][1]}};
              put_slice<2, false, WS>(w2, stg, slot, maps, outs, es, tile_tma, row_ok, row, srow,
                                  col, args.N, col_lim, (int)r0, 0, group, leader, pol_out);
            }
          }
        }
      } else if constexpr (T::kgrouped) {
        constexpr int NO = T::dual ? 2 : 1;
#pragma unroll 1
        for (int c = c_lo; c < c_end; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(t_row + c, g);
          if constexpr (T::dual) tmem_ld32(t_row + T::BN + c, u);
          tmem_ld_wait();
          uint32_t pk[NO][16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pk[0][i] = pack_bf16(__uint_as_float(g[2 * i]), __uint_as_float(g[2 * i + 1]));
            if constexpr (T::dual)
              pk[NO - 1][i] = pack_bf16(__uint_as_float(u[2 * i]), __uint_as_float(u[2 * i + 1]));
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint4 v[NO][2];
            slice_of<NO, 16>(pk, h, v);
            constexpr int es[2] = {2, 2};
            put_slice<NO, true, WS>(v, stg, slot, maps, outs, es, tile_tma, false, row, srow,
                                    ti.n0 + c + 16 * h, args.N, col_lim, (int)r0, ti.e, group,
                                    leader, pol_out);
          }
        }
      } else if constexpr (T::dense) {
        // one split: the result (+ bias); several: this split's fp32 partial, summed later
        const bool in_m = row < args.M;
        const bool whole = args.ksplit == 1;
        float* orow = args.outf + ((int64_t)ti.e * args.M + row) * args.N;
#pragma unroll 1
        for (int c = c_lo; c < c_end; c += 32) {
          uint32_t r[32];
          tmem_ld32(t_row + c, r);
          tmem_ld_wait();
          if (!in_m) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = ti.n0 + c + i;
            if (col < col_lim)
              orow[col] = __uint_as_float(r[i]) + (whole && args.bias ? args.bias[col] : 0.f);
          }
        }
      } else if constexpr (T::fused) {
        // gate/up tile: A = act(G, U) from the two 128-column accumulators,
        // bf16 in 16-column slices (each warpgroup 64 columns); down tile:
        // the row's score times the fp32 accumulator in 8-column slices
        // (each warpgroup 128 columns)
        const int fhalf = ti.ph ? 128 : 64;
        const int flo = group * fhalf;
        const int fN = ti.ph ? args.N2 : args.N;
        const int fend = min(flo + fhalf, fN - ti.n0);
        const int flim = ti.n0 + fend;
        if (ti.ph == 0) {
          const CUtensorMap* mA[1] = {&mapO2};
          uint8_t* oA[1] = {static_cast<uint8_t*>(args.out2)};
          constexpr int esA[1] = {2};
#pragma unroll 1
          for (int c = flo; c < fend; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(t_row + c, g);
            tmem_ld32(t_row + 128 + c, u);
            tmem_ld_wait();
            uint32_t pa[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pa[i] = pack_bf16(swiglu(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i]), args.act),
                                swiglu(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1]),
                                       args.act));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint4 v[1][2];
              v[0][0] = make_uint4(pa[8 * h + 0], pa[8 * h + 1], pa[8 * h + 2], pa[8 * h + 3]);
              v[0][1] = make_uint4(pa[8 * h + 4], pa[8 * h + 5], pa[8 * h + 6], pa[8 * h + 7]);
              put_slice<1, false, false>(v, stg, slot, mA, oA, esA, tile_tma, row_ok, row, srow,
                                         ti.n0 + c + 16 * h, fN, flim, (int)r0, 0, group, leader,
                                         pol_out);
            }
          }
        } else {
          float w = 0.0f;
          if (row_ok) {
            const int32_t p = args.src_pair[row];
            if (p >= 0) w = p < args.p_routed ? args.pair_w[p] : 1.0f;
          }
          const CUtensorMap* mY[1] = {&mapO3};
          uint8_t* oY[1] = {static_cast<uint8_t*>(args.out3)};
          constexpr int esY[1] = {4};
#pragma unroll 1
          for (int c = flo; c < fend; c += 32) {
            uint32_t r[32];
            tmem_ld32(t_row + c, r);
            tmem_ld_wait();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v[1][2];
              v[0][0] = make_uint4(__float_as_uint(__uint_as_float(r[8 * q + 0]) * w),
                                   __float_as_uint(__uint_as_float(r[8 * q + 1]) * w),
                                   __float_as_uint(__uint_as_float(r[8 * q + 2]) * w),
                                   __float_as_uint(__uint_as_float(r[8 * q + 3]) * w));
              v[0][1] = make_uint4(__float_as_uint(__uint_as_float(r[8 * q + 4]) * w),
                                   __float_as_uint(__uint_as_float(r[8 * q + 5]) * w),
                                   __float_as_uint(__uint_as_float(r[8 * q + 6]) * w),
                                   __float_as_uint(__uint_as_float(r[8 * q + 7]) * w));
              put_slice<1, false, false>(v, stg, slot, mY, oY, esY, tile_tma, row_ok, row, srow,
                                         ti.n0 + c + 8 * q, fN, flim, (int)r0, 0, group, leader,
                                         pol_out);
            }
          }
        }
      } else if constexpr (K == Kind::DownDgrad) {
        // dA = w * acc; dG = dA * U * h'(G), dU = dA * h(G), 16 columns at a
        // time: from two chunks of the slots (none past the half's last
        // column or for rows all past the group: zeros there, nothing is
        // stored), or in one CTA from registers, the next 16 columns' G and U
        // loaded while these are computed
        constexpr int es[2] = {2, 2};
        const int nch = (c_end > c_lo && r0 < ti.row_end) ? (c_end - c_lo + 7) >> 3 : 0;
        float dtw = 0.0f;   // this row's <dAu, h(G) U> over this warpgroup's columns
        float4 gn[4], un[4];
#pragma unroll 1
        for (int c = c_lo; c < c_end; c += 32) {
          uint32_t r[32];
          tmem_ld32(t_row + c, r);
          const int j0 = (c - c_lo) >> 3;
          if constexpr (G::gu_slots == 0) {
            if (c + 16 < c_end) load_gu(c + 16, gn, un);
            tmem_ld_wait();
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float gf[16], uf[16];
            if constexpr (G::gu_slots > 0) {
#pragma unroll
              for (int q = 0; q < 2; ++q) {
                if (j0 + 2 * h + q < nch) {
                  gu_get(gf + 8 * q, uf + 8 * q);
                } else {
#pragma unroll
                  for (int i = 0; i < 8; ++i) { gf[8 * q + i] = 0.0f; uf[8 * q + i] = 0.0f; }
                }
              }
              // every lane has read the two slots: they take the next chunks
              __syncwarp();
              if (lane == 0) fence_async_smem();
              gu_fill();
              if (h == 0) tmem_ld_wait();
            } else {
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                gf[4 * v + 0] = gc[v].x; gf[4 * v + 1] = gc[v].y;
                gf[4 * v + 2] = gc[v].z; gf[4 * v + 3] = gc[v].w;
                uf[4 * v + 0] = uc[v].x; uf[4 * v + 1] = uc[v].y;
                uf[4 * v + 2] = uc[v].z; uf[4 * v + 3] = uc[v].w;
              }
            }
            uint32_t pk[2][8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float dg[2], du[2];
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int q = 2 * i + j;
                const float au = __uint_as_float(r[16 * h + q]);
                const float f = au * rscale;
                // h = gc sigmoid(alpha gc), h' = s + alpha gc s (1 - s); the
                // clamps pass no gradient past their limits
                const float gc = fminf(gf[q], args.act.limit);
                const float uc = fminf(fmaxf(uf[q], -args.act.limit), args.act.limit) + args.act.c;
                const float sg = __fdividef(1.0f, 1.0f + __expf(-args.act.alpha * gc));
                const float hg = gc * sg;
                const float h1 = fmaf(args.act.alpha * gc, sg * (1.0f - sg), sg);
                // only the tile's real columns: past them the accumulator was
                // never written (the MMA's N stops at the tile width) and the
                // G, U registers may hold the previous half
                if (ti.n0 + c + 16 * h + q < col_lim) dtw = fmaf(au, hg * uc, dtw);
                dg[j] = gf[q] <= args.act.limit ? f * uc * h1 : 0.0f;
                du[j] = fabsf(uf[q]) <= args.act.limit ? f * hg : 0.0f;
              }
              pk[0][i] = pack_bf16(dg[0], dg[1]);
              pk[1][i] = pack_bf16(du[0], du[1]);
            }
            if constexpr (G::gu_slots == 0) {
#pragma unroll
              for (int v = 0; v < 4; ++v) { gc[v] = gn[v]; uc[v] = un[v]; }
              if (h == 0 && c + 32 < c_end) load_gu(c + 32, gn, un);
            }
            uint4 vv[2][2];
            slice_of<2, 8>(pk, 0, vv);
            put_slice<2, false, WS>(vv, stg, slot, maps, outs, es, tile_tma, row_ok, row, srow,
                                    ti.n0 + c + 16 * h, args.N, col_lim, (int)r0, 0, group,
                                    leader, pol_out);
          }
        }
        if (row_ok)
          args.dtw_part[row * args.dtw_slots + 2 * (ti.n0 / bn) + group] = dtw;
      } else {
        // single accumulator, fp32 output (DownFwd optionally row-scaled): 8-column slices
#pragma unroll 1
        for (int c = c_lo; c < c_end; c += 32) {
          uint32_t r[32];
          tmem_ld32(t_row + c, r);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v[1][2];
            v[0][0] = make_uint4(__float_as_uint(__uint_as_float(r[8 * q + 0]) * rscale),
                                 __float_as_uint(__uint_as_float(r[8 * q + 1]) * rscale),
                                 __float_as_uint(__uint_as_float(r[8 * q + 2]) * rscale),
                                 __float_as_uint(__uint_as_float(r[8 * q + 3]) * rscale));
            v[0][1] = make_uint4(__float_as_uint(__uint_as_float(r[8 * q + 4]) * rscale),
                                 __float_as_uint(__uint_as_float(r[8 * q + 5]) * rscale),
                                 __float_as_uint(__uint_as_float(r[8 * q + 6]) * rscale),
                                 __float_as_uint(__uint_as_float(r[8 * q + 7]) * rscale));
            constexpr int es[1] = {4};
            put_slice<1, false, WS>(v, stg, slot, maps, outs, es, tile_tma, row_ok, row, srow,
                                    ti.n0 + c + 8 * q, args.N, col_lim, (int)r0, 0, group,
                                    leader, pol_out);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !rank0)
          mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));   // rank 0's MMA waits on it
        else
          mbar_arrive(tempty_bar(acc));
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      if constexpr (T::fused) {
        // a gate/up tile publishes its rows of A: its TMA stores complete
        // (and its masked row stores are fenced) before the m-tile's count
        // goes up with release; down tiles of these rows wait for the count
        if (ti.ph == 0) {
          if (leader) {
            bulk_wait_all();
            fence_async_global();
          }
          __threadfence();
          epi_all(true);
          if (warp == 4 && lane == 0) red_release_gpu_add(args.ready + ti.mt, 1);
        }
      }
    }
    if (leader) bulk_wait_all();   // the unit's staged stores finish before the CTA exits
    if constexpr (K == Kind::DownDgrad) {
      // after an abort: the G/U loads still in flight land before shared memory goes away
      if (lane == 0)
        for (int q = gu_done; q < gu_issue; ++q)
          drain_wait(gu_bar(ew, q % NS), (uint32_t)((q / NS) & 1), args.status);
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();   // no remote arrival or copy is still to come
  tc_fence_after();
  if (warp == 2) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
#undef GEMM_CID
#undef GEMM_NCL
}

// ------------------------------------------------------------------ host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [outer, inner] matrix, box [box_outer, 64], 128-byte swizzle
static bool map2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer,
                  uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [E, d1, d0] (d0 innermost), box [1, box1, 64]
static bool map3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t E,
                  uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, E};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Maps for the epilogues' TMA stores: boxes of `rows` rows x 32 bytes (16 bf16
// or 8 fp32 columns: one staging slot, 128 rows per warpgroup or 32 per warp)
// with the 32-byte swizzle the slots are written in.
// 2-D over a row buffer [R, N]; esz = 2 (bf16) or 4 (fp32).
static bool map2d_out(CUtensorMap* m, const void* ptr, uint64_t N, uint64_t R, int esz = 2,
                      uint32_t rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {N, R};
  cuuint64_t strides[1] = {N * (uint64_t)esz};
  cuuint32_t box[2] = {(cuuint32_t)(32 / esz), rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, esz == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The down dgrad's loads of the saved G or U [R, N] (fp32): boxes of 8
// columns x 32 rows with the 32-byte swizzle, a whole 128-byte line brought
// into L2 per miss (the row's next chunks follow).
static bool map2d_gu(CUtensorMap* m, const float* ptr, uint64_t N, uint64_t R) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {N, R};
  cuuint64_t strides[1] = {N * 4};
  cuuint32_t box[2] = {8, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map over [E, M, N] (N innermost), boxes of one warp's 32 rows
static bool map3d_out(CUtensorMap* m, const void* ptr, uint64_t N, uint64_t M, uint64_t E,
                      uint32_t rows = 32) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {N, M, E};
  cuuint64_t strides[2] = {N * 2, N * M * 2};
  cuuint32_t box[3] = {16, rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// tiles_upper: an upper bound on the kernel's tiles (pair tiles for PAIR). A
// persistent grid: one CTA per SM, or for PAIR one two-CTA cluster per pair of
// SMs that can hold one at a time.
template <Kind K, bool PAIR>
static cudaError_t launch_kind(const CUtensorMap& a0, const CUtensorMap& a1,
                               const CUtensorMap& b0, const CUtensorMap& b1, const GemmArgs& args,
                               int64_t tiles_upper, cudaStream_t s,
                               const CUtensorMap* o0 = nullptr, const CUtensorMap* o1 = nullptr,
                               const CUtensorMap* o2 = nullptr, bool pdl = false,
                               const CUtensorMap* b2 = nullptr, const CUtensorMap* o3 = nullptr) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int units = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_kernel<K, PAIR>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    units = num_sms();
    if (PAIR && attr_err == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmemBytes;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<K, PAIR>, &cfg) != cudaSuccess ||
          n < 1) {
        cudaGetLastError();
        n = num_sms() / 2;
      }
      units = n;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  int64_t grid = units;
  if (tiles_upper < grid) grid = tiles_upper;
  if (grid < 1) grid = 1;
  // the router's timers bracket these GEMMs with their other kernels (route.cu)
  if constexpr (!Tr<K>::dense) timer_before(Tr<K>::kernel_id, s);
  const CUtensorMap& m0 = o0 ? *o0 : a0;
  const CUtensorMap& m1 = o1 ? *o1 : m0;
  const CUtensorMap& m2 = o2 ? *o2 : m0;
  const CUtensorMap& mb2 = b2 ? *b2 : b0;
  const CUtensorMap& m3 = o3 ? *o3 : m0;
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // as launch_pdl
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(2 * grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 2 : 1;
    cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<K, PAIR>, a0, a1, b0, b1, m0, m1, m2, mb2, m3,
                       args);
  } else {
    launch_pdl(pdl, grouped_gemm_kernel<K, PAIR>, dim3((unsigned)grid), dim3(kThreads), kSmemBytes,
               s, a0, a1, b0, b1, m0, m1, m2, mb2, m3, args);
  }
  note_launches(1);
  if constexpr (!Tr<K>::dense) timer_after(Tr<K>::kernel_id, s);
  return cudaGetLastError();
}

// CTA pairs (M = 256 MMAs over two SMs: half the B traffic per SM, a deeper
// ring) for the M-grouped kinds when the experts average at least 1024 rows,
// where 256-row tiles waste little; the gate/up forward and dgrad, which move
// two weight matrices per tile, and the down dgrad, whose pair form also
// loads G and U ahead by TMA, from 512 rows. Not by default for the K-grouped weight gradients: their rows (d or
// f, e.g. 2880 = 11.25 x 256) leave a mostly empty last 256-row tile.
// MOE_GEMM_PAIRS=0 or 1 in the environment turns pairs off or on for every
// grouped kind (a tuning and testing knob; the results are the same).
static int pairs_env() {
  static const int v = [] {
    const char* e = getenv("MOE_GEMM_PAIRS");
    return (e && (e[0] == '0' || e[0] == '1')) ? e[0] - '0' : -1;
  }();
  return v;
}
static bool pairs_mgrouped(const GroupedDims& g, int min_rows = 1024) {
  const int e = pairs_env();
  return e >= 0 ? e == 1 : g.P >= (int64_t)min_rows * g.E;
}
static bool pairs_kgrouped() { return pairs_env() == 1; }

// Tile width of a single-accumulator GEMM over N columns: the fewest 256-wide
// tiles, made equal in width and rounded up to `step` columns: 16 (the MMA's
// step) when B is K-major, 64 when B is N-major, whose TMA boxes are 64
// columns wide and stay on 128-byte lines only at multiples of 64.
static int pick_bn(int N, int step) {
  const int n = (N + 255) / 256;
  const int w = (N + n - 1) / n;
  return (w + step - 1) / step * step;
}

static GemmArgs base_args(const GroupedDims& g, int* status) {
  GemmArgs a{};
  a.offsets = g.offsets;
  a.E = g.E;
  a.R_cap = g.R_cap;
  a.src_pair = g.src_pair;
  a.status = status;
  return a;
}

// K chunks for a GEMM of `tiles` output tiles over `steps` k-steps: none while
// the tiles alone fill half the SMs; else as many as fit the SMs in one round,
// at least min_steps k-steps per chunk, at most 16 chunks, and normalised so
// that ceil(steps / chunk length) chunks of ceil(steps / chunks) steps are all
// non-empty.
static int ksplit_for(int64_t tiles, int64_t steps, int min_steps) {
  if (steps <= 0 || tiles <= 0 || 2 * tiles >= num_sms()) return 1;
  int64_t sp = (int64_t)num_sms() / tiles;   // one round of CTAs
  sp = sp > 16 ? 16 : sp;
  sp = sp > steps / min_steps ? steps / min_steps : sp;
  if (sp < 1) return 1;
  const int64_t len = (steps + sp - 1) / sp;
  return (int)((steps + len - 1) / len);
}

// The number of K chunks the router GEMM splits into (at least 4 k-steps each).
int router_ksplit(int64_t T, int d, int E) {
  const int bn = pick_bn(E, 64);
  return ksplit_for(((T + BM - 1) / BM) * ((E + bn - 1) / bn), 3 * ((d + BK - 1) / BK), 4);
}

// logits[T, E] = x[T, d] . (W_hi + W_mid + W_lo) + b, the three bf16 parts
// stacked along K in w_split [3d, E8] (E8 = E rounded up to 8). With ksplit > 1
// the K range is cut into chunks whose fp32 partials go to out[ksplit][T][E].
cudaError_t launch_router_gemm(const moe_bf16* x, const moe_bf16* w_split, const float* bias,
                               int64_t T, int d, int E, int E8, int ksplit, float* out,
                               int* status, cudaStream_t s) {
  CUtensorMap a0, b0;
  if (!map2d(&a0, x, d, T, BM) || !map2d(&b0, w_split, E8, 3 * (uint64_t)d, BK))
    return cudaErrorInvalidValue;
  GemmArgs a{};
  a.E = 1;
  a.M = (int)T;
  a.N = E;
  a.nk_seg = (d + BK - 1) / BK;
  a.nseg = 3;
  a.seg_koff = d;
  const int steps = a.nk_seg * a.nseg;
  a.ksteps_split = (steps + ksplit - 1) / ksplit;
  a.ksplit = (steps + a.ksteps_split - 1) / a.ksteps_split;   // no empty chunk
  if (a.ksplit != ksplit) return cudaErrorInvalidValue;
  a.outf = out;
  a.bias = bias;
  a.status = status;
  a.bn = pick_bn(E, 64);
  const int64_t tiles = ((T + BM - 1) / BM) * ((E + a.bn - 1) / a.bn) * a.ksplit;
  return launch_kind<Kind::RouterLogits, false>(a0, a0, b0, b0, a, tiles, s, nullptr, nullptr,
                                                  nullptr, pdl_for_tokens(T));
}

// The number of K chunks of the router-weight gradient GEMM (at least 8 k-steps each).
int router_wgrad_ksplit(int64_t T, int d, int N3) {
  const int bn = pick_bn(N3, 64);
  return ksplit_for((int64_t)((d + BM - 1) / BM) * ((N3 + bn - 1) / bn), (T + BK - 1) / BK, 8);
}

// part[s][d][N3] = sum over the tokens of chunk s of x[t, :]^T dl3[t, :]: the
// gradient of the router weight with dl's three bf16 parts side by side in N
// (dl3 [T, N3] bf16, N3 = 3 * E8); the chunks and parts are summed later.
cudaError_t launch_router_wgrad_gemm(const moe_bf16* x, const moe_bf16* dl3, int64_t T, int d,
                                     int N3, int ksplit, float* part, int* status,
                                     cudaStream_t s) {
  if (T == 0) return cudaMemsetAsync(part, 0, (size_t)ksplit * d * N3 * 4, s);
  CUtensorMap a0, b0;
  if (!map2d(&a0, x, d, T, BK) || !map2d(&b0, dl3, N3, T, BK)) return cudaErrorInvalidValue;
  GemmArgs a{};
  a.E = 1;
  a.M = d;
  a.N = N3;
  a.nk_seg = (int)((T + BK - 1) / BK);
  a.nseg = 1;
  a.seg_koff = 0;
  a.ksteps_split = (a.nk_seg + ksplit - 1) / ksplit;
  a.ksplit = (a.nk_seg + a.ksteps_split - 1) / a.ksteps_split;   // no empty chunk
  if (a.ksplit != ksplit) return cudaErrorInvalidValue;
  a.outf = part;
  a.status = status;
  a.bn = pick_bn(N3, 64);
  const int64_t tiles = (int64_t)((d + BM - 1) / BM) * ((N3 + a.bn - 1) / a.bn) * a.ksplit;
  return launch_kind<Kind::RouterWgrad, false>(a0, a0, b0, b0, a, tiles, s, nullptr, nullptr,
                                                 nullptr, pdl_for_tokens(T));
}

static int64_t mgrouped_tiles_upper(const GroupedDims& g, int N, int BN, int TM = BM) {
  // each expert's rows may end in a partial tile
  return ((g.R_cap + TM - 1) / TM + g.E) * ((N + BN - 1) / BN);
}

cudaError_t launch_gateup_fwd(const GroupedDims& g, const moe_bf16* xp, const moe_bf16* w_gate,
                              const moe_bf16* w_up, float* G, float* U, moe_bf16* A,
                              const ActParams& act, int* status, cudaStream_t s) {
  CUtensorMap a0, b0, b1, o0, o1, o2;
  if (!map2d(&a0, xp, g.d, g.R_cap, BM) || !map3d(&b0, w_gate, g.f, g.d, g.E, BK) ||
      !map3d(&b1, w_up, g.f, g.d, g.E, BK) || !map2d_out(&o0, G, g.f, g.R_cap, 4) ||
      !map2d_out(&o1, U, g.f, g.R_cap, 4) || !map2d_out(&o2, A, g.f, g.R_cap))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  const bool pdl = pdl_for_pairs(g.P);
  a.N = g.f;
  a.nk_seg = (g.d + BK - 1) / BK;
  a.out0 = G; a.out1 = U; a.out2 = A;
  a.act = Act{act.limit, act.alpha, act.c};
  // Few rows per expert (the weight-bound regime): 128-wide tiles leave too few
  // tiles to fill every SM's last round of weight streaming; halve them.
  const int64_t rows = (g.P + g.E - 1) / g.E;
  const int64_t tiles = (int64_t)g.E * ((rows + BM - 1) / BM) * ((g.f + 127) / 128);
  if (tiles < 8 * (int64_t)num_sms())
    return launch_kind<Kind::GateUpFwdNarrow, false>(
        a0, a0, b0, b1, a, mgrouped_tiles_upper(g, g.f, 64), s, &o0, &o1, &o2, pdl);
  if (pairs_mgrouped(g, 512))
    return launch_kind<Kind::GateUpFwd, true>(
        a0, a0, b0, b1, a, mgrouped_tiles_upper(g, g.f, 128, 2 * BM), s, &o0, &o1, &o2, pdl);
  return launch_kind<Kind::GateUpFwd, false>(a0, a0, b0, b1, a, mgrouped_tiles_upper(g, g.f, 128),
                                             s, &o0, &o1, &o2, pdl);
}

cudaError_t launch_down_fwd(const GroupedDims& g, const moe_bf16* A, const moe_bf16* w_down,
                            const float* row_w, float* yp, int* status, cudaStream_t s) {
  CUtensorMap a0, b0, o0;
  if (!map2d(&a0, A, g.f, g.R_cap, BM) || !map3d(&b0, w_down, g.d, g.f, g.E, BK) ||
      !map2d_out(&o0, yp, g.d, g.R_cap, 4))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  const bool pdl = pdl_for_pairs(g.P);
  a.N = g.d;
  a.nk_seg = (g.f + BK - 1) / BK;
  a.out0 = yp;
  a.row_w = row_w;
  // So few pairs that the 256-wide tiles of the experts that can hold rows
  // (at most min(E, P)) are fewer than the SMs (a few decoded tokens): halve
  // the tiles so more SMs stream the weights (measured: one token 43 -> 41 us
  // a step; from eight tokens on the wide tiles are faster)
  const int64_t groups = g.P < (int64_t)g.E ? g.P : (int64_t)g.E;
  const int64_t rows = groups > 0 ? (g.P + groups - 1) / groups : 0;
  const int64_t tiles = groups * ((rows + BM - 1) / BM) * ((g.d + 255) / 256);
  if (tiles < (int64_t)num_sms())
    return launch_kind<Kind::DownFwdNarrow, false>(a0, a0, b0, b0, a,
                                                   mgrouped_tiles_upper(g, g.d, 128), s, &o0,
                                                   nullptr, nullptr, pdl);
  if (pairs_mgrouped(g))
    return launch_kind<Kind::DownFwd, true>(a0, a0, b0, b0, a,
                                            mgrouped_tiles_upper(g, g.d, 256, 2 * BM), s, &o0,
                                            nullptr, nullptr, pdl);
  return launch_kind<Kind::DownFwd, false>(a0, a0, b0, b0, a, mgrouped_tiles_upper(g, g.d, 256), s,
                                           &o0, nullptr, nullptr, pdl);
}

// The fused expert forward's counts: one per m-tile of the tile table.
size_t fused_fwd_ws_bytes(int64_t R_cap, int E) {
  return (size_t)4 * (size_t)((R_cap + BM - 1) / BM + E + 1);
}

// The fused expert forward (one persistent launch, FusedFwd): gate/up tiles
// store A = act(G, U) (G and U stay in tensor memory); down tiles, once
// every gate/up tile of their rows has published its part of A, store
// Yp = score * (A . W_down[e]) in fp32. One CTA (or pair) per SM (pair of
// SMs) and a grid of at most that many, so every CTA is resident while
// others wait for it.
cudaError_t launch_fused_fwd(const GroupedDims& g, const moe_bf16* xp, const moe_bf16* w_gate,
                             const moe_bf16* w_up, const moe_bf16* w_down, const float* pair_w,
                             moe_bf16* A, float* yp, int* ready, const ActParams& act,
                             int* status, cudaStream_t s) {
  CUtensorMap ax, aa, b0, b1, b2, o2, o3;
  if (!g.src_pair) return cudaErrorInvalidValue;
  if (!map2d(&ax, xp, g.d, g.R_cap, BM) || !map2d(&aa, A, g.f, g.R_cap, BM) ||
      !map3d(&b0, w_gate, g.f, g.d, g.E, BK) || !map3d(&b1, w_up, g.f, g.d, g.E, BK) ||
      !map3d(&b2, w_down, g.d, g.f, g.E, BK) || !map2d_out(&o2, A, g.f, g.R_cap) ||
      !map2d_out(&o3, yp, g.d, g.R_cap, 4))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  a.N = g.f;
  a.nk_seg = (g.d + BK - 1) / BK;
  a.N2 = g.d;
  a.nk2 = (g.f + BK - 1) / BK;
  a.out2 = A;
  a.out3 = yp;
  a.ready = ready;
  a.p_routed = g.P_routed;
  a.pair_w = pair_w;
  a.act = Act{act.limit, act.alpha, act.c};
  cudaError_t e = cudaMemsetAsync(ready, 0, fused_fwd_ws_bytes(g.R_cap, g.E), s);
  if (e != cudaSuccess) return e;
  // CTA pairs from 512 rows per expert on average, as the five-call forward
  if (pairs_mgrouped(g, 512)) {
    const int64_t tiles = mgrouped_tiles_upper(g, g.f, 128, 2 * BM) +
                          mgrouped_tiles_upper(g, g.d, 256, 2 * BM);
    return launch_kind<Kind::FusedFwd, true>(ax, aa, b0, b1, a, tiles, s, nullptr, nullptr, &o2,
                                             false, &b2, &o3);
  }
  const int64_t tiles = mgrouped_tiles_upper(g, g.f, 128) + mgrouped_tiles_upper(g, g.d, 256);
  return launch_kind<Kind::FusedFwd, false>(ax, aa, b0, b1, a, tiles, s, nullptr, nullptr, &o2,
                                            false, &b2, &o3);
}

// Partial slots per row of the down dgrad's top-k weight gradient: one per
// n-tile and epilogue warpgroup.
int down_dgrad_dtw_slots(int f) {
  const int bn = pick_bn(f, 16);
  return 2 * ((f + bn - 1) / bn);
}

cudaError_t launch_down_dgrad(const GroupedDims& g, const moe_bf16* dyg, const float* pair_w,
                              const moe_bf16* w_down, const float* G, const float* U,
                              moe_bf16* dG, moe_bf16* dU, float* dtw_part,
                              const ActParams& act, int* status, cudaStream_t s) {
  CUtensorMap a0, b0, o0, o1, mg, mu;
  const int bn = pick_bn(g.f, 16);
  // pairs from 512 rows per expert on average: half the weight bytes per SM
  // from L2, and G and U loaded by TMA ahead of the epilogue (fewer rows: the
  // last 256-row tile of each group would be mostly empty)
  const bool pair = pairs_mgrouped(g, 512);
  // dA[r, c] = w(r) sum_j dyg[r, j] W_down[e][c, j]: B is W_down[e] read as
  // [N = f rows, K = d] (a pair's CTAs load bn / 2 rows each); G and U come
  // to the epilogue through the second A and B maps
  if (!g.src_pair) return cudaErrorInvalidValue;
  if (!map2d(&a0, dyg, g.d, g.R_cap, BM) ||
      !map3d(&b0, w_down, g.d, g.f, g.E, pair ? bn / 2 : bn) ||
      !map2d_out(&o0, dG, g.f, g.R_cap, 2, 32) || !map2d_out(&o1, dU, g.f, g.R_cap, 2, 32) ||
      !map2d_gu(&mg, G, g.f, g.R_cap) || !map2d_gu(&mu, U, g.f, g.R_cap))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  const bool pdl = pdl_for_pairs(g.P);
  a.N = g.f;
  a.nk_seg = (g.d + BK - 1) / BK;
  a.in0 = G; a.in1 = U;
  a.out0 = dG; a.out1 = dU;
  a.pair_w = pair_w;
  a.p_routed = g.P_routed;
  a.act = Act{act.limit, act.alpha, act.c};
  a.dtw_part = dtw_part;
  a.dtw_slots = down_dgrad_dtw_slots(g.f);
  a.bn = bn;
  if (pair)
    return launch_kind<Kind::DownDgrad, true>(
        a0, mg, b0, mu, a, mgrouped_tiles_upper(g, g.f, bn, 2 * BM), s, &o0, &o1, nullptr, pdl);
  return launch_kind<Kind::DownDgrad, false>(a0, mg, b0, mu, a, mgrouped_tiles_upper(g, g.f, bn),
                                             s, &o0, &o1, nullptr, pdl);
}

cudaError_t launch_gateup_dgrad(const GroupedDims& g, const moe_bf16* dG, const moe_bf16* dU,
                                const moe_bf16* w_gate, const moe_bf16* w_up, float* dxp,
                                int* status, cudaStream_t s) {
  CUtensorMap a0, a1, b0, b1, o0;
  const int bn = pick_bn(g.d, 16);
  const bool pair = pairs_mgrouped(g, 512);
  const int brows = pair ? bn / 2 : bn;   // a pair's CTAs load bn / 2 rows of B each
  // dXp[r, i] = sum_c dG[r, c] W_gate[e][i, c] + dU[r, c] W_up[e][i, c]:
  // B is W_gate[e] / W_up[e] read as [N = d rows, K = f]
  if (!map2d(&a0, dG, g.f, g.R_cap, BM) || !map2d(&a1, dU, g.f, g.R_cap, BM) ||
      !map3d(&b0, w_gate, g.f, g.d, g.E, brows) || !map3d(&b1, w_up, g.f, g.d, g.E, brows) ||
      !map2d_out(&o0, dxp, g.d, g.R_cap, 4))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  const bool pdl = pdl_for_pairs(g.P);
  a.N = g.d;
  a.nk_seg = (g.f + BK - 1) / BK;
  a.out0 = dxp;
  a.bn = bn;
  if (pair)
    return launch_kind<Kind::GateUpDgrad, true>(a0, a1, b0, b1, a,
                                                mgrouped_tiles_upper(g, g.d, bn, 2 * BM), s, &o0,
                                                nullptr, nullptr, pdl);
  return launch_kind<Kind::GateUpDgrad, false>(a0, a1, b0, b1, a, mgrouped_tiles_upper(g, g.d, bn),
                                               s, &o0, nullptr, nullptr, pdl);
}

cudaError_t launch_wgrad_down(const GroupedDims& g, const moe_bf16* A, const moe_bf16* dyp,
                              moe_bf16* dw_down, int* status, cudaStream_t s) {
  CUtensorMap a0, b0, o0;
  // dW_down[e] (f x d) = A_e^T . dYp_e: A read as [K = rows, M = f], B as [K = rows, N = d]
  if (!map2d(&a0, A, g.f, g.R_cap, BK) || !map2d(&b0, dyp, g.d, g.R_cap, BK) ||
      !map3d_out(&o0, dw_down, g.d, g.f, g.E))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  const bool pdl = pdl_for_pairs(g.P);
  a.M = g.f;
  a.N = g.d;
  a.out0 = dw_down;
  const int64_t nN = (g.d + 255) / 256;
  if (pairs_kgrouped())
    return launch_kind<Kind::WgradDown, true>(a0, a0, b0, b0, a,
                                              (int64_t)g.E * ((g.f + 2 * BM - 1) / (2 * BM)) * nN,
                                              s, &o0, nullptr, nullptr, pdl);
  return launch_kind<Kind::WgradDown, false>(a0, a0, b0, b0, a,
                                             (int64_t)g.E * ((g.f + BM - 1) / BM) * nN, s, &o0,
                                             nullptr, nullptr, pdl);
}

cudaError_t launch_wgrad_gateup(const GroupedDims& g, const moe_bf16* xp, const moe_bf16* dG,
                                const moe_bf16* dU, moe_bf16* dw_gate, moe_bf16* dw_up,
                                int* status, cudaStream_t s) {
  CUtensorMap a0, b0, b1, o0, o1;
  // dW_gate[e] (d x f) = Xp_e^T . dG_e: A read as [K = rows, M = d], B as [K = rows, N = f]
  if (!map2d(&a0, xp, g.d, g.R_cap, BK) || !map2d(&b0, dG, g.f, g.R_cap, BK) ||
      !map2d(&b1, dU, g.f, g.R_cap, BK) || !map3d_out(&o0, dw_gate, g.f, g.d, g.E) ||
      !map3d_out(&o1, dw_up, g.f, g.d, g.E))
    return cudaErrorInvalidValue;
  GemmArgs a = base_args(g, status);
  const bool pdl = pdl_for_pairs(g.P);
  a.M = g.d;
  a.N = g.f;
  a.out0 = dw_gate;
  a.out1 = dw_up;
  const int64_t nN = (g.f + 127) / 128;
  if (pairs_kgrouped())
    return launch_kind<Kind::WgradGateUp, true>(
        a0, a0, b0, b1, a, (int64_t)g.E * ((g.d + 2 * BM - 1) / (2 * BM)) * nN, s, &o0, &o1,
        nullptr, pdl);
  return launch_kind<Kind::WgradGateUp, false>(a0, a0, b0, b1, a,
                                               (int64_t)g.E * ((g.d + BM - 1) / BM) * nN, s, &o0,
                                               &o1, nullptr, pdl);
}

}  // namespace moe
