/*
 * moe.h — C ABI of the routed Mixture-of-Experts expert layer for one GB300
 * (sm_103a): router softmax / top-k, atomic-free permute into a padded
 * expert-grouped layout, grouped SwiGLU expert GEMMs, score-weighted
 * gather-sum combine, and the backward of all of them.
 *
 * Sources (the web pages this layer is built from):
 *   [HALO]  Halo "Performance" — §Levers that help (grouped GEMM, atomic-free
 *           expert permute, fused GLU), §Levers that do not help here
 *           (small-M experts are bound by weight bandwidth).
 *   [PLLM]  PocketLLM "Qwen4-Exp Heterogeneous TP4 Performance" — §Runtime
 *           architecture (512 routed experts, top-10 routing).
 *   [PRL]   prime-rl PR #3885 (DeepSeek-V4.1 Flash perf work) — §Changes:
 *           "Single-pass DeepEP local layout" (one gather into the padded
 *           expert-grouped layout, one fp32 score-weighted gather-sum back,
 *           gathers in backward), "FP8 routed experts" (grouped forward,
 *           dgrad and wgrad GEMMs), "FP8 Mega MoE" (K-grouped wgrad),
 *           "dispatch.type = mega_moe" (gradients for x, the top-k weights
 *           and the expert weights), the 32-bit offset overflow fix (element
 *           offsets here are 64-bit), "Spread balanced routing".
 *
 * Conventions shared by every entry point:
 *   - moe_bf16 is the raw 16-bit pattern of a bfloat16.
 *   - Every pointer is a DEVICE pointer unless stated otherwise; every buffer
 *     is owned by the caller. A pointer to an array sized by T (x, dy, y, dx,
 *     logits, the [T, k] arrays, dst_row) may be NULL when T = 0. No entry point allocates, frees or
 *     synchronises device memory (moe_status and the timer read are the only
 *     calls that synchronise). All work is enqueued on `stream` in order.
 *   - Matrices are row-major and densely packed.
 *   - T tokens of width d; E experts of ffn width f; top-k routing; pair
 *     p = t*k + j is token t's j-th choice; P = T*k.
 *   - The padded layout: expert e owns rows [offsets[e], offsets[e+1]) of
 *     every "row buffer" ([R_cap, ...]); its n_e real rows come first in
 *     ascending pair id, then zero padding up to a multiple of `align`.
 *     R_cap >= T*k + E*(align-1) bounds the padded size for any routing, so
 *     the host never needs the counts.
 *   - Shared experts (S >= 0 of them): experts every token goes through with
 *     weight 1, whose outputs are added to the routed ones ([PRL "Fused FP8
 *     shared expert"]: routed and shared outputs summed in the write-back).
 *     Their weights follow the E routed experts' in the same [E+S, ...]
 *     tensors; in the layout they are groups E .. E+S-1, each holding the T
 *     pairs T*k + s*T + t (t = 0 .. T-1, token order) after the T*k routed
 *     pairs t*k + j. With S shared experts R_cap >= T*(k+S) + (E+S)*(align-1)
 *     (moe_row_capacity(T, k + S, E + S, align)); k + S <= 32, E + S <= 1024.
 *   - Return codes below; MOE_ERR_ARG etc. are detected on the host before
 *     anything is enqueued. MOE_ERR_DEVICE_* are raised by kernels into a
 *     per-device status word and reported by moe_status().
 *   - Tuning: the expert GEMMs run some kinds as two-CTA clusters (one
 *     M = 256 tensor-core MMA over two SMs) where that is faster; the
 *     environment variable MOE_GEMM_PAIRS=0 or 1, read once per process,
 *     turns that off or on for every grouped GEMM. Results agree either way
 *     within rounding of the same fp32 accumulation.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;
typedef struct CUstream_st* moe_stream_t; /* the same handle as cudaStream_t */

/* The experts' gated activation (a HOST pointer to it is passed; NULL means
 * the plain SwiGLU, A = silu(G) * U [HALO §Levers that help, fused GLU]):
 *   A = h(min(G, limit)) * (clamp(U, -limit, limit) + up_offset),
 *   h(g) = g * sigmoid(alpha * g);
 * the clamped SwiGLU of [PRL "FP8 routed experts"], whose constants the pages
 * do not print; GPT-OSS-20B's are limit 7, alpha 1.702, up_offset 1. The plain
 * SwiGLU is {INFINITY, 1, 0}. No gradient passes a clamp at its limit.
 * limit must be > 0 (INFINITY allowed); alpha and up_offset finite. */
typedef struct {
  float limit;
  float alpha;
  float up_offset;
} moe_swiglu;

#define MOE_OK                 0
#define MOE_ERR_ARG            1 /* null required pointer, size <= 0, k > E, bad align, ... */
#define MOE_ERR_UNSUPPORTED    2 /* shape the kernels do not take (d or f not a multiple of 8, E > 1024) */
#define MOE_ERR_CAPACITY       3 /* R_cap < T*k + E*(align-1) */
#define MOE_ERR_CUDA           4 /* a CUDA runtime / driver call failed */
#define MOE_ERR_DEVICE_INDEX   5 /* device: an expert id outside [0, E) in a caller-supplied index */
#define MOE_ERR_DEVICE_TIMEOUT 6 /* device: a bounded wait inside a kernel gave up */

/* ------------------------------------------------------------------------
 * moe_route — router logits, top-k selection and renormalised weights.
 * [PLLM §Runtime architecture] top-k routing over many experts; the
 * softmax / top-k / renormalise formula is the plainest reading (the pages do
 * not write it out): l_t = x_t . W_r (+ b) in fp32; S_t = the k largest
 * logits by descending value, equal logits -> lower expert index first;
 * w_t,j = exp(l_S_j - l_S_0) / sum_j' exp(l_S_j' - l_S_0) (a softmax over
 * all E experts restricted to S_t and renormalised is the same number).
 *
 *  x          [T, d] bf16            w_router [d, E] fp32     bias [E] fp32 or NULL
 *  forced_idx [T, k] int32 or NULL:  when given, S_t is taken from it instead
 *             of the top-k (slot order as given; weights are still the
 *             renormalised softmax over it). [PRL "Spread balanced routing"]
 *             An id outside [0, E) raises MOE_ERR_DEVICE_INDEX (the slot's
 *             weight is written as 0).
 *  logits     [T, E] fp32 out        topk_idx [T, k] int32 out    topk_w [T, k] fp32 out
 *  ws         moe_workspace_size(MOE_WS_ROUTE, ...) bytes, 256-byte aligned:
 *             W_r split into three bf16 parts (hi + mid + lo reproduce the fp32
 *             value) so the logits run on the tensor cores from exact products
 *             with fp32 accumulation; for T <= 32 the logits run on the CUDA
 *             cores instead (fp32 products of the bf16 and fp32 values, summed
 *             in row slices, then the slices in order) and ws holds the
 *             slices' partial sums.
 * Limits: 1 <= k <= min(E, 32); E <= 1024; d a multiple of 8.
 * ------------------------------------------------------------------------ */
int moe_route(const moe_bf16* x, const float* w_router, const float* bias,
              const int32_t* forced_idx, int64_t T, int d, int E, int k,
              float* logits, int32_t* topk_idx, float* topk_w,
              void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute — the padded expert-grouped layout and the gather into it.
 * [PRL "Single-pass DeepEP local layout"] one gather of token copies into a
 * padded expert-grouped layout; [HALO §Levers that help] atomic-free expert
 * permute: a per-block histogram (warp match, no atomics), a fixed-order
 * exclusive scan over (block, expert), stable ranks — deterministic.
 *
 *  topk_idx [T, k] int32 in (ids outside [0, E) raise MOE_ERR_DEVICE_INDEX;
 *           such pairs are dropped from the layout, their dst_row is -1)
 *  S        shared experts (groups E .. E+S-1, every token in token order)
 *  x        [T, d] bf16 in
 *  counts   [E+S] int32 out: n_e (T for a shared expert)
 *  offsets  [E+S+1] int64 out: offsets[e] = sum_{e'<e} ceil(n_e'/align)*align
 *  dst_row  [T*(k+S)] int32 out: row of pair p
 *  src_pair [R_cap] int32 out: pair held by row r, -1 for padding and for
 *           rows past offsets[E]
 *  xp       [R_cap, d] bf16 out: xp[r] = x[src_pair[r] / k]; padding rows
 *           inside groups are 0; rows >= offsets[E] are not written
 *  align    power of two in [16, 256] (the grouped GEMMs consume rows in
 *           steps of 16, one bf16 MMA K-step, so every group must be a
 *           multiple of 16 rows)
 *  ws       workspace of moe_workspace_size(MOE_WS_PERMUTE, ...) bytes
 * ------------------------------------------------------------------------ */
int moe_permute(const int32_t* topk_idx, int64_t T, int k, int E, int S, int align,
                const moe_bf16* x, int d, int64_t R_cap,
                int32_t* counts, int64_t* offsets, int32_t* dst_row, int32_t* src_pair,
                moe_bf16* xp, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute_noalloc — moe_permute without a workspace argument (routed
 * experts only: S = 0).
 * (No counterpart on the source pages: this is a calling convention of this
 * library, not part of the method.)
 * For callers that cannot allocate device memory: a host application that
 * owns all device memory through its own fixed pool and forbids other
 * allocations, or a latency-critical path where cudaMalloc's implicit
 * device synchronisation and its possible failure under memory pressure are
 * not acceptable. The kernels' scratch lives in a 2 MiB array built into the
 * library (every GPU that loads the library keeps it until process exit), so
 * this call allocates nothing; the caller still passes every input and
 * output, with the meaning, layout and limits of moe_permute.
 *  - The scratch needed is 4*ceil(T*k/4096)*E + 4*T*k bytes (each part
 *    rounded up to 256); problems needing more than 2 MiB return
 *    MOE_ERR_UNSUPPORTED before anything is enqueued (T*k up to about 500k
 *    pairs at E = 64; use moe_permute with a workspace beyond that).
 *  - The first call on each device looks up the array's device address with
 *    cudaGetSymbolAddress (a host-side call with that device current); make
 *    that first call before any stream capture begins. The address is kept
 *    for the life of the process: after cudaDeviceReset on that device it is
 *    no longer valid, so do not call this entry point again in that process.
 *  - All calls share the one array, and it keeps the last call's contents:
 *    calls whose work overlaps on the GPU (different streams, or different
 *    host threads on one device) race on it and must be serialised by the
 *    caller. The kernels overwrite every scratch word before reading it, so
 *    nothing needs clearing between calls.
 * ------------------------------------------------------------------------ */
int moe_permute_noalloc(const int32_t* topk_idx, int64_t T, int k, int E, int align,
                        const moe_bf16* x, int d, int64_t R_cap,
                        int32_t* counts, int64_t* offsets, int32_t* dst_row, int32_t* src_pair,
                        moe_bf16* xp, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_expert_fwd — grouped gate/up GEMM with fused SwiGLU, grouped down GEMM.
 * [HALO §Levers that help] one grouped expert matmul instead of a loop, fused
 * GLU; [PRL "Kept expert activations"] G and U are kept for backward (in
 * fp32, so the backward's SwiGLU gradient starts from unrounded values).
 * Per expert e on its rows:  G = Xp.W_gate[e], U = Xp.W_up[e] (fp32
 * accumulation in tensor memory), A = act(G, U) from the fp32 accumulators,
 * Yp = A.W_down[e] (times row_w[r] in fp32 when row_w is given), kept in
 * fp32 so the combine's gather-sum rounds each output once.
 *
 *  xp [R_cap, d] bf16, offsets [E+S+1] int64 (from moe_permute)
 *  act: host pointer to the activation (moe_swiglu), or NULL: plain SwiGLU
 *  T, k, E, S: tokens, top-k, routed and shared experts (T*(k+S) pairs over
 *        E+S groups; sizes the tile schedule: with few rows per expert the
 *        gate/up GEMM uses narrower tiles)
 *  w_gate, w_up [E+S, d, f] bf16;  w_down [E+S, f, d] bf16
 *  row_w [R_cap] fp32 or NULL (NULL: Yp is the unscaled expert output, the
 *        layout the combine and moe_expert_bwd expect)
 *  g, u [R_cap, f] fp32 out;  a [R_cap, f] bf16 out (the down GEMM's operand);
 *  yp [R_cap, d] fp32 out
 * Rows of every group, padding included, are written; padding rows come out
 * 0 because their xp rows are 0. Rows >= offsets[E] are not written.
 * Limits: d, f multiples of 8 (16-byte rows for TMA); E <= 1024.
 * ------------------------------------------------------------------------ */
int moe_expert_fwd(const moe_bf16* xp, const int64_t* offsets, const float* row_w,
                   const moe_swiglu* act, int64_t T, int k, int E, int S, int d, int f,
                   int64_t R_cap,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   float* g, float* u, moe_bf16* a, float* yp,
                   moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_expert_fwd_fused — the expert GEMMs of the forward in one persistent
 * launch (inference: G and U are not kept for a backward).
 * [PRL "FP8 Mega MoE", "dispatch.type = mega_moe"] the routed-expert layer as
 * one fused op in expert-major order; [PRL "Single-pass DeepEP local
 * layout"] the score-weighted fp32 partials a gather-sum adds up.
 * Per expert e on its rows r of the layout: G = Xp.W_gate[e], U = Xp.W_up[e]
 * in fp32 (tensor memory only), A = act(G, U) rounded to bf16 into `a`; the
 * down tiles of a 128-row tile (256 in a CTA pair) wait (bounded, on a count
 * in ws) until every gate/up tile of those rows has stored its part of A,
 * then Yp = w(r) * (A.W_down[e]) in fp32, w(r) the pair's score topk_w[p]
 * for p = src_pair[r] (1 for a shared expert's pair, 0 for padding).
 * y = moe_combine(yp, dst_row, NULL, ...): the same gather-sum, weights 1.
 * A equals moe_expert_fwd's; Yp is its Yp times the score, rounded once.
 *
 *  xp [R_cap, d] bf16, src_pair [R_cap] int32, offsets [E+S+1] int64
 *     (moe_permute);  topk_w [T, k] fp32 (moe_route);  act: as in
 *     moe_expert_fwd;  T, k, E, S as in moe_expert_fwd
 *  w_gate, w_up [E+S, d, f] bf16;  w_down [E+S, f, d] bf16
 *  a [R_cap, f] bf16 out;  yp [R_cap, d] fp32 out (rows of every group;
 *     rows >= offsets[E+S] are not written)
 *  ws  moe_expert_fwd_fused_workspace_size(R_cap, E, S) bytes, 16-byte
 *      aligned; cleared by the call, so one call at a time per buffer
 * The launch holds one CTA per SM and its CTAs wait on one another: a
 * concurrent kernel that keeps SMs busy for longer than the wait limit
 * (1.5 s) makes the call report MOE_ERR_DEVICE_TIMEOUT instead of hanging.
 * Limits: d, f multiples of 8; E + S <= 1024; T >= 1 (T = 0 does nothing).
 * ------------------------------------------------------------------------ */
int moe_expert_fwd_fused(const moe_bf16* xp, const int32_t* src_pair, const int64_t* offsets,
                         const float* topk_w, const moe_swiglu* act, int64_t T, int k, int E,
                         int S, int d, int f, int64_t R_cap, const moe_bf16* w_gate,
                         const moe_bf16* w_up, const moe_bf16* w_down, moe_bf16* a, float* yp,
                         void* ws, size_t ws_bytes, moe_stream_t stream);
size_t moe_expert_fwd_fused_workspace_size(int64_t R_cap, int E, int S);

/* ------------------------------------------------------------------------
 * moe_combine — fp32 score-weighted gather-sum back to token order.
 * [PRL "Single-pass DeepEP local layout"] out[t] = sum_{j<k} w[t,j] *
 * rows[dst_row[t*k+j]] + sum_{s<S} rows[dst_row[T*k + s*T + t]] (the shared
 * experts with weight 1), accumulated in fp32 in slot order, rounded once to
 * bf16. With topk_w == NULL the weights are 1: that is the permute's
 * transpose (dx_t = sum over the token's pairs of dXp) used in backward.
 *  rows [R_cap, d] fp32 in (Yp or dXp);  dst_row [T*(k+S)] int32;
 *  topk_w [T, k] fp32 or NULL;  out [T, d] bf16 out
 * ------------------------------------------------------------------------ */
int moe_combine(const float* rows, const int32_t* dst_row, const float* topk_w,
                int64_t T, int k, int S, int d, moe_bf16* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_expert_bwd — backward of the combine and of the experts.
 * [PRL "Single-pass DeepEP local layout"] gathers in backward;
 * [PRL "FP8 routed experts"] grouped dgrad and wgrad; [PRL "FP8 Mega MoE"]
 * K-grouped wgrad; [PRL "dispatch.type = mega_moe"] gradient of the top-k
 * weights. Steps:
 *   combine transpose:  dyg[r] = dy[t(p)] (the gathered rows, an exact copy),
 *                       dyp[r] = w(p) * dy[t(p)] (bf16; w = 1 for a shared
 *                       expert's pair), both 0 on padding rows
 *   down dgrad:         dAu = dyg . W_down[e]^T (fp32 accumulator), and in its
 *                       epilogue dA = w(p) * dAu (so dA carries no bf16
 *                       rounding of w * dy), dg = dA * dact/dG,
 *                       du = dA * dact/dU, and for the routed pairs
 *                       d_topk_w[p] = <dy[t(p)], Yu> as <dAu, act(G, U)> from
 *                       the fp32 G and U (the expert output of the unrounded
 *                       A), summed over the column tiles in a fixed order
 *   gate/up dgrad:      dxp = dg . W_gate[e]^T + du . W_up[e]^T  (one K = 2f
 *                       sum, stored in fp32 so dx is rounded once)
 *   K-grouped wgrad:    dW_down[e] = A_e^T . dyp_e, dW_gate[e] = Xp_e^T . dg_e,
 *                       dW_up[e] = Xp_e^T . du_e   (an empty expert gets zeros)
 *  dy [T, d] bf16; src_pair [R_cap], dst_row [T*(k+S)] int32; topk_w [T, k]
 *  fp32; offsets [E+S+1]; act, T, k, E, S as in moe_expert_fwd; xp, a
 *  (bf16), g, u (fp32) as written by moe_permute / moe_expert_fwd; weights
 *  as in moe_expert_fwd.
 *  ws: moe_expert_bwd_workspace_size(R_cap, f) bytes, 256-byte aligned (the
 *  top-k weight gradient's per-tile partials; scratch after the call).
 *  Outputs (row buffers, caller-owned, may be reused after the call):
 *  dyg, dyp [R_cap, d] bf16; dg, du [R_cap, f] bf16; dxp [R_cap, d] fp32;
 *  d_topk_w [T, k] fp32 (pairs dropped from the layout get no value);
 *  dw_gate, dw_up [E+S, d, f], dw_down [E+S, f, d] bf16 (overwritten).
 * ------------------------------------------------------------------------ */
int moe_expert_bwd(const moe_bf16* dy, const int32_t* src_pair, const int32_t* dst_row,
                   const float* topk_w, const int64_t* offsets, const moe_swiglu* act,
                   int64_t T, int k, int E, int S, int d, int f, int64_t R_cap,
                   const moe_bf16* xp, const float* g, const float* u, const moe_bf16* a,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   moe_bf16* dyg, moe_bf16* dyp, moe_bf16* dg, moe_bf16* du, float* dxp,
                   float* d_topk_w, moe_bf16* dw_gate, moe_bf16* dw_up, moe_bf16* dw_down,
                   void* ws, size_t ws_bytes, moe_stream_t stream);
/* Workspace bytes of moe_expert_bwd for R_cap rows of ffn width f (0 for a
 * size <= 0). */
size_t moe_expert_bwd_workspace_size(int64_t R_cap, int f);

/* ------------------------------------------------------------------------
 * moe_route_bwd — backward of the router.
 * [PRL "dispatch.type = mega_moe"] gradients for x through the top-k weights.
 * dl_t,S_j = w_j (dw_j - sum_j' w_j' dw_j') on the selected experts (0
 * elsewhere; the selection is piecewise constant); then
 *   dx[t] += sum_j dl_t,j W_r[:, S_j]        (dxp == NULL: read-modify-write of
 *                                             bf16 dx, sum in fp32), or
 *   dx[t]  = sum_p dxp[dst_row[p]] + sum_j dl_t,j W_r[:, S_j]
 *                                            (dxp given: the permute's transpose
 *                                             over the token's k routed and S
 *                                             shared pairs fused in, fp32,
 *                                             rounded once)
 *   dW_r = x^T . dl   (dl as a dense [T, E] matrix; fp32 accumulation of
 *                      exact products on the tensor cores, fixed order)
 *   dbias[e] = sum over e's rows of the padded layout of dl (fp32, row order)
 *  d_topk_w, topk_w [T, k] fp32; topk_idx [T, k] int32; w_router [d, E] fp32;
 *  x [T, d] bf16: the layer input (16-byte aligned);
 *  offsets, src_pair from moe_permute (with the same `align` and S).
 *  dx_inout [T, d] bf16 (added to, or overwritten when dxp is given);
 *  dxp [R_cap, d] fp32 or NULL (from moe_expert_bwd); dst_row [T*(k+S)] int32
 *  (required with dxp); dw_router [d, E] fp32 out; dbias [E] fp32 out or NULL.
 *  ws: moe_workspace_size(MOE_WS_ROUTE_BWD, ...) bytes, 256-byte aligned.
 * ------------------------------------------------------------------------ */
int moe_route_bwd(const float* d_topk_w, const float* topk_w, const int32_t* topk_idx,
                  const float* w_router, const int64_t* offsets, const int32_t* src_pair,
                  const moe_bf16* x, int64_t T, int d, int E, int k, int S, int align,
                  moe_bf16* dx_inout, const float* dxp, const int32_t* dst_row,
                  float* dw_router, float* dbias,
                  void* ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_decode_fwd — the whole forward for a handful of tokens (decode), in one
 * cooperative kernel (routed experts with the plain SwiGLU; no shared experts).
 * [HALO §Levers that do not help here] small-M experts are bound by reading
 * their weights; [PLLM §Runtime architecture] top-k routing. For T <= 8 the
 * general path's seven launches cost more than the work: this call computes
 * the same forward as moe_route + moe_permute + moe_expert_fwd + moe_combine
 * (row_w == NULL) in one launch whose phases are separated by grid barriers:
 * router logits (fp32 dot products), top-k with renormalised weights (ties ->
 * lower index), then the gate/up and down products of every selected expert
 * with every token routed to it (each weight row read once, the rows of all
 * selected experts split evenly over every warp of the GPU), A = silu(G)*U
 * and the expert outputs kept in fp32, and y[t] = sum_j w[t,j] * (expert
 * output) in slot order, rounded to bf16 once. Two calls on one GPU give
 * bitwise equal results. The general path (the four calls above) is faster
 * on GB300 at the decode sizes measured; this call is the one-launch form.
 *  x [T, d] bf16; w_router [d, E] fp32; bias [E] fp32 or NULL;
 *  forced_idx [T, k] int32 or NULL (as in moe_route: ids outside [0, E) raise
 *  MOE_ERR_DEVICE_INDEX and the pair is dropped);
 *  w_gate, w_up [E, d, f] bf16; w_down [E, f, d] bf16;
 *  logits [T, E] fp32, topk_idx [T, k] int32, topk_w [T, k] fp32, y [T, d]
 *  bf16 out.
 *  ws: moe_decode_workspace_size(T, d, f, E, k) bytes, 256-byte aligned. The
 *  size depends on the current device's SM count: query it with the device
 *  that will run the call current.
 * Limits: T <= 8 (else MOE_ERR_UNSUPPORTED; T = 0 does nothing), d and f
 * multiples of 64, d <= 8192, f <= 16384, each cut into equal column blocks of
 * at most 4096 (else MOE_ERR_UNSUPPORTED), k <= 32, E <= 1024. Needs a device
 * that supports cooperative launch with one CTA of 544 threads and about
 * 200 KiB of shared memory per SM, and at most 256 SMs (else MOE_ERR_CUDA).
 * ------------------------------------------------------------------------ */
int moe_decode_fwd(const moe_bf16* x, const float* w_router, const float* bias,
                   const int32_t* forced_idx, int64_t T, int d, int f, int E, int k,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   float* logits, int32_t* topk_idx, float* topk_w, moe_bf16* y,
                   void* ws, size_t ws_bytes, moe_stream_t stream);
/* 0 for arguments the call rejects (T outside [0, 8], a size <= 0). */
size_t moe_decode_workspace_size(int64_t T, int d, int f, int E, int k);

/* ------------------------------------------------------------------------
 * Workspace sizes (bytes) for the calls that take `ws`. Any 256-byte-aligned
 * device buffer of at least this size works; its contents need no
 * initialisation and are scratch after the call.
 * ------------------------------------------------------------------------ */
#define MOE_WS_PERMUTE   1
#define MOE_WS_ROUTE_BWD 2
#define MOE_WS_ROUTE     3
size_t moe_workspace_size(int which, int64_t T, int d, int E, int k, int align);

/* Smallest valid R_cap: T*k + E*(align-1). */
int64_t moe_row_capacity(int64_t T, int k, int E, int align);

/* Synchronises `stream`, then reads and clears this device's status word.
 * Returns MOE_OK or the first MOE_ERR_DEVICE_* a kernel raised since the
 * last call (a CUDA error is reported as MOE_ERR_CUDA). */
int moe_status(moe_stream_t stream);

/* Human-readable name of a return code (static string). */
const char* moe_status_str(int code);

/* ------------------------------------------------------------------------
 * Kernel timer (measurement only). moe_timer_start(kernel, n) makes the
 * library record a CUDA event pair around each of the next n launches of
 * `kernel` (one of MOE_KERNEL_*; a group id covers every launch of that
 * step); moe_timer_read waits for them and returns the summed device time in
 * ms and the number of launches timed. One timer at a time per process.
 * Events are created in start and destroyed in read.
 * ------------------------------------------------------------------------ */
#define MOE_KERNEL_ROUTER_LOGITS 1
#define MOE_KERNEL_TOPK          2
#define MOE_KERNEL_PERMUTE       3
#define MOE_KERNEL_GATEUP_FWD    4
#define MOE_KERNEL_DOWN_FWD      5
#define MOE_KERNEL_COMBINE       6
#define MOE_KERNEL_COMBINE_BWD   7
#define MOE_KERNEL_DOWN_DGRAD    8
#define MOE_KERNEL_GATEUP_DGRAD  9
#define MOE_KERNEL_WGRAD_DOWN    10
#define MOE_KERNEL_WGRAD_GATEUP  11
#define MOE_KERNEL_ROUTE_BWD     12
#define MOE_KERNEL_DECODE        13
#define MOE_KERNEL_FUSED_FWD     14
int moe_timer_start(int kernel, int max_launches);
int moe_timer_read(float* total_ms, int* launches);

/* Number of kernels this library has enqueued in this process so far (all
 * devices, all streams). Measurement only. */
uint64_t moe_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
