// internal.h — host-side launchers of the kernels, called by the C ABI in
// api.cu after it has checked the arguments. Each launcher enqueues work on
// `s` and returns the cudaError_t of its launches.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Kernel timer hooks (api.cu): no-ops unless moe_timer_start armed `kernel`.
void timer_before(int kernel, cudaStream_t s);
void timer_after(int kernel, cudaStream_t s);
// Launch counter behind moe_kernel_launches().
void note_launches(int n);
// The per-device status word kernels raise errors into.
int* device_status_ptr();
int num_sms();

// route.cu
size_t route_ws_bytes(int64_t T, int d, int E);
// up to 32 tokens: routing on the CUDA cores, logits and top-k in two launches
inline bool route_is_small(int64_t T) { return T <= 32; }
cudaError_t launch_route_small(const moe_bf16* x, const float* w_router, const float* bias,
                               const int32_t* forced, int64_t T, int d, int E, int k,
                               float* logits, int32_t* topk_idx, float* topk_w, void* ws,
                               int* status, cudaStream_t s);
cudaError_t launch_router_logits(const moe_bf16* x, const float* w_router, const float* bias,
                                 int64_t T, int d, int E, float* logits, void* ws, int* status,
                                 cudaStream_t s);
cudaError_t launch_topk(const float* logits, const int32_t* forced_idx, int64_t T, int E, int k,
                        int32_t* topk_idx, float* topk_w, int* status, cudaStream_t s);
size_t route_bwd_ws_bytes(int64_t T, int d, int E, int k, int align);
cudaError_t launch_route_bwd(const float* d_topk_w, const float* topk_w, const int32_t* topk_idx,
                             const float* w_router, const int64_t* offsets,
                             const int32_t* src_pair, const moe_bf16* x, int64_t T, int d, int E,
                             int k, int S, int align, moe_bf16* dx_inout, const float* dxp,
                             const int32_t* dst_row, float* dw_router, float* dbias, void* ws,
                             int* status, cudaStream_t s);

// permute.cu
size_t permute_ws_bytes(int64_t T, int k, int E);
cudaError_t launch_permute(const int32_t* topk_idx, int64_t T, int k, int E, int S, int align,
                           const moe_bf16* x, int d, int64_t R_cap, int32_t* counts,
                           int64_t* offsets, int32_t* dst_row, int32_t* src_pair, moe_bf16* xp,
                           void* ws, int* status, cudaStream_t s);

// combine.cu
cudaError_t launch_combine(const float* rows, const int32_t* dst_row, const float* topk_w,
                           int64_t T, int k, int S, int d, moe_bf16* out, cudaStream_t s);
cudaError_t launch_combine_bwd(const moe_bf16* dy, const int32_t* src_pair, const float* topk_w,
                               const int64_t* offsets, int64_t T, int k, int E, int d,
                               int64_t R_cap, moe_bf16* dyg, moe_bf16* dyp, cudaStream_t s);
// d_topk_w[p] = sum over the slots, in order, of part[dst_row[p]][slot]
cudaError_t launch_dtw_finalize(const float* part, int slots, const int32_t* dst_row, int64_t P,
                                float* d_topk_w, cudaStream_t s);

// gemm.cu (tcgen05 grouped GEMMs)
constexpr int kDecodeMaxT = 8;        // tokens of one decode call
constexpr int kDecodeMaxD = 8192;     // x is kept in shared memory
constexpr int kDecodeMaxF = 16384;
size_t decode_ws_bytes(int64_t T, int d, int f, int E, int k);
bool decode_shape_ok(int d, int f);   // rows cut into equal column blocks of whole octets
cudaError_t launch_decode_fwd(const moe_bf16* x, const float* w_router, const float* bias,
                              const int32_t* forced, int T, int d, int f, int E, int k,
                              const moe_bf16* w_gate, const moe_bf16* w_up,
                              const moe_bf16* w_down, float* logits, int32_t* topk_idx,
                              float* topk_w, moe_bf16* y, void* ws, int* status,
                              cudaStream_t s);
int router_ksplit(int64_t T, int d, int E);
int router_wgrad_ksplit(int64_t T, int d, int N3);
cudaError_t launch_router_wgrad_gemm(const moe_bf16* x, const moe_bf16* dl3, int64_t T, int d,
                                     int N3, int ksplit, float* part, int* status,
                                     cudaStream_t s);
cudaError_t launch_router_gemm(const moe_bf16* x, const moe_bf16* w_split, const float* bias,
                               int64_t T, int d, int E, int E8, int ksplit, float* out,
                               int* status, cudaStream_t s);
// The experts' activation: A = h(min(G, L)) (clamp(U, -L, L) + c),
// h(g) = g sigmoid(alpha g); the plain SwiGLU is {inf, 1, 0}.
struct ActParams {
  float limit, alpha, c;
};
struct GroupedDims {
  const int64_t* offsets;
  int E, d, f;      // E: every group of the layout (routed and shared experts)
  int64_t R_cap;
  int64_t P;        // pairs of the layout (T * (k + S)): sizes the tile schedule
  int64_t P_routed = 0;   // routed pairs (T * k): the rest are shared, weight 1
  // the pair held by each row of the layout (-1: padding), or NULL: lets the
  // K-grouped weight gradients stop each expert's reduction at its real rows;
  // the down dgrad needs it (it finds each row's score through it)
  const int32_t* src_pair = nullptr;
};
cudaError_t launch_gateup_fwd(const GroupedDims& g, const moe_bf16* xp, const moe_bf16* w_gate,
                              const moe_bf16* w_up, float* G, float* U, moe_bf16* A,
                              const ActParams& act, int* status, cudaStream_t s);
cudaError_t launch_down_fwd(const GroupedDims& g, const moe_bf16* A, const moe_bf16* w_down,
                            const float* row_w, float* yp, int* status, cudaStream_t s);
size_t fused_fwd_ws_bytes(int64_t R_cap, int E);
cudaError_t launch_fused_fwd(const GroupedDims& g, const moe_bf16* xp, const moe_bf16* w_gate,
                             const moe_bf16* w_up, const moe_bf16* w_down, const float* pair_w,
                             moe_bf16* A, float* yp, int* ready, const ActParams& act,
                             int* status, cudaStream_t s);
int down_dgrad_dtw_slots(int f);
cudaError_t launch_down_dgrad(const GroupedDims& g, const moe_bf16* dyg, const float* pair_w,
                              const moe_bf16* w_down, const float* G, const float* U,
                              moe_bf16* dG, moe_bf16* dU, float* dtw_part,
                              const ActParams& act, int* status, cudaStream_t s);
cudaError_t launch_gateup_dgrad(const GroupedDims& g, const moe_bf16* dG, const moe_bf16* dU,
                                const moe_bf16* w_gate, const moe_bf16* w_up, float* dxp,
                                int* status, cudaStream_t s);
cudaError_t launch_wgrad_down(const GroupedDims& g, const moe_bf16* A, const moe_bf16* dyp,
                              moe_bf16* dw_down, int* status, cudaStream_t s);
cudaError_t launch_wgrad_gateup(const GroupedDims& g, const moe_bf16* xp, const moe_bf16* dG,
                                const moe_bf16* dU, moe_bf16* dw_gate, moe_bf16* dw_up,
                                int* status, cudaStream_t s);

}  // namespace moe
