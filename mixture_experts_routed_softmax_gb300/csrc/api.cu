// api.cu — the C ABI declared in include/moe.h: argument checks, the
// per-device status word, workspace sizes, the kernel timer, and the order
// in which each entry point launches its kernels.
#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

// Per-device status word: kernels raise MOE_ERR_DEVICE_* into it.
__device__ int g_moe_status;

namespace moe {

static constexpr int kMaxDevices = 64;

int* device_status_ptr() {
  static int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_status) != cudaSuccess) {
      cudaGetLastError();   // leave no stale error for the next call's launch check
      return nullptr;
    }
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

int num_sms() {
  static int sms[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  if (!sms[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = n > 0 ? n : 1;
  }
  return sms[dev];
}

static std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

// ------------------------------------------------------------ kernel timer --
struct Timer {
  std::mutex mu;
  int kernel = 0;
  int cap = 0;
  int count = 0;
  std::vector<cudaEvent_t> start, stop;
};
static Timer g_timer;

void timer_before(int kernel, cudaStream_t s) {
  if (g_timer.kernel != kernel) return;
  std::lock_guard<std::mutex> lock(g_timer.mu);
  if (g_timer.kernel == kernel && g_timer.count < g_timer.cap)
    cudaEventRecord(g_timer.start[g_timer.count], s);
}
void timer_after(int kernel, cudaStream_t s) {
  if (g_timer.kernel != kernel) return;
  std::lock_guard<std::mutex> lock(g_timer.mu);
  if (g_timer.kernel == kernel && g_timer.count < g_timer.cap)
    cudaEventRecord(g_timer.stop[g_timer.count++], s);
}

}  // namespace moe

using namespace moe;

static bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
// the activation's parameters (NULL: the plain SwiGLU); a limit <= 0, NaN or
// a NaN alpha / offset is rejected
static bool act_of(const moe_swiglu* a, ActParams* out) {
  if (!a) {
    *out = ActParams{INFINITY, 1.0f, 0.0f};
    return true;
  }
  if (!(a->limit > 0.0f) || a->alpha != a->alpha || a->up_offset != a->up_offset) return false;
  *out = ActParams{a->limit, a->alpha, a->up_offset};
  return true;
}
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static int cuda_code(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

extern "C" {

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int64_t moe_row_capacity(int64_t T, int k, int E, int align) {
  return T * k + (int64_t)E * (align - 1);
}

size_t moe_workspace_size(int which, int64_t T, int d, int E, int k, int align) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0) return 0;
  switch (which) {
    case MOE_WS_PERMUTE: return permute_ws_bytes(T, k, E);
    case MOE_WS_ROUTE_BWD: return (align > 0) ? route_bwd_ws_bytes(T, d, E, k, align) : 0;
    case MOE_WS_ROUTE: return route_ws_bytes(T, d, E);
    default: return 0;
  }
}

const char* moe_status_str(int code) {
  switch (code) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_ARG: return "MOE_ERR_ARG: invalid argument";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape not supported by the kernels";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY: R_cap below T*k + E*(align-1)";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    case MOE_ERR_DEVICE_INDEX: return "MOE_ERR_DEVICE_INDEX: expert id outside [0, E)";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded wait in a kernel gave up";
    default: return "unknown moe status code";
  }
}

int moe_status(moe_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return v;
}

int moe_timer_start(int kernel, int max_launches) {
  if (kernel < MOE_KERNEL_ROUTER_LOGITS || kernel > MOE_KERNEL_FUSED_FWD || max_launches <= 0)
    return MOE_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_timer.mu);
  if (g_timer.kernel != 0) return MOE_ERR_ARG;
  g_timer.start.assign(max_launches, nullptr);
  g_timer.stop.assign(max_launches, nullptr);
  for (int i = 0; i < max_launches; ++i) {
    if (cudaEventCreate(&g_timer.start[i]) != cudaSuccess ||
        cudaEventCreate(&g_timer.stop[i]) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  g_timer.cap = max_launches;
  g_timer.count = 0;
  g_timer.kernel = kernel;
  return MOE_OK;
}

int moe_timer_read(float* total_ms, int* launches) {
  if (!total_ms || !launches) return MOE_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_timer.mu);
  if (g_timer.kernel == 0) return MOE_ERR_ARG;
  int rc = MOE_OK;
  float sum = 0.f;
  for (int i = 0; i < g_timer.count; ++i) {
    float ms = 0.f;
    if (cudaEventSynchronize(g_timer.stop[i]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, g_timer.start[i], g_timer.stop[i]) != cudaSuccess)
      rc = MOE_ERR_CUDA;
    sum += ms;
  }
  *total_ms = sum;
  *launches = g_timer.count;
  for (int i = 0; i < g_timer.cap; ++i) {
    if (g_timer.start[i]) cudaEventDestroy(g_timer.start[i]);
    if (g_timer.stop[i]) cudaEventDestroy(g_timer.stop[i]);
  }
  g_timer.start.clear();
  g_timer.stop.clear();
  g_timer.kernel = 0;
  g_timer.cap = g_timer.count = 0;
  return rc;
}

int moe_route(const moe_bf16* x, const float* w_router, const float* bias,
              const int32_t* forced_idx, int64_t T, int d, int E, int k, float* logits,
              int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
              moe_stream_t stream) {
  if (!w_router || (T > 0 && (!x || !logits || !topk_idx || !topk_w))) return MOE_ERR_ARG;
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_ARG;
  if (k > kMaxTopK || E > kMaxExperts || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (T >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x)) return MOE_ERR_ARG;
  if (!ws || ws_bytes < route_ws_bytes(T, d, E) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  if (route_is_small(T))
    return cuda_code(launch_route_small(x, w_router, bias, forced_idx, T, d, E, k, logits,
                                        topk_idx, topk_w, ws, st, s));
  cudaError_t e = launch_router_logits(x, w_router, bias, T, d, E, logits, ws, st, s);
  if (e == cudaSuccess) e = launch_topk(logits, forced_idx, T, E, k, topk_idx, topk_w, st, s);
  return cuda_code(e);
}

int moe_permute(const int32_t* topk_idx, int64_t T, int k, int E, int S, int align,
                const moe_bf16* x, int d, int64_t R_cap, int32_t* counts, int64_t* offsets,
                int32_t* dst_row, int32_t* src_pair, moe_bf16* xp, void* ws, size_t ws_bytes,
                moe_stream_t stream) {
  if (!counts || !offsets || !src_pair || !xp || (T > 0 && (!topk_idx || !x || !dst_row)))
    return MOE_ERR_ARG;
  if (T < 0 || k <= 0 || E <= 0 || d <= 0 || k > E || S < 0) return MOE_ERR_ARG;
  if (!is_pow2(align) || align < 16 || align > 256) return MOE_ERR_ARG;
  if (E + S > kMaxExperts || k + S > kMaxTopK || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (R_cap < moe_row_capacity(T, k + S, E + S, align)) return MOE_ERR_CAPACITY;
  if (R_cap >= ((int64_t)1 << 31) || T * (k + S) >= ((int64_t)1 << 31))
    return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_ARG;
  const size_t need = permute_ws_bytes(T, k, E);
  if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  return cuda_code(launch_permute(topk_idx, T, k, E, S, align, x, d, R_cap, counts, offsets,
                                  dst_row, src_pair, xp, ws, st,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

static int check_expert_dims(int E, int d, int f, int64_t R_cap) {
  if (E <= 0 || d <= 0 || f <= 0 || R_cap <= 0) return MOE_ERR_ARG;
  if (E > kMaxExperts || d % 8 != 0 || f % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (R_cap >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int moe_expert_fwd(const moe_bf16* xp, const int64_t* offsets, const float* row_w,
                   const moe_swiglu* act, int64_t T, int k, int E, int S, int d, int f,
                   int64_t R_cap, const moe_bf16* w_gate, const moe_bf16* w_up,
                   const moe_bf16* w_down, float* g, float* u, moe_bf16* a, float* yp,
                   moe_stream_t stream) {
  if (!xp || !offsets || !w_gate || !w_up || !w_down || !g || !u || !a || !yp) return MOE_ERR_ARG;
  if (T < 0 || k <= 0 || k > E || S < 0) return MOE_ERR_ARG;
  ActParams ap;
  if (!act_of(act, &ap)) return MOE_ERR_ARG;
  int rc = check_expert_dims(E + S, d, f, R_cap);
  if (rc) return rc;
  if (R_cap < T * (k + S)) return MOE_ERR_CAPACITY;
  for (const void* p : {(const void*)xp, (const void*)w_gate, (const void*)w_up,
                        (const void*)w_down, (const void*)g, (const void*)u, (const void*)a,
                        (const void*)yp})
    if (!aligned16(p)) return MOE_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GroupedDims gd{offsets, E + S, d, f, R_cap, T * (k + S)};
  gd.P_routed = T * k;
  cudaError_t e = launch_gateup_fwd(gd, xp, w_gate, w_up, g, u, a, ap, st, s);
  if (e == cudaSuccess) e = launch_down_fwd(gd, a, w_down, row_w, yp, st, s);
  return cuda_code(e);
}

size_t moe_expert_fwd_fused_workspace_size(int64_t R_cap, int E, int S) {
  if (R_cap < 0 || E < 0 || S < 0) return 0;
  return fused_fwd_ws_bytes(R_cap, E + S);
}

int moe_expert_fwd_fused(const moe_bf16* xp, const int32_t* src_pair, const int64_t* offsets,
                         const float* topk_w, const moe_swiglu* act, int64_t T, int k, int E,
                         int S, int d, int f, int64_t R_cap, const moe_bf16* w_gate,
                         const moe_bf16* w_up, const moe_bf16* w_down, moe_bf16* a, float* yp,
                         void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (T < 0 || k <= 0 || k > E || S < 0) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!xp || !src_pair || !offsets || !topk_w || !w_gate || !w_up || !w_down || !a || !yp || !ws)
    return MOE_ERR_ARG;
  ActParams ap;
  if (!act_of(act, &ap)) return MOE_ERR_ARG;
  int rc = check_expert_dims(E + S, d, f, R_cap);
  if (rc) return rc;
  if (R_cap < T * (k + S)) return MOE_ERR_CAPACITY;
  if (ws_bytes < fused_fwd_ws_bytes(R_cap, E + S)) return MOE_ERR_ARG;
  for (const void* p : {(const void*)xp, (const void*)w_gate, (const void*)w_up,
                        (const void*)w_down, (const void*)a, (const void*)yp, (const void*)ws})
    if (!aligned16(p)) return MOE_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GroupedDims gd{offsets, E + S, d, f, R_cap, T * (k + S)};
  gd.P_routed = T * k;
  gd.src_pair = src_pair;
  return cuda_code(launch_fused_fwd(gd, xp, w_gate, w_up, w_down, topk_w, a, yp,
                                    static_cast<int*>(ws), ap, st, s));
}

int moe_combine(const float* rows, const int32_t* dst_row, const float* topk_w, int64_t T,
                int k, int S, int d, moe_bf16* out, moe_stream_t stream) {
  if (!rows || (T > 0 && (!dst_row || !out))) return MOE_ERR_ARG;
  if (T < 0 || k <= 0 || d <= 0 || S < 0) return MOE_ERR_ARG;
  if (k + S > kMaxTopK || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(rows) || !aligned16(out)) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  return cuda_code(launch_combine(rows, dst_row, topk_w, T, k, S, d, out,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

int moe_expert_bwd(const moe_bf16* dy, const int32_t* src_pair, const int32_t* dst_row,
                   const float* topk_w, const int64_t* offsets, const moe_swiglu* act,
                   int64_t T, int k, int E, int S, int d, int f, int64_t R_cap,
                   const moe_bf16* xp, const float* g,
                   const float* u, const moe_bf16* a,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   moe_bf16* dyg, moe_bf16* dyp, moe_bf16* dg, moe_bf16* du, float* dxp,
                   float* d_topk_w, moe_bf16* dw_gate, moe_bf16* dw_up, moe_bf16* dw_down,
                   void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!src_pair || !offsets || !xp || !g || !u || !a || !w_gate || !w_up || !w_down ||
      !dyg || !dyp || !dg || !du || !dxp || !dw_gate || !dw_up || !dw_down ||
      (T > 0 && (!dy || !dst_row || !topk_w || !d_topk_w)))
    return MOE_ERR_ARG;
  if (T < 0 || k <= 0 || k > E || S < 0) return MOE_ERR_ARG;
  ActParams ap;
  if (!act_of(act, &ap)) return MOE_ERR_ARG;
  int rc = check_expert_dims(E + S, d, f, R_cap);
  if (rc) return rc;
  if (R_cap < T * (k + S)) return MOE_ERR_CAPACITY;
  if (!ws || ws_bytes < moe_expert_bwd_workspace_size(R_cap, f) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_ARG;
  for (const void* p : {(const void*)dy, (const void*)xp, (const void*)g, (const void*)u,
                        (const void*)a, (const void*)w_gate, (const void*)w_up,
                        (const void*)w_down, (const void*)dyg, (const void*)dyp, (const void*)dg,
                        (const void*)du, (const void*)dxp, (const void*)dw_gate, (const void*)dw_up,
                        (const void*)dw_down})
    if (!aligned16(p)) return MOE_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  GroupedDims gd{offsets, E + S, d, f, R_cap, T * (k + S)};
  gd.P_routed = T * k;
  gd.src_pair = src_pair;
  float* part = static_cast<float*>(ws);
  cudaError_t e = launch_combine_bwd(dy, src_pair, topk_w, offsets, T, k, E + S, d, R_cap, dyg,
                                     dyp, s);
  if (e == cudaSuccess)
    e = launch_down_dgrad(gd, dyg, topk_w, w_down, g, u, dg, du, part, ap, st, s);
  if (e == cudaSuccess)
    e = launch_dtw_finalize(part, down_dgrad_dtw_slots(f), dst_row, T * k, d_topk_w, s);
  if (e == cudaSuccess) e = launch_gateup_dgrad(gd, dg, du, w_gate, w_up, dxp, st, s);
  if (e == cudaSuccess) e = launch_wgrad_down(gd, a, dyp, dw_down, st, s);
  if (e == cudaSuccess) e = launch_wgrad_gateup(gd, xp, dg, du, dw_gate, dw_up, st, s);
  return cuda_code(e);
}

size_t moe_expert_bwd_workspace_size(int64_t R_cap, int f) {
  if (R_cap <= 0 || f <= 0) return 0;
  return (size_t)R_cap * down_dgrad_dtw_slots(f) * sizeof(float);
}

size_t moe_decode_workspace_size(int64_t T, int d, int f, int E, int k) {
  if (T < 0 || T > kDecodeMaxT || d <= 0 || f <= 0 || E <= 0 || k <= 0) return 0;
  return decode_ws_bytes(T, d, f, E, k);
}

int moe_decode_fwd(const moe_bf16* x, const float* w_router, const float* bias,
                   const int32_t* forced_idx, int64_t T, int d, int f, int E, int k,
                   const moe_bf16* w_gate, const moe_bf16* w_up, const moe_bf16* w_down,
                   float* logits, int32_t* topk_idx, float* topk_w, moe_bf16* y,
                   void* ws, size_t ws_bytes, moe_stream_t stream) {
  if (!w_router || !w_gate || !w_up || !w_down ||
      (T > 0 && (!x || !logits || !topk_idx || !topk_w || !y)))
    return MOE_ERR_ARG;
  if (T < 0 || d <= 0 || f <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_ARG;
  if (T > kDecodeMaxT || k > kMaxTopK || E > kMaxExperts || d % 64 != 0 || f % 64 != 0 ||
      d > kDecodeMaxD || f > kDecodeMaxF || !decode_shape_ok(d, f))
    return MOE_ERR_UNSUPPORTED;
  for (const void* p : {(const void*)x, (const void*)w_gate, (const void*)w_up,
                        (const void*)w_down, (const void*)y})
    if (!aligned16(p)) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!ws || ws_bytes < decode_ws_bytes(T, d, f, E, k) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  return cuda_code(launch_decode_fwd(x, w_router, bias, forced_idx, (int)T, d, f, E, k, w_gate,
                                     w_up, w_down, logits, topk_idx, topk_w, y, ws, st,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int moe_route_bwd(const float* d_topk_w, const float* topk_w, const int32_t* topk_idx,
                  const float* w_router, const int64_t* offsets, const int32_t* src_pair,
                  const moe_bf16* x, int64_t T, int d, int E, int k, int S, int align,
                  moe_bf16* dx_inout, const float* dxp, const int32_t* dst_row,
                  float* dw_router, float* dbias, void* ws, size_t ws_bytes,
                  moe_stream_t stream) {
  if (!w_router || !offsets || !src_pair || !dw_router ||
      (T > 0 && (!d_topk_w || !topk_w || !topk_idx || !x || !dx_inout)))
    return MOE_ERR_ARG;
  if (dxp && ((T > 0 && !dst_row) || !aligned16(dxp))) return MOE_ERR_ARG;
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || S < 0) return MOE_ERR_ARG;
  if (!is_pow2(align) || align < 16 || align > 256) return MOE_ERR_ARG;
  if (k + S > kMaxTopK || E + S > kMaxExperts || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (moe_row_capacity(T, k + S, E + S, align) >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(dx_inout)) return MOE_ERR_ARG;
  const size_t need = route_bwd_ws_bytes(T, d, E, k, align);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_ARG;
  int* st = device_status_ptr();
  if (!st) return MOE_ERR_CUDA;
  return cuda_code(launch_route_bwd(d_topk_w, topk_w, topk_idx, w_router, offsets, src_pair, x,
                                    T, d, E, k, S, align, dx_inout, dxp, dst_row, dw_router, dbias,
                                    ws, st, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
