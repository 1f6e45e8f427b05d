// permute_noalloc.cu — moe_permute for callers that cannot allocate device
// memory: the same kernels, with their scratch in a fixed array that is part
// of the library image instead of a caller-supplied workspace.
//
// The scratch is a file-scope __device__ array of kNoAllocScratchBytes. Every
// GPU that loads the library holds it until the process exits. Host code
// must not pass the array's name to a kernel (on the host it is only a
// stand-in symbol): its device address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;   // 2 MiB

static __device__ __align__(256) unsigned char g_permute_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;

// Device address of the scratch array on the current device; nullptr on failure.
void* scratch_ptr() {
  static void* ptrs[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess) {
      cudaGetLastError();   // leave no stale error for the next call's launch check
      return nullptr;
    }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_idx, int64_t T, int k, int E, int align,
                                   const moe_bf16* x, int d, int64_t R_cap, int32_t* counts,
                                   int64_t* offsets, int32_t* dst_row, int32_t* src_pair,
                                   moe_bf16* xp, moe_stream_t stream) {
  if (!counts || !offsets || !src_pair || !xp || (T > 0 && (!topk_idx || !x || !dst_row)))
    return MOE_ERR_ARG;
  if (T < 0 || k <= 0 || E <= 0 || d <= 0 || k > E) return MOE_ERR_ARG;
  if (!is_pow2(align) || align < 16 || align > 256) return MOE_ERR_ARG;
  if (E > moe::kMaxExperts || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (R_cap < moe_row_capacity(T, k, E, align)) return MOE_ERR_CAPACITY;
  if (R_cap >= ((int64_t)1 << 31) || T * k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(xp)) return MOE_ERR_ARG;
  // the built-in scratch bounds the problem size
  if (moe::permute_ws_bytes(T, k, E) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
  void* ws = scratch_ptr();
  int* st = moe::device_status_ptr();
  if (!ws || !st) return MOE_ERR_CUDA;
  // The permute kernels write every scratch word before they read it, so the
  // previous call's leftovers need no clearing.
  const cudaError_t e = moe::launch_permute(topk_idx, T, k, E, 0, align, x, d, R_cap, counts,
                                            offsets, dst_row, src_pair, xp, ws, st,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
