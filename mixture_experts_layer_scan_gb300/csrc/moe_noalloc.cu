// Allocation-free variant of moe_forward.
//
// Some callers cannot hand the library a workspace: a plugin inside a host
// engine that owns and pre-plans every byte of device memory, a serving loop
// that may not take cudaMalloc's latency or its implicit device
// synchronisation in the middle of a step, or a plain C caller that has no
// device allocator at all.  moe_forward_noalloc serves them: it runs the same
// layer as moe_forward, with the workspace placed in a fixed-size array that
// lives in this library's own device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (MOE_NOALLOC_MAX_WORKSPACE bytes) until the process exits.
// Host code cannot use the array's name as a device address; its address on
// the current device is looked up once per device with cudaGetSymbolAddress
// (first call on that device) and cached.  cudaDeviceReset() makes the cached
// address stale; the library is not to be used on a device after a reset.
#include <mutex>

#include <cuda_runtime.h>

#include "moe_api.h"

namespace {

constexpr size_t kStaticScratchBytes = MOE_NOALLOC_MAX_WORKSPACE;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device (nullptr on failure).
void* static_scratch_for_current_device() {
  static void* ptr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return nullptr;
    ptr[dev] = p;
  }
  return ptr[dev];
}

}  // namespace

extern "C" int moe_forward_noalloc(const void* hidden, const void* router_w, const void* w13, const void* w2, int T,
                                   int H, int I, int E, int topk, int renorm, moe_dtype act_dtype, moe_dtype w_dtype,
                                   const void* w13_scale, const void* w2_scale, void* out,
                                   const moe_options* opts, moe_stream_t stream) {
  size_t need = 0;
  const int rc = moe_workspace_size(T, H, I, E, topk, act_dtype, w_dtype, opts, &need);
  if (rc != MOE_OK) return rc;
  if (T == 0) return MOE_OK;
  if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;  // shape too large for the fixed array
  void* ws = static_scratch_for_current_device();
  if (!ws) return MOE_ERR_CUDA;
  // moe_forward initialises every workspace word it reads before reading it
  // (the FP8 amax words, the test flag and the single-launch kernel's launch
  // tag are cleared on the stream), so the previous call's contents need no
  // clearing here.
  return moe_forward(hidden, router_w, w13, w2, T, H, I, E, topk, renorm, act_dtype, w_dtype, w13_scale, w2_scale,
                     out, ws, kStaticScratchBytes, opts, stream);
}
