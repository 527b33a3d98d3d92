// Router: gate GEMM (fp32 accumulation) and warp-shuffle softmax / top-k, as
// stand-alone kernels (the building blocks live in moe_route.cuh).
#include "moe_internal.h"
#include "moe_route.cuh"

namespace moe {

namespace {

constexpr int kRouterTT = 4;  // tokens per CTA

// logits[t][e] on the CUDA cores (decode batches and the fp32 layer): a CTA
// owns one expert and kRouterTT tokens.
template <typename TIn>
__global__ void __launch_bounds__(kRouterWarps * 32) k_router_logits(const TIn* __restrict__ X,
                                                                      const TIn* __restrict__ Wr, int T, int H, int E,
                                                                      float* __restrict__ logits) {
  pdl_enter();
  __shared__ float red[kRouterWarps * kRouterTT];
  router_block<TIn, kRouterTT>(X, Wr, T, H, E, blockIdx.x * kRouterTT, blockIdx.y, logits, red);
}

// The same with kRouterWideEB experts per CTA: for batches from kRouterWideMinTokens
// tokens, where one expert per CTA makes more CTAs than the SMs hold at once (2048 at 64
// tokens over 128 experts, about 2.7 waves; here 512, about 1.1).  Logits bit-identical.
constexpr int kRouterWideEB = 4;
constexpr int kRouterWideMinTokens = 32;
template <typename TIn>
__global__ void __launch_bounds__(kRouterWarps * 32) k_router_logits_wide(const TIn* __restrict__ X,
                                                                           const TIn* __restrict__ Wr, int T, int H,
                                                                           int E, float* __restrict__ logits) {
  pdl_enter();
  __shared__ float red[kRouterWarps * kRouterTT * kRouterWideEB];
  router_tile<TIn, kRouterTT, kRouterWideEB>(X, Wr, T, H, E, blockIdx.x * kRouterTT, blockIdx.y * kRouterWideEB,
                                              logits, red);
}

// One warp per token.
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k, int renorm,
                                              float* __restrict__ topk_w, int32_t* __restrict__ topk_ids) {
  pdl_enter();
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_warp<false>(logits + (size_t)t * E, E, k, renorm, topk_w + (size_t)t * k, topk_ids + (size_t)t * k);
}

// Test hook: wait (bounded, ~1 ms) for a flag nobody sets, then report a timeout.
__global__ void k_inject_timeout(const int* flag, int* status) {
  const uint64_t t0 = globaltimer_ns();
  while (*(volatile const int*)flag == 0) {
    if (globaltimer_ns() - t0 > 1000000ull) {
      report(status, MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_router_logits(const void* X, const void* Wr, int T, int H, int E, bool bf16, float* logits,
                                 cudaStream_t s) {
  if (T >= kRouterWideMinTokens) {
    const dim3 wgrid((T + kRouterTT - 1) / kRouterTT, (E + kRouterWideEB - 1) / kRouterWideEB);
    if (bf16)
      MOE_LAUNCH(k_router_logits_wide<__nv_bfloat16>, wgrid, dim3(kRouterWarps * 32), 0, s,
                 (const __nv_bfloat16*)X, (const __nv_bfloat16*)Wr, T, H, E, logits);
    else
      MOE_LAUNCH(k_router_logits_wide<float>, wgrid, dim3(kRouterWarps * 32), 0, s, (const float*)X,
                 (const float*)Wr, T, H, E, logits);
    return cudaGetLastError();
  }
  dim3 grid((T + kRouterTT - 1) / kRouterTT, E);
  if (bf16)
    MOE_LAUNCH(k_router_logits<__nv_bfloat16>, dim3(grid), dim3(kRouterWarps * 32), 0, s, 
        (const __nv_bfloat16*)X, (const __nv_bfloat16*)Wr, T, H, E, logits);
  else
    MOE_LAUNCH(k_router_logits<float>, dim3(grid), dim3(kRouterWarps * 32), 0, s, (const float*)X, (const float*)Wr, T, H, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int renorm, float* w, int32_t* ids,
                        cudaStream_t s) {
  const int warps = 8;
  MOE_LAUNCH(k_topk, dim3((T + warps - 1) / warps), dim3(warps * 32), 0, s, logits, T, E, k, renorm, w, ids);
  return cudaGetLastError();
}

cudaError_t launch_inject_timeout(const int* flag, int* status, cudaStream_t s) {
  k_inject_timeout<<<1, 1, 0, s>>>(flag, status);
  return cudaGetLastError();
}

}  // namespace moe
