// Router: gate GEMM (fp32 accumulation) and warp-shuffle softmax / top-k.
//
// "FusedMoE vs MegaMoE" (zwxr.cn), section 2: the router gives each token a
// weight distribution over the experts, and the k highest-weight experts
// process it.  The selection ranks the fp32 logits (softmax is strictly
// increasing, so this is the ranking of the probabilities); equal logits rank
// the lower expert index first.  Weights are softmax over all E experts,
// renormalised over the k chosen ones on request.
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;
constexpr int kRouterTT = 4;    // tokens per CTA
constexpr int kRouterEPW = 2;   // experts per warp
constexpr int kRouterHC = 1024; // hidden columns staged per pass

// logits[t][e] = sum_h X[t][h] * Wr[e][h]; a CTA covers kRouterTT tokens and
// kRouterWarps*kRouterEPW experts, staging the token rows in shared memory.
// Each lane accumulates a strided slice of h; the warp then reduces with a
// fixed butterfly, so the result does not depend on scheduling.
template <typename TIn>
__global__ void __launch_bounds__(kRouterWarps * 32) k_router_logits(const TIn* __restrict__ X,
                                                                      const TIn* __restrict__ Wr, int T, int H, int E,
                                                                      float* __restrict__ logits) {
  __shared__ float xs[kRouterTT][kRouterHC];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRouterTT;
  const int e0 = (blockIdx.y * kRouterWarps + warp) * kRouterEPW;
  float acc[kRouterEPW][kRouterTT];
#pragma unroll
  for (int a = 0; a < kRouterEPW; ++a)
#pragma unroll
    for (int b = 0; b < kRouterTT; ++b) acc[a][b] = 0.0f;

  for (int hc = 0; hc < H; hc += kRouterHC) {
    const int hn = min(kRouterHC, H - hc);
    __syncthreads();
    for (int i = threadIdx.x; i < kRouterTT * kRouterHC; i += blockDim.x) {
      const int tt = i / kRouterHC, h = i % kRouterHC;
      xs[tt][h] = (t0 + tt < T && h < hn) ? to_f32(X[(size_t)(t0 + tt) * H + hc + h]) : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < kRouterEPW; ++a) {
      const int e = e0 + a;
      if (e >= E) break;
      const TIn* w = Wr + (size_t)e * H + hc;
      for (int h = lane; h < hn; h += 32) {
        const float wv = to_f32(w[h]);
#pragma unroll
        for (int b = 0; b < kRouterTT; ++b) acc[a][b] = fmaf(wv, xs[b][h], acc[a][b]);
      }
    }
  }
#pragma unroll
  for (int a = 0; a < kRouterEPW; ++a)
#pragma unroll
    for (int b = 0; b < kRouterTT; ++b)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[a][b] += __shfl_xor_sync(0xffffffffu, acc[a][b], off);
  if (lane == 0) {
#pragma unroll
    for (int a = 0; a < kRouterEPW; ++a) {
      const int e = e0 + a;
      if (e >= E) break;
#pragma unroll
      for (int b = 0; b < kRouterTT; ++b)
        if (t0 + b < T) logits[(size_t)(t0 + b) * E + e] = acc[a][b];
    }
  }
}

// (value, index) order of the ranking: larger value first, lower index on ties.
__device__ __forceinline__ bool ranks_before(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// One warp per token.  k rounds of a warp arg-max over the experts not yet
// taken; each lane owns experts lane, lane+32, ... and a bit mask of the ones
// already taken.  Lane j keeps the j-th pick.
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k, int renorm,
                                              float* __restrict__ topk_w, int32_t* __restrict__ topk_ids) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  uint32_t taken = 0;  // bit q: expert lane + 32*q taken
  float my_v = 0.0f;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int q = 0, e = lane; e < E; ++q, e += 32) {
      if (taken & (1u << q)) continue;
      const float v = l[e];
      if (ranks_before(v, e, bv, bi)) { bv = v; bi = e; }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (bi < 0 || bi >= E) bi = 0;  // only reachable with NaN logits
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) { my_v = bv; my_i = bi; }
  }
  // softmax: m is the largest logit (the first pick)
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - m) : 0.0f;
  float denom;
  if (renorm) {
    denom = ex;
  } else {
    denom = 0.0f;
    for (int e = lane; e < E; e += 32) denom += expf(l[e] - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  if (lane < k) {
    topk_ids[(size_t)t * k + lane] = my_i;
    topk_w[(size_t)t * k + lane] = ex / denom;
  }
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
  dim3 grid((T + kRouterTT - 1) / kRouterTT, (E + kRouterWarps * kRouterEPW - 1) / (kRouterWarps * kRouterEPW));
  if (bf16)
    k_router_logits<__nv_bfloat16><<<grid, kRouterWarps * 32, 0, s>>>(
        (const __nv_bfloat16*)X, (const __nv_bfloat16*)Wr, T, H, E, logits);
  else
    k_router_logits<float><<<grid, kRouterWarps * 32, 0, s>>>((const float*)X, (const float*)Wr, T, H, E, logits);
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits, int T, int E, int k, int renorm, float* w, int32_t* ids,
                        cudaStream_t s) {
  const int warps = 8;
  k_topk<<<(T + warps - 1) / warps, warps * 32, 0, s>>>(logits, T, E, k, renorm, w, ids);
  return cudaGetLastError();
}

cudaError_t launch_inject_timeout(const int* flag, int* status, cudaStream_t s) {
  k_inject_timeout<<<1, 1, 0, s>>>(flag, status);
  return cudaGetLastError();
}

}  // namespace moe
