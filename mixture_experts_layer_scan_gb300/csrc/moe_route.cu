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
constexpr int kRouterTT = 4;  // tokens per CTA

// 16-byte vector of router inputs, widened to fp32.
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
    v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}
__device__ __forceinline__ void load16(const float* p, float (&v)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x;
  v[1] = u.y;
  v[2] = u.z;
  v[3] = u.w;
}

// logits[t][e] = sum_h X[t][h] * Wr[e][h] on the CUDA cores (decode batches and
// the fp32 layer).  A CTA owns one expert and kRouterTT tokens; its 8 warps
// split H into interleaved 16-byte vectors (one pass over Wr[e] per CTA),
// each warp reduces with a fixed butterfly and the 8 warp sums are added in
// warp order, so the result does not depend on scheduling.
template <typename TIn>
__global__ void __launch_bounds__(kRouterWarps * 32) k_router_logits(const TIn* __restrict__ X,
                                                                      const TIn* __restrict__ Wr, int T, int H, int E,
                                                                      float* __restrict__ logits) {
  pdl_enter();
  constexpr int V = 16 / sizeof(TIn);
  __shared__ float red[kRouterWarps][kRouterTT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRouterTT, e = blockIdx.y;
  const int nt = min(kRouterTT, T - t0);
  float acc[kRouterTT];
#pragma unroll
  for (int b = 0; b < kRouterTT; ++b) acc[b] = 0.0f;
  const TIn* w = Wr + (size_t)e * H;
  for (int h = (warp * 32 + lane) * V; h < H; h += kRouterWarps * 32 * V) {
    float wv[V];
    load16(w + h, wv);
#pragma unroll
    for (int b = 0; b < kRouterTT; ++b) {
      if (b < nt) {
        float xv[V];
        load16(X + (size_t)(t0 + b) * H + h, xv);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[b] = fmaf(wv[q], xv[q], acc[b]);
      }
    }
  }
#pragma unroll
  for (int b = 0; b < kRouterTT; ++b) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
    if (lane == 0) red[warp][b] = acc[b];
  }
  __syncthreads();
  if (threadIdx.x < nt) {
    float sum = 0.0f;
#pragma unroll
    for (int w8 = 0; w8 < kRouterWarps; ++w8) sum += red[w8][threadIdx.x];
    logits[(size_t)(t0 + threadIdx.x) * E + e] = sum;
  }
}

constexpr int kTopkCache = 8;  // logits per lane kept in registers by the top-k kernel

// (value, index) order of the ranking: larger value first, lower index on ties.
__device__ __forceinline__ bool ranks_before(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// One warp per token.  k rounds of a warp arg-max over the experts not yet
// taken; each lane owns experts lane, lane+32, ... and a bit mask of the ones
// already taken.  Lane j keeps the j-th pick.
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ logits, int T, int E, int k, int renorm,
                                              float* __restrict__ topk_w, int32_t* __restrict__ topk_ids) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  // the first kTopkCache logits of this lane stay in registers (all of them for E <= 256);
  // the scan order and arithmetic are those of a plain loop over e = lane, lane+32, ...
  float cache[kTopkCache];
#pragma unroll
  for (int q = 0; q < kTopkCache; ++q) cache[q] = (lane + 32 * q < E) ? l[lane + 32 * q] : -INFINITY;
  uint32_t taken = 0;  // bit q: expert lane + 32*q taken
  float my_v = 0.0f;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < kTopkCache; ++q) {
      const int e = lane + 32 * q;
      if (e < E && !(taken & (1u << q)) && ranks_before(cache[q], e, bv, bi)) { bv = cache[q]; bi = e; }
    }
    for (int q = kTopkCache, e = lane + 32 * kTopkCache; e < E; ++q, e += 32) {
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
  // softmax: m is the largest logit (the first pick); each lane sums its experts in ascending order
  const float m = __shfl_sync(0xffffffffu, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - m) : 0.0f;
  float denom;
  if (renorm) {
    denom = ex;
  } else {
    denom = 0.0f;
#pragma unroll
    for (int q = 0; q < kTopkCache; ++q)
      if (lane + 32 * q < E) denom += expf(cache[q] - m);
    for (int e = lane + 32 * kTopkCache; e < E; e += 32) denom += expf(l[e] - m);
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
