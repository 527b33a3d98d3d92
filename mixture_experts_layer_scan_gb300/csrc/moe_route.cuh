// Router building blocks shared by the stand-alone routing kernels and the
// single-launch decode kernel, so both compute bit-identical logits, weights
// and expert ids.
//
// "FusedMoE vs MegaMoE" (zwxr.cn), section 2: the router gives each token a
// weight distribution over the experts, and the k highest-weight experts
// process it.  The selection ranks the fp32 logits (softmax is strictly
// increasing, so this is the ranking of the probabilities); equal logits rank
// the lower expert index first.  Weights are softmax over all E experts,
// renormalised over the k chosen ones on request.
#pragma once

#include "moe_device.cuh"

namespace moe {

constexpr int kRouterWarps = 8;  // threads of a router block: kRouterWarps * 32

// 16-byte vector of router inputs, widened to fp32.
__device__ __forceinline__ void router_load16(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
    v[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}
__device__ __forceinline__ void router_load16(const float* p, float (&v)[4]) {
  const float4 u = *reinterpret_cast<const float4*>(p);
  v[0] = u.x;
  v[1] = u.y;
  v[2] = u.z;
  v[3] = u.w;
}

// logits[t][e] = sum_h X[t][h] * Wr[e][h] for tokens t0 .. t0+TT-1 (< T) of
// one expert, by kRouterWarps * 32 threads (all threads of the block must
// call).  The warps split H into interleaved 16-byte vectors (one pass over
// Wr[e]); each lane accumulates its vectors in order with fma, each warp
// reduces with a fixed butterfly and the warp sums are added in warp order,
// so the value of a logit depends neither on TT nor on scheduling.
// red: shared scratch of kRouterWarps * TT floats.
template <typename TIn, int TT>
__device__ __forceinline__ void router_block(const TIn* __restrict__ X, const TIn* __restrict__ Wr, int T, int H,
                                             int E, int t0, int e, float* __restrict__ logits, float* red) {
  constexpr int V = 16 / sizeof(TIn);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = min(TT, T - t0);
  float acc[TT];
#pragma unroll
  for (int b = 0; b < TT; ++b) acc[b] = 0.0f;
  const TIn* w = Wr + (size_t)e * H;
  for (int h = (warp * 32 + lane) * V; h < H; h += kRouterWarps * 32 * V) {
    float wv[V];
    router_load16(w + h, wv);
    // every token row is loaded (rows past the batch re-read its last row), so
    // the loads go out together; only the batch's tokens are stored
    float xv[TT][V];
#pragma unroll
    for (int b = 0; b < TT; ++b) router_load16(X + (size_t)(t0 + min(b, nt - 1)) * H + h, xv[b]);
#pragma unroll
    for (int b = 0; b < TT; ++b)
#pragma unroll
      for (int q = 0; q < V; ++q) acc[b] = fmaf(wv[q], xv[b][q], acc[b]);
  }
#pragma unroll
  for (int b = 0; b < TT; ++b) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
    if (lane == 0) red[warp * TT + b] = acc[b];
  }
  cta_sync();
  if ((int)threadIdx.x < nt) {
    float sum = 0.0f;
#pragma unroll
    for (int w8 = 0; w8 < kRouterWarps; ++w8) sum += red[w8 * TT + threadIdx.x];
    logits[(size_t)(t0 + threadIdx.x) * E + e] = sum;
  }
  cta_sync();  // red is free again
}

// The same logits for TT tokens and EB experts (e0 .. e0+EB-1, < E) per block, with
// the arithmetic of router_block for every logit: lane-sequential fma over its
// 16-byte vectors, the fixed butterfly, warp sums in warp order.  Inputs stay in
// registers as raw 16-byte vectors and are widened inside the fma loop.
// red: shared scratch of kRouterWarps * TT * EB floats.
__device__ __forceinline__ float router_elem(const uint4& u, int q, const __nv_bfloat16*) {
  const uint32_t w = q < 2 ? u.x : q < 4 ? u.y : q < 6 ? u.z : u.w;
  return bf16_bits_to_f32((q & 1) ? (w >> 16) : (w & 0xffffu));
}
__device__ __forceinline__ float router_elem(const uint4& u, int q, const float*) {
  return __uint_as_float(q == 0 ? u.x : q == 1 ? u.y : q == 2 ? u.z : u.w);
}

template <typename TIn, int TT, int EB>
__device__ __forceinline__ void router_tile(const TIn* __restrict__ X, const TIn* __restrict__ Wr, int T, int H,
                                            int E, int t0, int e0, float* __restrict__ logits, float* red) {
  constexpr int V = 16 / sizeof(TIn);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt = min(TT, T - t0), ne = min(EB, E - e0);
  float acc[EB][TT];
#pragma unroll
  for (int c = 0; c < EB; ++c)
#pragma unroll
    for (int b = 0; b < TT; ++b) acc[c][b] = 0.0f;
  for (int h = (warp * 32 + lane) * V; h < H; h += kRouterWarps * 32 * V) {
    // every row is loaded (rows past the batch or the experts re-read the last one)
    uint4 wr[EB], xr[TT];
#pragma unroll
    for (int c = 0; c < EB; ++c) wr[c] = *reinterpret_cast<const uint4*>(Wr + (size_t)(e0 + min(c, ne - 1)) * H + h);
#pragma unroll
    for (int b = 0; b < TT; ++b) xr[b] = *reinterpret_cast<const uint4*>(X + (size_t)(t0 + min(b, nt - 1)) * H + h);
#pragma unroll
    for (int q = 0; q < V; ++q) {
#pragma unroll
      for (int c = 0; c < EB; ++c) {
        const float w = router_elem(wr[c], q, X);
#pragma unroll
        for (int b = 0; b < TT; ++b) acc[c][b] = fmaf(w, router_elem(xr[b], q, X), acc[c][b]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < EB; ++c)
#pragma unroll
    for (int b = 0; b < TT; ++b) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[c][b] += __shfl_xor_sync(0xffffffffu, acc[c][b], off);
      if (lane == 0) red[(warp * EB + c) * TT + b] = acc[c][b];
    }
  cta_sync();
  if ((int)threadIdx.x < EB * TT) {
    const int c = threadIdx.x / TT, b = threadIdx.x % TT;
    if (c < ne && b < nt) {
      float sum = 0.0f;
#pragma unroll
      for (int w8 = 0; w8 < kRouterWarps; ++w8) sum += red[(w8 * EB + c) * TT + b];
      logits[(size_t)(t0 + b) * E + e0 + c] = sum;
    }
  }
  cta_sync();  // red is free again
}

constexpr int kTopkCache = 8;  // logits per lane kept in registers by the top-k

// (value, index) order of the ranking: larger value first, lower index on ties.
__device__ __forceinline__ bool ranks_before(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// logit loads: through L1, or L2 only (CG) when another block of the same
// kernel wrote them
template <bool CG>
__device__ __forceinline__ float topk_ld(const float* p) {
  if constexpr (CG)
    return __ldcg(p);
  else
    return *p;
}

// Top-k of one token's E logits by one warp (all 32 lanes call).  k rounds of
// a warp arg-max over the experts not yet taken; each lane owns experts lane,
// lane+32, ... and a bit mask of the ones already taken; lane j keeps the
// j-th pick and writes ids[j], w[j].
template <bool CG>
__device__ __forceinline__ void topk_warp(const float* __restrict__ l, int E, int k, int renorm,
                                          float* __restrict__ w_out, int32_t* __restrict__ id_out) {
  const int lane = threadIdx.x & 31;
  // the first kTopkCache logits of this lane stay in registers (all of them for E <= 256);
  // the scan order and arithmetic are those of a plain loop over e = lane, lane+32, ...
  float cache[kTopkCache];
#pragma unroll
  for (int q = 0; q < kTopkCache; ++q) cache[q] = topk_ld<CG>(l + min(lane + 32 * q, E - 1));  // loads go out together
#pragma unroll
  for (int q = 0; q < kTopkCache; ++q)
    if (lane + 32 * q >= E) cache[q] = -INFINITY;
  uint32_t taken = 0;  // bit q: expert lane + 32*q taken
  float my_v = 0.0f;
  int my_i = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < kTopkCache; ++q) {
      const int e = lane + 32 * q;
      if (e < E && !(taken & (1u << q)) && ranks_before(cache[q], e, bv, bi)) {
        bv = cache[q];
        bi = e;
      }
    }
    for (int q = kTopkCache, e = lane + 32 * kTopkCache; e < E; ++q, e += 32) {
      if (taken & (1u << q)) continue;
      const float v = topk_ld<CG>(l + e);
      if (ranks_before(v, e, bv, bi)) {
        bv = v;
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ranks_before(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (bi < 0 || bi >= E) bi = 0;  // only reachable with NaN logits
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_v = bv;
      my_i = bi;
    }
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
    for (int e = lane + 32 * kTopkCache; e < E; e += 32) denom += expf(topk_ld<CG>(l + e) - m);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);
  if (lane < k) {
    id_out[lane] = my_i;
    w_out[lane] = ex / denom;
  }
}

}  // namespace moe
