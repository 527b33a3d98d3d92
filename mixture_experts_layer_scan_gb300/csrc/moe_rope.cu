// Inverse rotary position embedding fused with per-head FP8 quantisation.
//
// "Mixture-of-Experts kernel engineering on Amazon SageMaker AI", section on
// the Triton JIT: the serving stack's _fused_inv_rope_fp8_quant_per_head kernel
// (fused rotary embedding + FP8 quantisation) was recompiled for every new
// token count until its variable-length arguments were exempted from
// specialisation.  This kernel is compiled once; every shape is a runtime
// argument.
//
// For each token t and head h, x = X[t][h][0:D] (bf16):
//   with R = rot_dim, half = R/2, (c_i, s_i) = cos_sin[pos[t]][i], [half + i]:
//     y_i        = x_i c_i + x_{half+i} s_i            i < half
//     y_{half+i} = x_{half+i} c_i - x_i s_i            (rotation by -angle: the inverse)
//     y_j        = x_j                                 R <= j < D (not rotated)
//   scale[t][h] = max_j |y_j| / 448 (1 when that is 0)
//   Q[t][h][j]  = e4m3(y_j * r), r = 1 / scale[t][h] (one correctly rounded fp32
//                 reciprocal per vector), round to nearest even, saturating
// Products, sums and the reciprocal are separate fp32 roundings (no fused
// multiply-add), so the codes are reproducible in plain fp32 arithmetic.
//
// Layouts with 16-byte granularity go to kernels where a group of lanes shares
// a vector and moves 8 elements per access: loads into registers on a persistent
// grid, or -- long vectors from 4 MB of input -- a shared-memory ring filled by
// bulk copies (below); others to one warp per vector with 4-byte accesses.  HBM
// bound: 3 bytes per element plus 4 per scale.
#include <algorithm>
#include <climits>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRopeWarps = 8;
constexpr int kRopeMaxPairs = 8;  // element pairs per lane and region: D <= 1024

// two floats -> two e4m3 codes (a in the low byte), round to nearest even, saturating
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t v) {
  return make_float2(bf16_bits_to_f32(v & 0xffffu), bf16_bits_to_f32(v >> 16));
}

__global__ void __launch_bounds__(kRopeWarps * 32)
    k_inv_rope_fp8(const uint32_t* __restrict__ X, int T, int heads, int D, int R, const int32_t* __restrict__ pos,
                   const float* __restrict__ cos_sin, int max_pos, uint16_t* __restrict__ Q,
                   float* __restrict__ scale, int* status) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int half = R / 2;
  const size_t nvec = (size_t)T * heads;
  for (size_t v = (size_t)blockIdx.x * kRopeWarps + (threadIdx.x >> 5); v < nvec;
       v += (size_t)gridDim.x * kRopeWarps) {
    const int t = (int)(v / heads);
    int p = pos[t];
    if (p < 0 || p >= max_pos) {
      if (lane == 0) report(status, MOE_ERR_DEVICE_INDEX);
      p = p < 0 ? 0 : max_pos - 1;
    }
    const uint32_t* xr = X + v * (D / 2);  // bf16 pairs of this vector
    const float* cs = cos_sin + (size_t)p * R;
    float2 a[kRopeMaxPairs], b[kRopeMaxPairs], c[kRopeMaxPairs];
    float amax = 0.0f;
    // rotated pairs: elements e, e+1 (e = 2 lane + 64 m < half) and their partners e + half
#pragma unroll
    for (int m = 0; m < kRopeMaxPairs; ++m) {
      const int e = 2 * lane + 64 * m;
      if (e < half) {
        const float2 x1 = bf16x2_to_f2(xr[e / 2]);
        const float2 x2 = bf16x2_to_f2(xr[(half + e) / 2]);
        const float2 co = *reinterpret_cast<const float2*>(cs + e);
        const float2 si = *reinterpret_cast<const float2*>(cs + half + e);
        a[m].x = __fadd_rn(__fmul_rn(x1.x, co.x), __fmul_rn(x2.x, si.x));
        a[m].y = __fadd_rn(__fmul_rn(x1.y, co.y), __fmul_rn(x2.y, si.y));
        b[m].x = __fsub_rn(__fmul_rn(x2.x, co.x), __fmul_rn(x1.x, si.x));
        b[m].y = __fsub_rn(__fmul_rn(x2.y, co.y), __fmul_rn(x1.y, si.y));
        amax = fmaxf(amax, fmaxf(fmaxf(fabsf(a[m].x), fabsf(a[m].y)), fmaxf(fabsf(b[m].x), fabsf(b[m].y))));
      }
    }
    // unrotated tail: elements j, j+1 (j = R + 2 lane + 64 m < D)
#pragma unroll
    for (int m = 0; m < kRopeMaxPairs; ++m) {
      const int j = R + 2 * lane + 64 * m;
      if (j < D) {
        c[m] = bf16x2_to_f2(xr[j / 2]);
        amax = fmaxf(amax, fmaxf(fabsf(c[m].x), fabsf(c[m].y)));
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = e4m3_scale_from_amax(amax);
    const float r = __fdiv_rn(1.0f, s);
    uint16_t* qr = Q + v * (D / 2);  // e4m3 code pairs of this vector
    auto code2 = [&](float2 y) -> uint16_t { return e4m3x2(__fmul_rn(y.x, r), __fmul_rn(y.y, r)); };
#pragma unroll
    for (int m = 0; m < kRopeMaxPairs; ++m) {
      const int e = 2 * lane + 64 * m;
      if (e < half) {
        qr[e / 2] = code2(a[m]);
        qr[(half + e) / 2] = code2(b[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < kRopeMaxPairs; ++m) {
      const int j = R + 2 * lane + 64 * m;
      if (j < D) qr[j / 2] = code2(c[m]);
    }
    if (lane == 0) scale[v] = s;
  }
}

// The same computation with 16-byte accesses: a vector is split into units
// of 8 elements -- a rotated unit is elements [8c, 8c+8) with their partners
// [half+8c, half+8c+8), a tail unit 8 unrotated elements -- and G lanes share
// a vector (U units each), so a warp works on 32/G vectors at once and every
// lane has U x (16..96) bytes of loads in flight.  Needs R % 16 == 0,
// (D - R) % 8 == 0 and 16-byte aligned rows and table.
__device__ __forceinline__ void bf16x8_to_f2(const uint4 u, float2 (&f)[4]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = bf16x2_to_f2(w[i]);
}

// packed fp32x2 multiply, round to nearest even per half
__device__ __forceinline__ uint64_t f2_bits(float2 a) {
  return (uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32);
}
__device__ __forceinline__ float2 f2_from(uint64_t d) {
  return make_float2(__uint_as_float((uint32_t)d), __uint_as_float((uint32_t)(d >> 32)));
}
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
  return f2_from(d);
}
__device__ __forceinline__ uint16_t e4m3x2_f2(float2 y) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
}

// One lane's share of a vector in the 16-byte kernels: units sub, sub + G, ...
// (raw[u][0] the unit's 8 elements, raw[u][1] their rotation partners), cs the
// token's cos/sin row (global or shared memory).  Products in packed fp32x2
// multiplies (each half an IEEE fp32 product rounded to nearest), sums in scalar
// adds with an explicit rounding, which are never fused with the products: the
// values of the scalar kernel above.  Returns the lane's max |y|.
template <int G, int U>
__device__ __forceinline__ float rope_lane(const uint4 (&raw)[U][2], const float4* cs, int sub, int nrot, int nunits,
                                           int half, bool valid, float2 (&ya)[U][4], float2 (&yb)[U][4]) {
  float amax = 0.0f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int unit = sub + G * u;
    if (valid && unit < nunits) {
      if (unit < nrot) {
        float2 x1[4], x2[4];
        bf16x8_to_f2(raw[u][0], x1);
        bf16x8_to_f2(raw[u][1], x2);
        const float4 c0 = cs[2 * unit], c1 = cs[2 * unit + 1];
        const float4 s0 = cs[(half + 8 * unit) / 4], s1 = cs[(half + 8 * unit) / 4 + 1];
        const float2 co[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w), make_float2(c1.x, c1.y),
                              make_float2(c1.z, c1.w)};
        const float2 si[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w), make_float2(s1.x, s1.y),
                              make_float2(s1.z, s1.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 p1 = f2_mul(x1[i], co[i]), p2 = f2_mul(x2[i], si[i]);
          const float2 p3 = f2_mul(x2[i], co[i]), p4 = f2_mul(x1[i], si[i]);
          ya[u][i] = make_float2(__fadd_rn(p1.x, p2.x), __fadd_rn(p1.y, p2.y));
          yb[u][i] = make_float2(__fsub_rn(p3.x, p4.x), __fsub_rn(p3.y, p4.y));
          amax = fmaxf(amax, fmaxf(fmaxf(fabsf(ya[u][i].x), fabsf(ya[u][i].y)),
                                   fmaxf(fabsf(yb[u][i].x), fabsf(yb[u][i].y))));
        }
      } else {
        bf16x8_to_f2(raw[u][0], ya[u]);
#pragma unroll
        for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(ya[u][i].x), fabsf(ya[u][i].y)));
      }
    }
  }
  return amax;
}

// The lane's codes: y * r (packed multiplies) to e4m3, 8 codes per uint2 store.
template <int G, int U>
__device__ __forceinline__ void rope_store(uint2* qr, const float2 (&ya)[U][4], const float2 (&yb)[U][4], float r,
                                           int sub, int nrot, int nunits, int half, int R) {
  const float2 r2 = make_float2(r, r);
  auto code8 = [&](const float2 (&y)[4]) -> uint2 {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      w[h] = (uint32_t)e4m3x2_f2(f2_mul(y[2 * h], r2)) | ((uint32_t)e4m3x2_f2(f2_mul(y[2 * h + 1], r2)) << 16);
    return make_uint2(w[0], w[1]);
  };
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int unit = sub + G * u;
    if (unit < nunits) {
      if (unit < nrot) {
        qr[unit] = code8(ya[u]);
        qr[(half + 8 * unit) / 8] = code8(yb[u]);
      } else {
        qr[(R + 8 * (unit - nrot)) / 8] = code8(ya[u]);
      }
    }
  }
}

// G lanes share a vector: max over the group, scale s = amax / 448 (1 for 0) and its
// IEEE reciprocal (the correctly rounded 1 / s).
template <int G>
__device__ __forceinline__ float rope_group_scale(float amax, float& r) {
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = e4m3_scale_from_amax(amax);
  r = __frcp_rn(s);
  return s;
}

// 32-bit vector indices (the host sends larger layouts to the scalar kernel).
template <int G, int U>
__global__ void __launch_bounds__(kRopeWarps * 32)
    k_inv_rope_fp8_v8(const uint4* __restrict__ X, uint32_t nvec, int heads, int D, int R,
                      const int32_t* __restrict__ pos, const float4* __restrict__ cos_sin, int max_pos,
                      uint2* __restrict__ Q, float* __restrict__ scale, int* status) {
  pdl_enter();
  const int lane = threadIdx.x & 31, sub = lane % G, grp = lane / G;
  const int half = R / 2, nrot = R / 16, nunits = nrot + (D - R) / 8;
  constexpr int VPW = 32 / G;  // vectors per warp at a time
  const uint32_t step = gridDim.x * kRopeWarps * VPW;
  const uint32_t uheads = (uint32_t)heads;
  // the 16-byte chunks of a unit: rotated (8 elements and their partners) or tail (8 elements)
  auto fetch = [&](uint32_t base, uint4 (&raw)[U][2], int& p) {
    const uint32_t v = base + grp;
    if (v >= nvec) return;
    p = __ldg(pos + v / uheads);
    const uint4* xr = X + (size_t)v * (D / 8);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int unit = sub + G * u;
      if (unit < nrot) {
        raw[u][0] = __ldg(xr + unit);
        raw[u][1] = __ldg(xr + (half + 8 * unit) / 8);
      } else if (unit < nunits) {
        raw[u][0] = __ldg(xr + (R + 8 * (unit - nrot)) / 8);
      }
    }
  };
  uint32_t base = (blockIdx.x * kRopeWarps + (threadIdx.x >> 5)) * VPW;
  uint4 nxt[U][2] = {};
  int nxt_p = 0;
  fetch(base, nxt, nxt_p);
  for (; base < nvec; base += step) {
    uint4 cur[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      cur[u][0] = nxt[u][0];
      cur[u][1] = nxt[u][1];
    }
    int p = nxt_p;
    fetch(base + step, nxt, nxt_p);  // the next vectors' loads overlap this one's arithmetic
    const uint32_t v = base + grp;
    const bool valid = v < nvec;
    if (p < 0 || p >= max_pos) {
      if (valid && sub == 0) report(status, MOE_ERR_DEVICE_INDEX);
      p = p < 0 ? 0 : max_pos - 1;
    }
    const float4* cs = cos_sin + (size_t)p * (R / 4);  // 4 floats per float4
    float2 ya[U][4], yb[U][4];
    const float amax = rope_lane<G, U>(cur, cs, sub, nrot, nunits, half, valid, ya, yb);
    float r;
    const float s = rope_group_scale<G>(amax, r);
    if (valid) {
      rope_store<G, U>(Q + (size_t)v * (D / 8), ya, yb, r, sub, nrot, nunits, half, R);
      if (sub == 0) scale[v] = s;
    }
  }
}

// The same layouts staged through shared memory, for long vectors (32 lanes to a
// vector).  Loading into registers keeps few bytes in flight per lane; here one
// producer warp streams chunks of CV consecutive vectors (about 16 KB) and the
// cos/sin rows of their tokens into a ring of shared-memory stages with untiled bulk
// copies (completion in bytes on an mbarrier), up to 8 stages in flight per SM
// whatever the registers, and NW consumer warps compute from shared memory.  (For
// short vectors the register kernel above measured faster: its 32 warps per SM hide
// the latency of the per-vector group reduction and scale better than the staged
// kernel's consumers.)  A chunk's vectors are spread over the consumer warps, G
// lanes per vector, VPT vectors per lane group.  One CTA per SM; every wait bounded.
template <int U>
constexpr int rope_tma_warps() { return U == 1 ? 27 : 15; }  // 28 warps of 72 registers / 16 of 128
constexpr int kRopeTmaMaxStages = 8;

template <int G, int U, int NW = rope_tma_warps<U>()>
__global__ void __launch_bounds__(32 * (NW + 1), 1)
    k_inv_rope_fp8_tma(const uint8_t* __restrict__ X, int heads, int D, int R, const int32_t* __restrict__ pos,
                       const float* __restrict__ cos_sin, int max_pos, uint2* __restrict__ Q,
                       float* __restrict__ scale, int* status, int nvec, int CV, int VPT, int nchunks, int stages,
                       uint32_t stage_bytes, uint32_t tab_off) {
  extern __shared__ uint8_t rope_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(rope_smem_raw) + 127) & ~uintptr_t(127));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + (uint32_t)stages * stage_bytes;
  const uint32_t bar_empty = bar_full + 8 * kRopeTmaMaxStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + (size_t)stages * stage_bytes + 16 * kRopeTmaMaxStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, NW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_enter();
  const int half = R / 2, nrot = R / 16, nunits = nrot + (D - R) / 8;
  const uint32_t vbytes = (uint32_t)D * 2;

  if (warp == 0) {
    // ---------------- producer ----------------
    // The positions of a chunk's tokens (lane j holds tokens j, j+32, ...) are loaded one
    // chunk ahead, so no copy waits on a dependent global load.
    constexpr int kPosRegs = 8;  // tokens per chunk up to 256 (the host checks)
    int pv[kPosRegs] = {};
    auto load_pos = [&](int c) {
      if (R == 0 || c >= nchunks) return;
      const int v0 = c * CV, nv = min(CV, nvec - v0);
      const int t0 = v0 / heads, ntok = (v0 + nv - 1) / heads - t0 + 1;
#pragma unroll
      for (int m = 0; m < kPosRegs; ++m)
        if (lane + 32 * m < ntok) pv[m] = pos[t0 + lane + 32 * m];
    };
    load_pos(blockIdx.x);
    uint32_t it = 0;
    bool ok = true;
    for (int c = blockIdx.x; c < nchunks; c += gridDim.x, ++it) {
      const int st = (int)(it % (uint32_t)stages);
      const uint32_t ph = (it / (uint32_t)stages) & 1u;
      if (it >= (uint32_t)stages && !mbar_wait_all(bar_empty + 8 * st, ph ^ 1u, abort_flag, status)) {
        ok = false;
        break;
      }
      const int v0 = c * CV, nv = min(CV, nvec - v0);
      const int t0 = v0 / heads, ntok = (v0 + nv - 1) / heads - t0 + 1;
      const uint32_t xb = (uint32_t)nv * vbytes, tb = R > 0 ? (uint32_t)ntok * (uint32_t)R * 4u : 0u;
      const uint32_t dst = sbase + (uint32_t)st * stage_bytes;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_full + 8 * st, xb + tb);
        bulk_g2s(dst, X + (size_t)v0 * vbytes, xb, bar_full + 8 * st);
      }
      __syncwarp();
      if (R > 0) {
#pragma unroll
        for (int m = 0; m < kPosRegs; ++m) {
          const int j = lane + 32 * m;
          if (j < ntok) {
            int p = pv[m];
            if (p < 0 || p >= max_pos) {
              report(status, MOE_ERR_DEVICE_INDEX);
              p = p < 0 ? 0 : max_pos - 1;
            }
            bulk_g2s(dst + tab_off + (uint32_t)j * (uint32_t)R * 4u, cos_sin + (size_t)p * R, (uint32_t)R * 4u,
                     bar_full + 8 * st);
          }
        }
      }
      __syncwarp();
      load_pos(c + (int)gridDim.x);
    }
    if (!ok && lane == 0) {  // let the copies in flight land before the CTA exits
      const uint32_t first = it > (uint32_t)stages ? it - (uint32_t)stages : 0u;
      for (uint32_t i = first; i < it; ++i)
        mbar_wait_drain(bar_full + 8 * (i % (uint32_t)stages), (i / (uint32_t)stages) & 1u, 100000000ull);
    }
  } else {
    // ---------------- consumers ----------------
    constexpr int VPW = 32 / G;  // vectors of a warp at a time
    const int cw = warp - 1, sub = lane % G, grp = lane / G;
    uint32_t it = 0;
    for (int c = blockIdx.x; c < nchunks; c += gridDim.x, ++it) {
      const int st = (int)(it % (uint32_t)stages);
      const uint32_t ph = (it / (uint32_t)stages) & 1u;
      if (!mbar_wait_all(bar_full + 8 * st, ph, abort_flag, status)) break;
      const int v0 = c * CV, nv = min(CV, nvec - v0);
      const int t0 = v0 / heads;
      const uint8_t* xs = smem + (size_t)st * stage_bytes;
      for (int k = 0; k < VPT; ++k) {  // (warp-uniform trip count: every lane reaches the shuffles)
        const int j = (cw * VPW + grp) * VPT + k;
        const bool valid = j < nv;
        const int jj = valid ? j : 0;  // (vector 0 of the chunk is always present)
        const int v = v0 + jj;
        const uint4* xr = reinterpret_cast<const uint4*>(xs + (size_t)jj * vbytes);
        const float4* cs = reinterpret_cast<const float4*>(xs + tab_off + (size_t)(v / heads - t0) * R * 4);
        uint4 raw[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int unit = sub + G * u;
          if (unit < nrot) {
            raw[u][0] = xr[unit];
            raw[u][1] = xr[(half + 8 * unit) / 8];
          } else if (unit < nunits) {
            raw[u][0] = xr[(R + 8 * (unit - nrot)) / 8];
          }
        }
        float2 ya[U][4], yb[U][4];
        const float amax = rope_lane<G, U>(raw, cs, sub, nrot, nunits, half, valid, ya, yb);
        float r;
        const float s = rope_group_scale<G>(amax, r);
        if (valid) {
          rope_store<G, U>(Q + (size_t)v * (D / 8), ya, yb, r, sub, nrot, nunits, half, R);
          if (sub == 0) scale[v] = s;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
    }
  }
}

// Host side of k_inv_rope_fp8_tma: chunk and stage sizes for this layout (a stage
// about 16 KB of vectors plus the cos/sin rows of the tokens they span).  Returns
// cudaErrorNotSupported when the layout does not fit the shared memory.
template <int G, int U>
cudaError_t launch_rope_tma(const void* X, int heads, int D, int R, const int32_t* pos, const float* cos_sin,
                            int max_pos, uint8_t* Q, float* scale, int* status, int nvec, int num_sms,
                            cudaStream_t s) {
  constexpr int kVpw = 32 / G, kNw = rope_tma_warps<U>();
  const int slots = kNw * kVpw;  // lane groups of the consumer warps
  const int vbytes = D * 2;
  const int VPT = std::max(1, 16384 / (vbytes * slots));
  const int CV = slots * VPT;
  const int max_tok = CV / heads + 2;  // tokens a run of CV consecutive vectors can touch
  if (max_tok > 256) return cudaErrorNotSupported;  // (the producer holds 8 positions a lane)
  const uint32_t tab_off = (uint32_t)(CV * vbytes + 15) / 16 * 16;
  const uint32_t stage_bytes = (tab_off + (uint32_t)(R > 0 ? max_tok * R * 4 : 0) + 127) / 128 * 128;
  const int stages = std::min<int>(kRopeTmaMaxStages, (int)((200u * 1024u) / stage_bytes));
  if (stages < 2) return cudaErrorNotSupported;
  const size_t smem = 128 + (size_t)stages * stage_bytes + 16 * kRopeTmaMaxStages + 16;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(k_inv_rope_fp8_tma<G, U>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const int nchunks = (nvec + CV - 1) / CV;
  const int grid = std::max(1, std::min(nchunks, num_sms > 0 ? num_sms : 152));
  MOE_LAUNCH(k_inv_rope_fp8_tma<G, U>, dim3(grid), dim3(32 * (kNw + 1)), smem, s, (const uint8_t*)X, heads,
             D, R, pos, cos_sin, max_pos, (uint2*)Q, scale, status, nvec, CV, VPT, nchunks, stages, stage_bytes,
             tab_off);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_inv_rope_fp8(const void* X, int T, int heads, int D, int R, const int32_t* pos,
                                const float* cos_sin, int max_pos, uint8_t* Q, float* scale, int* status,
                                int num_sms, cudaStream_t s) {
  const size_t nvec = (size_t)T * heads;
  const size_t cap = (size_t)(num_sms > 0 ? num_sms : 152) * 16;
  const int nunits = R / 16 + (D - R) / 8;
  const bool vec16 = R % 16 == 0 && (D - R) % 8 == 0 && nunits <= 128 && (reinterpret_cast<uintptr_t>(X) & 15) == 0 &&
                     (reinterpret_cast<uintptr_t>(Q) & 7) == 0 &&
                     (R == 0 || (reinterpret_cast<uintptr_t>(cos_sin) & 15) == 0);
  // (the 16-byte kernels index vectors in 32 bits)
  if (vec16 && nunits > 0 && nvec < (size_t)INT32_MAX) {
    int G = 4;
    while (G < 32 && G < nunits) G *= 2;
    const int U = (nunits + G - 1) / G;
    // long vectors (32 lanes each) from about 4 MB of input go through the staged kernel
    // (below that its prologue and the shared-memory carve-out it needs cost more than
    // the loads in flight save)
    if (G == 32 && nvec * (size_t)D * 2 >= ((size_t)4 << 20)) {
      cudaError_t e = cudaErrorNotSupported;
#define MOE_ROPE_TMA_CASE(GG, UU)                                                                                  \
  if (G == GG && U == UU)                                                                                          \
    e = launch_rope_tma<GG, UU>(X, heads, D, R, pos, cos_sin, max_pos, Q, scale, status, (int)nvec, num_sms, s);
      MOE_ROPE_TMA_CASE(32, 1)
      MOE_ROPE_TMA_CASE(32, 2)
      MOE_ROPE_TMA_CASE(32, 3)
      MOE_ROPE_TMA_CASE(32, 4)
#undef MOE_ROPE_TMA_CASE
      if (e != cudaErrorNotSupported) return e;
    }
    // a persistent grid: the blocks the SMs hold at once (the occupancy of this instance), so
    // every warp runs many grid-stride iterations and its one-ahead loads stay overlapped
    // (a grid of 16 blocks per SM ran in waves of about 3 iterations a warp: 7-20 % slower)
    const size_t per_block = (size_t)kRopeWarps * (32 / G);
    const size_t need = (nvec + per_block - 1) / per_block;
    const int sms = num_sms > 0 ? num_sms : 152;
#define MOE_ROPE_CASE(GG, UU)                                                                                   \
  if (G == GG && U == UU) {                                                                                     \
    static int resident = 0;                                                                                    \
    if (resident == 0) {                                                                                        \
      const cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, k_inv_rope_fp8_v8<GG, UU>, \
                                                                           kRopeWarps * 32, 0);                 \
      if (oe != cudaSuccess) return oe;                                                                         \
      if (resident < 1) resident = 1;                                                                           \
    }                                                                                                           \
    const size_t blocks = std::max<size_t>(1, std::min<size_t>(need, (size_t)sms * resident));                 \
    MOE_LAUNCH(k_inv_rope_fp8_v8<GG, UU>, dim3((unsigned)blocks), dim3(kRopeWarps * 32), 0, s, (const uint4*)X,     \
               (uint32_t)nvec, heads, D, R, pos, (const float4*)cos_sin, max_pos, (uint2*)Q, scale, status);      \
    return cudaGetLastError();                                                                                  \
  }
    MOE_ROPE_CASE(4, 1)
    MOE_ROPE_CASE(8, 1)
    MOE_ROPE_CASE(16, 1)
    MOE_ROPE_CASE(32, 1)
    MOE_ROPE_CASE(32, 2)
    MOE_ROPE_CASE(32, 3)
    MOE_ROPE_CASE(32, 4)
#undef MOE_ROPE_CASE
  }
  size_t blocks = (nvec + kRopeWarps - 1) / kRopeWarps;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  MOE_LAUNCH(k_inv_rope_fp8, dim3((unsigned)blocks), dim3(kRopeWarps * 32), 0, s, (const uint32_t*)X, T, heads, D, R,
             pos, cos_sin, max_pos, (uint16_t*)Q, scale, status);
  return cudaGetLastError();
}

}  // namespace moe
