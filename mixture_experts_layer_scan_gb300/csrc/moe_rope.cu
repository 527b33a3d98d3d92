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
//   Q[t][h][j]  = e4m3(y_j * r), r = 1 / scale[t][h] (one fp32 division per
//                 vector), round to nearest even, saturating
// Products, sums and the reciprocal are separate fp32 roundings (no fused
// multiply-add), so the codes are reproducible in plain fp32 arithmetic.
//
// Layouts with 16-byte granularity go to a kernel where a group of lanes shares
// a vector and moves 8 elements per access (below); others to one warp per
// vector with 4-byte accesses.  HBM bound: 3 bytes per element plus 4 per scale.
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
__device__ __forceinline__ void bf16x8_to_f(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
    f[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }
}

template <int G, int U>
__global__ void __launch_bounds__(kRopeWarps * 32)
    k_inv_rope_fp8_v8(const uint4* __restrict__ X, int T, int heads, int D, int R, const int32_t* __restrict__ pos,
                      const float4* __restrict__ cos_sin, int max_pos, uint2* __restrict__ Q,
                      float* __restrict__ scale, int* status) {
  pdl_enter();
  const int lane = threadIdx.x & 31, sub = lane % G, grp = lane / G;
  const int half = R / 2, nrot = R / 16, nunits = nrot + (D - R) / 8;
  const size_t nvec = (size_t)T * heads;
  constexpr int VPW = 32 / G;  // vectors per warp at a time
  const size_t step = (size_t)gridDim.x * kRopeWarps * VPW;
  // the 16-byte chunks of a unit: rotated (8 elements and their partners) or tail (8 elements)
  auto fetch = [&](size_t base, uint4 (&raw)[U][2], int& p) {
    const size_t v = base + grp;
    if (v >= nvec) return;
    p = __ldg(pos + v / heads);
    const uint4* xr = X + v * (D / 8);
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
  size_t base = ((size_t)blockIdx.x * kRopeWarps + (threadIdx.x >> 5)) * VPW;
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
    const size_t v = base + grp;
    const bool valid = v < nvec;
    const size_t vv = valid ? v : nvec - 1;
    if (p < 0 || p >= max_pos) {
      if (valid && sub == 0) report(status, MOE_ERR_DEVICE_INDEX);
      p = p < 0 ? 0 : max_pos - 1;
    }
    const float4* cs = cos_sin + (size_t)p * (R / 4);  // 4 floats per float4
    float ya[U][8], yb[U][8];
    float amax = 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int unit = sub + G * u;
      if (valid && unit < nunits) {
        if (unit < nrot) {
          float x1[8], x2[8];
          bf16x8_to_f(cur[u][0], x1);
          bf16x8_to_f(cur[u][1], x2);
          const float4 c0 = cs[2 * unit], c1 = cs[2 * unit + 1];
          const float4 s0 = cs[(half + 8 * unit) / 4], s1 = cs[(half + 8 * unit) / 4 + 1];
          const float co[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          const float si[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            ya[u][i] = __fadd_rn(__fmul_rn(x1[i], co[i]), __fmul_rn(x2[i], si[i]));
            yb[u][i] = __fsub_rn(__fmul_rn(x2[i], co[i]), __fmul_rn(x1[i], si[i]));
            amax = fmaxf(amax, fmaxf(fabsf(ya[u][i]), fabsf(yb[u][i])));
          }
        } else {
          bf16x8_to_f(cur[u][0], ya[u]);
#pragma unroll
          for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(ya[u][i]));
        }
      }
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = e4m3_scale_from_amax(amax);
    const float r = __fdiv_rn(1.0f, s);
    if (valid) {
      uint2* qr = Q + vv * (D / 8);  // 8 codes per uint2
      auto code8 = [&](const float (&y)[8]) -> uint2 {
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h)
          w[h] = (uint32_t)e4m3x2(__fmul_rn(y[4 * h], r), __fmul_rn(y[4 * h + 1], r)) |
                 ((uint32_t)e4m3x2(__fmul_rn(y[4 * h + 2], r), __fmul_rn(y[4 * h + 3], r)) << 16);
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
      if (sub == 0) scale[v] = s;
    }
  }
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
  if (vec16 && nunits > 0) {
    int G = 4;
    while (G < 32 && G < nunits) G *= 2;
    const int U = (nunits + G - 1) / G;
    const size_t per_block = (size_t)kRopeWarps * (32 / G);
    size_t blocks = (nvec + per_block - 1) / per_block;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
#define MOE_ROPE_CASE(GG, UU)                                                                                   \
  if (G == GG && U == UU) {                                                                                     \
    MOE_LAUNCH(k_inv_rope_fp8_v8<GG, UU>, dim3((unsigned)blocks), dim3(kRopeWarps * 32), 0, s, (const uint4*)X, T, \
               heads, D, R, pos, (const float4*)cos_sin, max_pos, (uint2*)Q, scale, status);                      \
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
