// fp32 grouped expert GEMMs on the CUDA cores (the fp32 layer; tcgen05 has no
// fp32-input kind that keeps a 1e-5 relative error).
//
// GEMM1: A[r][i] = SiLU(sum_h Xs[r][h] W13[e][i][h]) * (sum_h Xs[r][h] W13[e][I+i][h])
// GEMM2: Y[f][h] = sum_i A[r][i] W2[e][h][i],  f = sorted[r] (pair index)
// for every sorted row r of block b, e = eids[b]  ("FusedMoE vs MegaMoE",
// section 3.1: one launch computes every expert on its own rows).
#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kRows = 16;  // sorted rows per tile (= permutation block size of this path)
constexpr int kCols = 64;  // output columns per tile
constexpr int kKc = 32;    // reduction chunk

__global__ void __launch_bounds__(256) k_gemm1_simt(const float* __restrict__ Xs, const float* __restrict__ W13,
                                                    int H, int I, const int32_t* __restrict__ eids,
                                                    const int32_t* __restrict__ meta, float* __restrict__ A) {
  pdl_enter();
  __shared__ float xs[kRows][kKc + 1];
  __shared__ float wg[kCols][kKc + 1];
  __shared__ float wu[kCols][kKc + 1];
  const int b = blockIdx.x;
  if (b >= meta[META_NBLK]) return;
  const int e = eids[b];
  const int r0 = b * kRows, i0 = blockIdx.y * kCols;
  const int row = threadIdx.x / 16, cg = threadIdx.x % 16;
  const float* W = W13 + (size_t)e * 2 * I * H;
  float g[4] = {0, 0, 0, 0}, u[4] = {0, 0, 0, 0};
  for (int k0 = 0; k0 < H; k0 += kKc) {
    for (int idx = threadIdx.x; idx < kRows * kKc; idx += 256) {
      const int rr = idx / kKc, kk = idx % kKc;
      xs[rr][kk] = (k0 + kk < H) ? Xs[(size_t)(r0 + rr) * H + k0 + kk] : 0.0f;
    }
    for (int idx = threadIdx.x; idx < kCols * kKc; idx += 256) {
      const int c = idx / kKc, kk = idx % kKc;
      const bool in = (i0 + c < I) && (k0 + kk < H);
      wg[c][kk] = in ? W[(size_t)(i0 + c) * H + k0 + kk] : 0.0f;
      wu[c][kk] = in ? W[(size_t)(I + i0 + c) * H + k0 + kk] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKc; ++kk) {
      const float x = xs[row][kk];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        g[q] = fmaf(x, wg[cg * 4 + q][kk], g[q]);
        u[q] = fmaf(x, wu[cg * 4 + q][kk], u[q]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int i = i0 + cg * 4 + q;
    if (i < I) A[(size_t)(r0 + row) * I + i] = silu(g[q]) * u[q];
  }
}

__global__ void __launch_bounds__(256) k_gemm2_simt(const float* __restrict__ A, const float* __restrict__ W2,
                                                    int H, int I, int n_pairs, const int32_t* __restrict__ sorted,
                                                    const int32_t* __restrict__ eids,
                                                    const int32_t* __restrict__ meta, float* __restrict__ Y) {
  pdl_enter();
  __shared__ float as[kRows][kKc + 1];
  __shared__ float ws[kCols][kKc + 1];
  const int b = blockIdx.x;
  if (b >= meta[META_NBLK]) return;
  const int e = eids[b];
  const int r0 = b * kRows, h0 = blockIdx.y * kCols;
  const int row = threadIdx.x / 16, cg = threadIdx.x % 16;
  const float* W = W2 + (size_t)e * H * I;
  float y[4] = {0, 0, 0, 0};
  for (int k0 = 0; k0 < I; k0 += kKc) {
    for (int idx = threadIdx.x; idx < kRows * kKc; idx += 256) {
      const int rr = idx / kKc, kk = idx % kKc;
      as[rr][kk] = (k0 + kk < I) ? A[(size_t)(r0 + rr) * I + k0 + kk] : 0.0f;
    }
    for (int idx = threadIdx.x; idx < kCols * kKc; idx += 256) {
      const int c = idx / kKc, kk = idx % kKc;
      ws[c][kk] = (h0 + c < H && k0 + kk < I) ? W[(size_t)(h0 + c) * I + k0 + kk] : 0.0f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKc; ++kk) {
      const float a = as[row][kk];
#pragma unroll
      for (int q = 0; q < 4; ++q) y[q] = fmaf(a, ws[cg * 4 + q][kk], y[q]);
    }
    __syncthreads();
  }
  const int f = sorted[r0 + row];
  if (f >= n_pairs) return;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int h = h0 + cg * 4 + q;
    if (h < H) Y[(size_t)f * H + h] = y[q];
  }
}

}  // namespace

cudaError_t launch_gemm1_simt(const float* Xs, const float* W13, int H, int I, int B, const int32_t* eids,
                              const int32_t* meta, int cap, float* A, cudaStream_t s) {
  if (B != kRows) return cudaErrorInvalidValue;
  dim3 grid(cap / kRows, (I + kCols - 1) / kCols);
  MOE_LAUNCH(k_gemm1_simt, dim3(grid), dim3(256), 0, s, Xs, W13, H, I, eids, meta, A);
  return cudaGetLastError();
}

cudaError_t launch_gemm2_simt(const float* A, const float* W2, int H, int I, int B, int T, int k,
                              const int32_t* sorted, const int32_t* eids, const int32_t* meta, int cap, float* Y,
                              cudaStream_t s) {
  if (B != kRows) return cudaErrorInvalidValue;
  dim3 grid(cap / kRows, (H + kCols - 1) / kCols);
  MOE_LAUNCH(k_gemm2_simt, dim3(grid), dim3(256), 0, s, A, W2, H, I, T * k, sorted, eids, meta, Y);
  return cudaGetLastError();
}

}  // namespace moe
