// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// One persistent kernel covers every active expert of the layer in a single
// launch ("Mixture-of-Experts kernel engineering on Amazon SageMaker AI",
// intro: routing, data shuffle and expert networks as one batched GPU
// operation; "FusedMoE vs MegaMoE", section 3.2: the fused kernel must keep
// every SM busy although experts receive different token counts).
//
// Roles (192 threads):
//   warp 0      TMA producer: weight tile + sorted activation tile per
//               128-byte K block into a ring of shared-memory stages
//   warp 1      MMA issuer: tcgen05.mma into a tensor-memory accumulator
//               (two accumulators, so the epilogue of one tile overlaps the
//               main loop of the next)
//   warps 2-5   epilogue: tcgen05.ld -> registers -> scale / SiLU(gate)*up ->
//               global stores
//
// Orientation.  In swap-AB mode (thin decode batches) the MMA computes
// C^T[N,M] = B^T[N,K] A^T[K,M]: expert weight rows occupy the M slot and the
// expert's few tokens (padded to 16) the N slot, so no tensor-core row is
// spent on empty token rows (page 1, section "Swap-AB pour l'utilisation de
// WGMMA", Figure 1: the large expert N dimension moved into the fixed-size
// operand slot; Hopper's slot is 64 rows, tcgen05's is 128).  A swap-AB tile
// is 256 weight rows, issued as two M = 128 MMAs (accumulators D0 and D1)
// against one shared activation tile, so each stage's activation bytes serve
// twice the weight bytes.  In token-major mode (prefill) 128 sorted token rows
// fill M and 256 weight rows N.
//
// The weight tile is two TMA loads of `wbox` rows.  For GEMM1 they are the
// gate rows and the matching up rows, so SiLU(gate)*up pairs values held by
// one thread: TMEM lane i of D0 and D1 in swap-AB mode, columns c and wbox+c
// in token-major mode.
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

namespace {

constexpr int kTcThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kTileQueue = 8;   // claimed-tile slots between the producer and the other roles
constexpr int kClaimMinWaves = 4;  // claim tiles only from this many waves of them
constexpr uint32_t kTmemCols = 512;  // all of tensor memory: accumulator buffers

struct TcDev {
  int epi;
  int T, k, E, I, H;
  int kb_total, kb_per_split, splits, n_tiles;
  int w_rows_per_expert, w_pair_off, w_tile_rows, wbox, xbox;
  int stages;
  int gather;       // 1: activation rows gathered by token from an unsorted [T][K] tensor
  int early;        // 1: the tile list may be read and weights streamed before the dependency wait
  int nbuf;         // accumulator buffers (2: epilogue of one tile overlaps the next; 1 for wide swap tiles)
  int buf_cols;     // tensor-memory columns per buffer
  int d1_col;       // swap-AB: column of accumulator D1 (weight rows 128..255) inside a buffer
  int n_valid;      // router: valid output columns
  int x_lo_rows;    // >0: the activation operand also has a bf16 low part at row offset x_lo_rows
  int tm_rows;      // token-major: sorted rows per tile (128; 256 on CTA pairs)
  int prefetch_kb;  // swap-AB GEMM1: K blocks of this CTA's first tile to prefetch into L2 before the
                    // dependency wait, guessing that every expert is active (0: none)
  int stack_lo;     // swap-AB GEMM2 with a hi/lo activation: one MMA over the hi rows then the lo rows
                    // (N = xbox + npad), the two column groups summed in the epilogue
  uint32_t stage_bytes, w_bytes, bar_off;
  const int32_t* pblk;    // CTA pairs: tile chunks (first row << 1 | 1 for a 128-row chunk)
  unsigned* fin;          // nullable (bf16 split GEMM1): per-(expert, weight tile) arrival counters,
                          // zeroed by the permutation kernel; the CTA storing a tile's last split
                          // sums the splits and writes the intermediate (out_fin, out_fin_lo)
  void* out_fin;
  void* out_fin_lo;
  const unsigned* ready;  // nullable: expert e's weights are streamed once ready[e] == want[e]
  const unsigned* want;
  int* claim;             // nullable: tiles past the first wave may be claimed from this counter
  int* zero_word;         // nullable: set to 0 after the dependency wait (the next GEMM's counter)
  const int32_t* sorted;
  const int32_t* eids;
  const int32_t* meta;
  void* out;
  void* out_lo;     // GEMM1: low bf16 part of the intermediate (nullable)
  size_t out_split_stride;
  const float* w_scale;
  const unsigned* a_amax;
  unsigned* amax_out;
  int* status;
};

struct Tile {
  int e, xrow, ntok, npad, wr0, kb0, kb1, n, s;
};

template <bool SWAP, int EPI>
__device__ __forceinline__ int tile_count(const TcDev& p) {
  if constexpr (EPI == TC_EPI_LOGITS)
    return (p.T + 127) / 128 * p.n_tiles;
  else if constexpr (SWAP)
    return p.meta[META_NACT] * p.n_tiles * p.splits;
  else
    return (p.meta[META_NPP] / p.tm_rows) * p.n_tiles;
}

template <bool SWAP, int EPI>
__device__ __forceinline__ Tile tile_at(const TcDev& p, int t) {
  Tile d;
  if constexpr (EPI == TC_EPI_LOGITS) {
    // router: 128 consecutive (unsorted) tokens against the experts of column tile n
    // (2 wbox experts from n * w_tile_rows; the column tiles of a token tile are adjacent
    // in t, so its second read of the tokens comes from L2)
    d.n = t % p.n_tiles;
    d.s = 0;
    d.e = 0;
    d.xrow = (t / p.n_tiles) * 128;
    d.ntok = 128;
    d.npad = 128;
    d.kb0 = 0;
    d.kb1 = p.kb_total;
    d.wr0 = d.n * p.w_tile_rows;
    return d;
  } else if constexpr (SWAP) {
    const int per_e = p.n_tiles * p.splits;
    const int a = t / per_e;
    const int rem = t - a * per_e;
    d.n = rem / p.splits;
    d.s = rem - d.n * p.splits;
    d.e = p.meta[meta_active(p.E) + a];
    d.xrow = p.meta[meta_offsets(p.E) + d.e];
    d.ntok = p.meta[meta_counts(p.E) + d.e];
    d.npad = (d.ntok + 15) & ~15;
    d.kb0 = d.s * p.kb_per_split;
    d.kb1 = min(d.kb0 + p.kb_per_split, p.kb_total);
  } else {
    const int m = t / p.n_tiles;
    d.n = t - m * p.n_tiles;
    d.s = 0;
    d.e = p.eids[m];
    d.xrow = m * p.tm_rows;
    d.ntok = p.tm_rows;
    d.npad = p.tm_rows;
    d.kb0 = 0;
    d.kb1 = p.kb_total;
  }
  d.wr0 = d.e * p.w_rows_per_expert + d.n * p.w_tile_rows;
  return d;
}

// OR of a flag over the 128 epilogue threads (named barrier 1).
__device__ __forceinline__ bool epi_any(bool v) { return named_bar_any(1, 128, v); }

// The epilogue of one finished tile: thread lrow (an accumulator row, TMEM
// lane) reads its accumulator columns from tensor memory at tb and stores them
// in the tile's output format.
template <bool SWAP, bool FP8, int EPI>
__device__ __forceinline__ void epi_tile(const TcDev& p, const Tile& d, uint32_t tb, int lrow, float scale,
                                         int n_pairs, float& amax, volatile int* sm_word = nullptr) {
  if constexpr (SWAP && (EPI == TC_EPI_G1_BF16 || EPI == TC_EPI_G1_F32AMAX)) {
    // lane r of D0 / D1: gate / up of intermediate column i = n*128 + r, one column per token
    const int i = d.n * 128 + lrow;
    for (int c0 = 0; c0 < d.npad; c0 += 16) {
      float g[16], u[16];
      tmem_ld16(tb + (uint32_t)c0, g);
      tmem_ld16(tb + (uint32_t)(p.d1_col + c0), u);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        if (c < d.ntok) {
          const float a = silu(g[j] * scale) * (u[j] * scale);
          const size_t o = (size_t)(d.xrow + c) * p.I + i;
          if constexpr (EPI == TC_EPI_G1_BF16) {
            const __nv_bfloat16 hi = __float2bfloat16_rn(a);
            reinterpret_cast<__nv_bfloat16*>(p.out)[o] = hi;
            if (p.out_lo)
              reinterpret_cast<__nv_bfloat16*>(p.out_lo)[o] = __float2bfloat16_rn(a - __bfloat162float(hi));
          } else {
            reinterpret_cast<float*>(p.out)[o] = a;
            amax = fmaxf(amax, fabsf(a));
          }
        }
      }
    }
  } else if constexpr (SWAP && EPI == TC_EPI_G1_PART) {
    // raw fp32 split partials P[s][pair][col]: gate at col i, up at col I + i
    const int i = d.n * 128 + lrow;
    float* P = reinterpret_cast<float*>(p.out) + (size_t)d.s * p.out_split_stride;
    for (int c0 = 0; c0 < d.npad; c0 += 16) {
      float g[16], u[16];
      tmem_ld16(tb + (uint32_t)c0, g);
      tmem_ld16(tb + (uint32_t)(p.d1_col + c0), u);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (c0 + j < d.ntok) {
          float* row = P + (size_t)p.sorted[d.xrow + c0 + j] * (2 * p.I);
          row[i] = g[j];
          row[p.I + i] = u[j];
        }
      }
    }
    if constexpr (!FP8) {
      if (p.fin) {
        // Last arriver: once all 128 columns of this split are stored, count it; the
        // CTA bringing the tile's last split sums the splits in split order from 0,
        // then SiLU(gate)*up into the bf16 (hi, lo) intermediate -- the arithmetic of
        // the split-reduction kernel, so the results are the same bit for bit.
        // (sm_word: a shared-memory word of the CTA for the decision)
        named_bar_sync(1, 128);
        if (lrow == 0) {
          __threadfence();
          *sm_word = atomicAdd(p.fin + d.e * p.n_tiles + d.n, 1u) == (unsigned)(p.splits - 1);
        }
        named_bar_sync(1, 128);
        if (*sm_word) {
          __threadfence();
          const float* P0 = reinterpret_cast<const float*>(p.out);
          for (int c = 0; c < d.ntok; ++c) {
            const float* row = P0 + (size_t)p.sorted[d.xrow + c] * (2 * p.I);
            float g = 0.0f, u = 0.0f;
            for (int sp = 0; sp < p.splits; ++sp) {
              g += __ldcg(row + (size_t)sp * p.out_split_stride + i);
              u += __ldcg(row + (size_t)sp * p.out_split_stride + p.I + i);
            }
            const float a = silu(g) * u;
            const size_t o = (size_t)(d.xrow + c) * p.I + i;
            const __nv_bfloat16 hi = __float2bfloat16_rn(a);
            reinterpret_cast<__nv_bfloat16*>(p.out_fin)[o] = hi;
            if (p.out_fin_lo)
              reinterpret_cast<__nv_bfloat16*>(p.out_fin_lo)[o] = __float2bfloat16_rn(a - __bfloat162float(hi));
          }
        }
      }
    }
  } else if constexpr (SWAP && EPI == TC_EPI_G2_F32) {
    // Y[s][pair][h]: h = n*256 + r (D0) and n*256 + 128 + r (D1), pair = sorted[xrow + c]
    const int h0 = d.n * 256 + lrow;
    const bool h1_ok = h0 + 128 < p.H;
    float* Y = reinterpret_cast<float*>(p.out) + (size_t)d.s * p.out_split_stride;
    for (int c0 = 0; c0 < d.npad; c0 += 16) {
      float v0[16], v1[16];
      tmem_ld16(tb + (uint32_t)c0, v0);
      tmem_ld16(tb + (uint32_t)(p.d1_col + c0), v1);
      if (p.stack_lo) {  // + the low part's products, xbox columns further on
        float l0[16], l1[16];
        tmem_ld16(tb + (uint32_t)(p.xbox + c0), l0);
        tmem_ld16(tb + (uint32_t)(p.d1_col + p.xbox + c0), l1);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          v0[j] += l0[j];
          v1[j] += l1[j];
        }
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        if (c < d.ntok) {
          float* row = Y + (size_t)p.sorted[d.xrow + c] * p.H;
          row[h0] = v0[j] * scale;
          if (h1_ok) row[h0 + 128] = v1[j] * scale;
        }
      }
    }
  } else if constexpr (!SWAP && (EPI == TC_EPI_G1_BF16 || EPI == TC_EPI_G1_F32AMAX)) {
    // row = xrow + lrow; columns [0, wbox) gate, [wbox, 2 wbox) up of i = n*wbox + c
    const size_t row = (size_t)(d.xrow + lrow);
    const bool row_valid = p.sorted[row] < n_pairs;
    for (int c0 = 0; c0 < p.wbox; c0 += 16) {
      float g[16], u[16];
      tmem_ld16(tb + (uint32_t)c0, g);
      tmem_ld16(tb + (uint32_t)(p.wbox + c0), u);
      float a[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) a[j] = silu(g[j] * scale) * (u[j] * scale);
      const size_t o = row * p.I + (size_t)d.n * p.wbox + c0;
      if constexpr (EPI == TC_EPI_G1_BF16) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o);
        uint32_t hv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[j] = pack_bf16x2(a[2 * j], a[2 * j + 1]);
        dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        if (p.out_lo) {
          uint32_t lv[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            lv[j] = pack_bf16x2(a[2 * j] - bf16_bits_to_f32(hv[j] & 0xffffu),
                                a[2 * j + 1] - bf16_bits_to_f32(hv[j] >> 16));
          uint4* dl = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out_lo) + o);
          dl[0] = make_uint4(lv[0], lv[1], lv[2], lv[3]);
          dl[1] = make_uint4(lv[4], lv[5], lv[6], lv[7]);
        }
      } else {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_float4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
        if (row_valid) {  // padding rows hold token 0's values: keep them out of the amax
#pragma unroll
          for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(a[j]));
        }
      }
    }
  } else if constexpr (EPI == TC_EPI_LOGITS) {
    const int row = d.xrow + lrow;
    const int ncols = 2 * p.wbox;
    const int col0 = d.n * ncols;  // first expert of this column tile
    for (int c0 = 0; c0 < ncols; c0 += 16) {
      float v[16];
      tmem_ld16(tb + (uint32_t)c0, v);
      if (row < p.T) {
        float* dst = reinterpret_cast<float*>(p.out) + (size_t)row * p.n_valid + col0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (col0 + c0 + j < p.n_valid) dst[c0 + j] = v[j];
      }
    }
  } else if constexpr (!SWAP && EPI == TC_EPI_G2_F32) {
    // fp32 rows of Y: read in the 16x256b shape, thread t has two adjacent columns of
    // rows t/4 and 8 + t/4 (of each 16-lane half of the warp's quadrant) per 8-column
    // group; one exchange with the neighbouring thread leaves 4 adjacent columns of one
    // row in each thread, so a store instruction writes 32 contiguous bytes of each of
    // 16 rows instead of 16 bytes of each of 32
    const int ln = lrow & 31;
    const bool odd = (ln & 1) != 0;
    const int ncols = 2 * p.wbox;
    const int cofs = (ln & 2) * 2;  // first of the 4 columns this thread stores in a group
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = (lrow & ~31) + 16 * h + (ln >> 2) + (odd ? 8 : 0);
      const int f = p.sorted[d.xrow + row];
      float* dst = reinterpret_cast<float*>(p.out) + (size_t)(f < n_pairs ? f : 0) * p.H + (size_t)d.n * ncols + cofs;
      for (int c0 = 0; c0 < ncols; c0 += 32) {
        float v[16];
        tmem_ld_16x256b_x4(tb + ((uint32_t)(16 * h) << 16) + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float s0 = odd ? v[4 * j] : v[4 * j + 2];  // the pair the neighbour stores
          const float s1 = odd ? v[4 * j + 1] : v[4 * j + 3];
          const float r0 = __shfl_xor_sync(0xffffffffu, s0, 1);
          const float r1 = __shfl_xor_sync(0xffffffffu, s1, 1);
          const float4 o = odd ? make_float4(r0 * scale, r1 * scale, v[4 * j + 2] * scale, v[4 * j + 3] * scale)
                               : make_float4(v[4 * j] * scale, v[4 * j + 1] * scale, r0 * scale, r1 * scale);
          if (f < n_pairs) *reinterpret_cast<float4*>(dst + c0 + 8 * j) = o;
        }
      }
    }
  } else if constexpr (!SWAP && EPI == TC_EPI_G2_BF16) {
    const int f = p.sorted[d.xrow + lrow];
    const int ncols = 2 * p.wbox;
    for (int c0 = 0; c0 < ncols; c0 += 16) {
      float v[16];
      tmem_ld16(tb + (uint32_t)c0, v);
      if (f < n_pairs) {
        const size_t o = (size_t)f * p.H + (size_t)d.n * ncols + c0;
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o);
        dst[0] = make_uint4(pack_bf16x2(v[0] * scale, v[1] * scale), pack_bf16x2(v[2] * scale, v[3] * scale),
                            pack_bf16x2(v[4] * scale, v[5] * scale), pack_bf16x2(v[6] * scale, v[7] * scale));
        dst[1] = make_uint4(pack_bf16x2(v[8] * scale, v[9] * scale), pack_bf16x2(v[10] * scale, v[11] * scale),
                            pack_bf16x2(v[12] * scale, v[13] * scale), pack_bf16x2(v[14] * scale, v[15] * scale));
      }
    }
  }
}

template <bool SWAP, bool FP8, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmX16, const TcDev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.bar_off;
  const uint32_t bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t bar_tfull = bar_empty + 8 * kMaxStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_exit = bar_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (2 * kMaxStages + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // claimed tiles: the producer publishes each tile index (or the end) in a ring of
  // kTileQueue slots read by the MMA warp and the four epilogue warps
  const uint32_t bar_tq_full = bar_full + 8 * (2 * kMaxStages + 6) + 16;
  const uint32_t bar_tq_empty = bar_tq_full + 8 * kTileQueue;
  volatile int* tq = reinterpret_cast<volatile int*>(smem + p.bar_off + 8 * (2 * kMaxStages + 6) + 16 + 16 * kTileQueue);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int q = 0; q < kTileQueue; ++q) {
      mbar_init(bar_tq_full + 8 * q, 1);
      mbar_init(bar_tq_empty + 8 * q, 1 + 4);  // the MMA warp and the four epilogue warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 128);
    }  // (buffer 1 unused when nbuf == 1)
    mbar_init(bar_drain, 1);
    mbar_init(bar_exit, kTcThreads / 32);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    if (SWAP) tma_prefetch_desc(&tmX16);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if constexpr (SWAP && EPI != TC_EPI_LOGITS) {
    // While routing still runs, HBM is idle: when every expert is almost surely active
    // (the host sets prefetch_kb only then), the tile list is the identity over experts
    // and this CTA's first tile is known; its first K blocks go to L2 as a hint.  A wrong
    // guess only costs idle bandwidth.
    if (p.prefetch_kb > 0 && !p.early && threadIdx.x == 0) {
      const int per_e = p.n_tiles * p.splits;
      const int t = blockIdx.x;
      const int e = t / per_e;
      if (e < p.E) {
        const int rem = t - e * per_e;
        const int n = rem / p.splits, sp = rem - n * p.splits;
        const int wr0 = e * p.w_rows_per_expert + n * p.w_tile_rows;
        const int kb0 = sp * p.kb_per_split, kb1 = min(kb0 + min(p.kb_per_split, p.prefetch_kb), p.kb_total);
        for (int kb = kb0; kb < kb1; ++kb) {
          tma_prefetch_l2(&tmW, kb * (FP8 ? 128 : 64), wr0);
          tma_prefetch_l2(&tmW, kb * (FP8 ? 128 : 64), wr0 + p.w_pair_off);
        }
      }
    }
  }
  // Programmatic dependent launch: kernels of this library let their
  // dependents launch early, so nothing written by an earlier kernel may be
  // read before pdl_wait() -- except when the host sets `early`: for GEMM2
  // (launched only after GEMM1 has itself passed its wait, so the permutation
  // metadata is complete), for a GEMM1 behind a row gather that lets its
  // dependents launch only after its own wait (the same guarantee), and for the
  // router GEMM (which reads none).
  if (!p.early) pdl_wait();
  const int ntiles = tile_count<SWAP, EPI>(p);
  // Tiles past each CTA's first are claimed from a counter when there are at least
  // kClaimMinWaves waves of them: SMs that stream faster then take more tiles (FP8 decode
  // at 16 tokens, 5.8 waves: 886 against 910 us).  With fewer waves the static schedule
  // measured faster (fine-grained decode at 32 and 64 tokens, 2.1-2.7 waves).
  const bool claim = p.claim != nullptr && ntiles >= kClaimMinWaves * (int)gridDim.x;
  constexpr int KBLK = FP8 ? 128 : 64;  // elements per 128-byte K block

  if (warp == 0) {
    // ---------------- TMA producer (warp 0) ----------------
    // The warp waits for free stages together; lane 0 arms their barriers and
    // loads the weight tiles.  The activation tile is either one tiled load of consecutive
    // sorted rows (lane 0), or -- when the activations are gathered -- one
    // tile::gather4 load per group of 4 rows, issued by the 32 lanes in
    // parallel with the token row of each sorted (token, slot) pair.
    //
    // Expert weights do not depend on the preceding kernel: lane 0 streams the
    // first stages of weight tiles before waiting for it (programmatic
    // dependent launch), so this kernel's HBM stream starts while the previous
    // one drains.
    //
    // Swap-AB tiles load only the token rows the MMA reads (N = npad): gathered
    // tiles npad rows, pre-gathered ones a 16-row box when npad is 16, else the
    // full activation box.
    const int parts = p.x_lo_rows ? 2 : 1;
    auto x_rows = [&](const Tile& d) -> int {
      if constexpr (SWAP) return p.gather ? d.npad : (d.npad <= 16 ? 16 : p.xbox);
      return p.xbox;
    };
    auto stage_tx = [&](const Tile& d) -> uint32_t {
      return p.w_bytes + (uint32_t)(x_rows(d) * 128 * parts);
    };
    int pre = 0;
    if (p.early && !p.ready && lane == 0 && (int)blockIdx.x < ntiles) {
      const Tile d = tile_at<SWAP, EPI>(p, blockIdx.x);
      pre = min(p.stages, d.kb1 - d.kb0);
      for (int i = 0; i < pre; ++i) {
        const uint32_t sw = sbase + i * p.stage_bytes;
        const uint32_t fb = bar_full + 8 * i;
        mbar_arrive_expect_tx(fb, stage_tx(d));
        tma_load_2d(sw, &tmW, (d.kb0 + i) * KBLK, d.wr0, fb);
        tma_load_2d(sw + p.wbox * 128, &tmW, (d.kb0 + i) * KBLK, d.wr0 + p.w_pair_off, fb);
      }
    }
    pre = __shfl_sync(0xffffffffu, pre, 0);
    pdl_wait();
    if (p.zero_word && blockIdx.x == 0 && lane == 0) *p.zero_word = 0;
    const int n_pairs = p.T * p.k;
    const int npp = (EPI == TC_EPI_LOGITS) ? 0 : p.meta[META_NPP];
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int i = 0, t = blockIdx.x; ok; ++i) {
      if (claim) {
        // the first tile is blockIdx.x (its weights may already be on their way)
        if (i > 0) {
          int c = 0;
          if (lane == 0) c = atomicAdd(p.claim, 1);
          t = (int)gridDim.x + __shfl_sync(0xffffffffu, c, 0);
        }
        const int slot = i % kTileQueue;
        if (i >= kTileQueue &&
            !mbar_wait_all(bar_tq_empty + 8 * slot, ((uint32_t)(i / kTileQueue) & 1u) ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          tq[slot] = t;
          mbar_arrive(bar_tq_full + 8 * slot);
        }
        __syncwarp();
      } else if (i > 0) {
        t += gridDim.x;
      }
      if (t >= ntiles) break;
      const Tile d = tile_at<SWAP, EPI>(p, t);
      // expert cache: this expert's weights may still be on their way into its slot
      if (p.ready && !wait_word_all(p.ready + d.e, p.want[d.e], abort_flag, p.status)) {
        ok = false;
        break;
      }
      int rows[2][4];  // token rows of this lane's gather groups g = lane and lane + 32
      if (p.gather) {
#pragma unroll
        for (int gi = 0; gi < 2; ++gi)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = d.xrow + 4 * (lane + 32 * gi) + i;
            const int f = (r < npp) ? p.sorted[r] : n_pairs;
            rows[gi][i] = (f < n_pairs) ? f / p.k : 0;  // padding rows read token 0; never stored
          }
      }
      for (int kb = d.kb0; kb < d.kb1; ++kb) {
        const uint32_t sw = sbase + stage * p.stage_bytes;
        const uint32_t fb = bar_full + 8 * stage;
        if ((int)issued >= pre) {  // (the first `pre` stages already hold their weight tiles)
          if (!mbar_wait_all(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(fb, stage_tx(d));
            tma_load_2d(sw, &tmW, kb * KBLK, d.wr0, fb);
            tma_load_2d(sw + p.wbox * 128, &tmW, kb * KBLK, d.wr0 + p.w_pair_off, fb);
          }
          __syncwarp();
        }
        if (p.gather) {
          const int groups_d = x_rows(d) / 4;
#pragma unroll
          for (int gi = 0; gi < 2; ++gi) {
            const int g = lane + 32 * gi;
            if (g < groups_d)
              tma_gather4(sw + p.w_bytes + (uint32_t)g * 512u, &tmX, kb * KBLK, rows[gi][0], rows[gi][1],
                          rows[gi][2], rows[gi][3], fb);
          }
        } else if (SWAP && x_rows(d) == 16 && p.xbox > 16) {
          if (lane == 0) {
            tma_load_2d(sw + p.w_bytes, &tmX16, kb * KBLK, d.xrow, fb);
            if (p.x_lo_rows)
              tma_load_2d(sw + p.w_bytes + p.xbox * 128, &tmX16, kb * KBLK, d.xrow + p.x_lo_rows, fb);
          }
        } else if (lane == 0) {
          tma_load_2d(sw + p.w_bytes, &tmX, kb * KBLK, d.xrow, fb);
          if (p.x_lo_rows) tma_load_2d(sw + p.w_bytes + p.xbox * 128, &tmX, kb * KBLK, d.xrow + p.x_lo_rows, fb);
        }
        __syncwarp();
        ++issued;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) {
      // every load of this CTA is issued: the next kernel may start its prologue
      pdl_launch_dependents();
      if (!ok) {  // let the copies already in flight land before the CTA exits
        const uint32_t first = issued > (uint32_t)p.stages ? issued - p.stages : 0u;
        for (uint32_t i = first; i < issued; ++i)
          mbar_wait_drain(bar_full + 8 * (i % p.stages), (i / p.stages) & 1u, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // The whole warp runs the loop and waits together; lane 0 issues the MMAs
    // and their commits (a commit tracks the MMAs of its own thread).
    pdl_wait();
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true, any = false;
    for (int i = 0, t = blockIdx.x; ok; ++i) {
      if (claim) {
        const int slot = i % kTileQueue;
        if (!mbar_wait_all(bar_tq_full + 8 * slot, (uint32_t)(i / kTileQueue) & 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        t = tq[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tq_empty + 8 * slot);
      } else if (i > 0) {
        t += gridDim.x;
      }
      if (t >= ntiles) break;
      const Tile d = tile_at<SWAP, EPI>(p, t);
      // (stacked hi/lo: the B rows are the xbox hi rows, then the lo rows, all in one MMA)
      const int N = SWAP ? (p.stack_lo ? p.xbox + d.npad : d.npad) : 2 * p.wbox;
      const uint32_t idesc = idesc_make(128, N, FP8);
      if (!mbar_wait_all(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + (uint32_t)(acc * p.buf_cols);
      for (int kb = d.kb0; kb < d.kb1; ++kb) {
        if (!mbar_wait_all(bar_full + 8 * stage, phase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sw = sbase + stage * p.stage_bytes;
          const uint32_t sx = sw + p.w_bytes;
          // the optional low bf16 part of the activations goes into the same fp32
          // accumulator: W (x_hi + x_lo) carries ~16 significant bits of the intermediate
          const int parts = (p.x_lo_rows && !p.stack_lo) ? 2 : 1;
          for (int part = 0; part < parts; ++part) {
            const uint32_t sxp = sx + (uint32_t)(part * p.xbox * 128);
            if constexpr (SWAP) {
              // D0 += W[rows 0..127] X^T, D1 += W[rows 128..255] X^T
              const uint32_t w1 = sw + (uint32_t)(p.wbox * 128);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc_in = (part > 0 || kb > d.kb0 || kk > 0) ? 1u : 0u;
                const uint64_t bdesc = sdesc_k_sw128(sxp + kk * 32);
                tc_mma<FP8>(dt, sdesc_k_sw128(sw + kk * 32), bdesc, idesc, acc_in);
                tc_mma<FP8>(dt + (uint32_t)p.d1_col, sdesc_k_sw128(w1 + kk * 32), bdesc, idesc, acc_in);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                tc_mma<FP8>(dt, sdesc_k_sw128(sxp + kk * 32), sdesc_k_sw128(sw + kk * 32), idesc,
                            (part > 0 || kb > d.kb0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(bar_empty + 8 * stage);
        }
        __syncwarp();
        any = true;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar_tfull + 8 * acc);
      __syncwarp();
      if (++acc == p.nbuf) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && any) {  // the tensor core must be idle before tensor memory is freed
      if (lane == 0) tc_commit(bar_drain);
      __syncwarp();
      mbar_wait_drain(bar_drain, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    pdl_wait();
    const int q = warp & 3;        // tensor-memory lane quadrant this warp may read
    const int lrow = q * 32 + lane; // accumulator row of this thread
    float a_scale = 1.0f;
    if constexpr (FP8) a_scale = e4m3_scale_from_amax(__uint_as_float(*p.a_amax));
    float amax = 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int n_pairs = p.T * p.k;
    for (int i = 0, t = blockIdx.x;; ++i) {
      if (claim) {
        const int slot = i % kTileQueue;
        const bool okq = mbar_wait_all(bar_tq_full + 8 * slot, (uint32_t)(i / kTileQueue) & 1u, abort_flag, p.status);
        if (epi_any(!okq)) break;
        t = tq[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tq_empty + 8 * slot);
      } else if (i > 0) {
        t += gridDim.x;
      }
      if (t >= ntiles) break;
      const Tile d = tile_at<SWAP, EPI>(p, t);
      const bool ok = mbar_wait_all(bar_tfull + 8 * acc, acc_phase, abort_flag, p.status);
      if (epi_any(!ok)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.buf_cols);
      const float scale = FP8 ? a_scale * p.w_scale[d.e] : 1.0f;

      epi_tile<SWAP, FP8, EPI>(p, d, tb, lrow, scale, n_pairs, amax,
                               reinterpret_cast<volatile int*>(tmem_slot + 2));
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == p.nbuf) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (EPI == TC_EPI_G1_F32AMAX) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (lane == 0 && amax > 0.0f) atomicMax(p.amax_out, __float_as_uint(amax));
    }
  }

  // Each warp reports the end of its role on an mbarrier; warp 1 frees tensor
  // memory once every warp has.  (A CTA-wide bar.sync here, reached by warps
  // coming out of different roles, was seen to release before all warps had
  // arrived.)
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_exit);
  if (warp == 1) {
    mbar_wait_drain(bar_exit, 0, 2 * kWaitLimitNs);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Token-major grouped GEMM on CTA pairs (tcgen05 cta_group::2)
// ---------------------------------------------------------------------------
// A cluster of two CTAs computes a tile of 256 sorted token rows x 256 weight
// rows.  CTA r stages token rows [128r, 128r + 128) of the tile and weight box r
// (GEMM1: the 128 gate rows, then the matching 128 up rows; GEMM2: rows
// [128r, 128r + 128) of the 256) in its own shared memory.  CTA 0 issues one
// M = 256, N = 256 MMA per K step; it reads both CTAs' halves and leaves each
// CTA's 128 token rows x 256 columns of the result in that CTA's tensor memory,
// so the epilogue pairs gate and up exactly as the single-CTA tile does.
// The permutation pads experts to 128 rows; an expert with an odd number of
// 128-row blocks ends in a 128-row tile, run as M = 128 MMAs: CTA r stages token
// rows [64r, 64r + 64), and the result lands in CTA r's tensor memory as row
// 64r + (lane mod 64) with columns 0-127 of N in lanes 0-63 and 128-255 in lanes
// 64-127.  For GEMM1 each CTA's weight half is then 64 gate rows followed by the
// matching 64 up rows, so gate and up of a column still meet in one thread.  Per 64-element K block an
// SM now writes and reads 32 KB of operands instead of 48 KB: the shared-memory
// bandwidth that bounds the single-CTA token-major tile ("FusedMoE vs
// MegaMoE", section 3.2: weight tiles staged in shared memory, every SM busy).
// Synchronisation: full[s] lives in CTA 0 and counts both CTAs' TMA bytes;
// empty[s] and tfull[b] live in both CTAs and are signalled by CTA 0's commits;
// tempty[b] in CTA 0 takes one arrival per epilogue warp of either CTA.
// Every wait is bounded; both CTAs meet at a cluster barrier before freeing
// tensor memory and exiting.
constexpr int kPairEpiArrivals = 8;  // epilogue warps of both CTAs

// CTA-pair tile t: chunk t / n_tiles of the permutation (256 rows, or 128 for an
// expert's last odd block: tail), weight tile t % n_tiles.
__device__ __forceinline__ Tile pair_tile_at(const TcDev& p, int t, bool& tail) {
  Tile d;
  const int c = t / p.n_tiles;
  d.n = t - c * p.n_tiles;
  d.s = 0;
  const int v = p.pblk[c];
  d.xrow = v >> 1;
  tail = (v & 1) != 0;
  d.e = p.eids[d.xrow / 128];
  d.ntok = d.npad = tail ? 128 : 256;
  d.kb0 = 0;
  d.kb1 = p.kb_total;
  d.wr0 = d.e * p.w_rows_per_expert + d.n * p.w_tile_rows;
  return d;
}

// Epilogue of a 128-row tail tile on a CTA pair: this thread's tensor-memory lane
// holds row 64 * rank + (lrow mod 64) of the tile and the half lrow / 64 of N.
template <bool FP8, int EPI>
__device__ __forceinline__ void epi_pair_tail(const TcDev& p, const Tile& d, uint32_t tb, int lrow, uint32_t rank,
                                              float scale, int n_pairs, float& amax) {
  const int hf = lrow >> 6;
  const size_t row = (size_t)(d.xrow + 64 * (int)rank + (lrow & 63));
  if constexpr (EPI == TC_EPI_G1_BF16 || EPI == TC_EPI_G1_F32AMAX) {
    // columns [0, 64): gate of intermediate column i = n*128 + 64*hf + c; [64, 128): its up
    const bool row_valid = p.sorted[row] < n_pairs;
    for (int c0 = 0; c0 < 64; c0 += 16) {
      float g[16], u[16];
      tmem_ld16(tb + (uint32_t)c0, g);
      tmem_ld16(tb + (uint32_t)(64 + c0), u);
      float a[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) a[j] = silu(g[j] * scale) * (u[j] * scale);
      const size_t o = row * p.I + (size_t)d.n * 128 + (size_t)(64 * hf + c0);
      if constexpr (EPI == TC_EPI_G1_BF16) {
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) + o);
        uint32_t hv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) hv[j] = pack_bf16x2(a[2 * j], a[2 * j + 1]);
        dst[0] = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        dst[1] = make_uint4(hv[4], hv[5], hv[6], hv[7]);
      } else {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o);
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = make_float4(a[4 * j], a[4 * j + 1], a[4 * j + 2], a[4 * j + 3]);
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(a[j]));
        }
      }
    }
  } else {
    // fp32 Y row of pair sorted[row], columns h = n*256 + 128*hf + c
    const int f = p.sorted[row];
    for (int c0 = 0; c0 < 128; c0 += 16) {
      float v[16];
      tmem_ld16(tb + (uint32_t)c0, v);
      if (f < n_pairs) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + (size_t)f * p.H +
                                                (size_t)d.n * 256 + (size_t)(128 * hf + c0));
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dst[j] = make_float4(v[4 * j] * scale, v[4 * j + 1] * scale, v[4 * j + 2] * scale, v[4 * j + 3] * scale);
      }
    }
  }
}

template <bool FP8, int EPI>
__global__ void __launch_bounds__(kTcThreads, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmW64, const __grid_constant__ CUtensorMap tmX64, const TcDev p) {
  constexpr bool G1 = EPI != TC_EPI_G2_F32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.bar_off;
  const uint32_t bar_empty = bar_full + 8 * kMaxStages;
  const uint32_t bar_tfull = bar_empty + 8 * kMaxStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (2 * kMaxStages + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, kPairEpiArrivals);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW64);
    tma_prefetch_desc(&tmX64);
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  cta_sync();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (!p.early) pdl_wait();
  const int ntiles = p.meta[META_NPB] * p.n_tiles;
  constexpr int KBLK = FP8 ? 128 : 64;  // elements per 128-byte K block
  const uint32_t half_bytes = 128u * 128u;  // a 128-row box of 128 bytes

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    // Each CTA loads its weight box and its token rows; completion is counted on
    // CTA 0's full barrier, which CTA 0 arms for both CTAs' bytes.
    const uint32_t wrow_off = rank ? (uint32_t)p.w_pair_off : 0u;
    // this CTA's weight half of one K block: GEMM1 tail tiles take 64 gate rows and
    // the matching 64 up rows, every other tile one 128-row box
    auto load_w = [&](uint32_t sw, const Tile& d, bool tail, int kb, uint32_t fb0) {
      if (G1 && tail) {
        tma_load_2d_pair(sw, &tmW64, kb * KBLK, d.wr0 + 64 * (int)rank, fb0);
        tma_load_2d_pair(sw + half_bytes / 2, &tmW64, kb * KBLK, d.wr0 + p.w_pair_off + 64 * (int)rank, fb0);
      } else {
        tma_load_2d_pair(sw, &tmW, kb * KBLK, d.wr0 + (int)wrow_off, fb0);
      }
    };
    int pre = 0;
    if (p.early && lane == 0 && pair < ntiles) {
      bool tail;
      const Tile d = pair_tile_at(p, pair, tail);
      pre = min(p.stages, d.kb1 - d.kb0);
      for (int i = 0; i < pre; ++i) {
        const uint32_t fb = bar_full + 8 * i;
        if (leader) mbar_arrive_expect_tx(fb, (tail ? 3u : 4u) * half_bytes);
        load_w(sbase + i * p.stage_bytes, d, tail, d.kb0 + i, mapa_shared(fb, 0));
      }
    }
    pre = __shfl_sync(0xffffffffu, pre, 0);
    pdl_wait();
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool ok = true;
    for (int t = pair; t < ntiles && ok; t += npairs) {
      bool tail;
      const Tile d = pair_tile_at(p, t, tail);
      for (int kb = d.kb0; kb < d.kb1; ++kb) {
        const uint32_t sw = sbase + stage * p.stage_bytes;
        const uint32_t fb = bar_full + 8 * stage;
        if ((int)issued >= pre) {
          if (!mbar_wait_all(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            // both CTAs' weight halves, plus token rows of 128 (64 in a tail tile) per CTA
            if (leader) mbar_arrive_expect_tx(fb, (tail ? 3u : 4u) * half_bytes);
            load_w(sw, d, tail, kb, mapa_shared(fb, 0));
          }
          __syncwarp();
        }
        if (lane == 0) {
          if (tail)
            tma_load_2d_pair(sw + half_bytes, &tmX64, kb * KBLK, d.xrow + 64 * (int)rank, mapa_shared(fb, 0));
          else
            tma_load_2d_pair(sw + half_bytes, &tmX, kb * KBLK, d.xrow + 128 * (int)rank, mapa_shared(fb, 0));
        }
        __syncwarp();
        ++issued;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) {
      pdl_launch_dependents();
      if (!ok && leader) {  // let the copies already in flight land before the CTA exits
        const uint32_t first = issued > (uint32_t)p.stages ? issued - p.stages : 0u;
        for (uint32_t i = first; i < issued; ++i)
          mbar_wait_drain(bar_full + 8 * (i % p.stages), (i / p.stages) & 1u, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (CTA 0) ----------------
    if (leader) {
      pdl_wait();
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true, any = false;
      for (int t = pair; t < ntiles && ok; t += npairs) {
        bool tail;
        const Tile d = pair_tile_at(p, t, tail);
        const uint32_t idesc = idesc_make(tail ? 128 : 256, 256, FP8);
        if (!mbar_wait_all(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dt = tmem_base + (uint32_t)(acc * p.buf_cols);
        for (int kb = d.kb0; kb < d.kb1; ++kb) {
          if (!mbar_wait_all(bar_full + 8 * stage, phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t sw = sbase + stage * p.stage_bytes;
            const uint32_t sx = sw + half_bytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc_mma_pair<FP8>(dt, sdesc_k_sw128(sx + kk * 32), sdesc_k_sw128(sw + kk * 32), idesc,
                               (kb > d.kb0 || kk > 0) ? 1u : 0u);
            tc_commit_pair(bar_empty + 8 * stage);                  // this CTA's copy of the stage
            tc_commit_pair(mapa_shared(bar_empty + 8 * stage, 1));  // the peer's
          }
          __syncwarp();
          any = true;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if (lane == 0) {
          tc_commit_pair(bar_tfull + 8 * acc);
          tc_commit_pair(mapa_shared(bar_tfull + 8 * acc, 1));
        }
        __syncwarp();
        if (++acc == p.nbuf) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok && any) {  // the tensor cores must be idle before tensor memory is freed
        if (lane == 0) tc_commit_pair(bar_drain);
        __syncwarp();
        mbar_wait_drain(bar_drain, 0, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
    pdl_wait();
    const int q = warp & 3;
    const int lrow = q * 32 + lane;
    float a_scale = 1.0f;
    if constexpr (FP8) a_scale = e4m3_scale_from_amax(__uint_as_float(*p.a_amax));
    float amax = 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int n_pairs = p.T * p.k;
    for (int t = pair; t < ntiles; t += npairs) {
      bool tail;
      Tile d = pair_tile_at(p, t, tail);
      const bool ok = mbar_wait_all(bar_tfull + 8 * acc, acc_phase, abort_flag, p.status);
      if (epi_any(!ok)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.buf_cols);
      const float scale = FP8 ? a_scale * p.w_scale[d.e] : 1.0f;
      if (tail) {
        epi_pair_tail<FP8, EPI>(p, d, tb, lrow, rank, scale, n_pairs, amax);
      } else {
        d.xrow += 128 * (int)rank;  // this CTA's 128 token rows of the tile
        epi_tile<false, FP8, EPI>(p, d, tb, lrow, scale, n_pairs, amax);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(bar_tempty + 8 * acc);
        else
          mbar_arrive_cluster(mapa_shared(bar_tempty + 8 * acc, 0));
      }
      if (++acc == p.nbuf) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if constexpr (EPI == TC_EPI_G1_F32AMAX) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      if (lane == 0 && amax > 0.0f) atomicMax(p.amax_out, __float_as_uint(amax));
    }
  }

  // Both CTAs finish every role (and with it every read of the other CTA's
  // shared memory or tensor memory) before either frees tensor memory or exits.
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// INT4 weight-only grouped GEMM (swap-AB): dequantisation in the main loop
// ---------------------------------------------------------------------------
// "FusedMoE vs MegaMoE" (zwxr.cn), section 6.3: quantised expert weights
// (INT4) cut the bytes the fused kernel streams.  Weights are 4-bit codes q in
// [-8, 7] with one bf16 scale per (weight row, 128 elements of K); the weight
// the MMA sees is bf16(q * s).  Packing: each 32-bit word holds 8 consecutive
// K elements, element e in nibble (e even ? e/2 : 4 + e/2), two's complement.
// Scales are stored group-major per expert ([E][K/128][rows]), so the 256
// scales of a tile's group are two contiguous 256-byte runs.
//
// With thin token batches every MMA re-reads its 128 x 16 weight operand, so
// dequantised weights staged in shared memory would cost four times the HBM
// bytes in shared-memory bandwidth (the limit of a first version of this
// kernel).  The converters therefore write the bf16 weights to tensor memory
// and the MMA takes its A operand from there; shared memory only carries the
// packed codes, the scales and the activation tiles.
//
// A raw stage is one 128-element group of K for the tile's 256 weight rows:
// 16 KB of codes (two TMA boxes of 128 rows x 64 bytes, 64-byte swizzle), the
// activation tiles of its two 64-element K blocks and the 256 scales of the
// group, all prefetched by the producer.
// Roles (448 threads):
//   warp 0      TMA producer: raw stages into their ring
//   warps 6-13  converters, one weight row per thread (the warp's tensor-memory
//               lane quarter): expand a raw stage's codes to bf16 in a
//               tensor-memory A buffer (per K block j and 128-row half h, the 32
//               columns from 64 j + 32 h), signal it
//   warp 1      MMA issuer (tcgen05 kind::f16, A from tensor memory, B = the
//               activation tile in shared memory, fp32 accumulators)
//   warps 2-5   epilogue (shared with k_gemm_tc)
// Tensor memory: accumulator buffers in columns [0, 256), A buffers of 128
// columns from column 256.  The MMA issuer synchronises once per raw stage
// (16 MMAs, 32 with the hi/lo activation split): with thin token tiles the
// issuing thread, which shares its scheduler with converter warps, is the
// critical path, so it runs as few instructions per MMA as possible.
// Conversion: a nibble n becomes the bf16 bit pattern of 128 + (n ^ 8)
// = 128 + q + 8 by one logic operation; subtracting 136 is exact; the product
// with the scale is the one rounding (bf16x2 multiply, nearest even).
constexpr int kW4Threads = 448;
constexpr int kW4ConvWarps = 8;
constexpr int kW4KPerStage = 128;                   // K elements per raw stage (64 bytes of codes per row)
constexpr uint32_t kW4CodeBytes = 2u * 128u * 64u;  // codes of one raw stage
constexpr uint32_t kW4ScaleBytes = 1024u;           // 512 bytes of scales, padded to keep stages 1 KB aligned
constexpr int kW4ABufs = 2;                         // tensor-memory A buffers (one raw stage, 128 columns, each)
constexpr uint32_t kW4ACol = 256;                   // first column of the A buffers

// 8 packed codes (one word, nibble order above) times the bf16 scale pair sc -> 4 bf16x2 (K order)
__device__ __forceinline__ void w4_dequant8(uint32_t w, uint32_t sc, uint32_t* o) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t t = ((w >> (4 * j)) & 0x000F000Fu) ^ 0x43084308u;  // bf16x2 (128 + q + 8)
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&t);
    v = __hsub2(v, __floats2bfloat162_rn(136.0f, 136.0f));             // q, exact
    v = __hmul2(v, *reinterpret_cast<const __nv_bfloat162*>(&sc));    // q * s, rounded once
    o[j] = *reinterpret_cast<uint32_t*>(&v);
  }
}

template <int EPI>
__global__ void __launch_bounds__(kW4Threads, 1)
    k_gemm_w4(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const __grid_constant__ CUtensorMap tmS, const TcDev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_rfull = sbase + p.bar_off;            // raw stage: codes + activations + scales landed
  const uint32_t bar_rempty = bar_rfull + 8 * kMaxStages;  // raw stage: converted and read by the MMA
  const uint32_t bar_afull = bar_rempty + 8 * kMaxStages;  // A buffer: bf16 weights stored
  const uint32_t bar_aempty = bar_afull + 8 * 4;           // A buffer: consumed by the MMA
  const uint32_t bar_tfull = bar_aempty + 8 * 4;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_exit = bar_drain + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (2 * kMaxStages + 8 + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar_rfull + 8 * s, 1);
      mbar_init(bar_rempty + 8 * s, kW4ConvWarps + 1);  // the converter warps + the MMA's commit
    }
    for (int b = 0; b < kW4ABufs; ++b) {
      mbar_init(bar_afull + 8 * b, kW4ConvWarps);
      mbar_init(bar_aempty + 8 * b, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 128);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_exit, kW4Threads / 32);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmS);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (!p.early) pdl_wait();
  const int ntiles = tile_count<true, EPI>(p);
  const uint32_t xbytes = (uint32_t)p.xbox * 128u;  // one activation part of one 64-element K block
  const int parts = p.x_lo_rows ? 2 : 1;
  const uint32_t scale_off = kW4CodeBytes + 2u * (uint32_t)parts * xbytes;  // scales inside a raw stage
  const int groups_k = p.kb_total;                                          // scale groups per row

  if (warp == 0) {
    // ---------------- TMA producer: raw stages (codes + activations + scales) ----------------
    pdl_wait();
    const int n_pairs = p.T * p.k;
    const int npp = p.meta[META_NPP];
    const int groups = p.xbox / 4;  // gather4 groups per activation tile
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile d = tile_at<true, EPI>(p, t);
      int rows[4] = {0, 0, 0, 0};  // token rows of this lane's gather group
      if (p.gather) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = d.xrow + 4 * lane + i;
          const int f = (r < npp) ? p.sorted[r] : n_pairs;
          rows[i] = (f < n_pairs) ? f / p.k : 0;  // padding rows read token 0; never stored
        }
      }
      const int r0 = d.n * p.w_tile_rows;  // first weight row of the tile inside its expert
      for (int rs = d.kb0; rs < d.kb1; ++rs) {
        if (!mbar_wait_all(bar_rempty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t sw = sbase + stage * p.stage_bytes;
        const uint32_t fb = bar_rfull + 8 * stage;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, scale_off + 512u);
          tma_load_2d(sw, &tmW, rs * 64, d.wr0, fb);
          tma_load_2d(sw + kW4CodeBytes / 2, &tmW, rs * 64, d.wr0 + p.w_pair_off, fb);
          tma_load_2d(sw + scale_off, &tmS, r0, d.e * groups_k + rs, fb);
          tma_load_2d(sw + scale_off + 256u, &tmS, r0 + p.w_pair_off, d.e * groups_k + rs, fb);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const uint32_t dst = sw + kW4CodeBytes + (uint32_t)(j * parts) * xbytes;
          const int kel = rs * kW4KPerStage + 64 * j;
          if (p.gather) {
            if (lane < groups)
              tma_gather4(dst + (uint32_t)lane * 512u, &tmX, kel, rows[0], rows[1], rows[2], rows[3], fb);
          } else if (lane == 0) {
            tma_load_2d(dst, &tmX, kel, d.xrow, fb);
            if (p.x_lo_rows) tma_load_2d(dst + xbytes, &tmX, kel, d.xrow + p.x_lo_rows, fb);
          }
        }
        __syncwarp();
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (lane == 0) pdl_launch_dependents();
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------- converters ----------------
    pdl_wait();
    const int q = warp & 3;                // tensor-memory lane quarter of this warp
    const int h = (warp - 6) >> 2;         // 128-row half: gate / up (GEMM1), rows 0-127 / 128-255 (GEMM2)
    const int r = q * 32 + lane;           // row inside the half = tensor-memory lane
    const uint32_t ta = tmem_base + ((uint32_t)(q * 32) << 16) + kW4ACol + (uint32_t)h * 32u;
    int stage = 0, b = 0;
    uint32_t phase = 0, bphase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile d = tile_at<true, EPI>(p, t);
      for (int rs = d.kb0; rs < d.kb1 && ok; ++rs) {
        if (!mbar_wait_all(bar_rfull + 8 * stage, phase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const uint32_t sw = sbase + stage * p.stage_bytes;
        uint32_t sc;
        asm volatile("ld.shared.u16 %0, [%1];" : "=r"(sc) : "r"(sw + scale_off + (uint32_t)(h * 128 + r) * 2u));
        sc |= sc << 16;  // bf16x2 (s, s)
        const uint32_t src = sw + (uint32_t)h * (kW4CodeBytes / 2) + (uint32_t)r * 64u;
        uint32_t wv[16];  // the row's 128 codes: 16-byte chunk c of the 64-byte row sits at chunk c ^ ((r >> 1) & 3)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t chunk = (uint32_t)c ^ (uint32_t)((r >> 1) & 3);
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(wv[4 * c]), "=r"(wv[4 * c + 1]), "=r"(wv[4 * c + 2]), "=r"(wv[4 * c + 3])
                       : "r"(src + chunk * 16u));
        }
        uint32_t a0[32], a1[32];  // K blocks 0 and 1; column m: K elements 2m, 2m+1 of the block
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) {
          w4_dequant8(wv[w8], sc, a0 + 4 * w8);
          w4_dequant8(wv[8 + w8], sc, a1 + 4 * w8);
        }
        if (!mbar_wait_all(bar_aempty + 8 * b, bphase ^ 1u, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st32_nowait(ta + (uint32_t)b * 128u, a0);
        tmem_st32_nowait(ta + (uint32_t)b * 128u + 64u, a1);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_afull + 8 * b);
        if (++b == kW4ABufs) {
          b = 0;
          bphase ^= 1u;
        }
        if (lane == 0) mbar_arrive(bar_rempty + 8 * stage);  // codes and scales of this stage read
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    pdl_wait();
    int stage = 0, b = 0, acc = 0;
    uint32_t phase = 0, bphase = 0, acc_phase = 0;
    bool ok = true, any = false;
    for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
      const Tile d = tile_at<true, EPI>(p, t);
      // (stacked hi/lo activation: one MMA over the xbox hi rows then the lo rows)
      const uint32_t idesc = idesc_make(128, p.stack_lo ? p.xbox + d.npad : d.npad, false);
      if (!mbar_wait_all(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + (uint32_t)(acc * p.buf_cols);
      for (int rs = d.kb0; rs < d.kb1 && ok; ++rs) {
        if (!mbar_wait_all(bar_rfull + 8 * stage, phase, abort_flag, p.status)) {  // activations landed
          ok = false;
          break;
        }
        if (!mbar_wait_all(bar_afull + 8 * b, bphase, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sw = sbase + stage * p.stage_bytes;
          const uint32_t ab = tmem_base + kW4ACol + (uint32_t)b * 128u;
          const uint32_t d1 = dt + (uint32_t)p.d1_col;
          for (int j = 0; j < 2; ++j) {
            const uint64_t bd = sdesc_k_sw128(sw + kW4CodeBytes + (uint32_t)(j * parts) * xbytes);
            tc_mma_ts_kblock(dt, d1, ab + (uint32_t)j * 64u, bd, idesc, (rs > d.kb0 || j > 0) ? 1u : 0u);
            if (parts > 1 && !p.stack_lo)
              tc_mma_ts_kblock(dt, d1, ab + (uint32_t)j * 64u, bd + (xbytes >> 4), idesc, 1u);
          }
          tc_commit(bar_aempty + 8 * b);
          tc_commit(bar_rempty + 8 * stage);  // the stage's activations are read
        }
        __syncwarp();
        any = true;
        if (++b == kW4ABufs) {
          b = 0;
          bphase ^= 1u;
        }
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) tc_commit(bar_tfull + 8 * acc);
      __syncwarp();
      if (++acc == p.nbuf) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && any) {
      if (lane == 0) tc_commit(bar_drain);
      __syncwarp();
      mbar_wait_drain(bar_drain, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    pdl_wait();
    const int q = warp & 3;
    const int lrow = q * 32 + lane;
    float amax = 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    const int n_pairs = p.T * p.k;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile d = tile_at<true, EPI>(p, t);
      const bool ok = mbar_wait_all(bar_tfull + 8 * acc, acc_phase, abort_flag, p.status);
      if (epi_any(!ok)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.buf_cols);
      epi_tile<true, false, EPI>(p, d, tb, lrow, 1.0f, n_pairs, amax);
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == p.nbuf) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar_exit);
  if (warp == 1) {
    mbar_wait_drain(bar_exit, 0, 2 * kWaitLimitNs);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <bool SWAP, bool FP8, int EPI>
cudaError_t launch_inst(const CUtensorMap& mw, const CUtensorMap& mx, const CUtensorMap& mx16, const TcDev& p,
                        int grid, size_t smem, cudaStream_t s, int max_grid) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = k_gemm_tc<SWAP, FP8, EPI>;
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  (void)max_grid;
  return cudaLaunchKernelEx(&cfg, kern, mw, mx, mx16, p);
}

// CTA-pair kernels: clusters of 2, a persistent grid of as many pairs as can be
// resident at once (an SM left over in a GPC cannot take half a pair).
template <bool FP8, int EPI>
cudaError_t launch_pair_inst(const CUtensorMap& mw, const CUtensorMap& mx, const CUtensorMap& mw64,
                             const CUtensorMap& mx64, const TcDev& p, int tiles, size_t smem, cudaStream_t s) {
  static bool attr_set[64] = {};
  static int max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = k_gemm_pair<FP8, EPI>;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(2);
  if (max_clusters[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = -1;
    }
    max_clusters[dev] = n;
  }
  if (max_clusters[dev] < 1) return cudaErrorInvalidConfiguration;
  const int pairs = std::max(1, std::min(tiles, max_clusters[dev]));
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, mw, mx, mw64, mx64, p);
}

}  // namespace

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D K-major tensor [rows][K] of 1- or 2-byte elements, box = 128 bytes of K x box_rows, 128-byte swizzle.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t K, uint64_t rows, uint32_t box_rows,
                        uint32_t box_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  if (box_bytes != 128 && box_bytes != 64 && box_bytes != 256) return false;
  const cuuint64_t dims[2] = {K, rows};
  const cuuint64_t strides[1] = {K * (uint64_t)elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)(box_bytes / elem_bytes), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                             : (box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int EPI>
static cudaError_t launch_w4_inst(const CUtensorMap& mw, const CUtensorMap& mx, const CUtensorMap& ms, const TcDev& p,
                                  int grid, size_t smem, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  auto kern = k_gemm_w4<EPI>;
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  return launch_pdl(kern, dim3(grid), dim3(kW4Threads), smem, s, mw, mx, ms, p);
}

// INT4 weights: swap-AB only; K splits and tile K ranges in raw stages of 128 elements.
static cudaError_t launch_gemm_w4(const TcGemmArgs& a, cudaStream_t s) {
  if (!a.swap || a.fp8 || a.K % kW4KPerStage || a.xbox > 128 || a.xbox % 16 || !a.w4_scale)
    return cudaErrorInvalidValue;
  CUtensorMap mw, mx, ms;
  if (!make_tensor_map_2d(&mw, a.W, 1, (uint64_t)a.K / 2, (uint64_t)a.E * a.w_rows_per_expert, 128u, 64u))
    return cudaErrorInvalidValue;
  // scales [E][K/128][rows]: boxes of 128 consecutive rows of one group
  if (!make_tensor_map_2d(&ms, a.w4_scale, 2, (uint64_t)a.w_rows_per_expert, (uint64_t)a.E * (a.K / 128), 1u, 256u))
    return cudaErrorInvalidValue;
  if (a.gather) {
    if (a.xbox % 4 || a.xbox > 128 || a.x_lo_rows) return cudaErrorInvalidValue;
    if (!make_tensor_map_2d(&mx, a.X, 2, (uint64_t)a.K, (uint64_t)a.T, 1u)) return cudaErrorInvalidValue;
  } else if (!make_tensor_map_2d(&mx, a.X, 2, (uint64_t)a.K, (uint64_t)a.cap + (uint64_t)a.x_lo_rows,
                                 (uint32_t)a.xbox)) {
    return cudaErrorInvalidValue;
  }
  TcDev p = {};
  p.tm_rows = 128;
  p.epi = a.epi;
  p.T = a.T;
  p.k = a.k;
  p.E = a.E;
  p.I = a.I;
  p.H = a.H;
  p.kb_total = a.K / kW4KPerStage;
  p.kb_per_split = a.kb_per_split;
  p.splits = a.splits;
  p.n_tiles = a.n_tiles;
  p.w_rows_per_expert = a.w_rows_per_expert;
  p.w_pair_off = a.w_pair_off;
  p.w_tile_rows = a.w_tile_rows;
  p.wbox = a.wbox;
  p.xbox = a.xbox;
  p.sorted = a.sorted;
  p.eids = a.eids;
  p.meta = a.meta;
  p.out = a.out;
  p.gather = a.gather ? 1 : 0;
  p.early = a.early ? 1 : 0;
  p.out_lo = a.out_lo;
  p.x_lo_rows = a.x_lo_rows;
  p.out_split_stride = a.out_split_stride;
  p.status = a.status;
  // accumulators: D0 and D1 of xbox columns each; two buffers while they fit below the A buffers
  // (a stacked hi/lo activation needs xbox + npad columns per accumulator)
  p.stack_lo = (a.x_lo_rows && a.xbox <= 64) ? 1 : 0;
  p.d1_col = p.stack_lo ? 2 * a.xbox : a.xbox;
  p.buf_cols = 2 * p.d1_col;
  p.nbuf = 2 * p.buf_cols <= (int)kW4ACol ? 2 : 1;
  if (a.x_lo_rows && !p.stack_lo && p.buf_cols > (int)kW4ACol) return cudaErrorInvalidValue;
  const int parts = a.x_lo_rows ? 2 : 1;
  // codes + two K blocks of activations + scales
  p.stage_bytes = kW4CodeBytes + 2u * (uint32_t)a.xbox * 128u * parts + kW4ScaleBytes;
  const uint32_t bar_bytes = 8 * (2 * kMaxStages + 8 + 6) + 16;
  const uint32_t total = 227 * 1024 - 1024 - bar_bytes;
  int stages = (int)(total / p.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  p.stages = stages;
  p.bar_off = (uint32_t)stages * p.stage_bytes;
  const size_t smem = 1024 + (size_t)p.bar_off + bar_bytes;
  const long upper = (long)std::min(a.E, a.T * a.k) * a.n_tiles * a.splits;
  int grid = (int)std::min<long>(upper, a.num_sms);
  if (grid < 1) grid = 1;
  if (a.epi == TC_EPI_G1_BF16) return launch_w4_inst<TC_EPI_G1_BF16>(mw, mx, ms, p, grid, smem, s);
  if (a.epi == TC_EPI_G1_PART) return launch_w4_inst<TC_EPI_G1_PART>(mw, mx, ms, p, grid, smem, s);
  if (a.epi == TC_EPI_G2_F32) return launch_w4_inst<TC_EPI_G2_F32>(mw, mx, ms, p, grid, smem, s);
  return cudaErrorInvalidValue;
}

// Token-major GEMM1 / GEMM2 on CTA pairs: tiles of 256 sorted rows (the
// permutation block) x 256 weight rows, each CTA staging half of each operand.
static cudaError_t launch_gemm_pair(const TcGemmArgs& a, cudaStream_t s) {
  if (a.swap || a.gather || a.x_lo_rows || a.w4 || a.epi == TC_EPI_LOGITS || a.wbox != 128 || a.xbox != 128 ||
      !a.pblk)
    return cudaErrorInvalidValue;
  const int eb = a.fp8 ? 1 : 2;
  CUtensorMap mw, mx, mw64, mx64;
  if (!make_tensor_map_2d(&mw, a.W, eb, (uint64_t)a.K, (uint64_t)a.E * a.w_rows_per_expert, 128u) ||
      !make_tensor_map_2d(&mx, a.X, eb, (uint64_t)a.K, (uint64_t)a.cap, 128u) ||
      !make_tensor_map_2d(&mw64, a.W, eb, (uint64_t)a.K, (uint64_t)a.E * a.w_rows_per_expert, 64u) ||
      !make_tensor_map_2d(&mx64, a.X, eb, (uint64_t)a.K, (uint64_t)a.cap, 64u))
    return cudaErrorInvalidValue;
  TcDev p = {};
  p.epi = a.epi;
  p.T = a.T;
  p.k = a.k;
  p.E = a.E;
  p.I = a.I;
  p.H = a.H;
  p.kb_total = a.K * eb / 128;
  p.kb_per_split = p.kb_total;
  p.splits = 1;
  p.n_tiles = a.n_tiles;
  p.w_rows_per_expert = a.w_rows_per_expert;
  p.w_pair_off = a.w_pair_off;
  p.w_tile_rows = a.w_tile_rows;
  p.wbox = 128;
  p.xbox = 128;
  p.tm_rows = 128;
  p.pblk = a.pblk;
  p.sorted = a.sorted;
  p.eids = a.eids;
  p.meta = a.meta;
  p.out = a.out;
  p.early = a.early ? 1 : 0;
  p.out_split_stride = a.out_split_stride;
  p.w_scale = a.w_scale;
  p.a_amax = a.a_amax;
  p.amax_out = a.amax_out;
  p.status = a.status;
  p.w_bytes = 128u * 128u;
  p.stage_bytes = 2u * 128u * 128u;  // this CTA's weight box and token rows
  const uint32_t bar_bytes = 8 * (2 * kMaxStages + 6) + 16;
  int stages = (int)((227 * 1024 - 1024 - bar_bytes) / p.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  p.stages = stages;
  p.bar_off = (uint32_t)stages * p.stage_bytes;
  p.d1_col = 0;
  p.buf_cols = 256;
  p.nbuf = 2;
  const size_t smem = 1024 + (size_t)p.bar_off + bar_bytes;
  const int tiles = (int)std::max<long>(1, (long)(a.cap / 128) * a.n_tiles);
  if (a.fp8) {
    if (a.epi == TC_EPI_G1_F32AMAX)
      return launch_pair_inst<true, TC_EPI_G1_F32AMAX>(mw, mx, mw64, mx64, p, tiles, smem, s);
    if (a.epi == TC_EPI_G2_F32) return launch_pair_inst<true, TC_EPI_G2_F32>(mw, mx, mw64, mx64, p, tiles, smem, s);
  } else {
    if (a.epi == TC_EPI_G1_BF16)
      return launch_pair_inst<false, TC_EPI_G1_BF16>(mw, mx, mw64, mx64, p, tiles, smem, s);
    if (a.epi == TC_EPI_G2_F32) return launch_pair_inst<false, TC_EPI_G2_F32>(mw, mx, mw64, mx64, p, tiles, smem, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(const TcGemmArgs& a, cudaStream_t s) {
  if (a.w4) return a.ready ? cudaErrorInvalidValue : launch_gemm_w4(a, s);
  if (a.pair) return a.ready ? cudaErrorInvalidValue : launch_gemm_pair(a, s);
  const int eb = a.fp8 ? 1 : 2;
  CUtensorMap mw, mx;
  if (!make_tensor_map_2d(&mw, a.W, eb, (uint64_t)a.K, (uint64_t)a.E * a.w_rows_per_expert, (uint32_t)a.wbox))
    return cudaErrorInvalidValue;
  if (a.gather) {
    // tile::gather4 needs a one-row box: 4 such rows per instruction
    if (a.xbox % 4 || a.xbox > 256 || a.x_lo_rows) return cudaErrorInvalidValue;
    if (!make_tensor_map_2d(&mx, a.X, eb, (uint64_t)a.K, (uint64_t)a.T, 1u)) return cudaErrorInvalidValue;
  }
  if (!a.gather && !make_tensor_map_2d(&mx, a.X, eb, (uint64_t)a.K, (uint64_t)a.cap + (uint64_t)a.x_lo_rows,
                                       (uint32_t)a.xbox)) {
    return cudaErrorInvalidValue;
  }

  // swap-AB: a 16-row box for the tiles of experts with at most 16 tokens
  CUtensorMap mx16 = mx;
  if (a.swap && !a.gather && a.xbox > 16 &&
      !make_tensor_map_2d(&mx16, a.X, eb, (uint64_t)a.K, (uint64_t)a.cap + (uint64_t)a.x_lo_rows, 16u))
    return cudaErrorInvalidValue;

  TcDev p = {};
  p.tm_rows = 128;
  p.prefetch_kb = a.prefetch_kb;
  p.stack_lo = (a.swap && a.x_lo_rows && !a.fp8 && a.xbox <= 64) ? 1 : 0;
  p.epi = a.epi;
  p.T = a.T;
  p.k = a.k;
  p.E = a.E;
  p.I = a.I;
  p.H = a.H;
  p.kb_total = a.K * eb / 128;
  p.kb_per_split = a.kb_per_split;
  p.splits = a.splits;
  p.n_tiles = a.n_tiles;
  p.w_rows_per_expert = a.w_rows_per_expert;
  p.w_pair_off = a.w_pair_off;
  p.w_tile_rows = a.w_tile_rows;
  p.wbox = a.wbox;
  p.xbox = a.xbox;
  p.sorted = a.sorted;
  p.eids = a.eids;
  p.meta = a.meta;
  p.out = a.out;
  p.gather = a.gather ? 1 : 0;
  p.early = a.early ? 1 : 0;
  p.claim = a.claim;
  p.zero_word = a.zero_word;
  p.n_valid = a.n_valid;
  p.out_lo = a.out_lo;
  p.x_lo_rows = a.x_lo_rows;
  p.out_split_stride = a.out_split_stride;
  p.w_scale = a.w_scale;
  p.a_amax = a.a_amax;
  p.amax_out = a.amax_out;
  p.status = a.status;
  p.ready = a.ready;
  p.want = a.ready ? a.want : nullptr;
  p.fin = a.fin;
  p.out_fin = a.out_fin;
  p.out_fin_lo = a.out_fin_lo;
  if (a.fin && (!a.swap || a.fp8 || a.epi != TC_EPI_G1_PART || !a.out_fin)) return cudaErrorInvalidValue;

  p.w_bytes = (uint32_t)(2 * a.wbox * 128);
  p.stage_bytes = p.w_bytes + (uint32_t)(a.xbox * 128) * (a.x_lo_rows ? 2u : 1u);
  const uint32_t bar_bytes = 8 * (2 * kMaxStages + 6) + 16 + 16 * kTileQueue + 4 * kTileQueue;
  const uint32_t budget = 227 * 1024 - 1024 - bar_bytes;
  int stages = (int)(budget / p.stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  p.stages = stages;
  p.bar_off = (uint32_t)stages * p.stage_bytes;
  if (a.swap) {
    // D0 and D1 of xbox columns each; two buffers while they fit in 512 columns
    if (a.xbox > 256) return cudaErrorInvalidValue;
    p.d1_col = a.xbox <= 128 ? 128 : 256;
    p.buf_cols = 2 * p.d1_col;
    p.nbuf = (2 * p.buf_cols <= (int)kTmemCols) ? 2 : 1;
  } else {
    p.d1_col = 0;
    p.buf_cols = 256;
    p.nbuf = 2;
  }
  const size_t smem = 1024 + (size_t)p.bar_off + bar_bytes;

  long upper;
  if (a.epi == TC_EPI_LOGITS)
    upper = (long)(a.T + 127) / 128 * a.n_tiles;
  else if (a.swap)
    upper = (long)std::min(a.E, a.T * a.k) * a.n_tiles * a.splits;
  else
    upper = (long)(a.cap / 128) * a.n_tiles;
  int grid = (int)std::min<long>(upper, a.num_sms);
  if (grid < 1) grid = 1;

#define MOE_TC_CASE(SW, F8, EP)                      \
  if (a.swap == SW && a.fp8 == F8 && a.epi == EP) \
    return launch_inst<SW, F8, EP>(mw, mx, mx16, p, grid, smem, s, a.num_sms);
  MOE_TC_CASE(true, false, TC_EPI_G1_BF16)
  MOE_TC_CASE(true, false, TC_EPI_G1_PART)
  MOE_TC_CASE(true, false, TC_EPI_G2_F32)
  MOE_TC_CASE(true, true, TC_EPI_G1_F32AMAX)
  MOE_TC_CASE(true, true, TC_EPI_G1_PART)
  MOE_TC_CASE(true, true, TC_EPI_G2_F32)
  MOE_TC_CASE(false, false, TC_EPI_G1_BF16)
  MOE_TC_CASE(false, false, TC_EPI_G2_F32)
  MOE_TC_CASE(false, true, TC_EPI_G1_F32AMAX)
  MOE_TC_CASE(false, true, TC_EPI_G2_F32)
  MOE_TC_CASE(false, false, TC_EPI_LOGITS)
#undef MOE_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace moe
