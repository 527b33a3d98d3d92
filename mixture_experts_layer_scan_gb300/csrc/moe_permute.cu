// Token-to-expert permutation, activation gather, split-K / FP8 activation
// passes and the routing-weighted combine.
//
// "FusedMoE vs MegaMoE" (zwxr.cn), section 2.3: routing scatters the tokens
// of a batch to experts and the results must be put back in token order;
// section 3.1: the fused design sorts tokens by expert, builds an index of
// which rows belong to which expert, computes, then reorders and sums the
// results with the routing weights.
#include <algorithm>
#include <cooperative_groups.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace cg = cooperative_groups;

namespace moe {

namespace {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kGatherThreads = 64;  // two warps (tokens) per CTA: short batches spread over SMs

// Exclusive scan over blockDim.x (= 1024) values, one per thread; returns the
// exclusive prefix of the caller and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* scratch /* >= 33 ints */, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += n;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = (lane < (int)(blockDim.x >> 5)) ? scratch[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += n;
    }
    scratch[lane] = wi - w;  // exclusive prefix of each warp
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  const int res = scratch[warp] + incl - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// Stable counting sort of the (token, slot) pairs by expert, run by one
// thread-block cluster of `csize` CTAs x 1024 threads (csize = 1 for decode
// batches).  CTA r owns the contiguous chunk r of the flat pair indices and
// its warp w the contiguous sub-chunk w of that.  Pass 1 counts per warp and
// expert with warp match (no atomics, so counts do not depend on timing).
// Each CTA then reads the other CTAs' per-expert totals straight from their
// shared memory (distributed shared memory of the cluster), which gives every
// warp its first slot inside every expert; pass 2 writes each pair there, so
// inside an expert the flat indices stay in ascending order.  No global
// scratch is needed.
__global__ void __launch_bounds__(kAlignThreads, 1)
    k_align(const int32_t* __restrict__ ids, int T, int k, int E, int B, int32_t* __restrict__ sorted,
            int32_t* __restrict__ eids, int32_t* __restrict__ npp_out, int32_t* __restrict__ counts_out,
            int32_t* __restrict__ meta, int* status, int skip_minus_one, int32_t* __restrict__ pblk,
            unsigned* __restrict__ zero_words, int n_zero, int32_t* __restrict__ inv) {
  pdl_enter();
  // counters of the next kernels of this call start at zero (e.g. GEMM1's split arrivals)
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x) zero_words[i] = 0u;
  cg::cluster_group cluster = cg::this_cluster();
  const int csize = (int)cluster.num_blocks();
  const int crank = (int)cluster.block_rank();
  extern __shared__ int sm[];
  int* wc = sm;                       // [kAlignWarps][E] per-warp counts, then per-warp bases
  int* ctot = wc + kAlignWarps * E;   // [E] this CTA's per-expert counts (read by the whole cluster)
  int* off = ctot + E;                // [E+1] padded offsets
  int* cnt = off + E + 1;             // [E] per-expert counts of the whole batch
  int* cbase = cnt + E;               // [E] pairs of this expert in lower-ranked CTAs
  int* scan_tmp = cbase + E;          // [33]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = T * k;
  const int C = (n + csize - 1) / csize;
  const int cbeg = min(n, crank * C), cend = min(n, cbeg + C);
  const int L = (cend - cbeg + kAlignWarps - 1) / kAlignWarps;
  const int beg = min(cend, cbeg + warp * L), end = min(cend, beg + L);

  for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) wc[i] = 0;
  __syncthreads();

  // pass 1: per-warp histogram
  bool bad = false;
  for (int base = beg; base < end; base += 32) {
    const int f = base + lane;
    int e = -1;
    if (f < end) {
      e = ids[f];
      // -1 marks a pair another pass handles (skip_minus_one): dropped without a flag
      if (e < 0 || e >= E) { bad = bad || !(skip_minus_one && e == -1); e = -1; }
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && lane == __ffs(grp) - 1) wc[warp * E + e] += __popc(grp);
    __syncwarp();
  }
  if (bad) report(status, MOE_ERR_DEVICE_INDEX);
  __syncthreads();

  // this CTA's totals and per-warp bases (exclusive over warps)
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
    for (int w = 0; w < kAlignWarps; ++w) {
      const int c = wc[w * E + e];
      wc[w * E + e] = run;
      run += c;
    }
    ctot[e] = run;
  }
  cluster.sync();  // every CTA's ctot is complete
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int tot = 0, below = 0;
    for (int r = 0; r < csize; ++r) {
      const int v = *cluster.map_shared_rank(ctot + e, r);
      if (r < crank) below += v;
      tot += v;
    }
    cnt[e] = tot;
    cbase[e] = below;
  }
  cluster.sync();  // remote reads done: no CTA touches another's shared memory after this

  // padded offsets and active list (E <= 1024 = blockDim); identical in every CTA
  {
    const int e = threadIdx.x;
    const int c = (e < E) ? cnt[e] : 0;
    const int padded = (c + B - 1) / B * B;
    int total_pad = 0, total_act = 0;
    const int o = block_exclusive_scan(padded, scan_tmp, &total_pad);
    const int a = block_exclusive_scan(c > 0 ? 1 : 0, scan_tmp, &total_act);
    if (e < E) {
      off[e] = o;
      if (crank == 0) {
        if (meta) {
          meta[meta_offsets(E) + e] = o;
          meta[meta_counts(E) + e] = c;
          if (c > 0) meta[meta_active(E) + a] = e;
        }
        if (counts_out) counts_out[e] = c;
      }
    }
    if (e == 0) {
      off[E] = total_pad;
      if (crank == 0) {
        *npp_out = total_pad;
        if (meta) {
          meta[META_NPP] = total_pad;
          meta[META_NBLK] = total_pad / B;
          meta[META_NACT] = total_act;
          meta[meta_offsets(E) + E] = total_pad;
        }
      }
    }
  }
  __syncthreads();

  // CTA-pair tiles (pblk non-null, B = 128): every expert's padded run in chunks of
  // 256 rows, the last one 128 rows when the run has an odd number of blocks;
  // pblk[p] = (first row << 1) | (1 for a 128-row chunk), meta word 3 = chunks
  if (pblk) {
    const int e = threadIdx.x;
    const int padded = (e < E) ? off[e + 1] - off[e] : 0;
    const int np = (padded + 255) / 256;
    int total_np = 0;
    const int ps = block_exclusive_scan(np, scan_tmp, &total_np);
    if (crank == 0) {
      for (int j = 0; j < np; ++j) pblk[ps + j] = ((off[e] + 256 * j) << 1) | (padded - 256 * j == 128 ? 1 : 0);
      if (e == 0 && meta) meta[META_NPB] = total_np;
    }
  }

  // pass 2: stable scatter
  for (int base = beg; base < end; base += 32) {
    const int f = base + lane;
    int e = -1;
    if (f < end) {
      e = ids[f];
      if (e < 0 || e >= E) e = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    int slot = 0;
    if (e >= 0) slot = off[e] + cbase[e] + wc[warp * E + e] + __popc(grp & ((1u << lane) - 1u));
    __syncwarp();
    if (e >= 0) {
      sorted[slot] = f;
      if (lane == __ffs(grp) - 1) wc[warp * E + e] += __popc(grp);
    }
    if (inv && f < end) inv[f] = e >= 0 ? slot : -1;  // pair -> sorted row (-1: left out)
    __syncwarp();
  }

  // block -> expert map and sentinel padding, blocks spread over the cluster
  const int total = off[E];
  const int nblk = total / B;
  for (int b = crank * blockDim.x + threadIdx.x; b < nblk; b += csize * blockDim.x) {
    int lo = 0, hi = E - 1;  // last expert with off[e] <= b*B: the owner of block b
    const int pos = b * B;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= pos) lo = mid; else hi = mid - 1;
    }
    eids[b] = lo;
    const int fill_from = max(pos, off[lo] + cnt[lo]);
    for (int q = fill_from; q < pos + B; ++q) sorted[q] = n;
  }
}

// The same permutation for batches of at most 32 pairs (decode), by one warp: each
// lane holds one pair, warp match gives every pair's expert group, its size and the
// pair's rank inside it (lower flat index first: the same stable order), and the group
// leaders -- the active experts -- find their padded offsets by comparing expert ids
// over the warp and write their own block map entries and sentinel rows.  The leaders'
// (expert, offset, count) sorted by expert give every expert's offset and count.  No
// block barrier and no second read of the ids:
// the general kernel's phases cost about 0.5 us each at this size.  Outputs equal the
// general kernel's (pblk is not produced here).
constexpr int kAlignSmallThreads = 128;

__global__ void __launch_bounds__(kAlignSmallThreads)
    k_align_small(const int32_t* __restrict__ ids, int n, int E, int B, int32_t* __restrict__ sorted,
                  int32_t* __restrict__ eids, int32_t* __restrict__ npp_out, int32_t* __restrict__ counts_out,
                  int32_t* __restrict__ meta, int* status, int skip_minus_one, unsigned* __restrict__ zero_words,
                  int n_zero, int32_t* __restrict__ inv) {
  pdl_enter();
  for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero_words[i] = 0u;
  if (threadIdx.x >= 32) return;
  __shared__ int s_e[32], s_off[32], s_c[32];  // active experts in ascending order
  const int lane = threadIdx.x;
  int e = -1;
  if (lane < n) {
    e = ids[lane];
    if (e < 0 || e >= E) {
      if (!(skip_minus_one && e == -1)) report(status, MOE_ERR_DEVICE_INDEX);
      e = -1;
    }
  }
  const unsigned grp = __match_any_sync(0xffffffffu, e);
  const int c = __popc(grp);
  const bool leader = e >= 0 && lane == __ffs(grp) - 1;
  const unsigned leaders = __ballot_sync(0xffffffffu, leader);
  const int pad = (c + B - 1) / B * B;
  // experts below mine among the active ones, and their padded rows
  int below = 0, off = 0;
  for (int j = 0; j < 32; ++j) {
    const int ej = __shfl_sync(0xffffffffu, e, j);
    const int pj = __shfl_sync(0xffffffffu, pad, j);
    if (((leaders >> j) & 1u) && ej < e) {
      ++below;
      off += pj;
    }
  }
  int total = leader ? pad : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  const int nact = __popc(leaders);
  if (leader) {
    s_e[below] = e;
    s_off[below] = off;
    s_c[below] = c;
    if (meta) meta[meta_active(E) + below] = e;
  }
  if (e >= 0) {
    const int slot = off + __popc(grp & ((1u << lane) - 1u));
    sorted[slot] = lane;
    if (inv) inv[lane] = slot;
  } else if (inv && lane < n) {
    inv[lane] = -1;
  }
  // block -> expert map and sentinel rows: each active expert's leader writes its own run
  if (leader) {
    for (int b = off / B; b < (off + pad) / B; ++b) eids[b] = e;
    for (int q = off + c; q < off + pad; ++q) sorted[q] = n;
  }
  __syncwarp();
  // every expert's offset and count: those of the first active expert at or above it
  // (lane x visits x, x + 32, ...: the active index lo only moves forward)
  int lo = 0;
  for (int x = lane; x < E; x += 32) {
    while (lo < nact && s_e[lo] < x) ++lo;
    const int cnt = (lo < nact && s_e[lo] == x) ? s_c[lo] : 0;
    if (meta) {
      meta[meta_offsets(E) + x] = lo < nact ? s_off[lo] : total;
      meta[meta_counts(E) + x] = cnt;
    }
    if (counts_out) counts_out[x] = cnt;
  }
  if (lane == 0) {
    *npp_out = total;
    if (meta) {
      meta[META_NPP] = total;
      meta[META_NBLK] = total / B;
      meta[META_NACT] = nact;
      meta[meta_offsets(E) + E] = total;
    }
  }
}

// The same permutation for 33 to 1024 pairs by one CTA, one pair per thread (pair f
// in thread f): warp match gives each pair's rank inside its warp and the warp's
// count of its expert (wc[warp][e], also added into the expert's total); a pair's
// stable slot is its expert's offset plus the counts of the lower warps plus its
// rank.  One warp scans the padded counts into offsets; every expert's thread then
// writes its block-map entries and sentinel rows.  Three block barriers (the general
// kernel has about a dozen).  Outputs equal the general kernel's (pblk not produced).
__global__ void __launch_bounds__(kAlignThreads, 1)
    k_align_mid(const int32_t* __restrict__ ids, int n, int E, int B, int32_t* __restrict__ sorted,
                int32_t* __restrict__ eids, int32_t* __restrict__ npp_out, int32_t* __restrict__ counts_out,
                int32_t* __restrict__ meta, int* status, int skip_minus_one, unsigned* __restrict__ zero_words,
                int n_zero, int32_t* __restrict__ inv) {
  pdl_enter();
  for (int i = threadIdx.x; i < n_zero; i += blockDim.x) zero_words[i] = 0u;
  extern __shared__ int sm[];
  int* wc = sm;            // [kAlignWarps][E] counts of each expert in each warp
  int* cnt = wc + kAlignWarps * E;  // [E]
  int* off = cnt + E;      // [E + 1]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) wc[i] = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  const int f = threadIdx.x;
  int e = -1;
  if (f < n) {
    e = ids[f];
    if (e < 0 || e >= E) {
      if (!(skip_minus_one && e == -1)) report(status, MOE_ERR_DEVICE_INDEX);
      e = -1;
    }
  }
  __syncthreads();
  const unsigned grp = __match_any_sync(0xffffffffu, e);
  const int rank = __popc(grp & ((1u << lane) - 1u));
  if (e >= 0 && lane == __ffs(grp) - 1) {
    wc[warp * E + e] = __popc(grp);
    atomicAdd(&cnt[e], __popc(grp));  // (a total: the order of the additions does not matter)
  }
  __syncthreads();
  int below = 0;  // pairs of my expert in lower warps
  if (e >= 0)
    for (int w = 0; w < warp; ++w) below += wc[w * E + e];
  if (warp == 0) {
    // offsets: lane l scans experts [l*per, l*per + per) after a warp scan of the lane sums
    const int per = (E + 31) / 32, x0 = min(E, lane * per), x1 = min(E, x0 + per);
    int lp = 0, la = 0;
    for (int x = x0; x < x1; ++x) {
      const int c = cnt[x];
      lp += (c + B - 1) / B * B;
      la += c > 0 ? 1 : 0;
    }
    int ip = lp, ia = la;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, ip, o), ua = __shfl_up_sync(0xffffffffu, ia, o);
      if (lane >= o) {
        ip += up;
        ia += ua;
      }
    }
    const int total = __shfl_sync(0xffffffffu, ip, 31), nact = __shfl_sync(0xffffffffu, ia, 31);
    int rp = ip - lp, ra = ia - la;
    for (int x = x0; x < x1; ++x) {
      const int c = cnt[x];
      off[x] = rp;
      if (meta) {
        meta[meta_offsets(E) + x] = rp;
        meta[meta_counts(E) + x] = c;
        if (c > 0) meta[meta_active(E) + ra] = x;
      }
      if (counts_out) counts_out[x] = c;
      ra += c > 0 ? 1 : 0;
      rp += (c + B - 1) / B * B;
    }
    if (lane == 0) {
      off[E] = total;
      *npp_out = total;
      if (meta) {
        meta[META_NPP] = total;
        meta[META_NBLK] = total / B;
        meta[META_NACT] = nact;
        meta[meta_offsets(E) + E] = total;
      }
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int slot = off[e] + below + rank;
    sorted[slot] = f;
    if (inv) inv[f] = slot;
  } else if (inv && f < n) {
    inv[f] = -1;
  }
  // block map and sentinel rows, one expert per thread
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    const int c = cnt[x];
    if (c == 0) continue;
    const int o = off[x], pad = (c + B - 1) / B * B;
    for (int b = o / B; b < (o + pad) / B; ++b) eids[b] = x;
    for (int q = o + c; q < o + pad; ++q) sorted[q] = n;
  }
}

// amax over n bf16 values (bit pattern of a non-negative float, atomicMax on
// the bits is order independent).
__global__ void k_amax_bf16(const uint16_t* __restrict__ X, size_t n, unsigned* amax_bits) {
  pdl_enter();
  float m = 0.0f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(bf16_bits_to_f32(X[i])));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, __float_as_uint(m));
}

// Gather of token rows into expert order, 16-byte vectors, token by token: a
// warp reads token t's row once and stores it at the sorted rows of its k pairs
// (inv[t*k + j]; -1 for a pair left out), so every row is read from memory once
// however many experts it goes to.  Rows holding the sentinel (expert padding)
// are then zero-filled.
__global__ void __launch_bounds__(kGatherThreads) k_gather_scatter(const uint4* __restrict__ X, int vec_per_row,
                                                                   int T, int k, int n_pairs,
                                                                   const int32_t* __restrict__ inv,
                                                                   const int32_t* __restrict__ sorted,
                                                                   const int32_t* __restrict__ meta,
                                                                   uint4* __restrict__ Xs) {
  pdl_enter();
  constexpr int kUnroll = 8;  // 16-byte loads of one lane in flight before its stores
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  // (every loop bound below is the same in all lanes of a warp, so all 32 lanes reach
  // each shuffle and ballot; only the loads and stores depend on the lane)
  for (int t = gw; t < T; t += nwarps) {
    const int my_row = lane < k ? inv[(size_t)t * k + lane] : -1;  // k <= 32
    const uint4* src = X + (size_t)t * vec_per_row;
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * kUnroll) {
      uint4 buf[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = v0 + 32 * u + lane;
        if (v < vec_per_row) buf[u] = src[v];
      }
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_row, j);
        if (r < 0) continue;
        uint4* dst = Xs + (size_t)r * vec_per_row;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + 32 * u + lane;
          if (v < vec_per_row) dst[v] = buf[u];
        }
      }
    }
  }
  const int npp = meta[META_NPP];
  for (int r0 = gw * 32; r0 < npp; r0 += nwarps * 32) {
    const int r = r0 + lane;
    unsigned pad = __ballot_sync(0xffffffffu, r < npp && sorted[r] >= n_pairs);
    while (pad) {
      const int b = __ffs(pad) - 1;
      pad &= pad - 1;
      uint4* dst = Xs + (size_t)(r0 + b) * vec_per_row;
      for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// Gather of token rows into expert order, 16-byte vectors, row by row: one warp
// per sorted row (grid-stride), rows holding the sentinel zero-filled.  For short
// batches, whose token rows stay in L2, this spreads the copies over the most warps.
__global__ void __launch_bounds__(256) k_gather_copy(const uint4* __restrict__ X, int vec_per_row, int k,
                                                     int n_pairs, const int32_t* __restrict__ sorted,
                                                     const int32_t* __restrict__ meta, uint4* __restrict__ Xs,
                                                     int late) {
  // late: dependents launch only once the permutation is complete (after this kernel's own
  // dependency wait), so GEMM1 may read its tile list and stream weights before its wait;
  // otherwise they launch at once (GEMM1 then prefetches guessed weights into L2 meanwhile)
  if (!late) pdl_launch_dependents();
  pdl_wait();
  if (late) pdl_launch_dependents();
  // one warp per row; each lane has kGatherUnroll 16-byte loads in flight before its stores
  constexpr int kGatherUnroll = 8;
  const int npp = meta[META_NPP];
  const int lane = threadIdx.x & 31;
  const int nwarps = gridDim.x * (blockDim.x >> 5);
  for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < npp; r += nwarps) {
    const int f = sorted[r];
    const bool real = f < n_pairs;
    const uint4* src = X + (size_t)(real ? f / k : 0) * vec_per_row;
    uint4* dst = Xs + (size_t)r * vec_per_row;
    for (int v0 = lane; v0 < vec_per_row; v0 += 32 * kGatherUnroll) {
      uint4 buf[kGatherUnroll];
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const int v = v0 + 32 * u;
        buf[u] = (real && v < vec_per_row) ? src[v] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u) {
        const int v = v0 + 32 * u;
        if (v < vec_per_row) dst[v] = buf[u];
      }
    }
  }
}

// Gather + dynamic per-tensor e4m3 quantisation: code = e4m3(x / s), s = amax/448.
__global__ void k_gather_quant(const uint4* __restrict__ X, int vec_per_row /* 8 bf16 each */, int k, int n_pairs,
                               const int32_t* __restrict__ sorted, const int32_t* __restrict__ meta,
                               const unsigned* __restrict__ amax_bits, uint2* __restrict__ Xq, int late) {
  if (!late) pdl_launch_dependents();  // (late: as in k_gather_copy)
  pdl_wait();
  if (late) pdl_launch_dependents();
  const int npp = meta[META_NPP];
  const float s = e4m3_scale_from_amax(__uint_as_float(*amax_bits));
  for (int r = blockIdx.x; r < npp; r += gridDim.x) {
    const int f = sorted[r];
    uint2* dst = Xq + (size_t)r * vec_per_row;
    if (f < n_pairs) {
      const uint4* src = X + (size_t)(f / k) * vec_per_row;
      for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) {
        const uint4 x = src[v];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t q[2] = {0, 0};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t bits = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
          q[j >> 2] |= (uint32_t)f32_to_e4m3(bf16_bits_to_f32(bits) / s) << (8 * (j & 3));
        }
        dst[v] = make_uint2(q[0], q[1]);
      }
    } else {
      for (int v = threadIdx.x; v < vec_per_row; v += blockDim.x) dst[v] = make_uint2(0, 0);
    }
  }
}

// Dynamic per-tensor e4m3 quantisation of the layer input (token order; the
// GEMM gathers the rows it needs): code = e4m3(x / s), s = amax/448.
__global__ void k_quant_x(const uint4* __restrict__ X, size_t nvec, const unsigned* __restrict__ amax_bits,
                          uint2* __restrict__ Xq) {
  pdl_enter();
  const float s = e4m3_scale_from_amax(__uint_as_float(*amax_bits));
  for (size_t v = (size_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (size_t)gridDim.x * blockDim.x) {
    const uint4 x = X[v];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t q[2] = {0, 0};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t bits = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xffffu);
      q[j >> 2] |= (uint32_t)f32_to_e4m3(bf16_bits_to_f32(bits) / s) << (8 * (j & 3));
    }
    Xq[v] = make_uint2(q[0], q[1]);
  }
}

// Split-K reduction of GEMM1 partials (fixed split order), scale, SiLU(gate)*up.
// blockIdx.x walks the sorted rows, blockIdx.y a 1024-column chunk of I; each
// thread owns 4 consecutive columns (16-byte partial loads).
__global__ void __launch_bounds__(256)
    k_reduce_act(const float* __restrict__ P, int splits, size_t split_stride, int I, int B, int n_pairs,
                 const int32_t* __restrict__ sorted, const int32_t* __restrict__ eids,
                 const int32_t* __restrict__ meta, const float* __restrict__ w_scale,
                 const unsigned* __restrict__ a_amax_bits, int out_mode, void* __restrict__ A_out,
                 void* __restrict__ A_lo, unsigned* __restrict__ amax_bits) {
  pdl_enter();
  const int npp = meta[META_NPP];
  const int i = blockIdx.y * 1024 + threadIdx.x * 4;
  float m = 0.0f;
  if (i < I) {
    for (int r = blockIdx.x; r < npp; r += gridDim.x) {
      const int f = sorted[r];
      float a[4] = {0.f, 0.f, 0.f, 0.f};
      if (f < n_pairs) {  // padding rows have no partials: zeros, outside the amax
        float scale = 1.0f;
        if (w_scale) scale = e4m3_scale_from_amax(__uint_as_float(*a_amax_bits)) * w_scale[eids[r / B]];
        const float* row = P + (size_t)f * 2 * I;  // partials are indexed by pair
        float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
        for (int sp = 0; sp < splits; ++sp) {
          const float4 gv = *reinterpret_cast<const float4*>(row + (size_t)sp * split_stride + i);
          const float4 uv = *reinterpret_cast<const float4*>(row + (size_t)sp * split_stride + I + i);
          g[0] += gv.x; g[1] += gv.y; g[2] += gv.z; g[3] += gv.w;
          u[0] += uv.x; u[1] += uv.y; u[2] += uv.z; u[3] += uv.w;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (w_scale) {
            g[c] *= scale;
            u[c] *= scale;
          }
          a[c] = silu(g[c]) * u[c];
          m = fmaxf(m, fabsf(a[c]));
        }
      }
      const size_t o = (size_t)r * I + i;
      if (out_mode == 0) {
        const uint32_t h01 = pack_bf16x2(a[0], a[1]), h23 = pack_bf16x2(a[2], a[3]);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(A_out) + o) = make_uint2(h01, h23);
        if (A_lo) {
          const uint32_t l01 = pack_bf16x2(a[0] - bf16_bits_to_f32(h01 & 0xffffu), a[1] - bf16_bits_to_f32(h01 >> 16));
          const uint32_t l23 = pack_bf16x2(a[2] - bf16_bits_to_f32(h23 & 0xffffu), a[3] - bf16_bits_to_f32(h23 >> 16));
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(A_lo) + o) = make_uint2(l01, l23);
        }
      } else {
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(A_out) + o) = make_float4(a[0], a[1], a[2], a[3]);
      }
    }
  }
  if (out_mode == 1) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0 && m > 0.0f) atomicMax(amax_bits, __float_as_uint(m));
  }
}

// A_q = e4m3(A / s), s = amax/448, rows below num_post_pad.
__global__ void k_quant_act(const float4* __restrict__ A, int vec_per_row, const int32_t* __restrict__ meta,
                            const unsigned* __restrict__ amax_bits, uint32_t* __restrict__ Aq) {
  pdl_enter();
  const int npp = meta[META_NPP];
  const float s = e4m3_scale_from_amax(__uint_as_float(*amax_bits));
  const size_t total = (size_t)npp * vec_per_row;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = A[i];
    Aq[i] = (uint32_t)f32_to_e4m3(v.x / s) | ((uint32_t)f32_to_e4m3(v.y / s) << 8) |
            ((uint32_t)f32_to_e4m3(v.z / s) << 16) | ((uint32_t)f32_to_e4m3(v.w / s) << 24);
  }
}

// out[t][h] = sum_j w[t][j] * (sum_s Y[s][t*k+j][h]): splits summed in s order,
// then the k routed outputs accumulated in j order, fp32, one rounding at the
// end.  8 consecutive h per thread; the loads of four (j, s) rows are issued
// before their use so each thread keeps 8 x 16 bytes in flight.
template <bool Y_BF16>
__device__ __forceinline__ void load8(const void* Yv, size_t idx, float (&y)[8]) {
  if constexpr (Y_BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(Yv) + idx);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      y[2 * i] = bf16_bits_to_f32(w[i] & 0xffffu);
      y[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(Yv) + idx);
    const float4 b = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(Yv) + idx + 4);
    y[0] = a.x; y[1] = a.y; y[2] = a.z; y[3] = a.w;
    y[4] = b.x; y[5] = b.y; y[6] = b.z; y[7] = b.w;
  }
}

// G consecutive lanes share one output vector: lane g accumulates the routed
// slots j = g, g+G, ... (each one the sum of its K-split partials, in split
// order), then the G partial sums are added in a fixed butterfly.  The order of
// every addition is fixed, so the result is the same on every run.
template <bool Y_BF16, bool OUT_BF16, int G>
__global__ void __launch_bounds__(256) k_combine(const void* __restrict__ Yv, int splits, size_t split_stride,
                                                 const float* __restrict__ w, int T, int k, int H,
                                                 void* __restrict__ out) {
  pdl_enter();
  const int hv = H / 8;
  const size_t total = (size_t)T * hv * G;  // a multiple of G: groups never straddle the tail
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int g = (int)(i % G);
    const size_t o = i / G;
    const int t = (int)(o / hv), h = (int)(o % hv) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float yj[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    // this lane's (j, split) rows, j-major: j = g, g+G, ...; four loads in flight
    const int rows = ((k - g + G - 1) / G) * splits;
    for (int r0 = 0; r0 < rows; r0 += 4) {
      float y[4][8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q;
        if (r < rows) {
          const int j = g + (r / splits) * G, sp = r % splits;
          load8<Y_BF16>(Yv, (size_t)sp * split_stride + ((size_t)t * k + j) * H + h, y[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int r = r0 + q;
        if (r < rows) {
#pragma unroll
          for (int c = 0; c < 8; ++c) yj[c] += y[q][c];
          if (r % splits == splits - 1) {
            const float wj = w[(size_t)t * k + g + (r / splits) * G];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              acc[c] = fmaf(wj, yj[c], acc[c]);
              yj[c] = 0.f;
            }
          }
        }
      }
    }
    if constexpr (G > 1) {
      const unsigned mask = __activemask();
#pragma unroll
      for (int off = 1; off < G; off <<= 1)
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] += __shfl_xor_sync(mask, acc[c], off);
    }
    if (g != 0) continue;
    if constexpr (OUT_BF16) {
      uint4 v;
      v.x = pack_bf16x2(acc[0], acc[1]);
      v.y = pack_bf16x2(acc[2], acc[3]);
      v.z = pack_bf16x2(acc[4], acc[5]);
      v.w = pack_bf16x2(acc[6], acc[7]);
      *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + (size_t)t * H + h) = v;
    } else {
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + (size_t)t * H + h);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

// Scalar fallback of the combine for H not divisible by 4 (fp32 path only).
template <bool Y_BF16, bool OUT_BF16>
__global__ void k_combine_scalar(const void* __restrict__ Yv, int splits, size_t split_stride,
                                 const float* __restrict__ w, int T, int k, int H, void* __restrict__ out) {
  pdl_enter();
  const size_t total = (size_t)T * H;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / H), h = (int)(i % H);
    float acc = 0.f;
    for (int j = 0; j < k; ++j) {
      const size_t f = (size_t)t * k + j;
      float y = 0.f;
      for (int s = 0; s < splits; ++s) {
        if constexpr (Y_BF16)
          y += bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(Yv)[(size_t)s * split_stride + f * H + h]);
        else
          y += reinterpret_cast<const float*>(Yv)[(size_t)s * split_stride + f * H + h];
      }
      acc = fmaf(w[f], y, acc);
    }
    if constexpr (OUT_BF16)
      reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(acc);
    else
      reinterpret_cast<float*>(out)[i] = acc;
  }
}

int grid_for(size_t work, int threads, int cap_blocks = 152 * 16) {
  size_t b = (work + threads - 1) / threads;
  if (b < 1) b = 1;
  if (b > (size_t)cap_blocks) b = cap_blocks;
  return (int)b;
}

}  // namespace

cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int B, int32_t* sorted, int32_t* eids,
                         int32_t* npp, int32_t* counts, int32_t* meta, int* status, cudaStream_t s,
                         bool skip_minus_one, int32_t* pblk, unsigned* zero_words, int n_zero, int32_t* inv) {
  if (pblk && B != 128) return cudaErrorInvalidValue;
  if (n_zero > 0 && !zero_words) return cudaErrorInvalidValue;
  if ((long)T * k <= 32 && !pblk) {
    MOE_LAUNCH(k_align_small, dim3(1), dim3(kAlignSmallThreads), 0, s, ids, T * k, E, B, sorted, eids, npp, counts,
               meta, status, skip_minus_one ? 1 : 0, zero_words, n_zero, inv);
    return cudaGetLastError();
  }
  if ((long)T * k <= kAlignThreads && !pblk) {
    static bool mid_configured[64] = {};
    int mdev = 0;
    cudaGetDevice(&mdev);
    if (mdev < 0 || mdev >= 64 || !mid_configured[mdev]) {
      cudaError_t e = cudaFuncSetAttribute(k_align_mid, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (e != cudaSuccess) return e;
      if (mdev >= 0 && mdev < 64) mid_configured[mdev] = true;
    }
    const size_t msmem = (size_t)(kAlignWarps * E + 2 * E + 1) * sizeof(int);
    MOE_LAUNCH(k_align_mid, dim3(1), dim3(kAlignThreads), msmem, s, ids, T * k, E, B, sorted, eids, npp, counts, meta,
               status, skip_minus_one ? 1 : 0, zero_words, n_zero, inv);
    return cudaGetLastError();
  }
  const size_t smem = (size_t)(kAlignWarps * E + 4 * E + 1 + 33) * sizeof(int);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_align, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  // one CTA up to 4096 pairs, then a cluster of up to 8 CTAs (about 4096 pairs each)
  const long n = (long)T * k;
  const int csize = (int)std::min<long>(8, std::max<long>(1, (n + 4095) / 4096));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(csize);
  cfg.blockDim = dim3(kAlignThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  // programmatic dependent launch, like every kernel of the library: the CTAs launch
  // while the top-k kernel drains and wait (griddepcontrol.wait) before reading its ids
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_align, ids, T, k, E, B, sorted, eids, npp, counts, meta, status,
                            skip_minus_one ? 1 : 0, pblk, zero_words, n_zero, inv);
}

cudaError_t launch_amax_bf16(const void* X, size_t n, unsigned* amax_bits, cudaStream_t s) {
  MOE_LAUNCH(k_amax_bf16, dim3(grid_for(n, 256)), dim3(256), 0, s, (const uint16_t*)X, n, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* X, int T, int H, int k, int elem_bytes, int mode, const unsigned* amax_bits,
                          const int32_t* sorted, const int32_t* inv, const int32_t* meta, int cap, void* Xs,
                          bool late, cudaStream_t s) {
  const int grid = cap < 152 * 8 ? (cap > 0 ? cap : 1) : 152 * 8;
  if (mode == 0) {
    const int vpr = H * elem_bytes / 16;
    if (inv) {
      if (k > 32) return cudaErrorInvalidValue;
      constexpr int wpb = kGatherThreads / 32;
      const int blocks = std::max(1, std::min((T + wpb - 1) / wpb, 152 * 32));  // one warp per token
      MOE_LAUNCH(k_gather_scatter, dim3(blocks), dim3(kGatherThreads), 0, s, (const uint4*)X, vpr, T, k, T * k, inv,
                 sorted, meta, (uint4*)Xs);
    } else {
      const int rows_grid = std::max(1, std::min((cap + 7) / 8, 152 * 8));  // 8 warps (rows) per CTA
      MOE_LAUNCH(k_gather_copy, dim3(rows_grid), dim3(256), 0, s, (const uint4*)X, vpr, k, T * k, sorted, meta,
                 (uint4*)Xs, late ? 1 : 0);
    }
  } else {
    const int vpr = H / 8;
    MOE_LAUNCH(k_gather_quant, dim3(grid), dim3(128), 0, s, (const uint4*)X, vpr, k, T * k, sorted, meta, amax_bits,
               (uint2*)Xs, late ? 1 : 0);
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_x(const void* X, size_t n, const unsigned* amax_bits, uint8_t* Xq, cudaStream_t s) {
  MOE_LAUNCH(k_quant_x, dim3(grid_for(n / 8, 256)), dim3(256), 0, s, (const uint4*)X, n / 8, amax_bits, (uint2*)Xq);
  return cudaGetLastError();
}

cudaError_t launch_reduce_act(const float* P, int splits, size_t split_stride, int I, int B, int n_pairs,
                              const int32_t* sorted, const int32_t* eids, const int32_t* meta, int cap,
                              const float* w_scale, const unsigned* a_amax_bits, int out_mode, void* A_out,
                              void* A_lo, unsigned* amax_bits, cudaStream_t s) {
  const int chunks = (I + 1023) / 1024;
  const int rows = std::max(1, std::min(cap, std::max(1, 152 * 8 / chunks)));
  MOE_LAUNCH(k_reduce_act, dim3(rows, chunks), dim3(256), 0, s, P, splits, split_stride, I, B, n_pairs, sorted, eids,
             meta, w_scale, a_amax_bits, out_mode, A_out, A_lo, amax_bits);
  return cudaGetLastError();
}

cudaError_t launch_quant_act(const float* A, int I, const int32_t* meta, int cap, const unsigned* amax_bits,
                             uint8_t* Aq, cudaStream_t s) {
  const int vpr = I / 4;
  MOE_LAUNCH(k_quant_act, dim3(grid_for((size_t)cap * vpr, 256)), dim3(256), 0, s, (const float4*)A, vpr, meta, amax_bits,
                                                               (uint32_t*)Aq);
  return cudaGetLastError();
}

int combine_lanes(int T, int H, int k) {
  // small batches: split each output's routed slots over G lanes for more parallelism
  const size_t vecs = (size_t)T * (H / 8);
  return vecs >= (size_t)152 * 2048 ? 1 : (k >= 4 ? 4 : (k >= 2 ? 2 : 1));
}

template <bool YB, bool OB>
static cudaError_t combine_vec(const void* Y, int splits, size_t split_stride, const float* w, int T, int k, int H,
                               void* out, cudaStream_t s) {
  const int G = combine_lanes(T, H, k);
  const size_t vecs = (size_t)T * (H / 8);
  const int grid = grid_for(vecs * G, 256);
  if (G == 4) MOE_LAUNCH(k_combine<YB, OB, 4>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  else if (G == 2) MOE_LAUNCH(k_combine<YB, OB, 2>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  else MOE_LAUNCH(k_combine<YB, OB, 1>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* Y, int y_bf16, int splits, size_t split_stride, const float* w, int T, int k,
                           int H, void* out, int out_bf16, cudaStream_t s) {
  if (H % 8 == 0) {
    if (y_bf16 && out_bf16) return combine_vec<true, true>(Y, splits, split_stride, w, T, k, H, out, s);
    if (y_bf16) return combine_vec<true, false>(Y, splits, split_stride, w, T, k, H, out, s);
    if (out_bf16) return combine_vec<false, true>(Y, splits, split_stride, w, T, k, H, out, s);
    return combine_vec<false, false>(Y, splits, split_stride, w, T, k, H, out, s);
  }
  const int grid = grid_for((size_t)T * H, 256);
  if (y_bf16 && out_bf16) MOE_LAUNCH(k_combine_scalar<true, true>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  else if (y_bf16) MOE_LAUNCH(k_combine_scalar<true, false>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  else if (out_bf16) MOE_LAUNCH(k_combine_scalar<false, true>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  else MOE_LAUNCH(k_combine_scalar<false, false>, dim3(grid), dim3(256), 0, s, Y, splits, split_stride, w, T, k, H, out);
  return cudaGetLastError();
}

}  // namespace moe
