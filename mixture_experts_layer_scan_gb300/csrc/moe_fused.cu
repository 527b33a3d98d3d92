// Single-launch decode layer: router, top-k, permutation, both expert GEMMs
// and the weighted combine in one cooperative persistent kernel (bf16,
// swap-AB orientation).
//
// "Mixture-of-Experts kernel engineering on Amazon SageMaker AI", intro: the
// routing, the data shuffle and the expert networks become one batched GPU
// operation; "FusedMoE vs MegaMoE" (zwxr.cn), section 3.1: one fused kernel
// sorts the tokens by expert, computes, then reorders and sums the results
// with the routing weights.  At decode sizes the layer's multi-kernel
// sequence spends more time in launch gaps and pipeline fill than in
// streaming expert weights; here every phase boundary is a grid barrier or a
// per-expert counter inside one launch.
//
// Phases (every CTA, 256 threads):
//   0  router logits, (expert, 4-token group) units spread over the CTAs
//   -- grid barrier --
//   1  top-k and softmax weights, one warp per token (up to 8 tokens: every
//      CTA ranks all tokens itself and skips the next barrier)
//   -- grid barrier --
//   2  every CTA builds the expert tables of the batch in shared memory
//      (stable counting sort of the (token, slot) pairs); batches over 32
//      tokens also gather their token rows into expert order, then
//   -- grid barrier --
//   3  one tile list: all GEMM1 tiles, then all GEMM2 tiles, dealt round-robin
//      to the CTAs (each CTA runs its GEMM1 tiles before its GEMM2 tiles).
//      Warp 0 streams weight and activation tiles with TMA, warp 1 issues
//      tcgen05.mma, warps 2-5 run the epilogues:
//        GEMM1 tile (expert e, 128 intermediate columns, K split s): SiLU(gate)*up
//          into the bf16 intermediate (hi + lo parts); with K splits, fp32
//          partials, and the CTA that completes the last split of a tile sums
//          them in split order.  A finished tile sets its ready flag.
//        GEMM2 tile (expert e, 256 hidden rows, K split s): fp32 Y rows; its
//          producer streams the W2 tiles at once and loads the intermediate
//          columns of each K block once the GEMM1 tile that produces them is
//          final.  For every token of the tile a counter per (token, 256
//          hidden rows) counts the arrived (slot, split) outputs.
//      Warps 6-7, and every other warp once its role is done, run the combine:
//      they claim (token, 128 hidden rows) units from a grid-wide counter, wait
//      for the unit's count and write the weighted sum over the k slots.
//
// Every arithmetic step is the one the multi-kernel path performs, in the same
// order (same tiles, K splits, MMA sequence, split-order sums, combine order),
// so both paths give bit-identical outputs.
//
// The blocks wait on one another, so the kernel is launched cooperatively (all
// CTAs resident).  Every wait is bounded (a timeout records
// MOE_ERR_DEVICE_TIMEOUT and the kernel winds down).  The barrier and
// dependency counters live in the workspace: CTA 0 zeroes them at the start of
// each launch and then publishes the launch's grid id (%gridid, unique per
// launch in a context); no CTA touches a counter before it has seen that id.
// The host clears the tag word on the stream before each launch, so stale
// workspace contents can never pass for the tag.
#include <algorithm>

#include "moe_device.cuh"
#include "moe_internal.h"
#include "moe_route.cuh"

namespace moe {

namespace {

constexpr int kFThreads = 256;  // 8 warps
constexpr int kFMaxStages = 8;
constexpr int kFRouterTT = 16;  // tokens per router unit
constexpr uint32_t kFTmemCols = 512;
constexpr int kFBarBytes = 256;  // mbarriers + small shared words

// words of the sync region: three grid barriers, the exit count, the next free
// combine unit, then the dependency counters
enum { SYNC_BAR0 = 0, SYNC_EXIT = 3, SYNC_CNEXT = 4, SYNC_NBAR = 8 };

struct FusedDev {
  int T, H, I, E, k, renorm;
  int n1, s1, kbs1, kbt1;  // GEMM1: tiles per expert (I/128), K splits, K blocks per split, K blocks
  int n2, s2, kbs2, kbt2;  // GEMM2: tiles per expert (ceil(H/256)), ...
  int xbox;                // activation rows per tile load (tokens rounded up to 16)
  int gather;              // 1: GEMM1 gathers token rows with tile::gather4; 0: rows gathered into Xs
  int act_split;           // intermediate stored as bf16 hi + lo
  int cap;                 // rows of Xs and of each intermediate part
  int combine_g;           // lanes per output of the stand-alone combine (1, 2, 4): same sum order here
  int stages;
  uint32_t stage_bytes, bar_off, tab_off;
  const __nv_bfloat16* X;
  const __nv_bfloat16* Wr;
  float* logits;
  float* topk_w;
  int32_t* topk_ids;
  __nv_bfloat16* Xs;     // [cap][H] token rows in expert order (gather == 0)
  __nv_bfloat16* aint;   // [cap][I] hi part, then [cap][I] lo part
  float* p1;             // GEMM1 K-split partials [s1][T*k][2I]
  size_t p1_stride;
  float* y;              // GEMM2 outputs [s2][T*k][H]
  size_t y_stride;
  __nv_bfloat16* out;    // [T][H]
  unsigned long long* trace;  // nullable: MOE_TRACE_WORDS %globaltimer stamps per CTA
  unsigned long long* go;  // grid id of the launch whose counters are zeroed
  unsigned* sync;          // SYNC_NBAR barrier words, arr1[E*n1], ready1[E*n1], cnt2[T*n2]
  int nsync;
  int* status;
};

// shared words after the mbarriers
enum { SW_TMEM = 0, SW_ABORT = 1, SW_FLAG = 2, SW_LAST = 3, SW_NACT = 4, SW_NPP = 5 };

__device__ __forceinline__ uint64_t grid_id() {
  uint64_t g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return g;
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const unsigned long long* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(unsigned long long* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// generic-proxy global writes before this point are ordered before later
// async-proxy (TMA) accesses, and vice versa
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// atomic add with release (this thread's earlier writes, and those ordered
// before it by a CTA barrier, become visible to an acquirer of the new value)
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned atom_acq_rel_add(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}


// The same wait by a whole warp: every lane polls, the outcome is decided
// warp-wide each round (see mbar_wait_all).
__device__ __forceinline__ bool warp_wait_geq(const unsigned* p, unsigned target, volatile int* abort, int* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (__all_sync(0xffffffffu, ld_acquire_u32(p) >= target)) return true;
    if (it == 0) t0 = globaltimer_ns();
    if ((it & 15u) == 15u) {
      const bool give_up = (abort && *abort) || (globaltimer_ns() - t0 > kWaitLimitNs);
      if (__any_sync(0xffffffffu, give_up)) {
        if ((threadIdx.x & 31) == 0 && !(abort && *abort)) {
          if (abort) *abort = 1;
          report(status, MOE_ERR_DEVICE_TIMEOUT);
        }
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool warp_wait_tag(const unsigned long long* p, uint64_t tag, int* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (__all_sync(0xffffffffu, ld_acquire_u64(p) == tag)) return true;
    if (it == 0) t0 = globaltimer_ns();
    if ((it & 15u) == 15u && __any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitLimitNs)) {
      if ((threadIdx.x & 31) == 0) report(status, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Grid barrier number b (each barrier of a launch has its own zeroed word).
// Thread 0 first waits for CTA 0 to have zeroed this launch's counters, then
// arrives and waits for all CTAs; the CTA's own writes are ordered before its
// arrival by the CTA barrier + release, and the other CTAs' writes before its
// later reads by the acquire + CTA barrier.  Returns false (for the whole CTA)
// on timeout.
__device__ bool grid_barrier(const FusedDev& p, int b, uint64_t gid, int* sw) {
  cta_sync();
  if (threadIdx.x < 32) {  // warp 0, all lanes together
    bool ok = warp_wait_tag(p.go, gid, p.status);
    if (ok) {
      if (threadIdx.x == 0) red_release_add(p.sync + SYNC_BAR0 + b, 1u);
      __syncwarp();
      ok = warp_wait_geq(p.sync + SYNC_BAR0 + b, gridDim.x, nullptr, p.status);
    }
    if (threadIdx.x == 0) sw[SW_FLAG] = ok ? 1 : 0;
  }
  cta_sync();
  return sw[SW_FLAG] != 0;
}

__device__ __forceinline__ void stamp(const FusedDev& p, int ev) {
  if (p.trace) p.trace[blockIdx.x * MOE_TRACE_WORDS + ev] = globaltimer_ns();
}

// One output tile of the fused tile list.
struct FTile {
  int g2;          // 0: GEMM1 tile, 1: GEMM2 tile
  int e, n, s;     // expert, weight tile, K split
  int xrow;        // first padded row of the expert (intermediate / Xs rows)
  int lbase;       // first entry of the expert in the stable pair list
  int ntok, npad;  // tokens of the expert, rounded up to 16
  int wr0, pair_off;
  int kb0, kb1;
};

__device__ __forceinline__ FTile ftile_at(const FusedDev& p, int t, int n_g1, const int* act, const int* cnt,
                                          const int* off, const int* poff) {
  FTile d;
  int per, kbs, kbt;
  if (t < n_g1) {
    d.g2 = 0;
    per = p.n1 * p.s1;
    kbs = p.kbs1;
    kbt = p.kbt1;
  } else {
    t -= n_g1;
    d.g2 = 1;
    per = p.n2 * p.s2;
    kbs = p.kbs2;
    kbt = p.kbt2;
  }
  const int splits = d.g2 ? p.s2 : p.s1;
  const int a = t / per;
  const int rem = t - a * per;
  d.n = rem / splits;
  d.s = rem - d.n * splits;
  d.e = act[a];
  d.xrow = poff[d.e];
  d.lbase = off[d.e];
  d.ntok = cnt[d.e];
  d.npad = (d.ntok + 15) & ~15;
  d.kb0 = d.s * kbs;
  d.kb1 = min(d.kb0 + kbs, kbt);
  if (d.g2) {
    d.wr0 = d.e * p.H + d.n * 256;
    d.pair_off = 128;
  } else {
    d.wr0 = d.e * 2 * p.I + d.n * 128;
    d.pair_off = p.I;
  }
  return d;
}

// OR of a flag over the 128 epilogue threads (named barrier 1) / the 64 combine threads (named barrier 2).
__device__ __forceinline__ bool f_epi_any(bool v) { return named_bar_any(1, 128, v); }
__device__ __forceinline__ bool f_comb_any(bool v) { return named_bar_any(2, 64, v); }

// out[t][h4 .. h4+3] for one token, with the arithmetic of the stand-alone
// combine: lane g of G sums the slots j = g, g+G, ... (each the sum of its
// K-split outputs in split order) with fma, then the G partial sums are added
// in its butterfly order.  The (slot, split) rows are visited in their natural
// order, which keeps every lane's chain in order; their 16-byte loads go out
// eight rows at a time (the tail of a batch re-reads the last row).
template <int G>
__device__ __forceinline__ void combine_unit(const FusedDev& p, int t, int h4, const float* wsm) {
  float acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[g][q] = 0.0f;
  float yj[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const int rows = p.k * p.s2;
  const float* ybase = p.y + (size_t)t * p.k * p.H + h4;
  for (int r0 = 0; r0 < rows; r0 += 8) {
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = min(r0 + i, rows - 1);
      const int j = r / p.s2, sp = r - j * p.s2;
      v[i] = __ldcg(reinterpret_cast<const float4*>(ybase + (size_t)sp * p.y_stride + (size_t)j * p.H));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = r0 + i;
      if (r < rows) {
        const int j = r / p.s2, sp = r - j * p.s2;
        yj[0] += v[i].x;
        yj[1] += v[i].y;
        yj[2] += v[i].z;
        yj[3] += v[i].w;
        if (sp == p.s2 - 1) {
          const float w = wsm[j];
          const int gj = j % G;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if (g == gj) {
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[g][q] = fmaf(w, yj[q], acc[g][q]);
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) yj[q] = 0.0f;
        }
      }
    }
  }
  float o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if constexpr (G == 4)
      o[q] = (acc[0][q] + acc[1][q]) + (acc[2][q] + acc[3][q]);
    else if constexpr (G == 2)
      o[q] = acc[0][q] + acc[1][q];
    else
      o[q] = acc[0][q];
  }
  *reinterpret_cast<uint2*>(p.out + (size_t)t * p.H + h4) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
}

// The combine as a pool of work: a warp whose own role is finished claims the
// next unit (token t, 128 hidden rows) from a grid-wide counter, waits until
// all k slots x s2 splits of GEMM2 output for those rows have arrived, and
// writes their weighted sum (4 hidden rows per lane).
__device__ __forceinline__ void combine_worker(const FusedDev& p, const unsigned* cnt2, const float* tws, bool ok,
                                               volatile int* abort_flag, bool stamp_first) {
  const int lane = threadIdx.x & 31;
  const int units = ok ? p.T * p.n2 * 2 : 0;
  const unsigned target = (unsigned)(p.k * p.s2);
  bool first = stamp_first;
  for (;;) {
    unsigned u = 0;
    if (lane == 0) u = atomicAdd(p.sync + SYNC_CNEXT, 1u);
    u = __shfl_sync(0xffffffffu, u, 0);
    if ((int)u >= units) break;
    const int t = (int)u / (2 * p.n2);
    const int rem = (int)u - t * 2 * p.n2;
    const int nn = rem >> 1, half = rem & 1;
    if (!warp_wait_geq(cnt2 + t * p.n2 + nn, target, abort_flag, p.status)) break;
    if (first && lane == 0) stamp(p, MOE_TRACE_COMB_FIRST);
    first = false;
    const int h4 = nn * 256 + half * 128 + 4 * lane;
    if (h4 < p.H) {
      if (p.combine_g == 4)
        combine_unit<4>(p, t, h4, tws + t * p.k);
      else if (p.combine_g == 2)
        combine_unit<2>(p, t, h4, tws + t * p.k);
      else
        combine_unit<1>(p, t, h4, tws + t * p.k);
    }
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kFThreads, 1)
    k_decode_fused(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW2,
                   const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA,
                   const FusedDev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + p.bar_off;
  const uint32_t bar_empty = bar_full + 8 * kFMaxStages;
  const uint32_t bar_tfull = bar_empty + 8 * kFMaxStages;
  const uint32_t bar_tempty = bar_tfull + 16;
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_exit = bar_drain + 8;
  int* sw = reinterpret_cast<int*>(smem + p.bar_off + 8 * (2 * kFMaxStages + 6));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sw + SW_ABORT);

  const int T = p.T, E = p.E, k = p.k;
  const int n = T * k;
  // shared tables
  float* red = reinterpret_cast<float*>(smem + p.tab_off);  // [kRouterWarps * kFRouterTT]
  int* sid = reinterpret_cast<int*>(red + kRouterWarps * kFRouterTT);  // [n] expert of each pair
  int* rank = sid + n;        // [n] rank of the pair inside its expert
  int* plist = rank + n;      // [n] pairs in expert order (stable)
  int* prow = plist + n;      // [n] padded row of each plist entry
  int* cnt = prow + n;        // [E] pairs per expert
  int* off = cnt + E;         // [E+1] first plist entry of each expert
  int* poff = off + E + 1;    // [E+1] first padded row of each expert (blocks of 16)
  int* act = poff + E + 1;    // [E] active experts, ascending
  float* tws = reinterpret_cast<float*>(act + E);  // [n] routing weights of every pair

  unsigned* arr1 = p.sync + SYNC_NBAR;        // [E * n1] GEMM1 split arrivals
  unsigned* ready1 = arr1 + E * p.n1;         // [E * n1] 1 once a GEMM1 tile's intermediate columns are final
  unsigned* cnt2 = ready1 + E * p.n1;         // [T * n2] arrived GEMM2 outputs per (token, hidden tile)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 128);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_exit, kFThreads / 32);
    sw[SW_ABORT] = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW1);
    tma_prefetch_desc(&tmW2);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) tmem_alloc(smem_u32(sw + SW_TMEM), kFTmemCols);
  const uint64_t gid = grid_id();
  if (blockIdx.x == 0) {
    // this launch's counters start at zero; published under the launch's grid id
    for (int i = threadIdx.x; i < p.nsync; i += blockDim.x) p.sync[i] = 0u;
    __threadfence();
    cta_sync();
    if (threadIdx.x == 0) st_release_u64(p.go, gid);
  }
  tc_fence_before();
  cta_sync();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)sw[SW_TMEM];
  bool ok = true;
  if (threadIdx.x == 0) stamp(p, MOE_TRACE_START);

  // ---------------- phase 0: router logits ----------------
  {
    const int units = ((T + kFRouterTT - 1) / kFRouterTT) * E;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const int e = u % E, t0 = (u / E) * kFRouterTT;
      router_block<__nv_bfloat16, kFRouterTT>(p.X, p.Wr, T, p.H, E, t0, e, p.logits, red);
    }
  }
  if (threadIdx.x == 0) stamp(p, MOE_TRACE_ROUTER);
  ok = grid_barrier(p, 0, gid, sw);
  if (threadIdx.x == 0) stamp(p, MOE_TRACE_BARRIER0);

  // ---------------- phase 1: top-k ----------------
  // Up to one token per warp: every CTA ranks all tokens itself, into shared
  // memory (same code, same logits, same result in every CTA; no barrier).
  // Longer batches: one warp per token over the grid, then a grid barrier.
  const bool local_topk = T <= kFThreads / 32;
  if (ok) {
    if (local_topk) {
      if (warp < T) topk_warp<true>(p.logits + (size_t)warp * E, E, k, p.renorm, tws + warp * k, sid + warp * k);
      if (lane == 0) stamp(p, MOE_TRACE_TOPK);
      cta_sync();
      if (threadIdx.x == 0) stamp(p, MOE_TRACE_BARRIER1);
    } else {
      for (int t = blockIdx.x * (kFThreads / 32) + warp; t < T; t += gridDim.x * (kFThreads / 32))
        topk_warp<true>(p.logits + (size_t)t * E, E, k, p.renorm, p.topk_w + (size_t)t * k,
                        p.topk_ids + (size_t)t * k);
      if (lane == 0) stamp(p, MOE_TRACE_TOPK);
      ok = grid_barrier(p, 1, gid, sw);
      if (threadIdx.x == 0) stamp(p, MOE_TRACE_BARRIER1);
    }
  }

  // ---------------- phase 2: expert tables (every CTA) ----------------
  if (ok) {
    bool bad = false;
    for (int f = threadIdx.x; f < n; f += blockDim.x) {
      int e;
      if (local_topk) {
        e = sid[f];
      } else {
        e = __ldcg(p.topk_ids + f);
        tws[f] = __ldcg(p.topk_w + f);
      }
      if (e < 0 || e >= E) {
        bad = true;
        e = -1;
      }
      sid[f] = e;
    }
    if (bad) report(p.status, MOE_ERR_DEVICE_INDEX);
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    cta_sync();
    if (warp == 0) {
      // ranks inside each expert in ascending pair order (warp match, no atomics)
      for (int base = 0; base < n; base += 32) {
        const int f = base + lane;
        const int e = (f < n) ? sid[f] : -1;
        const unsigned grp = __match_any_sync(0xffffffffu, e);
        if (e >= 0) rank[f] = cnt[e] + __popc(grp & ((1u << lane) - 1u));
        __syncwarp();
        if (e >= 0 && lane == __ffs(grp) - 1) cnt[e] += __popc(grp);
        __syncwarp();
      }
    }
    cta_sync();
    if (warp == 0) {
      // exclusive scans: list offsets, padded row offsets (blocks of 16), active experts
      int run = 0, prun = 0, arun = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int c = (e < E) ? cnt[e] : 0;
        const int pc = (c + 15) & ~15;
        const int a = c > 0 ? 1 : 0;
        int ic = c, ip = pc, ia = a;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x1 = __shfl_up_sync(0xffffffffu, ic, o);
          const int x2 = __shfl_up_sync(0xffffffffu, ip, o);
          const int x3 = __shfl_up_sync(0xffffffffu, ia, o);
          if (lane >= o) {
            ic += x1;
            ip += x2;
            ia += x3;
          }
        }
        if (e < E) {
          off[e] = run + ic - c;
          poff[e] = prun + ip - pc;
          if (a) act[arun + ia - 1] = e;
        }
        run += __shfl_sync(0xffffffffu, ic, 31);
        prun += __shfl_sync(0xffffffffu, ip, 31);
        arun += __shfl_sync(0xffffffffu, ia, 31);
      }
      if (lane == 0) {
        off[E] = run;
        poff[E] = prun;
        sw[SW_NACT] = arun;
        sw[SW_NPP] = prun;
      }
    }
    cta_sync();
    for (int f = threadIdx.x; f < n; f += blockDim.x) {
      const int e = sid[f];
      if (e >= 0) {
        const int q = off[e] + rank[f];
        plist[q] = f;
        prow[q] = poff[e] + rank[f];
      }
    }
    cta_sync();
    if (threadIdx.x == 0) stamp(p, MOE_TRACE_TABLES);
    if (!p.gather) {
      // token rows into expert order, spread over all CTAs (16-byte vectors)
      const int vpr = p.H / 8;
      const int nvalid = off[E];
      const size_t total = (size_t)nvalid * vpr;
      const uint4* X4 = reinterpret_cast<const uint4*>(p.X);
      uint4* Xs4 = reinterpret_cast<uint4*>(p.Xs);
      for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
           i += (size_t)gridDim.x * blockDim.x) {
        const int q = (int)(i / vpr), v = (int)(i - (size_t)q * vpr);
        Xs4[(size_t)prow[q] * vpr + v] = X4[(size_t)(plist[q] / k) * vpr + v];
      }
      fence_proxy_async_global();
      ok = grid_barrier(p, 2, gid, sw);
    }
    if (threadIdx.x == 0) stamp(p, MOE_TRACE_GATHERED);
  }


  // ---------------- phase 3: expert GEMMs ----------------
  const int nact = sw[SW_NACT];
  const int n_g1 = nact * p.n1 * p.s1;
  const int ntiles = ok ? n_g1 + nact * p.n2 * p.s2 : 0;
  constexpr uint32_t kWBytes = 2u * 128u * 128u;  // two 128-row weight loads of 128 bytes of K
  const uint32_t x1_bytes = (uint32_t)p.xbox * 128u;
  const uint32_t x2_bytes = x1_bytes * (p.act_split ? 2u : 1u);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    int stage = 0;
    uint32_t phase = 0, issued = 0;
    bool okp = true;
    const int groups = p.xbox / 4;  // gather4 groups per activation tile (<= 16)
    int pend_stage[kFMaxStages], pend_kb[kFMaxStages];
    bool g1_stamped = false, ready_stamped = false;
    for (int t = blockIdx.x; t < ntiles && okp; t += gridDim.x) {
      const FTile d = ftile_at(p, t, n_g1, act, cnt, off, poff);
      const CUtensorMap* tmw = d.g2 ? &tmW2 : &tmW1;
      if (d.g2 && !g1_stamped && lane == 0) {
        stamp(p, MOE_TRACE_G1_ISSUED);
        g1_stamped = true;
      }
      int rows[4] = {0, 0, 0, 0};  // token rows of this lane's gather group (GEMM1, gather mode)
      if (!d.g2 && p.gather) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * lane + i;
          rows[i] = (r < d.ntok) ? plist[d.lbase + r] / k : 0;  // padding rows read token 0; never stored
        }
      }
      // GEMM2: weight tiles go out at once; the intermediate columns of K block kb
      // (GEMM1 tile kb/2 of the expert) once that tile is final.  Stages still
      // waiting for their columns queue up in order (lane 0 keeps the queue).
      int qhead = 0, npend = 0;
      const unsigned* rdy = ready1 + d.e * p.n1;
      auto load_a = [&](int st, int kb) {
        if (!ready_stamped) {
          stamp(p, MOE_TRACE_G2_READY);
          ready_stamped = true;
        }
        const uint32_t sx = sbase + st * p.stage_bytes + kWBytes;
        const uint32_t fb = bar_full + 8 * st;
        tma_load_2d(sx, &tmA, kb * 64, d.xrow, fb);
        if (p.act_split) tma_load_2d(sx + x1_bytes, &tmA, kb * 64, d.xrow + p.cap, fb);
      };
      auto flush_ready = [&]() {  // lane 0: the queued loads whose columns are final, in order
        bool fenced = false;
        while (npend > 0 && ld_acquire_u32(rdy + (pend_kb[qhead] >> 1)) != 0u) {
          if (!fenced) {
            fence_proxy_async_global();
            fenced = true;
          }
          load_a(pend_stage[qhead], pend_kb[qhead]);
          qhead = (qhead + 1) % kFMaxStages;
          --npend;
        }
      };
      for (int kb = d.kb0; kb < d.kb1; ++kb) {
        if (npend == p.stages) {
          // every stage holds weights waiting for intermediate columns: wait for the oldest
          const int head_kb = __shfl_sync(0xffffffffu, pend_kb[qhead], 0);
          if (!warp_wait_geq(rdy + (head_kb >> 1), 1u, abort_flag, p.status)) {
            okp = false;
            break;
          }
          if (lane == 0) flush_ready();
          npend = __shfl_sync(0xffffffffu, npend, 0);
        }
        if (!mbar_wait_all(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.status)) {
          okp = false;
          break;
        }
        if (lane == 0) {
          const uint32_t sws = sbase + stage * p.stage_bytes;
          const uint32_t fb = bar_full + 8 * stage;
          mbar_arrive_expect_tx(fb, kWBytes + (d.g2 ? x2_bytes : x1_bytes));
          tma_load_2d(sws, tmw, kb * 64, d.wr0, fb);
          tma_load_2d(sws + kWBytes / 2, tmw, kb * 64, d.wr0 + d.pair_off, fb);
          if (d.g2) {
            flush_ready();
            if (npend == 0 && ld_acquire_u32(rdy + (kb >> 1)) != 0u) {
              fence_proxy_async_global();
              load_a(stage, kb);
            } else {
              const int slot = (qhead + npend) % kFMaxStages;
              pend_stage[slot] = stage;
              pend_kb[slot] = kb;
              ++npend;
            }
          } else if (!p.gather) {
            tma_load_2d(sws + kWBytes, &tmX, kb * 64, d.xrow, fb);
          }
        }
        npend = __shfl_sync(0xffffffffu, npend, 0);
        if (!d.g2 && p.gather && lane < groups)
          tma_gather4(sbase + stage * p.stage_bytes + kWBytes + (uint32_t)lane * 512u, &tmX, kb * 64, rows[0],
                      rows[1], rows[2], rows[3], bar_full + 8 * stage);
        __syncwarp();
        ++issued;
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      while (okp && npend > 0) {
        const int head_kb = __shfl_sync(0xffffffffu, pend_kb[qhead], 0);
        if (!warp_wait_geq(rdy + (head_kb >> 1), 1u, abort_flag, p.status)) {
          okp = false;
          break;
        }
        if (lane == 0) flush_ready();
        npend = __shfl_sync(0xffffffffu, npend, 0);
      }
      __syncwarp();
    }
    if (lane == 0) {
      if (!g1_stamped) stamp(p, MOE_TRACE_G1_ISSUED);
      stamp(p, MOE_TRACE_ISSUED);
    }
    if (lane == 0 && !okp) {
      // let the copies already in flight land before the CTA exits (pending
      // stages never receive their intermediate: their waits time out)
      const uint32_t first = issued > (uint32_t)p.stages ? issued - p.stages : 0u;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_drain(bar_full + 8 * (i % p.stages), (i / p.stages) & 1u, 100000000ull);
    }
    __syncwarp();
    combine_worker(p, cnt2, tws, ok, abort_flag, false);
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // the whole warp runs the loop and waits together; lane 0 issues the MMAs and their commits
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool okm = true, any = false;
    for (int t = blockIdx.x; t < ntiles && okm; t += gridDim.x) {
      const FTile d = ftile_at(p, t, n_g1, act, cnt, off, poff);
      // GEMM2 with a hi/lo intermediate: one MMA over the xbox hi rows then the lo rows
      const bool stacked = d.g2 && p.act_split;
      const uint32_t idesc = idesc_make(128, stacked ? p.xbox + d.npad : d.npad, false);
      if (!mbar_wait_all(bar_tempty + 8 * acc, acc_phase ^ 1u, abort_flag, p.status)) {
        okm = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + (uint32_t)(acc * 256);
      const int parts = 1;
      for (int kb = d.kb0; kb < d.kb1; ++kb) {
        if (!mbar_wait_all(bar_full + 8 * stage, phase, abort_flag, p.status)) {
          okm = false;
          break;
        }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sws = sbase + stage * p.stage_bytes;
          const uint32_t sx = sws + kWBytes;
          // D0 += W[rows 0..127] X^T, D1 += W[rows 128..255] X^T (GEMM2 with a hi/lo intermediate: X^T
          // is the hi rows then the lo rows, whose products the epilogue adds)
          for (int part = 0; part < parts; ++part) {
            const uint32_t sxp = sx + (uint32_t)part * x1_bytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc_in = (part > 0 || kb > d.kb0 || kk > 0) ? 1u : 0u;
              const uint64_t bdesc = sdesc_k_sw128(sxp + kk * 32);
              tc_mma<false>(dt, sdesc_k_sw128(sws + kk * 32), bdesc, idesc, acc_in);
              tc_mma<false>(dt + 128u, sdesc_k_sw128(sws + kWBytes / 2 + kk * 32), bdesc, idesc, acc_in);
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
      if (!okm) break;
      if (lane == 0) tc_commit(bar_tfull + 8 * acc);
      __syncwarp();
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) stamp(p, MOE_TRACE_MMA_DONE);
    if (!okm && any) {  // the tensor core must be idle before tensor memory is freed
      if (lane == 0) tc_commit(bar_drain);
      __syncwarp();
      mbar_wait_drain(bar_drain, 0, 100000000ull);
    }
    __syncwarp();
    combine_worker(p, cnt2, tws, ok, abort_flag, false);
  } else if (warp < 6) {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;          // tensor-memory lane quadrant of this warp
    const int lrow = q * 32 + lane;  // accumulator row of this thread
    const int I = p.I, H = p.H;
    __nv_bfloat16* a_hi = p.aint;
    __nv_bfloat16* a_lo = p.act_split ? p.aint + (size_t)p.cap * I : nullptr;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const FTile d = ftile_at(p, t, n_g1, act, cnt, off, poff);
      const bool okw = mbar_wait_all(bar_tfull + 8 * acc, acc_phase, abort_flag, p.status);
      if (f_epi_any(!okw)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256);
      if (!d.g2) {
        // lane r of D0 / D1: gate / up of intermediate column i = n*128 + r, one column per token
        const int i = d.n * 128 + lrow;
        float* P = p.p1 + (size_t)d.s * p.p1_stride;
        for (int c0 = 0; c0 < d.npad; c0 += 16) {
          float g[16], u[16];
          tmem_ld16(tb + (uint32_t)c0, g);
          tmem_ld16(tb + 128u + (uint32_t)c0, u);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c = c0 + j;
            if (c < d.ntok) {
              if (p.s1 == 1) {
                const float a = silu(g[j] * 1.0f) * (u[j] * 1.0f);
                const size_t o = (size_t)(d.xrow + c) * I + i;
                const __nv_bfloat16 hi = __float2bfloat16_rn(a);
                a_hi[o] = hi;
                if (a_lo) a_lo[o] = __float2bfloat16_rn(a - __bfloat162float(hi));
              } else {
                float* row = P + (size_t)plist[d.lbase + c] * (2 * I);
                row[i] = g[j];
                row[I + i] = u[j];
              }
            }
          }
        }
      } else {
        // Y[s][pair][h]: h = n*256 + r (D0) and n*256 + 128 + r (D1)
        const int h0 = d.n * 256 + lrow;
        const bool h1_ok = h0 + 128 < H;
        float* Y = p.y + (size_t)d.s * p.y_stride;
        for (int c0 = 0; c0 < d.npad; c0 += 16) {
          float v0[16], v1[16];
          tmem_ld16(tb + (uint32_t)c0, v0);
          tmem_ld16(tb + 128u + (uint32_t)c0, v1);
          if (p.act_split) {  // + the low part's products, xbox columns further on
            float l0[16], l1[16];
            tmem_ld16(tb + (uint32_t)(p.xbox + c0), l0);
            tmem_ld16(tb + 128u + (uint32_t)(p.xbox + c0), l1);
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
              float* row = Y + (size_t)plist[d.lbase + c] * H;
              row[h0] = v0[j] * 1.0f;
              if (h1_ok) row[h0 + 128] = v1[j] * 1.0f;
            }
          }
        }
      }
      // the accumulator buffer is free for the next tile
      tc_fence_before();
      mbar_arrive(bar_tempty + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }

      if (!d.g2) {
        bool finished = true;
        if (p.s1 > 1) {
          // the CTA that brings the last split of this tile sums the partials in split order
          named_bar_sync(1, 128);
          if (lrow == 0) {
            const unsigned old = atom_acq_rel_add(arr1 + d.e * p.n1 + d.n, 1u);
            sw[SW_LAST] = (old == (unsigned)(p.s1 - 1)) ? 1 : 0;
          }
          named_bar_sync(1, 128);
          finished = sw[SW_LAST] != 0;
          if (finished) {
            // (token, split) rows in natural order, so each token's splits add up in
            // split order from 0; their loads go out eight rows at a time
            const int i = d.n * 128 + lrow;
            const int rows = d.ntok * p.s1;
            float g = 0.0f, u = 0.0f;
            for (int r0 = 0; r0 < rows; r0 += 8) {
              float pg[8], pu[8];
#pragma unroll
              for (int q2 = 0; q2 < 8; ++q2) {
                const int r = min(r0 + q2, rows - 1);  // (the tail of a batch re-reads the last row)
                const int c = r / p.s1, sp = r - c * p.s1;
                const float* row = p.p1 + (size_t)sp * p.p1_stride + (size_t)plist[d.lbase + c] * 2 * I;
                pg[q2] = __ldcg(row + i);
                pu[q2] = __ldcg(row + I + i);
              }
#pragma unroll
              for (int q2 = 0; q2 < 8; ++q2) {
                const int r = r0 + q2;
                if (r < rows) {
                  const int c = r / p.s1, sp = r - c * p.s1;
                  g += pg[q2];
                  u += pu[q2];
                  if (sp == p.s1 - 1) {
                    const float a = silu(g) * u;
                    const size_t o = (size_t)(d.xrow + c) * I + i;
                    const __nv_bfloat16 hi = __float2bfloat16_rn(a);
                    a_hi[o] = hi;
                    if (a_lo) a_lo[o] = __float2bfloat16_rn(a - __bfloat162float(hi));
                    g = 0.0f;
                    u = 0.0f;
                  }
                }
              }
            }
          }
          named_bar_sync(1, 128);  // every thread has read SW_LAST
        }
        if (finished) {
          // the intermediate columns of this tile are complete: count the tile for GEMM2 (read by TMA)
          fence_proxy_async_global();
          named_bar_sync(1, 128);
          if (lrow == 0) red_release_add(ready1 + d.e * p.n1 + d.n, 1u);
        }
        if (lrow == 0) stamp(p, MOE_TRACE_G1_DONE);
      } else {
        // count this tile's outputs per (token, hidden tile) for the combine warps
        named_bar_sync(1, 128);
        if (lrow < d.ntok) red_release_add(cnt2 + (plist[d.lbase + lrow] / k) * p.n2 + d.n, 1u);
      }
    }
    if (lrow == 0) stamp(p, MOE_TRACE_EPI_DONE);
    combine_worker(p, cnt2, tws, ok, abort_flag, false);
  } else {
    // ---------------- combine (warps 6, 7; every other warp once its role is done) ----------------
    combine_worker(p, cnt2, tws, ok, abort_flag, warp == 6);
    if (lane == 0 && warp == 6) stamp(p, MOE_TRACE_COMB_DONE);
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
    tmem_dealloc(tmem_base, kFTmemCols);
    if (lane == 0) {
      stamp(p, MOE_TRACE_END);
      if (ok) {
        // the last CTA out withdraws the launch tag, so no later launch can take
        // this launch's counters for its own
        if (atom_acq_rel_add(p.sync + SYNC_EXIT, 1u) == gridDim.x - 1) st_release_u64(p.go, 0ull);
      }
    }
  }
}

}  // namespace

}  // namespace moe

namespace moe {

size_t fused_sync_bytes(int T, int H, int I, int E) {
  const size_t words = SYNC_NBAR + 2 * (size_t)E * (I / 128) + (size_t)T * ((H + 255) / 256);
  return 256 + (words * 4 + 255) / 256 * 256;  // launch tag in the first 256 bytes, then the counters
}

size_t fused_table_bytes(int T, int E, int k) {
  const size_t n = (size_t)T * k;
  const size_t words = kRouterWarps * kFRouterTT + 5 * n + 4 * (size_t)E + 2;
  return (words * 4 + 15) / 16 * 16;
}

cudaError_t launch_decode_fused(const FusedArgs& a, cudaStream_t s) {
  if (a.xbox < 16 || a.xbox > 64 || a.xbox % 16 || (a.gather && a.xbox > 32) || a.H % 128 || a.I % 128 ||
      a.num_sms <= 0)
    return cudaErrorInvalidValue;
  CUtensorMap mw1, mw2, mx, ma;
  if (!make_tensor_map_2d(&mw1, a.w13, 2, (uint64_t)a.H, (uint64_t)a.E * 2 * a.I, 128u) ||
      !make_tensor_map_2d(&mw2, a.w2, 2, (uint64_t)a.I, (uint64_t)a.E * a.H, 128u) ||
      !make_tensor_map_2d(&ma, a.aint, 2, (uint64_t)a.I, (uint64_t)a.cap * (a.act_split ? 2 : 1),
                          (uint32_t)a.xbox))
    return cudaErrorInvalidValue;
  if (a.gather ? !make_tensor_map_2d(&mx, a.X, 2, (uint64_t)a.H, (uint64_t)a.T, 1u)
               : !make_tensor_map_2d(&mx, a.Xs, 2, (uint64_t)a.H, (uint64_t)a.cap, (uint32_t)a.xbox))
    return cudaErrorInvalidValue;

  FusedDev p = {};
  p.T = a.T;
  p.H = a.H;
  p.I = a.I;
  p.E = a.E;
  p.k = a.k;
  p.renorm = a.renorm;
  p.n1 = a.I / 128;
  p.s1 = a.s1;
  p.kbs1 = a.kbs1;
  p.kbt1 = a.H / 64;
  p.n2 = (a.H + 255) / 256;
  p.s2 = a.s2;
  p.kbs2 = a.kbs2;
  p.kbt2 = a.I / 64;
  p.xbox = a.xbox;
  p.gather = a.gather ? 1 : 0;
  p.act_split = a.act_split ? 1 : 0;
  p.cap = a.cap;
  p.combine_g = a.combine_g;
  p.X = static_cast<const __nv_bfloat16*>(a.X);
  p.Wr = static_cast<const __nv_bfloat16*>(a.Wr);
  p.logits = a.logits;
  p.topk_w = a.topk_w;
  p.topk_ids = a.topk_ids;
  p.Xs = static_cast<__nv_bfloat16*>(a.Xs);
  p.aint = static_cast<__nv_bfloat16*>(a.aint);
  p.p1 = a.p1;
  p.p1_stride = a.p1_stride;
  p.y = a.y;
  p.y_stride = a.y_stride;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.go = static_cast<unsigned long long*>(a.sync);
  p.sync = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(a.sync) + 256);
  p.nsync = SYNC_NBAR + 2 * a.E * p.n1 + a.T * p.n2;
  p.status = a.status;
  p.trace = static_cast<unsigned long long*>(a.trace);

  p.stage_bytes = 2u * 128u * 128u + (uint32_t)a.xbox * 128u * (a.act_split ? 2u : 1u);
  const size_t tab = fused_table_bytes(a.T, a.E, a.k);
  const size_t budget = 227 * 1024 - 1024 - kFBarBytes - tab;
  int stages = (int)(budget / p.stage_bytes);
  if (stages > kFMaxStages) stages = kFMaxStages;
  if (stages < 2) return cudaErrorInvalidValue;
  p.stages = stages;
  p.bar_off = (uint32_t)stages * p.stage_bytes;
  p.tab_off = p.bar_off + kFBarBytes;
  const size_t smem = 1024 + (size_t)p.tab_off + tab;

  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_decode_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_fused, kFThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // one CTA per SM at most; fewer when the batch has fewer tiles than SMs
  const long act_upper = std::min<long>(a.E, (long)a.T * a.k);
  const long tiles_upper = act_upper * ((long)p.n1 * p.s1 + (long)p.n2 * p.s2);
  const int grid = (int)std::max<long>(1, std::min<long>(tiles_upper, a.num_sms));

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the CTAs wait on one another: all must be resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_fused, mw1, mw2, mx, ma, p);
}

}  // namespace moe
