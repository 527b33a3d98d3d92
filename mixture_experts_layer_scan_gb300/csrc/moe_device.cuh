// Device-side helpers shared by the kernels of the MoE library (sm_103a).
//
// Number conversions, bounded waits, and thin wrappers over the Blackwell
// PTX the grouped GEMM uses (mbarrier, TMA, tcgen05).  Every wait in this
// library is bounded: it gives up after a time limit, records
// MOE_ERR_DEVICE_TIMEOUT in the per-device status word and lets the kernel
// return, so a bug can never leave a GPU spinning forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe_api.h"

namespace moe {

// ---------------------------------------------------------------------------
// element conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// two floats -> packed bf16x2 (round to nearest even), low half = a
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// float -> e4m3 code, round to nearest even, saturating to +-448 (OCP E4M3)
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// dynamic per-tensor e4m3 scale from an amax (same formula the oracle states)
__device__ __forceinline__ float e4m3_scale_from_amax(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ---------------------------------------------------------------------------
// status word (one int per device, owned by the host layer)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound of any single wait inside a kernel: a healthy wait in this
// library lasts microseconds; 2 s means something is broken.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------------------
// shared-memory address and mbarrier helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Raise the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up (returns
// false) when *abort is raised by another role of the CTA, or after
// kWaitLimitNs, in which case it raises *abort and records a timeout.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        report(status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// The same wait by all 32 lanes of a warp together: every lane polls, and
// the outcome (done / gave up) is decided warp-wide each round, so the warp
// never splits into a spinning lane and lanes parked elsewhere.  Roles that
// issue from one lane wait this way and predicate only the issue itself.
__device__ __forceinline__ bool mbar_wait_all(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    if (it == 0) t0 = globaltimer_ns();
    if ((it & 31u) == 31u) {
      const bool give_up = *abort || (globaltimer_ns() - t0 > kWaitLimitNs);
      if (__any_sync(0xffffffffu, give_up)) {
        if ((threadIdx.x & 31) == 0 && !*abort) {
          *abort = 1;
          report(status, MOE_ERR_DEVICE_TIMEOUT);
        }
        return false;
      }
    }
  }
}

// Warp-wide bounded wait until the global word *word equals want (acquire).
// Used for words written by another engine (a copy stream's in-order writes
// after the data they announce); the data is then read through TMA, so the
// async proxy is ordered after the observation.
__device__ __forceinline__ bool wait_word_all(const unsigned* word, unsigned want, volatile int* abort, int* status) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(word) : "memory");
    if (__all_sync(0xffffffffu, v == want)) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      return true;
    }
    if (it == 0) t0 = globaltimer_ns();
    if ((it & 15u) == 15u) {
      const bool give_up = *abort || (globaltimer_ns() - t0 > kWaitLimitNs);
      if (__any_sync(0xffffffffu, give_up)) {
        if ((threadIdx.x & 31) == 0 && !*abort) {
          *abort = 1;
          report(status, MOE_ERR_DEVICE_TIMEOUT);
        }
        return false;
      }
    }
    __nanosleep(256);
  }
}

// Drain wait used on the abort path only: ignores the abort flag, own limit.
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// Untiled bulk copy global -> shared (the CTA's own shared memory), completion
// counted in bytes on an mbarrier.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t smem_dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ---------------------------------------------------------------------------
// TMA (tiled 2-D bulk tensor copy global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t smem_dst, const void* tmap, int c_inner, int c_row,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
      "[%2];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c_inner), "r"(c_row)
      : "memory");
}

// Rank of this CTA in its cluster, and a barrier over every thread of the cluster.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive once on an mbarrier of another CTA of the cluster (release, cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}

// CTA pairs (tcgen05 cta_group::2): a 2-D tile into this CTA's shared memory
// whose completion (bytes) is counted on an mbarrier of either CTA of the pair
// (bar_cluster_addr, e.g. CTA 0's barrier mapped with mapa_shared).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t smem_dst, const void* tmap, int c_inner, int c_row,
                                                 uint32_t bar_cluster_addr) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar_cluster_addr), "r"(c_inner), "r"(c_row)
      : "memory");
}

// Four rows (row0..row3) of a 2-D tensor whose map has a one-row box, each
// box-width wide from column c_inner, into consecutive rows at smem_dst.
__device__ __forceinline__ void tma_gather4(uint32_t smem_dst, const void* tmap, int c_inner, int row0, int row1,
                                            int row2, int row3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(smem_dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c_inner), "r"(row0), "r"(row1), "r"(row2), "r"(row3), "r"(bar)
      : "memory");
}

// Prefetch a 2-D tile of a tensor into L2 (a hint: no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2(const void* tmap, int c_inner, int c_row) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
               "r"(c_inner), "r"(c_row)
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, accumulators in tensor memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// CTA pairs: both CTAs of the pair allocate together (each CTA's warp issues
// the instruction with the same column count; both receive the same address).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A * B on a CTA pair, issued by CTA 0: A (M = 256) is rows 0-127 in CTA
// 0's shared memory and rows 128-255 at the same offset in CTA 1's; B likewise
// holds N/2 rows in each CTA; each CTA's tensor memory receives its 128 rows of D.
template <bool FP8>
__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  if constexpr (FP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// CTA pairs: arrive once on the mbarrier at bar_cluster_addr (this CTA's or the
// peer's) when the pair MMAs issued so far by this thread complete.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar_cluster_addr) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_cluster_addr)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 128 bytes, 8-row / 1024-byte swizzle atoms).
//   bits  0-13 start address >> 4     bits 16-29 leading byte offset >> 4 (unused here)
//   bits 32-45 stride byte offset >> 4 (1024: next 8-row group)
//   bits 46-48 fixed 0b001            bits 61-63 swizzle mode (2 = 128-byte)
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1u << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor: fp32 accumulator, K-major A and B, shape M x N.
// kind::f16 with bf16 operands (bits 7-9 and 10-12 = 1), or kind::f8f6f4
// with e4m3 operands (format 0).
__device__ __forceinline__ uint32_t idesc_make(int M, int N, bool fp8) {
  uint32_t d = 0;
  d |= 1u << 4;  // D format F32
  if (!fp8) {
    d |= 1u << 7;   // A = BF16
    d |= 1u << 10;  // B = BF16
  }
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

template <bool FP8>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  if constexpr (FP8) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// D (+)= A * B with A (M rows in lanes, K along 32-bit columns, two bf16 per
// column, lower K in the low half) read from tensor memory at a_tmem and B
// from shared memory (kind::f16, bf16 operands).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The 8 MMAs of one 64-element K block of a 256-row swap-AB tile, A from
// tensor memory, issued as one block: D0 (+)= A[a .. a+31] x B and
// D1 (+)= A[a+32 .. a+63] x B, four K steps of 16 (8 columns of A, 32 bytes of
// the 128-byte-swizzled B rows each).  accumulate = 0 starts both accumulators.
__device__ __forceinline__ void tc_mma_ts_kblock(uint32_t d0, uint32_t d1, uint32_t a, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, t;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t.reg .b64 b1, b2, b3;\n\t"
      "setp.ne.b32 p, %5, 0;\n\tsetp.ne.b32 t, %4, 0;\n\t"
      "add.u32 a1, %2, 32;\n\tadd.u32 a2, %2, 8;\n\tadd.u32 a3, %2, 40;\n\tadd.u32 a4, %2, 16;\n\t"
      "add.u32 a5, %2, 48;\n\tadd.u32 a6, %2, 24;\n\tadd.u32 a7, %2, 56;\n\t"
      "add.u64 b1, %3, 2;\n\tadd.u64 b2, %3, 4;\n\tadd.u64 b3, %3, 6;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %3, %4, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [a1], %3, %4, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b1, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [a3], b1, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b2, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [a5], b2, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b3, %4, t;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%1], [a7], b3, %4, t;\n\t}" ::"r"(d0),
      "r"(d1), "r"(a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 registers per thread -> 32 lanes x 32 consecutive 32-bit columns of tensor
// memory; complete (visible to the tensor core) after tmem_wait_st().
__device__ __forceinline__ void tmem_st32_nowait(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Arrive once on an mbarrier when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns of tensor memory -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 lanes x 32 columns in the 16x256b shape (four 8-column groups): thread t
// holds, for group j, v[4j], v[4j+1] = (lane t/4, columns 8j + 2(t%4), +1) and
// v[4j+2], v[4j+3] = (lane 8 + t/4, the same columns), lanes counted from taddr's.
__device__ __forceinline__ void tmem_ld_16x256b_x4(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// CTA and named barriers for warp-specialised code.  Every lane of a warp
// reaches the barrier, but possibly not together (lane 0 may still be issuing
// MMAs or storing a flag): __syncwarp() first reconverges the warp, then the
// .aligned barrier, whose arrivals count whole warps, is well defined.  (An
// aligned barrier reached by a diverged warp can release early; the
// non-aligned form is defined but can stall for microseconds while the warp
// scheduler switches to the lagging lanes.)
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void cta_sync() {
  __syncwarp();
  __syncthreads();
}
// OR of a flag over the nthreads threads of named barrier id.
__device__ __forceinline__ bool named_bar_any(int id, int nthreads, bool v) {
  __syncwarp();
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Programmatic dependent launch: wait for the preceding kernel's results /
// allow the next kernel to start its prologue.  Every kernel of the layer is
// launched with programmatic stream serialisation; each one lets its
// dependents launch early and calls pdl_wait() before it reads anything the
// previous kernel wrote (the wait returns once that kernel has completed and
// its memory is visible), so only launch latency and prologues overlap.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_launch_dependents();
  pdl_wait();
}

// Host: launch a kernel with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl(...) inside a function returning cudaError_t: return the error if any.
#define MOE_LAUNCH(...)                                  \
  do {                                                   \
    const cudaError_t moe_launch_err_ = launch_pdl(__VA_ARGS__); \
    if (moe_launch_err_ != cudaSuccess) return moe_launch_err_;  \
  } while (0)

}  // namespace moe
