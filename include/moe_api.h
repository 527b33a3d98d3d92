/*
 * moe_api.h -- C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer forward.
 *
 * The layer (one call of moe_forward) is the fused MoE operation the pages
 * describe: token routing, the data shuffle that groups tokens by expert, the
 * expert networks and the routing-weighted sum back to token order, run as one
 * batched GPU operation instead of a loop over experts
 *   ("Mixture-of-Experts kernel engineering on Amazon SageMaker AI", intro;
 *    "FusedMoE vs MegaMoE" (zwxr.cn), sections 2 and 3.1).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named *hidden*, *router_w*, *w13*, *w2*, *out*, *logits*,
 *    *topk_*, *sorted_ids*, *expert_ids*, *num_post_pad*, *expert_counts*,
 *    *workspace* and the FP8 scales are DEVICE pointers of the current CUDA
 *    device.  The caller owns all of them; the library never allocates,
 *    frees or retains device memory across calls (it keeps one status word
 *    per device, see moe_get_status).  The library caches per-device state
 *    (that word's address, kernel attributes); cudaDeviceReset() invalidates
 *    it, so the library must not be used on a device after a reset.
 *  - All arrays are dense row-major with no padding between rows.  Device
 *    pointers must be 16-byte aligned (MOE_ERR_ALIGNMENT otherwise).
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  A return of MOE_OK means "validated and
 *    enqueued"; faults found by the kernels themselves (an expert id out of
 *    range, a bounded wait that ran out) are reported by moe_get_status.
 *  - Results are deterministic: the same inputs give bitwise-identical outputs
 *    on every call (fixed reduction orders, no floating-point atomics).
 *  - Shapes are runtime arguments; no call compiles or specialises code for a
 *    new token count (page 1, section "Élimination de la recompilation JIT de
 *    Triton": recompiling per num_tokens cost 9 % TTFT at 8-way TP).
 *  - T = 0 is a valid, empty call (nothing is enqueued, MOE_OK).
 *
 * Notation: T tokens, H hidden size, I expert intermediate size, E experts,
 * k = topk experts per token, B = block (token-tile) size of the permutation.
 */
#ifndef MOE_API_H
#define MOE_API_H

#include <stddef.h>
#include <stdint.h>

#if defined(MOE_BUILD_LIBRARY) && defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */
typedef struct CUevent_st* moe_event_t;   /* same type as cudaEvent_t */

/* Element types.  BF16 is stored as 16-bit bfloat16, E4M3 as 8-bit OCP E4M3
 * codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, max 448).
 * INT4 (expert weights only): 4-bit two's complement codes q in [-8, 7], eight
 * consecutive K elements per little-endian 32-bit word, element e of the word in
 * nibble (e even ? e/2 : 4 + e/2); one bf16 scale s per (weight row, 128 K
 * elements); the weight is q * s rounded once to bf16 (nearest even). */
typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_E4M3 = 2, MOE_INT4 = 3 } moe_dtype;

/* Return codes (0 or negative). */
enum {
  MOE_OK = 0,
  MOE_ERR_ARG = -1,            /* bad size, null pointer, bad enum */
  MOE_ERR_UNSUPPORTED = -2,    /* valid but not implemented (dtype pair, shape rule) */
  MOE_ERR_WORKSPACE = -3,      /* workspace smaller than moe_workspace_size() */
  MOE_ERR_CUDA = -4,           /* a CUDA runtime call failed (launch, no device ...) */
  MOE_ERR_DEVICE_TIMEOUT = -5, /* a kernel's bounded wait ran out (from moe_get_status) */
  MOE_ERR_DEVICE_INDEX = -6,   /* a kernel met an expert id outside [0, E) (moe_get_status) */
  MOE_ERR_ALIGNMENT = -7       /* a device pointer is not 16-byte aligned */
};

/* Orientation of the grouped expert GEMMs.
 * SWAP_AB computes C^T[N,M] = B^T[N,K] * A^T[K,M]: the expert weight rows fill
 * the tensor core's fixed 128-row M slot and the few tokens of an expert
 * take the flexible N slot (page 1, section "Swap-AB pour l'utilisation de
 * WGMMA", Figure 1; re-derived here for tcgen05, whose M slot is 128).
 * TOKEN_MAJOR puts 128 sorted token rows in the M slot (prefill).
 * AUTO picks SWAP_AB for T <= 64 and TOKEN_MAJOR above. */
typedef enum { MOE_ORIENT_AUTO = 0, MOE_ORIENT_SWAP_AB = 1, MOE_ORIENT_TOKEN_MAJOR = 2 } moe_orientation;

/* Stages of moe_forward, for the optional timing events below. */
typedef enum {
  MOE_STAGE_ROUTE = 0,   /* router GEMM + softmax/top-k (+ renorm) */
  MOE_STAGE_ALIGN = 1,   /* histogram / scan / stable scatter */
  MOE_STAGE_GATHER = 2,  /* activation rows in expert order (+ FP8 input quantisation) */
  MOE_STAGE_GEMM1 = 3,   /* grouped GEMM on w13 with the SiLU(gate)*up epilogue */
  MOE_STAGE_ACT = 4,     /* split-K reduction / FP8 intermediate quantisation (may be empty) */
  MOE_STAGE_GEMM2 = 5,   /* grouped GEMM on w2 */
  MOE_STAGE_COMBINE = 6, /* routing-weighted sum back to token order */
  MOE_NUM_STAGES = 7
} moe_stage;

/* Phase stamps of the single-launch kernel (moe_options.trace), per CTA. */
typedef enum {
  MOE_TRACE_START = 0,      /* kernel entry, after the prologue */
  MOE_TRACE_ROUTER = 1,     /* router logits of this CTA written */
  MOE_TRACE_BARRIER0 = 2,   /* all logits visible */
  MOE_TRACE_TOPK = 3,       /* top-k of this CTA's tokens written */
  MOE_TRACE_BARRIER1 = 4,   /* all routing visible */
  MOE_TRACE_TABLES = 5,     /* expert tables built in shared memory */
  MOE_TRACE_GATHERED = 6,   /* token rows in expert order (after the third barrier; = TABLES without it) */
  MOE_TRACE_G1_ISSUED = 7,  /* producer: loads of every GEMM1 tile of this CTA issued */
  MOE_TRACE_G2_READY = 8,   /* producer: first GEMM2 tile found its intermediate complete */
  MOE_TRACE_ISSUED = 9,     /* producer: every load issued */
  MOE_TRACE_MMA_DONE = 10,  /* MMA issuer: last tile committed */
  MOE_TRACE_G1_DONE = 11,   /* epilogue: last GEMM1 tile of this CTA signalled */
  MOE_TRACE_EPI_DONE = 12,  /* epilogue: last tile stored */
  MOE_TRACE_COMB_FIRST = 13,/* combine: first unit's outputs all arrived */
  MOE_TRACE_COMB_DONE = 14, /* combine: last unit written */
  MOE_TRACE_END = 15,       /* CTA done */
  MOE_TRACE_WORDS = 16
} moe_trace_event;

/* Optional knobs of moe_forward / moe_workspace_size.  Pass NULL for defaults
 * (all-zero struct == defaults).  The same options must be given to
 * moe_workspace_size and to the moe_forward calls that use that workspace. */
typedef struct {
  int orientation;    /* moe_orientation; SWAP_AB needs T <= 256 */
  int split_k;        /* 0 = automatic; n > 0 forces n K-splits in SWAP_AB mode */
  int inject_timeout; /* test hook: 1 makes the first kernel wait on a device flag that
                         nothing sets, with a ~1 ms bound; the call then reports
                         MOE_ERR_DEVICE_TIMEOUT through moe_get_status and writes
                         nothing else.  0 in normal use. */
  int act_split;      /* bf16 and INT4 weights: 0 = automatic (bf16: hi/lo in SWAP_AB, single in
                         TOKEN_MAJOR; INT4: single), 1 = intermediate stored as one bf16,
                         2 = as bf16 hi + bf16 lo (a - bf16(a)), GEMM2 then runs both parts into
                         one fp32 accumulator */
  void* trace;        /* nullable device buffer of MOE_TRACE_WORDS uint64 per SM: when the call
                         runs as a single launch, CTA c writes %globaltimer stamps (ns) of its
                         phases to trace[c * MOE_TRACE_WORDS + moe_trace_event]; events a CTA
                         does not reach are left as they were (zero the buffer first) */
  int single_launch;  /* bf16 SWAP_AB batches: 0 = automatic, 1 = run the whole layer as one
                         cooperative kernel (MOE_ERR_UNSUPPORTED where it does not apply:
                         it needs the bf16 path in SWAP_AB mode, T <= 64, T*topk <= 512,
                         E <= 256), 2 = always the multi-kernel sequence.  Both give
                         bit-identical outputs. */
  /* Nullable CUDA events recorded on `stream` right before / after the
   * kernels of each stage (the caller creates and owns them). */
  moe_event_t stage_begin[MOE_NUM_STAGES];
  moe_event_t stage_end[MOE_NUM_STAGES];
  int cta_pair;       /* TOKEN_MAJOR tensor-core GEMMs: 0 = automatic (CTA pairs when H % 256 == 0),
                         1 = CTA pairs (MOE_ERR_UNSUPPORTED where they do not apply), 2 = single CTAs.
                         On CTA pairs (tcgen05 cta_group::2) two SMs compute a 256-token x
                         256-weight-row tile together, each staging half of both operands, and the
                         permutation pads experts to 256 rows; on single CTAs, tiles of 128 tokens. */
} moe_options;

/* What moe_forward will run for a shape (filled by moe_plan_info). */
typedef struct {
  int orientation;      /* MOE_ORIENT_SWAP_AB or MOE_ORIENT_TOKEN_MAJOR (0 on the fp32 path) */
  /* (cta_pair below: 1 if the TOKEN_MAJOR GEMMs run on CTA pairs) */
  int block;            /* permutation block size B */
  int splits_gemm1;     /* K splits of GEMM1 / GEMM2 */
  int splits_gemm2;
  int act_split;        /* 1 if the bf16 intermediate is stored as hi + lo */
  int kernel_launches;  /* kernels one moe_forward call launches */
  int single_launch;    /* 1 if the whole layer runs as one cooperative kernel */
  size_t workspace_bytes;
  int cta_pair;         /* 1 if the TOKEN_MAJOR GEMMs run on CTA pairs */
} moe_plan;

/* Human-readable text of a return code (static storage). */
MOE_API const char* moe_strerror(int code);

/* Bytes of device workspace moe_forward needs for this shape, dtype pair and
 * options (written to *bytes).  Depends only on its arguments. */
MOE_API int moe_workspace_size(int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                       const moe_options* opts, size_t* bytes);

/* Describes the kernels and workspace moe_forward uses for these arguments
 * (host only, no device work).  Same argument rules as moe_workspace_size. */
MOE_API int moe_plan_info(int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                          const moe_options* opts, moe_plan* info);

/* Capacities of the permutation outputs for (T, topk, E, block):
 *   sorted_cap = T*topk + min(E, T*topk)*(block-1)     (int32 entries)
 *   blocks_cap = sorted_cap / block                     (int32 entries) */
MOE_API int moe_align_capacity(int T, int topk, int E, int block, size_t* sorted_cap, size_t* blocks_cap);

/* Router: steps 1-2 of the layer
 *   ("FusedMoE vs MegaMoE", section 2: the router gives every token a weight
 *    distribution over experts and the k highest experts are chosen).
 *   logits_out[T][E] (fp32, required: the library allocates nothing, and the router writes the
 *   logits there before ranking them; NULL returns MOE_ERR_ARG)
 *                      = hidden[T][H] . router_w[E][H]^T, fp32 accumulation;
 *   p = softmax over all E; topk_ids[T][topk] (int32) = the topk largest p in
 *   descending order, equal values ranked by lower expert index (ranking is on
 *   the fp32 logit, which orders like p); topk_w[T][topk] (fp32) = p of those
 *   experts, divided by their sum when renorm != 0.
 * hidden and router_w have type act_dtype (MOE_F32 or MOE_BF16); H must be a multiple
 * of 8 (bf16) or 4 (fp32).  Long bf16 batches (T >= 256, E <= 256, H % 128 == 0) run the
 * logits on the tensor cores, shorter ones on the CUDA cores; both accumulate in fp32.
 * Limits: 1 <= topk <= min(E, 32), E <= 1024. */
MOE_API int moe_route(const void* hidden, const void* router_w, int T, int H, int E, int topk, int renorm,
              moe_dtype act_dtype, float* logits_out, float* topk_w, int32_t* topk_ids, moe_stream_t stream);

/* Step 2 alone, from given fp32 logits[T][E] (same ranking and weights as
 * moe_route).  Lets routing be compared exactly on identical logits. */
MOE_API int moe_topk_from_logits(const float* logits, int T, int E, int topk, int renorm, float* topk_w,
                         int32_t* topk_ids, moe_stream_t stream);

/* Step 3: token-to-expert permutation
 *   ("FusedMoE vs MegaMoE", section 3.1: sort routed tokens by expert and
 *    build the index of which rows belong to which expert; page 1, section
 *    "Routage backend...": variable token bucketing onto expert tiles).
 * For every (token t, slot j) pair the flat index f = t*topk + j.  Experts are
 * laid out in ascending order; inside an expert its f values ascend (stable);
 * each expert's run is padded with the sentinel T*topk to a multiple of
 * `block`; experts without tokens get no block.
 *   sorted_ids[sorted_cap]   int32, entries [0, *num_post_pad) written
 *   expert_ids[blocks_cap]   int32, expert of each block, [0, *num_post_pad/block) written
 *   num_post_pad[1]          int32, total padded length
 *   expert_counts[E]         int32, tokens per expert (nullable)
 * Ids outside [0, E) are dropped and flagged as MOE_ERR_DEVICE_INDEX (moe_get_status).
 * Limits: E <= 1024, 1 <= block <= 1024, T*topk < 2^31. */
MOE_API int moe_align(const int32_t* topk_ids, int T, int topk, int E, int block, int32_t* sorted_ids, int32_t* expert_ids,
              int32_t* num_post_pad, int32_t* expert_counts, moe_stream_t stream);

/* The whole layer forward, steps 1-7, on `stream`:
 *   route -> align -> gather -> GEMM1 (w13) + SiLU(gate)*up -> GEMM2 (w2) -> combine
 *   out[t] = sum_j topk_w[t][j] * W2[e_j] . (SiLU(W13[e_j][0:I] . x_t) * (W13[e_j][I:2I] . x_t))
 *   ("FusedMoE vs MegaMoE", sections 2 and 3.1; page 1, sections on Swap-AB and FP8).
 * Arguments:
 *   hidden   [T][H]      act_dtype (MOE_F32 or MOE_BF16)
 *   router_w [E][H]      act_dtype
 *   w13      [E][2I][H]  w_dtype; rows [0, I) are the gate, rows [I, 2I) the up projection
 *   w2       [E][H][I]   w_dtype
 *   w13_scale, w2_scale  MOE_E4M3 weights: [E] fp32 per-expert dequantisation scales;
 *                        MOE_INT4 weights: bf16 group scales, group-major per expert,
 *                        [E][H/128][2I] and [E][I/128][H]; ignored otherwise
 *   (MOE_INT4: w13 [E][2I][H/2] and w2 [E][H][I/2] bytes of packed codes)
 *   out      [T][H]      act_dtype
 *   workspace            >= moe_workspace_size(...) bytes, 256-byte aligned, contents ignored
 * Supported dtype pairs:
 *   (F32, F32)   fp32 CUDA-core path, any H, I >= 1
 *   (BF16, BF16) tcgen05 tensor-core path (kind::f16, fp32 accumulation in TMEM)
 *   (BF16, E4M3) tcgen05 kind::f8f6f4 path: the input is quantised to e4m3 with one
 *                dynamic scale amax/448, the intermediate likewise; the scales are applied
 *                in the GEMM epilogues (page 1, section "Routage backend pour la
 *                quantisation des tenseurs FP8": scaling fused where the data is used)
 *   (BF16, INT4) tcgen05 kind::f16 path with the codes expanded to bf16 weights in
 *                tensor memory inside the GEMM main loop (the MMA takes its weight operand
 *                from there; "FusedMoE vs MegaMoE", section 6.3: quantised expert
 *                weights); SWAP_AB orientation only,
 *                T <= 128, H % 256 == 0 and I % 256 == 0 (else MOE_ERR_UNSUPPORTED)
 *   tensor-core paths need H % 128 == 0 and I % 128 == 0.
 * The intermediate SiLU(gate)*up is stored in bf16 (as a bf16 hi + lo pair in SWAP_AB
 * mode, see moe_options.act_split; fp32 on the fp32 path; e4m3 on the FP8 path);
 * accumulation is fp32 throughout; out is rounded once.
 * Single launch (moe_options.single_launch): thin bf16 decode batches may run all
 * seven steps in one cooperative kernel ("Mixture-of-Experts kernel engineering on
 * Amazon SageMaker AI", intro: routing, shuffle and expert networks as one batched
 * operation); its stage events then bracket that one kernel (recorded as GEMM1, the
 * other stages empty).  All its CTAs must be resident at once: the call fails with
 * MOE_ERR_CUDA if the device cannot hold them (e.g. while another kernel occupies SMs
 * under MPS limits). */
MOE_API int moe_forward(const void* hidden, const void* router_w, const void* w13, const void* w2, int T, int H, int I, int E,
                int topk, int renorm, moe_dtype act_dtype, moe_dtype w_dtype, const void* w13_scale,
                const void* w2_scale, void* out, void* workspace, size_t workspace_bytes, const moe_options* opts,
                moe_stream_t stream);

/* The layer from host memory to host memory, on `stream`:
 *   1. hidden_host -> hidden_dev, T*H elements of act_dtype, by a copy kernel that reads the
 *      host memory directly (cudaMemcpyAsync when the byte count or an address is not a
 *      multiple of 16),
 *   2. moe_forward(hidden_dev, ..., out, ...) exactly as above, with `out` the device
 *      address of out_host: the layer's last kernel stores the output into host memory.
 * hidden_host and out_host are page-locked host memory that the device can address
 * (cudaHostAlloc, cudaMallocHost or cudaHostRegister on a system with unified addressing;
 * MOE_ERR_ARG otherwise); out_host 16-byte aligned (MOE_ERR_ALIGNMENT).  hidden_dev is a
 * device staging buffer of T*H elements (16-byte aligned) owned by the caller.  Every
 * other argument is moe_forward's.  The call returns once the work is enqueued: out_host
 * holds the result when the work enqueued on `stream` has completed (cudaStreamSynchronize,
 * an event).  Errors: those of moe_forward, MOE_ERR_ARG for a null, pageable or unmapped
 * host buffer, MOE_ERR_CUDA when the copy cannot be enqueued.  T == 0 is a no-op. */
MOE_API int moe_forward_host(const void* hidden_host, void* hidden_dev, const void* router_w, const void* w13,
                             const void* w2, int T, int H, int I, int E, int topk, int renorm, moe_dtype act_dtype,
                             moe_dtype w_dtype, const void* w13_scale, const void* w2_scale, void* out_host,
                             void* workspace, size_t workspace_bytes, const moe_options* opts, moe_stream_t stream);

/* Inverse rotary position embedding fused with per-head FP8 quantisation
 *   ("Mixture-of-Experts kernel engineering on Amazon SageMaker AI", section on
 *    the Triton JIT: the serving stack's _fused_inv_rope_fp8_quant_per_head kernel,
 *    rotary embedding + FP8 quantisation fused; here every shape is a runtime argument).
 * For token t, head h, x = x[t][h][0:head_dim] (bf16), R = rot_dim, half = R/2 and
 * (c_i, s_i) = (cos_sin[positions[t]][i], cos_sin[positions[t]][half + i]):
 *   y_i = x_i c_i + x_{half+i} s_i,  y_{half+i} = x_{half+i} c_i - x_i s_i   (i < half: the
 *   rotation by minus the position's angle, rotate-half pairing), y_j = x_j for j >= R;
 *   scale_out[t][h] = max_j |y_j| / 448 (1.0 when that is 0), fp32;
 *   q_out[t][h][j] = e4m3(y_j * r), r = 1 / scale_out[t][h] once per vector (round to nearest
 *   even, saturating to +-448).
 * Every product, sum and the reciprocal is one fp32 rounding (no fused multiply-add).
 * Arguments:
 *   x          [T][heads][head_dim] bf16, 4-byte aligned
 *   positions  [T] int32, each in [0, max_pos); others are clamped and flagged
 *              MOE_ERR_DEVICE_INDEX (moe_get_status)
 *   cos_sin    [max_pos][rot_dim] fp32, 16-byte aligned: cos of the rot_dim/2 angles, then their sin
 *              (may be NULL when rot_dim == 0)
 *   q_out      [T][heads][head_dim] e4m3 codes;  scale_out [T][heads] fp32
 * Limits: head_dim even, rot_dim % 4 == 0, rot_dim <= min(head_dim, 1024),
 *   head_dim - rot_dim <= 512.  T = 0 is a successful no-op. */
MOE_API int moe_inv_rope_fp8_quant(const void* x, int T, int heads, int head_dim, int rot_dim,
                                   const int32_t* positions, const float* cos_sin, int max_pos, uint8_t* q_out,
                                   float* scale_out, moe_stream_t stream);

/* Steps 3-7 of the layer on a routing the caller provides (its own router, or
 * expert ids remapped to the slots of an expert cache): the same permutation,
 * expert GEMMs and combine as moe_forward, which it matches bit for bit given
 * moe_forward's routing.
 *   topk_w   [T][topk] fp32 routing weights (used as given, no renormalisation)
 *   topk_ids [T][topk] int32 expert ids in [0, E); ids outside are dropped and flagged
 *            MOE_ERR_DEVICE_INDEX
 * Other arguments, the workspace (moe_workspace_size with the same E) and the options
 * as moe_forward; the multi-kernel sequence always (single_launch = 1 is refused). */
MOE_API int moe_forward_routed(const void* hidden, const float* topk_w, const int32_t* topk_ids, const void* w13,
                               const void* w2, int T, int H, int I, int E, int topk, moe_dtype act_dtype,
                               moe_dtype w_dtype, const void* w13_scale, const void* w2_scale, void* out,
                               void* workspace, size_t workspace_bytes, const moe_options* opts, moe_stream_t stream);

/* Expert cache ("FusedMoE vs MegaMoE", section 4: MegaMoE keeps expert weights
 * in host memory, stages the experts a batch needs into GPU memory with an LRU
 * policy and overlaps the copies with computation on separate CUDA streams
 * synchronised by events; sections 4.1 and 4.2).  The cache owns a pool of
 * n_slots expert slots in device memory; the full weights stay in host memory
 * (on a GB300 the Grace CPU's, over NVLink-C2C).  Each moe_forward_cached call
 * routes the batch on the GPU, reads the expert ids back (one host
 * synchronisation per call), keeps the experts already resident, copies the
 * missing ones into free slots or the slots of the least recently used experts
 * the call does not need, and runs the expert part of the layer over the slots.
 * By default (MOE_CACHE_COPY_OVERLAP) the copies run on the cache's copy stream
 * while the expert kernels already compute the resident experts: a per-slot
 * readiness word, written on the copy stream after each weight matrix lands,
 * gates the GEMMs' weight streaming per expert (a bounded wait).  A call needing
 * more distinct experts than slots runs in passes of at most n_slots experts
 * (resident ones first) with one combine at the end.  Results equal
 * moe_forward's on the same weights given the same plan (the expert count of the
 * plan is n_slots).  Prediction of future experts is not built. */
typedef struct moe_expert_cache moe_expert_cache;
typedef struct {
  unsigned long long calls, hits, misses, evictions, bytes_h2d;
  unsigned long long passes; /* expert passes run (one per call unless a call needs more experts than slots) */
} moe_cache_stats_t;

/* How a cache brings missing experts in (moe_cache_set_copy_mode). */
enum {
  MOE_CACHE_COPY_OVERLAP = 0, /* copy engine on the copy stream, overlapped with the expert kernels (default) */
  MOE_CACHE_COPY_SERIAL = 1,  /* copy engine; the expert kernels start after every copy of the pass */
  MOE_CACHE_COPY_KERNEL = 2   /* a copy kernel on the caller's stream reads the host weights directly
                                 (needs host memory the device can address), then the expert kernels */
};

/* host_w13 [E][2I][H], host_w2 [E][H][I] in host memory (registered as page-locked
 * by the cache unless already pinned, unregistered at destroy); w_dtype MOE_BF16 or
 * MOE_E4M3 (then host_w13_scale / host_w2_scale [E] fp32, read at each miss).
 * topk <= n_slots <= E device slots; calls take T <= max_tokens tokens.  FP8 calls
 * must fit in one pass (at most n_slots distinct experts, else MOE_ERR_UNSUPPORTED):
 * their intermediate scale spans every pair of the call.  H % 128 == 0, I % 128 == 0.
 * The cache allocates its device and pinned buffers here (cudaMalloc), none per call. */
MOE_API int moe_cache_create(const void* host_w13, const void* host_w2, const float* host_w13_scale,
                             const float* host_w2_scale, int E, int H, int I, moe_dtype w_dtype, int n_slots,
                             int max_tokens, int topk, moe_expert_cache** cache);
/* MOE_CACHE_COPY_*; MOE_ERR_UNSUPPORTED for MOE_CACHE_COPY_KERNEL when the device cannot
 * address the host weights. */
MOE_API int moe_cache_set_copy_mode(moe_expert_cache* cache, int mode);
MOE_API int moe_cache_destroy(moe_expert_cache* cache);
/* Workspace bytes of a moe_forward_cached call with T tokens. */
MOE_API int moe_cache_workspace_size(const moe_expert_cache* cache, int T, moe_dtype act_dtype,
                                     const moe_options* opts, size_t* bytes);
/* The layer on hidden [T][H] with router_w [E][H] (act_dtype) into out [T][H]; the
 * call blocks until the batch's routing is known.  Calls on one cache are serialised. */
MOE_API int moe_forward_cached(moe_expert_cache* cache, const void* hidden, const void* router_w, int T, int renorm,
                               moe_dtype act_dtype, void* out, void* workspace, size_t workspace_bytes,
                               const moe_options* opts, moe_stream_t stream);
MOE_API int moe_cache_stats(const moe_expert_cache* cache, moe_cache_stats_t* stats);
/* The cache's copy kernel on its own: copies `bytes` (a multiple of 16) from src_host,
 * page-locked host memory the device can address (reads cross NVLink-C2C on a GB300),
 * to the device buffer dst, on `stream`; both 16-byte aligned.  MOE_ERR_UNSUPPORTED if the
 * device cannot address src_host. */
MOE_API int moe_copy_from_host(const void* src_host, void* dst, size_t bytes, moe_stream_t stream);

/* The cache's slot policy alone, host only (no device work): over n_calls calls of
 * `pairs` expert ids each (ids [n_calls][pairs]), writes the slot of every id during
 * its pass (slot_ids [n_calls][pairs]) and, per call, the expert last copied into each
 * slot or -1 (loaded_expert [n_calls][n_slots]); totals of hits and misses (distinct
 * experts per pass found / not found in a slot). */
MOE_API int moe_cache_lru_plan(int E, int n_slots, int n_calls, int pairs, const int32_t* ids, int32_t* slot_ids,
                               int32_t* loaded_expert, unsigned long long* hits, unsigned long long* misses);

/* Allocation-free form of moe_forward (the pages have no counterpart; it is an
 * interface convenience of this library).
 *
 * For callers that cannot allocate device memory when they run the layer --
 * a plugin whose host engine owns and plans all device memory, a serving loop
 * that may not take cudaMalloc's latency or implicit synchronisation, a C
 * caller without a device allocator.  Same arguments and results as
 * moe_forward, without the workspace: the workspace is a fixed array of
 * MOE_NOALLOC_MAX_WORKSPACE bytes in this library's device memory, which every
 * GPU that loads the library keeps until the process exits.
 *  - Shapes whose moe_workspace_size() exceeds MOE_NOALLOC_MAX_WORKSPACE are
 *    rejected with MOE_ERR_WORKSPACE before anything is enqueued.  For
 *    example, bf16 decode batches of up to 64 tokens of a Mixtral-shaped
 *    layer (hidden 4096, 8 experts, FFN 14336: 29.5 MiB) or of a fine-grained
 *    one (hidden 2048, 128 experts, FFN 768, top-8: 26.7 MiB) fit; an FP8
 *    layer with hidden 4096, 64 experts, FFN 8192, top-8 at 64 tokens needs
 *    71 MiB and prefill batches need far more -- use moe_forward for those.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture on that device.  cudaDeviceReset() invalidates the cached
 *    address (and the library's other per-device state): do not call the
 *    library on a device after resetting it in the same process.
 *  - Every call on a device uses the same array and finds the previous call's
 *    contents in it; the layer initialises every word it reads (the FP8 amax
 *    words, the timeout test flag and the single-launch kernel's launch tag
 *    are cleared on the stream first), so nothing needs clearing by the
 *    caller.  Calls whose GPU work overlaps (different streams, or several
 *    host threads) race on the array: issue them on one stream.
 *  - Allocates nothing, frees nothing, and calls no allocating library routine. */
#define MOE_NOALLOC_MAX_WORKSPACE (32u << 20)
MOE_API int moe_forward_noalloc(const void* hidden, const void* router_w, const void* w13, const void* w2, int T, int H,
                                int I, int E, int topk, int renorm, moe_dtype act_dtype, moe_dtype w_dtype,
                                const void* w13_scale, const void* w2_scale, void* out, const moe_options* opts,
                                moe_stream_t stream);

/* Synchronises `stream`, then reads and clears this device's status word.
 * Returns MOE_OK, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_DEVICE_INDEX or MOE_ERR_CUDA. */
MOE_API int moe_get_status(moe_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
MOE_API int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_API_H */
