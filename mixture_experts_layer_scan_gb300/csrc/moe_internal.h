// Internal host-side interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe_api.h"

namespace moe {

// Per-call routing metadata written by the permutation kernel (int32 words):
//   [0] num_post_pad  [1] number of blocks  [2] number of active experts
//   [3] number of CTA-pair chunks (token-major on CTA pairs; see launch_align)
//   [4, 4+E)          active experts, ascending
//   [4+E, 5+2E)       padded start offset of every expert (E+1 entries, last = num_post_pad)
//   [5+2E, 5+3E)      tokens per expert
enum { META_NPP = 0, META_NBLK = 1, META_NACT = 2, META_NPB = 3, META_HDR = 4 };
inline int meta_words(int E) { return META_HDR + 3 * E + 1; }
__host__ __device__ inline int meta_active(int E) { (void)E; return META_HDR; }
__host__ __device__ inline int meta_offsets(int E) { return META_HDR + E; }
__host__ __device__ inline int meta_counts(int E) { return META_HDR + 2 * E + 1; }

// ---- routing ----------------------------------------------------------------
cudaError_t launch_router_logits(const void* X, const void* Wr, int T, int H, int E, bool bf16, float* logits,
                                 cudaStream_t s);
cudaError_t launch_topk(const float* logits, int T, int E, int k, int renorm, float* w, int32_t* ids,
                        cudaStream_t s);
cudaError_t launch_inject_timeout(const int* flag, int* status, cudaStream_t s);

// ---- permutation / data movement ----------------------------------------------
// skip_minus_one: ids equal to -1 are pairs handled elsewhere (dropped silently); other ids
// outside [0, E) are dropped and flagged MOE_ERR_DEVICE_INDEX.
// pblk (nullable, B = 128, capacity sorted_cap / 128): the chunks of the CTA-pair GEMM tiles,
// every expert's padded run split into 256-row chunks with a 128-row last chunk where the
// run has an odd number of blocks: pblk[c] = (first row << 1) | (1 for 128 rows); their
// count goes to meta[META_NPB].  inv (nullable, T*k words): the sorted row of each
// pair, -1 for a pair left out.
cudaError_t launch_align(const int32_t* ids, int T, int k, int E, int B, int32_t* sorted, int32_t* eids,
                         int32_t* npp, int32_t* counts, int32_t* meta, int* status, cudaStream_t s,
                         bool skip_minus_one = false, int32_t* pblk = nullptr, unsigned* zero_words = nullptr,
                         int n_zero = 0, int32_t* inv = nullptr);
// dst (device) = bytes of page-locked host memory read by the device at src (its device
// address); a kernel launched like the library's others (bytes and both addresses 16-byte
// multiples, else cudaErrorInvalidValue)
cudaError_t launch_copy_from_host(const void* src, void* dst, size_t bytes, int sms, cudaStream_t s);
// amax over n bf16 values -> *amax_bits (float bits, must be zeroed before)
cudaError_t launch_amax_bf16(const void* X, size_t n, unsigned* amax_bits, cudaStream_t s);
// Xs[r] = X[sorted[r]/k] (zero rows for the sentinel) for r < num_post_pad;
// mode 0: copy elements of elem_bytes, token by token through inv when it is given
// (launch_align's inverse map; k <= 32: every token row read once), else row by row;
// mode 1: bf16 -> e4m3 with scale amax/448 (inv unused).
// late (row-by-row copy and mode 1): let dependents launch only after this kernel's own
// dependency wait, so the permutation is complete when the next kernel starts.
cudaError_t launch_gather(const void* X, int T, int H, int k, int elem_bytes, int mode, const unsigned* amax_bits,
                          const int32_t* sorted, const int32_t* inv, const int32_t* meta, int cap, void* Xs,
                          bool late, cudaStream_t s);
// split-K reduction of the GEMM1 partials P[split][pair][2I] + scale + SiLU(gate)*up
// into sorted rows (row r holds pair sorted[r]).
//   out_mode 0: bf16 A_int   1: fp32 A (+ amax into amax_bits)
// Padding rows (sentinel pairs) become zero and stay out of the amax.
// out_mode 0 with A_lo != nullptr also writes the low bf16 part a - bf16(a).
cudaError_t launch_reduce_act(const float* P, int splits, size_t split_stride, int I, int B, int n_pairs,
                              const int32_t* sorted, const int32_t* eids, const int32_t* meta, int cap,
                              const float* w_scale, const unsigned* a_amax_bits, int out_mode, void* A_out,
                              void* A_lo, unsigned* amax_bits, cudaStream_t s);
// Xq[i] = e4m3(X[i] / (amax/448)) for the n bf16 values of X (n % 8 == 0)
cudaError_t launch_quant_x(const void* X, size_t n, const unsigned* amax_bits, uint8_t* Xq, cudaStream_t s);
// A_q[r][i] = e4m3(A[r][i] / (amax/448)) for r < num_post_pad
cudaError_t launch_quant_act(const float* A, int I, const int32_t* meta, int cap, const unsigned* amax_bits,
                             uint8_t* Aq, cudaStream_t s);
// out[t] = sum_j w[t][j] * sum_s Y[s][t*k+j]   (Y fp32 or bf16, out fp32 or bf16)
cudaError_t launch_combine(const void* Y, int y_bf16, int splits, size_t split_stride, const float* w, int T, int k,
                           int H, void* out, int out_bf16, cudaStream_t s);
// lanes G that share one output vector in the combine (H % 8 == 0); fixes its addition order
int combine_lanes(int T, int H, int k);

// ---- fp32 CUDA-core grouped GEMMs ---------------------------------------------
cudaError_t launch_gemm1_simt(const float* Xs, const float* W13, int H, int I, int B, const int32_t* eids,
                              const int32_t* meta, int cap, float* A, cudaStream_t s);
cudaError_t launch_gemm2_simt(const float* A, const float* W2, int H, int I, int B, int T, int k,
                              const int32_t* sorted, const int32_t* eids, const int32_t* meta, int cap, float* Y,
                              cudaStream_t s);

// ---- tcgen05 grouped GEMM --------------------------------------------------------
enum TcEpilogue {
  TC_EPI_G1_BF16 = 0,    // GEMM1: SiLU(gate)*up -> bf16 A_int
  TC_EPI_G1_PART = 1,    // GEMM1: raw fp32 partials [split][pair][2I] (gate cols [0,I), up [I,2I))
  TC_EPI_G1_F32AMAX = 2, // GEMM1: scaled SiLU(gate)*up -> fp32 A + amax (FP8 path)
  TC_EPI_G2_F32 = 3,     // GEMM2: fp32 Y[split][pair][H]
  TC_EPI_G2_BF16 = 4,    // GEMM2: bf16 Y[pair][H]
  TC_EPI_LOGITS = 5      // router: fp32 logits[T][n_valid] of unsorted token rows (token-major only)
};

struct TcGemmArgs {
  bool swap;        // swap-AB orientation (weights in the M slot)
  bool fp8;         // e4m3 operands (kind::f8f6f4), else bf16 (kind::f16)
  int epi;          // TcEpilogue
  // problem
  int T, k, E, I, H;
  int K;            // reduction length in elements
  int w_rows_per_expert;
  int w_pair_off;   // row offset of the second weight load from the first
  int w_tile_rows;  // weight rows advanced per output tile
  int wbox;         // rows per weight load (tile = two loads)
  int xbox;         // token rows per activation load
  int n_tiles;      // output tiles per expert (or per 128-row block)
  int splits;       // K splits (swap mode)
  int kb_per_split; // k-blocks (128 bytes of K) per split
  int cap;          // rows of the sorted activation buffer (T for the router)
  bool gather;      // X is the unsorted [T][K] tensor; rows are gathered by token (tile::gather4)
  bool early;       // tile list and weights may be read before the dependency wait: only when every
                    // kernel that wrote the metadata finished before the preceding kernel could launch
  int n_valid;      // router: number of output columns (experts) to store
  // tensors
  const void* W;    // weights viewed as [E * w_rows_per_expert][K]
  const void* X;    // sorted activations [cap][K]
  const int32_t* sorted;
  const int32_t* eids;
  const int32_t* meta;
  void* out;
  void* out_lo;             // GEMM1 bf16: low part of the intermediate, a - bf16(a) (nullable)
  int x_lo_rows;            // GEMM2: >0 when X holds a low bf16 part at rows [x_lo_rows, x_lo_rows + cap)
  size_t out_split_stride;  // elements between split partial buffers
  const float* w_scale;     // [E] (FP8)
  const unsigned* a_amax;   // amax bits of the activation operand (FP8)
  unsigned* amax_out;       // amax bits of the produced intermediate (FP8 GEMM1)
  int* status;
  int num_sms;
  bool pair;                // token-major on CTA pairs (tcgen05 cta_group::2), tiles from pblk
  const int32_t* pblk;      // CTA-pair chunks (launch_align)
  int prefetch_kb;          // swap-AB GEMM1: L2 prefetch of the first tile's first K blocks before the
                            // dependency wait, on the guess that all experts are active (0: off)
  bool w4;                  // INT4 weight codes (swap-AB), dequantised to bf16 in the main loop
  const void* w4_scale;     // bf16 group scales [E][K / 128][w_rows_per_expert]
  // bf16 swap-AB GEMM1 with K splits: arrival counters [E][n_tiles] (zeroed by launch_align) that
  // let the CTA storing a tile's last split write the finished intermediate (out_fin / out_fin_lo)
  unsigned* fin;
  void* out_fin;
  void* out_fin_lo;
  // expert cache: before streaming expert e's weights the producer waits (bounded) until
  // ready[e] == want[e] (words written by the cache's copy stream after each copy); nullable
  const unsigned* ready;
  const unsigned* want;
  // swap-AB k_gemm_tc: tiles past the first wave may be claimed from *claim (zeroed each call
  // by the preceding GEMM through zero_word, after its dependency wait); nullable
  int* claim;
  int* zero_word;
};
cudaError_t launch_gemm_tc(const TcGemmArgs& a, cudaStream_t s);

// 2-D K-major tensor map [rows][K] of 1- or 2-byte elements: box of box_bytes
// of K x box_rows; 128 and 64 bytes are swizzled with the same span, 256 bytes
// are not swizzled.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t K, uint64_t rows,
                        uint32_t box_rows, uint32_t box_bytes = 128);

// ---- inverse rotary embedding + per-head FP8 quantisation ----------------------------
cudaError_t launch_inv_rope_fp8(const void* X, int T, int heads, int D, int R, const int32_t* pos,
                                const float* cos_sin, int max_pos, uint8_t* Q, float* scale, int* status,
                                int num_sms, cudaStream_t s);

// ---- single-launch decode layer (bf16, swap-AB) ----------------------------------
struct FusedArgs {
  int T, H, I, E, k, renorm;
  int s1, kbs1, s2, kbs2;  // K splits and K blocks (128 bytes) per split of GEMM1 / GEMM2
  int xbox;                // tokens rounded up to 16 (<= 64)
  bool gather;             // GEMM1 gathers token rows itself (xbox <= 32); else rows go to Xs first
  bool act_split;          // intermediate as bf16 hi + lo
  int cap;                 // rows of Xs / of each intermediate part
  int combine_g;           // lanes per output of the stand-alone combine (same sum order)
  const void* X;           // [T][H] bf16
  const void* Wr;          // [E][H] bf16
  const void* w13;         // [E][2I][H] bf16
  const void* w2;          // [E][H][I] bf16
  float* logits;           // [T][E]
  float* topk_w;           // [T][k]
  int32_t* topk_ids;       // [T][k]
  void* Xs;                // [cap][H] (gather == false)
  void* aint;              // [cap][I] (x2 with act_split)
  float* p1;               // [s1][T*k][2I] (s1 > 1)
  size_t p1_stride;
  float* y;                // [s2][T*k][H]
  size_t y_stride;
  void* out;               // [T][H] bf16
  void* sync;              // fused_sync_bytes(E, I, H, T) bytes, 256-aligned
  void* trace;             // nullable: MOE_TRACE_WORDS uint64 per CTA
  int* status;
  int num_sms;
};
// bytes of the launch tag and counters the single-launch kernel keeps in the workspace
size_t fused_sync_bytes(int T, int H, int I, int E);
// shared memory the single-launch kernel needs beyond its stage ring
size_t fused_table_bytes(int T, int E, int k);
cudaError_t launch_decode_fused(const FusedArgs& a, cudaStream_t s);

// status word of the current device
int* status_word();

// ---- expert cache passes (moe_cache.cu) -----------------------------------------------
// Per-slot readiness words: GEMM1 streams slot e's w13 once ready13[e] == want[e], GEMM2
// its w2 once ready2[e] == want[e].  Null members: no waiting.
struct SlotGate {
  const unsigned* ready13;
  const unsigned* ready2;
  const unsigned* want;
};
// Steps of the layer on a given routing (as moe_forward_routed), for the expert cache:
//   experts: permutation + GEMMs of the pairs whose id is not -1 (ids -1 are skipped
//            silently: another pass computes them); Y rows of those pairs are written
//   combine: the weighted sum of every pair's Y rows into out
// The plan depends only on (T, H, I, E, topk, dtypes, options), so passes over disjoint
// pair sets with the same arguments share the workspace's Y buffers and one combine.
int forward_routed_pass(const void* hidden, const float* topk_w, const int32_t* ids, const void* w13, const void* w2,
                        int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                        const void* w13_scale, const void* w2_scale, void* out, void* workspace,
                        size_t workspace_bytes, const moe_options* opts, cudaStream_t stream, bool experts,
                        bool combine, const SlotGate* gate);

}  // namespace moe
