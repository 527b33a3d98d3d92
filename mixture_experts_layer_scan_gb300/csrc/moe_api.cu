// C ABI of the fused MoE layer forward: argument checks, workspace layout,
// choice of kernels, and the launch sequence of one layer call.
//
// Declared in include/moe_api.h; every entry point is extern "C", takes plain
// pointers and sizes, and enqueues work on the caller's stream.
#include <algorithm>
#include <mutex>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// One status word per device: kernels record the first fault they see here
// (MOE_ERR_DEVICE_TIMEOUT / MOE_ERR_DEVICE_INDEX); moe_get_status reads and
// clears it.
static __device__ int g_status_word;

constexpr int kMaxDevices = 64;

int* status_word() {
  static int* ptr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptr[dev] = static_cast<int*>(p);
  }
  return ptr[dev];
}

static int num_sms() {
  static int sms[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return sms[dev];
}

// SM count used to plan K splits.  A fixed constant (the 152 SMs of a GB300)
// so that the workspace size depends only on the arguments.
constexpr int kPlanSms = 152;
// Router logits go through the tensor-core GEMM from this many tokens on.
constexpr int kRouterTcMinTokens = 256;
// From this many tokens on, the row gather goes token by token (each token row read
// once, stored at its k sorted rows); shorter batches gather row by row over more warps.
constexpr int kGatherTokenOrderMinTokens = 4096;
// Largest swap-AB activation tile whose rows GEMM1 gathers itself.
constexpr int kGatherInGemmMaxRows = 32;
// Single-launch decode kernel limits (shared-memory tables, one token column per epilogue thread).
constexpr int kFusedMaxTokens = 64;
constexpr int kFusedMaxPairs = 512;
constexpr int kFusedMaxExperts = 256;
// Largest batch whose single-launch GEMM1 keeps the K splits of the multi-kernel plan.
constexpr int kFusedSplitMaxTokens = 8;
// Largest batch whose split GEMM1 is summed by the last-arriving CTA of each tile.
constexpr int kFinMaxTokens = 8;
// moe_options.single_launch == 0 picks the single-launch kernel for eligible shapes.
constexpr bool kFusedAuto = false;

enum Path { PATH_F32 = 0, PATH_BF16 = 1, PATH_FP8 = 2, PATH_W4 = 3 };

struct Plan {
  int path = 0;
  bool swap = false;
  int B = 16;
  long cap = 0, nblk_cap = 0;
  int xbox = 128;
  int s1 = 1, kb1 = 1, s2 = 1, kb2 = 1;
  int wbox2 = 128;  // token-major GEMM2 weight rows per load (N = 2 * wbox2)
  bool y_bf16 = false;
  bool act_split = false;  // bf16 intermediate stored as hi + lo parts (two MMAs in GEMM2)
  bool gather_in_gemm = false;  // GEMM1 gathers its activation rows itself (TMA tile::gather4)
  bool fused = false;           // the whole layer as one cooperative kernel
  bool pair = false;            // token-major GEMMs on CTA pairs (256-row permutation blocks)
  bool fin = false;             // bf16 swap-AB GEMM1 splits summed by the last-arriving CTA (no reduction kernel)
  size_t o_sync = 0;
  size_t o_logits = 0, o_tw = 0, o_tid = 0, o_meta = 0, o_sorted = 0, o_eids = 0, o_xs = 0, o_aint = 0, o_af32 = 0,
         o_p1 = 0, o_y = 0, o_misc = 0, o_pblk = 0, o_fin = 0, o_inv = 0, total = 0;
  size_t p1_stride = 0, y_stride = 0;
};

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// K splits of a swap-AB GEMM with base_tiles (expert x 128-row) tiles of
// kb_total 128-byte K blocks.  The persistent kernel gives each CTA
// ceil(tiles / SMs) tiles, so the step time follows
//   ceil(base_tiles * s / SMs) * (ceil(kb_total / s) + 1)
// (the +1 stands for the per-tile fill and epilogue); take the s in [1, 16]
// with at least 2 K blocks per split that minimises it, fewest splits on ties.
// split_penalty (in K blocks) charges an extra reduction kernel, if splitting
// needs one.
static int choose_splits(long base_tiles, int kb_total, int forced, int split_penalty) {
  if (forced > 0) return std::max(1, std::min(forced, kb_total));
  int best = 1;
  long best_t = -1;
  for (int s = 1; s <= 16 && s <= std::max(1, kb_total / 2); ++s) {
    const int kbs = (kb_total + s - 1) / s;
    const int se = (kb_total + kbs - 1) / kbs;
    if (se != s) continue;
    const long waves = (base_tiles * s + kPlanSms - 1) / kPlanSms;
    const long t = waves * (kbs + 1) + (s > 1 ? split_penalty : 0);
    if (best_t < 0 || t < best_t) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

// K splits of swap-AB GEMM2 (no reduction kernel: the combine sums the splits).  The
// waves of (expert, tile, split) units share HBM: a wave of n < SMs units streams each
// unit at min(kSmStreamCap, SMs / n) times a full wave's per-unit rate, so a last,
// partial wave -- or a single wave of a few large tiles -- costs less than a full one.
// Step time in K-block units of a full wave:
//   sum over waves of ceil(kb_total / s) / min(kSmStreamCap, SMs / units in the wave) + 1.
// (Measured on the decode layers: one 128-tile wave of whole rows beats 7 or 8 splits,
// while 32 tiles want about 4.)  The tile count is the upper bound min(E, T*k) of active
// experts, which is exact for one token and near certain from 4E pairs on; in between
// (4 tokens of top-2 over 8 experts activate about 5.5) a plan trusting it leaves SMs
// idle, so those batches keep the wave count alone.
constexpr double kSmStreamCap = 1.25;
static int choose_splits_shared(long base_tiles, int kb_total, int forced) {
  if (forced > 0) return std::max(1, std::min(forced, kb_total));
  int best = 1;
  double best_t = -1.0;
  for (int s = 1; s <= 16 && s <= std::max(1, kb_total / 2); ++s) {
    const int kbs = (kb_total + s - 1) / s;
    const int se = (kb_total + kbs - 1) / kbs;
    if (se != s) continue;
    double t = 0.0;
    for (long left = base_tiles * s; left > 0; left -= kPlanSms) {
      const long n = std::min<long>(left, kPlanSms);
      t += kbs / std::min(kSmStreamCap, (double)kPlanSms / (double)n) + 1.0;
    }
    if (best_t < 0.0 || t < best_t - 1e-9) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

static int check_shape(int T, int H, int I, int E, int topk) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || E > 1024 || topk < 1 || topk > E || topk > 32) return MOE_ERR_ARG;
  const long long n = (long long)T * topk;
  if (n + (long long)std::min<long long>(E, n) * 127 >= (1ll << 31)) return MOE_ERR_ARG;
  return MOE_OK;
}

static int make_plan(int T, int H, int I, int E, int topk, moe_dtype act, moe_dtype w, const moe_options* opts,
                     Plan* pl) {
  int rc = check_shape(T, H, I, E, topk);
  if (rc) return rc;
  Plan p;
  if (act == MOE_F32 && w == MOE_F32) {
    p.path = PATH_F32;
    if (H % 4) return MOE_ERR_UNSUPPORTED;
  } else if (act == MOE_BF16 && w == MOE_BF16) {
    p.path = PATH_BF16;
  } else if (act == MOE_BF16 && w == MOE_E4M3) {
    p.path = PATH_FP8;
  } else if (act == MOE_BF16 && w == MOE_INT4) {
    p.path = PATH_W4;
  } else {
    return (act > MOE_INT4 || w > MOE_INT4 || act < 0 || w < 0) ? MOE_ERR_ARG : MOE_ERR_UNSUPPORTED;
  }
  const int orient = opts ? opts->orientation : MOE_ORIENT_AUTO;
  if (orient < 0 || orient > 2) return MOE_ERR_ARG;
  const int act_mode = opts ? opts->act_split : 0;
  if (act_mode < 0 || act_mode > 2) return MOE_ERR_ARG;
  const long n = (long)T * topk;
  if (p.path != PATH_F32) {
    if (H % 128 || I % 128) return MOE_ERR_UNSUPPORTED;
    p.swap = orient == MOE_ORIENT_SWAP_AB ||
             (orient == MOE_ORIENT_AUTO && (T <= 64 || (p.path == PATH_W4 && T <= 128)));
    if (p.swap && T > 256) return MOE_ERR_UNSUPPORTED;
    // INT4 weights: swap-AB batches of up to 128 tokens, whole 256-row weight tiles
    if (p.path == PATH_W4 && (!p.swap || T > 128 || H % 256 || I % 256)) return MOE_ERR_UNSUPPORTED;
    const int eb = p.path == PATH_FP8 ? 1 : 2;
    if (p.swap) {
      p.B = 16;
      p.xbox = std::max(16, (T + 15) / 16 * 16);
      const long act_upper = std::min<long>(E, n);
      const int forced = opts ? opts->split_k : 0;
      if (forced < 0) return MOE_ERR_ARG;
      // K blocks: 128 bytes of K for bf16 / e4m3 operands, 128-element raw stages (one scale group) for INT4
      const int kbt1 = p.path == PATH_W4 ? H / 128 : H * eb / 128;
      const int kbt2 = p.path == PATH_W4 ? I / 128 : I * eb / 128;
      // swap-AB tiles: 128 gate + 128 up rows (GEMM1), 256 rows of w2 (GEMM2)
      p.s1 = choose_splits(act_upper * (I / 128), kbt1, forced, 8);
      p.kb1 = (kbt1 + p.s1 - 1) / p.s1;
      p.s1 = (kbt1 + p.kb1 - 1) / p.kb1;
      // (INT4 GEMMs are bound by the MMA rate, not by a shared HBM stream: wave counts only)
      const bool active_known = T == 1 || n >= 4L * E;
      p.s2 = (p.path != PATH_W4 && active_known) ? choose_splits_shared(act_upper * ((H + 255) / 256), kbt2, forced)
                                                 : choose_splits(act_upper * ((H + 255) / 256), kbt2, forced, 0);
      p.kb2 = (kbt2 + p.s2 - 1) / p.s2;
      p.s2 = (kbt2 + p.kb2 - 1) / p.kb2;
      p.y_bf16 = false;
    } else {
      const int pair_mode = opts ? opts->cta_pair : 0;
      if (pair_mode < 0 || pair_mode > 2) return MOE_ERR_ARG;
      p.pair = pair_mode != 2 && H % 256 == 0;
      if (pair_mode == 1 && !p.pair) return MOE_ERR_UNSUPPORTED;
      p.B = 128;
      p.xbox = 128;
      p.s1 = p.s2 = 1;
      p.kb1 = H * eb / 128;
      p.kb2 = I * eb / 128;
      p.wbox2 = (H % 256 == 0) ? 128 : 64;
      p.y_bf16 = false;
    }
    // hi/lo intermediate: by default where it is free (bf16 swap-AB decode
    // streams weights from HBM; the second MMA only uses idle tensor-core time).
    // The INT4 GEMMs are bound by the MMA instruction rate, where GEMM2's second
    // MMA costs about 10 %: there it is on request only (act_split = 2).
    p.act_split = (p.path == PATH_BF16 && (act_mode == 2 || (act_mode == 0 && p.swap))) ||
                  (p.path == PATH_W4 && act_mode == 2);
    // GEMM1 gathers token rows itself (one tile::gather4 per 4 rows) when the
    // activation tile is short; for wider tiles the per-stage TMA instruction
    // count outweighs the saved kernel, so rows are gathered beforehand.
    p.gather_in_gemm = p.swap && p.xbox <= kGatherInGemmMaxRows;
  } else {
    p.B = 16;
    p.swap = false;
  }
  p.cap = n + std::min<long>(E, n) * (p.B - 1);
  p.nblk_cap = p.cap / p.B;
  const int single = opts ? opts->single_launch : 0;
  if (single < 0 || single > 2) return MOE_ERR_ARG;
  const bool fused_ok = p.path == PATH_BF16 && p.swap && T <= kFusedMaxTokens && n <= kFusedMaxPairs &&
                        E <= kFusedMaxExperts;
  if (single == 1 && !fused_ok) return MOE_ERR_UNSUPPORTED;
  p.fused = fused_ok && (single == 1 || (single == 0 && kFusedAuto));
  if (p.fused && T > kFusedSplitMaxTokens && !(opts && opts->split_k > 0)) {
    // in the single launch the CTA finishing a tile's last K split sums the
    // splits for all of the expert's tokens; past a few tokens that serial
    // reduction costs more than the splits gain, so GEMM1 runs unsplit
    p.s1 = 1;
    p.kb1 = H * (p.path == PATH_FP8 ? 1 : 2) / 128;
  }

  const size_t A = 256;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1), A);
    return at;
  };
  const size_t xb = p.path == PATH_F32 ? 4 : (p.path == PATH_FP8 ? 1 : 2);  // activation element bytes
  p.o_logits = take((size_t)T * E * 4);
  p.o_tw = take((size_t)n * 4);
  p.o_tid = take((size_t)n * 4);
  p.o_meta = take((size_t)meta_words(E) * 4);
  p.o_sorted = take((size_t)p.cap * 4);
  p.o_eids = take((size_t)std::max<long>(p.nblk_cap, 1) * 4);
  // gathered activation rows: the fp32 path gathers into sorted order; the
  // tensor-core paths gather inside GEMM1 (FP8 keeps a token-order e4m3 copy)
  size_t xs_bytes = (size_t)p.cap * H * xb;                      // rows gathered into expert order
  if (p.gather_in_gemm) xs_bytes = p.path == PATH_FP8 ? (size_t)T * H : 0;  // token order (FP8: e4m3 copy)
  p.o_xs = take(xs_bytes);
  p.o_aint = take((size_t)p.cap * I * xb * (p.act_split ? 2 : 1));
  if (p.path == PATH_FP8) p.o_af32 = take((size_t)p.cap * I * 4);
  if (p.s1 > 1) {
    p.p1_stride = (size_t)n * 2 * I;
    p.o_p1 = take(p.p1_stride * p.s1 * 4);
  }
  p.y_stride = (size_t)n * H;
  p.o_y = take(p.y_stride * p.s2 * (p.y_bf16 ? 2 : 4));
  p.o_misc = take(256);
  if (p.pair) p.o_pblk = take((size_t)std::max<long>(p.nblk_cap, 1) * 4);
  // pair -> sorted row, for the token-order gather of long batches
  if (p.gather_in_gemm || p.path == PATH_FP8 || T < kGatherTokenOrderMinTokens) p.o_inv = 0;
  else p.o_inv = take((size_t)n * 4);
  // (the last arriver sums the splits token by token: a chain of L2 round trips that
  // outgrows the separate reduction kernel past a few tokens)
  p.fin = p.path == PATH_BF16 && p.swap && p.s1 > 1 && !p.fused && T <= kFinMaxTokens;
  if (p.fin) p.o_fin = take((size_t)E * (I / 128) * 4);
  if (p.fused) p.o_sync = take(fused_sync_bytes(T, H, I, E));
  p.total = o;
  *pl = p;
  return MOE_OK;
}

static bool misaligned(const void* p, uintptr_t a = 16) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

static int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static void record(moe_event_t ev, cudaStream_t s) {
  if (ev) cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), s);
}

// Router logits: the tensor-core GEMM for long bf16 batches (128 tokens per
// tile, all experts in the N slot), the CUDA-core kernel otherwise.
static cudaError_t launch_router(const void* X, const void* Wr, int T, int H, int E, moe_dtype act, float* logits,
                                 int* status, cudaStream_t s) {
  const int sms = num_sms();
  if (act == MOE_BF16 && T >= kRouterTcMinTokens && E <= 256 && H % 128 == 0 && sms > 0) {
    TcGemmArgs g = {};
    g.swap = false;
    g.fp8 = false;
    g.epi = TC_EPI_LOGITS;
    g.T = T;
    g.k = 1;
    g.E = 1;
    g.H = H;
    g.K = H;
    g.W = Wr;
    g.w_rows_per_expert = E;
    // experts in nt column tiles of N = epad / nt when the token tiles alone would leave
    // SMs idle (N a multiple of 16, each of the tile's two weight boxes a multiple of 8 rows)
    const int epad = (E + 15) / 16 * 16;
    const int row_tiles = (T + 127) / 128;
    int nt = 1;
    while (nt < 4 && epad % (32 * nt) == 0 && 2 * nt * row_tiles <= sms) nt *= 2;
    g.wbox = epad / (2 * nt);
    g.w_pair_off = g.wbox;
    g.w_tile_rows = 2 * g.wbox;
    g.xbox = 128;
    g.n_tiles = nt;
    g.splits = 1;
    g.kb_per_split = H * 2 / 128;
    g.cap = T;
    g.X = X;
    g.out = logits;
    g.n_valid = E;
    g.early = true;  // the router reads no earlier kernel's output before its dependency wait except weights
    g.status = status;
    g.num_sms = sms;
    return launch_gemm_tc(g, s);
  }
  return launch_router_logits(X, Wr, T, H, E, act == MOE_BF16, logits, s);
}

enum { STEPS_ROUTE = 1, STEPS_EXPERTS = 2, STEPS_COMBINE = 4, STEPS_ALL = 7 };

// The launch sequence of one layer call on a planned, validated workspace.
// steps selects routing (S1-S2), the expert part (S3-S6, which reads the
// routing from the workspace or tw_in / tid_in) and the combine (S7).
// E_router is the router's expert count and logits_override an optional
// logits buffer (both differ from the plan's when the experts are cache
// slots).  gate (nullable) makes the GEMMs wait for per-slot readiness words;
// skip_minus_one drops pairs whose id is -1 from the permutation.
static int forward_steps(const Plan& pl, int steps, const void* hidden, const void* router_w, int E_router,
                         float* logits_override, const float* tw_in, const int32_t* tid_in, const void* w13,
                         const void* w2, int T, int H, int I, int E, int topk, int renorm, moe_dtype act_dtype,
                         const void* w13_scale, const void* w2_scale, void* out, void* workspace,
                         const moe_options* opts, int* st, int sms, cudaStream_t s, const SlotGate* gate = nullptr,
                         bool skip_minus_one = false) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* logits = logits_override ? logits_override : reinterpret_cast<float*>(ws + pl.o_logits);
  // the routing: written here by steps 1-2, or given by the caller for the expert steps alone
  float* tw = tw_in ? const_cast<float*>(tw_in) : reinterpret_cast<float*>(ws + pl.o_tw);
  int32_t* tid = tid_in ? const_cast<int32_t*>(tid_in) : reinterpret_cast<int32_t*>(ws + pl.o_tid);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + pl.o_meta);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + pl.o_sorted);
  int32_t* eids = reinterpret_cast<int32_t*>(ws + pl.o_eids);
  int32_t* pblk = pl.pair ? reinterpret_cast<int32_t*>(ws + pl.o_pblk) : nullptr;
  int32_t* inv = pl.o_inv ? reinterpret_cast<int32_t*>(ws + pl.o_inv) : nullptr;
  unsigned* fin = pl.fin ? reinterpret_cast<unsigned*>(ws + pl.o_fin) : nullptr;
  void* xs = ws + pl.o_xs;
  void* aint = ws + pl.o_aint;
  float* af32 = reinterpret_cast<float*>(ws + pl.o_af32);
  float* p1 = reinterpret_cast<float*>(ws + pl.o_p1);
  void* y = ws + pl.o_y;
  unsigned* amax = reinterpret_cast<unsigned*>(ws + pl.o_misc);  // [0] input amax, [1] intermediate amax
  int* flag = reinterpret_cast<int*>(ws + pl.o_misc + 64);
  const moe_options* o = opts;
  const int cap = (int)pl.cap;
  const int n = T * topk;
  cudaError_t e = cudaSuccess;
#define MOE_TRY(x)                 \
  do {                             \
    e = (x);                       \
    if (e != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

  if (steps == STEPS_ALL && pl.fused && !(o && o->inject_timeout)) {
    // steps 1-7 in one cooperative kernel; its events bracket the kernel as GEMM1
    if (o) {
      for (int st = MOE_STAGE_ROUTE; st < MOE_STAGE_GEMM1; ++st) {
        record(o->stage_begin[st], s);
        record(o->stage_end[st], s);
      }
      record(o->stage_begin[MOE_STAGE_GEMM1], s);
    }
    FusedArgs fa = {};
    fa.T = T;
    fa.H = H;
    fa.I = I;
    fa.E = E;
    fa.k = topk;
    fa.renorm = renorm != 0;
    fa.s1 = pl.s1;
    fa.kbs1 = pl.kb1;
    fa.s2 = pl.s2;
    fa.kbs2 = pl.kb2;
    fa.xbox = pl.xbox;
    fa.gather = pl.gather_in_gemm;
    fa.act_split = pl.act_split;
    fa.cap = cap;
    fa.combine_g = combine_lanes(T, H, topk);
    fa.X = hidden;
    fa.Wr = router_w;
    fa.w13 = w13;
    fa.w2 = w2;
    fa.logits = logits;
    fa.topk_w = tw;
    fa.topk_ids = tid;
    fa.Xs = xs;
    fa.aint = aint;
    fa.p1 = p1;
    fa.p1_stride = pl.p1_stride;
    fa.y = reinterpret_cast<float*>(y);
    fa.y_stride = pl.y_stride;
    fa.out = out;
    fa.sync = ws + pl.o_sync;
    fa.trace = o ? o->trace : nullptr;
    fa.status = st;
    fa.num_sms = sms;
    // The launch tag starts at zero: the workspace may hold anything (a previous call of
    // another shape), and other CTAs start once the tag equals this launch's grid id.
    if (cudaMemsetAsync(fa.sync, 0, sizeof(unsigned long long), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (launch_decode_fused(fa, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (o) {
      record(o->stage_end[MOE_STAGE_GEMM1], s);
      for (int st = MOE_STAGE_ACT; st < MOE_NUM_STAGES; ++st) {
        record(o->stage_begin[st], s);
        record(o->stage_end[st], s);
      }
    }
    return MOE_OK;
  }

  if ((steps & STEPS_ROUTE) && o && o->inject_timeout) {
    MOE_TRY(cudaMemsetAsync(flag, 0, sizeof(int), s));
    MOE_TRY(launch_inject_timeout(flag, st, s));
    return MOE_OK;
  }

  // 1-2. router
  if (steps & STEPS_ROUTE) {
    if (o) record(o->stage_begin[MOE_STAGE_ROUTE], s);
    MOE_TRY(launch_router(hidden, router_w, T, H, E_router, act_dtype, logits, st, s));
    MOE_TRY(launch_topk(logits, T, E_router, topk, renorm != 0, tw, tid, s));
    if (o) record(o->stage_end[MOE_STAGE_ROUTE], s);
  }
  // routing leaves HBM idle: when every expert is almost surely active (T*k at least
  // 8 E pairs), each swap-AB GEMM1 CTA prefetches its first tile's first weights into L2
  // while the routing runs (a hint: a wrong guess costs only idle bandwidth).  Otherwise
  // the row gather lets GEMM1 launch only once the permutation is complete, and GEMM1
  // streams its first weight stages into shared memory while the gather runs.
  const bool g1_prefetch = pl.swap && !gate && (long)T * topk >= 8L * E;
  const bool g1_early = pl.swap && pl.path != PATH_W4 && !pl.gather_in_gemm && !inv && !gate && !g1_prefetch;

  if (!(steps & (STEPS_EXPERTS | STEPS_COMBINE))) return MOE_OK;
  if (!(steps & STEPS_EXPERTS)) goto combine_step;

  // 3. permutation
  if (o) record(o->stage_begin[MOE_STAGE_ALIGN], s);
  // the permutation kernel also zeroes the counters of this call's later kernels: the split
  // arrival counters (last-arriver sums) or the two FP8 amax words, so that no memset node
  // breaks the chain of programmatically dependent launches
  {
    unsigned* zero_words = pl.fin ? fin : (pl.path == PATH_FP8 ? amax : nullptr);
    const int n_zero = pl.fin ? E * (I / 128) : (pl.path == PATH_FP8 ? 2 : 0);
    MOE_TRY(launch_align(tid, T, topk, E, pl.B, sorted, eids, meta + META_NPP, nullptr, meta, st, s, skip_minus_one,
                         pblk, zero_words, n_zero, inv));
  }
  if (o) record(o->stage_end[MOE_STAGE_ALIGN], s);

  // 4. activations: the fp32 path gathers rows into expert order here; the
  // tensor-core paths gather inside GEMM1 (FP8: quantise the input to e4m3 first)
  if (o) record(o->stage_begin[MOE_STAGE_GATHER], s);
  if (pl.path == PATH_FP8) {
    MOE_TRY(launch_amax_bf16(hidden, (size_t)T * H, amax, s));
    if (pl.gather_in_gemm)
      MOE_TRY(launch_quant_x(hidden, (size_t)T * H, amax, (uint8_t*)xs, s));
    else
      MOE_TRY(launch_gather(hidden, T, H, topk, 2, 1, amax, sorted, nullptr, meta, cap, xs, g1_early, s));
  } else if (!pl.gather_in_gemm) {
    MOE_TRY(launch_gather(hidden, T, H, topk, pl.path == PATH_F32 ? 4 : 2, 0, nullptr, sorted, inv, meta, cap, xs,
                          g1_early, s));
  }
  if (o) record(o->stage_end[MOE_STAGE_GATHER], s);

  if (pl.path == PATH_F32) {
    if (o) record(o->stage_begin[MOE_STAGE_GEMM1], s);
    MOE_TRY(launch_gemm1_simt((const float*)xs, (const float*)w13, H, I, pl.B, eids, meta, cap, (float*)aint, s));
    if (o) record(o->stage_end[MOE_STAGE_GEMM1], s);
    if (o) record(o->stage_begin[MOE_STAGE_ACT], s);
    if (o) record(o->stage_end[MOE_STAGE_ACT], s);
    if (o) record(o->stage_begin[MOE_STAGE_GEMM2], s);
    MOE_TRY(launch_gemm2_simt((const float*)aint, (const float*)w2, H, I, pl.B, T, topk, sorted, eids, meta, cap,
                              (float*)y, s));
    if (o) record(o->stage_end[MOE_STAGE_GEMM2], s);
  } else {
    const bool fp8 = pl.path == PATH_FP8;
    const bool w4 = pl.path == PATH_W4;
    TcGemmArgs g = {};
    g.swap = pl.swap;
    g.fp8 = fp8;
    g.w4 = w4;
    g.T = T;
    g.k = topk;
    g.E = E;
    g.I = I;
    g.H = H;
    g.cap = cap;
    g.sorted = sorted;
    g.eids = eids;
    g.meta = meta;
    g.status = st;
    g.num_sms = sms;
    g.want = gate ? gate->want : nullptr;
    g.pair = pl.pair;
    g.pblk = pblk;

    // 5. GEMM1 on w13 (+ SiLU(gate)*up)
    TcGemmArgs g1 = g;
    g1.K = H;
    g1.W = w13;
    g1.X = (fp8 || !pl.gather_in_gemm) ? (const void*)xs : hidden;
    g1.gather = pl.gather_in_gemm;
    g1.w_rows_per_expert = 2 * I;
    g1.w_pair_off = I;
    g1.wbox = 128;
    g1.w_tile_rows = 128;
    g1.xbox = pl.xbox;
    g1.n_tiles = I / 128;
    g1.splits = pl.s1;
    g1.kb_per_split = pl.kb1;
    g1.w_scale = static_cast<const float*>(w13_scale);
    g1.w4_scale = w4 ? w13_scale : nullptr;
    g1.a_amax = amax;
    g1.amax_out = amax + 1;
    g1.ready = gate ? gate->ready13 : nullptr;
    // the routing-phase L2 prefetch: about 64 MB over the grid
    if (g1_prefetch) {
      const long kb_bytes = 2L * 128 * 128;  // both 128-row boxes of one K block
      g1.prefetch_kb = (int)std::max<long>(1, (64L << 20) / (kb_bytes * std::max(1, sms)));
    }
    g1.early = g1_early;
    // swap-AB GEMM2 may claim its tiles past the first wave from a counter that GEMM1 zeroes
    int* g2_claim = (pl.swap && pl.path != PATH_W4 && !gate) ? reinterpret_cast<int*>(ws + pl.o_misc + 128) : nullptr;
    g1.zero_word = g2_claim;
    void* aint_lo = pl.act_split ? (void*)((uint16_t*)aint + (size_t)cap * I) : nullptr;
    if (pl.s1 > 1) {
      g1.epi = TC_EPI_G1_PART;
      g1.out = p1;
      g1.out_split_stride = pl.p1_stride;
      if (pl.fin) {
        g1.fin = fin;
        g1.out_fin = aint;
        g1.out_fin_lo = aint_lo;
      }
    } else {
      g1.epi = fp8 ? TC_EPI_G1_F32AMAX : TC_EPI_G1_BF16;
      g1.out = fp8 ? (void*)af32 : aint;
      g1.out_lo = aint_lo;
    }
    if (o) record(o->stage_begin[MOE_STAGE_GEMM1], s);
    MOE_TRY(launch_gemm_tc(g1, s));
    if (o) record(o->stage_end[MOE_STAGE_GEMM1], s);

    // split-K reduction / FP8 quantisation of the intermediate
    if (o) record(o->stage_begin[MOE_STAGE_ACT], s);
    if (pl.s1 > 1 && !pl.fin)
      MOE_TRY(launch_reduce_act(p1, pl.s1, pl.p1_stride, I, pl.B, n, sorted, eids, meta, cap,
                                fp8 ? static_cast<const float*>(w13_scale) : nullptr, amax, fp8 ? 1 : 0,
                                fp8 ? (void*)af32 : aint, aint_lo, amax + 1,
                                s));
    if (fp8) MOE_TRY(launch_quant_act(af32, I, meta, cap, amax + 1, (uint8_t*)aint, s));
    if (o) record(o->stage_end[MOE_STAGE_ACT], s);

    // 6. GEMM2 on w2
    TcGemmArgs g2 = g;
    g2.K = I;
    g2.W = w2;
    g2.X = aint;
    g2.x_lo_rows = pl.act_split ? cap : 0;
    g2.w_rows_per_expert = H;
    g2.wbox = pl.swap ? 128 : pl.wbox2;
    g2.w_pair_off = g2.wbox;
    g2.w_tile_rows = 2 * g2.wbox;
    g2.xbox = pl.xbox;
    g2.n_tiles = (H + g2.w_tile_rows - 1) / g2.w_tile_rows;
    g2.splits = pl.s2;
    g2.kb_per_split = pl.kb2;
    g2.w_scale = static_cast<const float*>(w2_scale);
    g2.w4_scale = w4 ? w2_scale : nullptr;
    g2.a_amax = amax + 1;
    g2.out = y;
    g2.out_split_stride = pl.y_stride;
    g2.epi = pl.y_bf16 ? TC_EPI_G2_BF16 : TC_EPI_G2_F32;
    g2.ready = gate ? gate->ready2 : nullptr;
    // GEMM2's predecessor is GEMM1 or a kernel GEMM1 let launch, and GEMM1 lets
    // its dependents launch only after its own dependency wait: the permutation
    // metadata is complete by then, so GEMM2 may stream weights early.
    g2.early = true;
    g2.claim = g2_claim;
    if (o) record(o->stage_begin[MOE_STAGE_GEMM2], s);
    MOE_TRY(launch_gemm_tc(g2, s));
    if (o) record(o->stage_end[MOE_STAGE_GEMM2], s);
  }

  if (!(steps & STEPS_COMBINE)) return MOE_OK;

combine_step:
  // 7. combine
  if (o) record(o->stage_begin[MOE_STAGE_COMBINE], s);
  MOE_TRY(launch_combine(y, pl.y_bf16 ? 1 : 0, pl.s2, pl.y_stride, tw, T, topk, H, out, act_dtype == MOE_BF16 ? 1 : 0,
                         s));
  if (o) record(o->stage_end[MOE_STAGE_COMBINE], s);
#undef MOE_TRY
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported dtype pair or shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait timed out";
    case MOE_ERR_DEVICE_INDEX: return "expert id out of range";
    case MOE_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    default: return "unknown error";
  }
}

int moe_version(void) { return 100; }

int moe_workspace_size(int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                       const moe_options* opts, size_t* bytes) {
  if (!bytes) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(T, H, I, E, topk, act_dtype, w_dtype, opts, &p);
  if (rc) return rc;
  *bytes = p.total;
  return MOE_OK;
}

int moe_plan_info(int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                  const moe_options* opts, moe_plan* info) {
  if (!info) return MOE_ERR_ARG;
  Plan p;
  const int rc = make_plan(T, H, I, E, topk, act_dtype, w_dtype, opts, &p);
  if (rc) return rc;
  info->orientation = p.path == PATH_F32 ? 0 : (p.swap ? MOE_ORIENT_SWAP_AB : MOE_ORIENT_TOKEN_MAJOR);
  info->block = p.B;
  info->splits_gemm1 = p.s1;
  info->splits_gemm2 = p.s2;
  info->act_split = p.act_split ? 1 : 0;
  // router logits, top-k, align, GEMM1, GEMM2, combine (+ the row gather unless
  // GEMM1 gathers; + amax and quantisation kernels on the FP8 path; + the
  // split-K reduction)
  int n = 6;
  if (!p.gather_in_gemm) n += 1;            // row gather (FP8: with input quantisation)
  if (p.path == PATH_FP8) n += p.gather_in_gemm ? 3 : 2;  // input amax (+ input quantisation), intermediate quantisation
  if (p.s1 > 1 && !p.fin) n += 1;
  if (p.fused) n = 1;
  info->kernel_launches = T > 0 ? n : 0;
  info->single_launch = p.fused ? 1 : 0;
  info->workspace_bytes = p.total;
  info->cta_pair = p.pair ? 1 : 0;
  return MOE_OK;
}

int moe_align_capacity(int T, int topk, int E, int block, size_t* sorted_cap, size_t* blocks_cap) {
  if (T < 0 || topk < 1 || E < 1 || block < 1 || !sorted_cap || !blocks_cap) return MOE_ERR_ARG;
  const long long n = (long long)T * topk;
  const long long cap = n + std::min<long long>(E, n) * (block - 1);
  if (cap >= (1ll << 31)) return MOE_ERR_ARG;
  *sorted_cap = (size_t)cap;
  *blocks_cap = (size_t)(cap / block);
  return MOE_OK;
}

int moe_route(const void* hidden, const void* router_w, int T, int H, int E, int topk, int renorm,
              moe_dtype act_dtype, float* logits_out, float* topk_w, int32_t* topk_ids, moe_stream_t stream) {
  if (T < 0 || H < 1 || E < 1 || E > 1024 || topk < 1 || topk > E || topk > 32) return MOE_ERR_ARG;
  if (act_dtype != MOE_F32 && act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (H % (act_dtype == MOE_BF16 ? 8 : 4)) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!hidden || !router_w || !logits_out || !topk_w || !topk_ids) return MOE_ERR_ARG;
  if (misaligned(hidden) || misaligned(router_w) || misaligned(logits_out) || misaligned(topk_w) ||
      misaligned(topk_ids))
    return MOE_ERR_ALIGNMENT;
  int* st = status_word();
  if (!st) return MOE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_router(hidden, router_w, T, H, E, act_dtype, logits_out, st, s);
  if (e == cudaSuccess) e = launch_topk(logits_out, T, E, topk, renorm != 0, topk_w, topk_ids, s);
  return cuda_rc(e);
}

int moe_topk_from_logits(const float* logits, int T, int E, int topk, int renorm, float* topk_w, int32_t* topk_ids,
                         moe_stream_t stream) {
  if (T < 0 || E < 1 || E > 1024 || topk < 1 || topk > E || topk > 32) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!logits || !topk_w || !topk_ids) return MOE_ERR_ARG;
  if (misaligned(logits) || misaligned(topk_w) || misaligned(topk_ids)) return MOE_ERR_ALIGNMENT;
  return cuda_rc(launch_topk(logits, T, E, topk, renorm != 0, topk_w, topk_ids, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_align(const int32_t* topk_ids, int T, int topk, int E, int block, int32_t* sorted_ids, int32_t* expert_ids,
              int32_t* num_post_pad, int32_t* expert_counts, moe_stream_t stream) {
  if (T < 0 || topk < 1 || E < 1 || E > 1024 || block < 1 || block > 1024) return MOE_ERR_ARG;
  size_t cap = 0, bcap = 0;
  if (moe_align_capacity(T, topk, E, block, &cap, &bcap) != MOE_OK) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!topk_ids || !sorted_ids || !expert_ids || !num_post_pad) return MOE_ERR_ARG;
  if (misaligned(topk_ids) || misaligned(sorted_ids) || misaligned(expert_ids) || misaligned(num_post_pad) ||
      (expert_counts && misaligned(expert_counts)))
    return MOE_ERR_ALIGNMENT;
  int* st = status_word();
  if (!st) return MOE_ERR_CUDA;
  return cuda_rc(launch_align(topk_ids, T, topk, E, block, sorted_ids, expert_ids, num_post_pad, expert_counts,
                              nullptr, st, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_forward(const void* hidden, const void* router_w, const void* w13, const void* w2, int T, int H, int I, int E,
                int topk, int renorm, moe_dtype act_dtype, moe_dtype w_dtype, const void* w13_scale,
                const void* w2_scale, void* out, void* workspace, size_t workspace_bytes, const moe_options* opts,
                moe_stream_t stream) {
  Plan pl;
  int rc = make_plan(T, H, I, E, topk, act_dtype, w_dtype, opts, &pl);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  if (!hidden || !router_w || !w13 || !w2 || !out || !workspace) return MOE_ERR_ARG;
  if ((pl.path == PATH_FP8 || pl.path == PATH_W4) && (!w13_scale || !w2_scale)) return MOE_ERR_ARG;
  if (misaligned(hidden) || misaligned(router_w) || misaligned(w13) || misaligned(w2) || misaligned(out) ||
      misaligned(workspace, 256) || (w13_scale && misaligned(w13_scale, 4)) || (w2_scale && misaligned(w2_scale, 4)))
    return MOE_ERR_ALIGNMENT;
  if (workspace_bytes < pl.total) return MOE_ERR_WORKSPACE;
  int* st = status_word();
  const int sms = num_sms();
  if (!st || sms <= 0) return MOE_ERR_CUDA;

  return forward_steps(pl, STEPS_ALL, hidden, router_w, E, nullptr, nullptr, nullptr, w13, w2, T, H, I, E, topk, renorm,
                       act_dtype, w13_scale, w2_scale, out, workspace, opts, st, sms,
                       reinterpret_cast<cudaStream_t>(stream));
}

// Page-locked host memory and the address at which the device reaches it
// (nullptr for anything else: pageable memory, device memory, unknown pointers).
static void* host_mapped(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // (not a sticky error: clear it)
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int moe_forward_host(const void* hidden_host, void* hidden_dev, const void* router_w, const void* w13, const void* w2,
                     int T, int H, int I, int E, int topk, int renorm, moe_dtype act_dtype, moe_dtype w_dtype,
                     const void* w13_scale, const void* w2_scale, void* out_host, void* workspace,
                     size_t workspace_bytes, const moe_options* opts, moe_stream_t stream) {
  Plan pl;
  int rc = make_plan(T, H, I, E, topk, act_dtype, w_dtype, opts, &pl);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  if (!hidden_host || !out_host || !hidden_dev) return MOE_ERR_ARG;
  void* in_mapped = host_mapped(hidden_host);
  void* out_mapped = host_mapped(out_host);
  if (!in_mapped || !out_mapped) return MOE_ERR_ARG;
  if (misaligned(hidden_dev) || misaligned(out_mapped)) return MOE_ERR_ALIGNMENT;
  const size_t bytes = (size_t)T * H * (act_dtype == MOE_F32 ? 4 : 2);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the batch comes in through a copy kernel that reads the host memory directly: a
  // kernel in the library's chain of programmatically dependent launches, where a
  // copy-engine node would end the chain (sizes that are not whole 16-byte vectors
  // take the copy engine)
  const cudaError_t ce = (bytes % 16 == 0 && !misaligned(in_mapped))
                             ? launch_copy_from_host(in_mapped, hidden_dev, bytes, num_sms(), s)
                             : cudaMemcpyAsync(hidden_dev, hidden_host, bytes, cudaMemcpyHostToDevice, s);
  if (ce != cudaSuccess) return MOE_ERR_CUDA;
  // the layer's last kernel stores the output straight into the host buffer
  return moe_forward(hidden_dev, router_w, w13, w2, T, H, I, E, topk, renorm, act_dtype, w_dtype, w13_scale, w2_scale,
                     out_mapped, workspace, workspace_bytes, opts, stream);
}

int moe_forward_routed(const void* hidden, const float* topk_w, const int32_t* topk_ids, const void* w13,
                       const void* w2, int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                       const void* w13_scale, const void* w2_scale, void* out, void* workspace,
                       size_t workspace_bytes, const moe_options* opts, moe_stream_t stream) {
  moe_options o = opts ? *opts : moe_options{};
  o.single_launch = 2;  // the single launch routes inside its kernel
  if (opts && opts->single_launch == 1) return MOE_ERR_UNSUPPORTED;
  if (opts && opts->inject_timeout) return MOE_ERR_ARG;
  Plan pl;
  int rc = make_plan(T, H, I, E, topk, act_dtype, w_dtype, &o, &pl);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  if (!hidden || !topk_w || !topk_ids || !w13 || !w2 || !out || !workspace) return MOE_ERR_ARG;
  if ((pl.path == PATH_FP8 || pl.path == PATH_W4) && (!w13_scale || !w2_scale)) return MOE_ERR_ARG;
  if (misaligned(hidden) || misaligned(topk_w, 4) || misaligned(topk_ids, 4) || misaligned(w13) || misaligned(w2) ||
      misaligned(out) || misaligned(workspace, 256) || (w13_scale && misaligned(w13_scale, 4)) ||
      (w2_scale && misaligned(w2_scale, 4)))
    return MOE_ERR_ALIGNMENT;
  if (workspace_bytes < pl.total) return MOE_ERR_WORKSPACE;
  int* st = status_word();
  const int sms = num_sms();
  if (!st || sms <= 0) return MOE_ERR_CUDA;
  return forward_steps(pl, STEPS_EXPERTS | STEPS_COMBINE, hidden, nullptr, E, nullptr, topk_w, topk_ids, w13, w2, T,
                       H, I, E, topk, 0, act_dtype, w13_scale, w2_scale, out, workspace, opts ? &o : nullptr, st, sms,
                       reinterpret_cast<cudaStream_t>(stream));
}

int moe_inv_rope_fp8_quant(const void* x, int T, int heads, int head_dim, int rot_dim, const int32_t* positions,
                           const float* cos_sin, int max_pos, uint8_t* q_out, float* scale_out, moe_stream_t stream) {
  if (T < 0 || heads < 1 || head_dim < 2 || head_dim % 2 || rot_dim < 0 || rot_dim % 4 || rot_dim > head_dim ||
      rot_dim > 1024 || head_dim - rot_dim > 512 || max_pos < 1)
    return MOE_ERR_ARG;
  if ((long long)T * heads * head_dim >= (1ll << 40)) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !positions || (rot_dim > 0 && !cos_sin) || !q_out || !scale_out) return MOE_ERR_ARG;
  if (misaligned(x, 4) || misaligned(positions, 4) || (cos_sin && misaligned(cos_sin, 16)) || misaligned(q_out, 2) ||
      misaligned(scale_out, 4))
    return MOE_ERR_ALIGNMENT;
  int* st = status_word();
  const int sms = num_sms();
  if (!st) return MOE_ERR_CUDA;
  return cuda_rc(launch_inv_rope_fp8(x, T, heads, head_dim, rot_dim, positions, cos_sin, max_pos, q_out, scale_out,
                                     st, sms, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_get_status(moe_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int* st = status_word();
  if (!st) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, st, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(st, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return v;
}

}  // extern "C"

namespace moe {

int forward_routed_pass(const void* hidden, const float* topk_w, const int32_t* ids, const void* w13, const void* w2,
                        int T, int H, int I, int E, int topk, moe_dtype act_dtype, moe_dtype w_dtype,
                        const void* w13_scale, const void* w2_scale, void* out, void* workspace,
                        size_t workspace_bytes, const moe_options* opts, cudaStream_t stream, bool experts,
                        bool combine, const SlotGate* gate) {
  moe_options o = opts ? *opts : moe_options{};
  o.single_launch = 2;
  if (gate) o.cta_pair = 2;  // readiness waits live in the single-CTA GEMMs (smaller or equal workspace)
  if (o.inject_timeout) return MOE_ERR_ARG;
  Plan pl;
  int rc = make_plan(T, H, I, E, topk, act_dtype, w_dtype, &o, &pl);
  if (rc) return rc;
  if (T == 0 || (!experts && !combine)) return MOE_OK;
  if (!hidden || !topk_w || !ids || !out || !workspace || (experts && (!w13 || !w2))) return MOE_ERR_ARG;
  if (workspace_bytes < pl.total) return MOE_ERR_WORKSPACE;
  int* st = status_word();
  const int sms = num_sms();
  if (!st || sms <= 0) return MOE_ERR_CUDA;
  const int steps = (experts ? STEPS_EXPERTS : 0) | (combine ? STEPS_COMBINE : 0);
  return forward_steps(pl, steps, hidden, nullptr, E, nullptr, topk_w, ids, w13, w2, T, H, I, E, topk, 0, act_dtype,
                       w13_scale, w2_scale, out, workspace, &o, st, sms, stream, gate, true);
}

}  // namespace moe
