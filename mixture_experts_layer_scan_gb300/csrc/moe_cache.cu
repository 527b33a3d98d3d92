// Expert cache: expert weights resident in host memory, a pool of HBM slots
// holding the recently used experts ("FusedMoE vs MegaMoE" (zwxr.cn), section
// 4: MegaMoE keeps the expert weights in host memory, stages the experts a
// batch needs into GPU memory with an LRU policy, and overlaps the copies with
// computation on separate CUDA streams synchronised by events; sections 4.1
// and 4.2).  On a GB300 the host memory is the Grace CPU's, reached over
// NVLink-C2C.
//
// One moe_forward_cached call:
//   1. the router (S1-S2) runs on the GPU into cache-owned buffers;
//   2. the host reads the expert ids back (the call's one host synchronisation);
//   3. the host plans passes and slots (ExpertCacheLru below): experts already
//      in a slot are hits; missing ones take a free slot or evict the least
//      recently used expert the pass does not need.  A call needing more
//      distinct experts than there are slots runs in passes of at most n_slots
//      experts (resident experts first), each pass computing the Y rows of its
//      experts' (token, expert) pairs; one combine follows the last pass;
//   4. missing experts are copied host -> slot on a copy stream, after the
//      kernels that last read the slot: one cudaMemcpyAsync per weight matrix,
//      each followed by a 4-byte copy of the slot's new version number into a
//      readiness word (w13 of every missing expert first, then w2);
//   5. the ids, rewritten as slot ids (-1 for pairs of other passes), go up
//      (read from pinned memory by a copy kernel: a copy-engine upload would
//      queue behind the expert copies) and the expert part of the layer runs
//      over the slot pool.  Its GEMM
//      producers wait (bounded) for a slot's readiness word to reach the
//      version this pass needs before streaming that expert's weights, so the
//      tiles of resident experts start at once while the missing ones copy.
// Copy modes: MOE_CACHE_COPY_OVERLAP (above, the default), MOE_CACHE_COPY_SERIAL
// (the expert kernels wait for all copies through an event) and
// MOE_CACHE_COPY_KERNEL (a copy kernel on the compute stream reads the host
// weights over NVLink-C2C, then the expert kernels run).
// The prediction of future experts from past routing is not built.
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// Slot bookkeeping, host only.  Deterministic.  A call whose distinct experts
// fit in the pool is one pass visiting its experts in order of first
// appearance: a hit refreshes the expert's use time; a miss takes the lowest
// free slot, else evicts the slot with the oldest use time among those the
// pass does not need.  A larger call is split into passes of n_slots experts,
// the experts resident at the start of the call first, then the others, each
// group in order of first appearance.
struct ExpertCacheLru {
  int E = 0, n_slots = 0;
  std::vector<int> slot_expert;   // [n_slots] expert held, -1 empty
  std::vector<int> expert_slot;   // [E] slot of the expert, -1 absent
  std::vector<unsigned long long> last_use;  // [n_slots]
  unsigned long long clock = 0, hits = 0, misses = 0, evictions = 0, passes = 0;

  void init(int e, int s) {
    E = e;
    n_slots = s;
    slot_expert.assign(s, -1);
    expert_slot.assign(e, -1);
    last_use.assign(s, 0);
  }

  // The distinct experts of ids[n] grouped into passes (see above).
  int plan_passes(const int32_t* ids, int n, std::vector<std::vector<int>>* groups) const {
    std::vector<int> needed;
    std::vector<char> seen(E, 0);
    for (int i = 0; i < n; ++i) {
      const int e = ids[i];
      if (e < 0 || e >= E) return MOE_ERR_DEVICE_INDEX;
      if (!seen[e]) {
        seen[e] = 1;
        needed.push_back(e);
      }
    }
    groups->clear();
    if ((int)needed.size() <= n_slots) {
      groups->push_back(needed);
      return MOE_OK;
    }
    std::vector<int> order;
    for (const int e : needed)
      if (expert_slot[e] >= 0) order.push_back(e);
    for (const int e : needed)
      if (expert_slot[e] < 0) order.push_back(e);
    for (size_t i = 0; i < order.size(); i += n_slots)
      groups->push_back(std::vector<int>(order.begin() + i, order.begin() + std::min(order.size(), i + n_slots)));
    return MOE_OK;
  }

  // Slots for the experts of one pass (|set| <= n_slots); loads receives the
  // (expert, slot) pairs to copy.
  void assign_pass(const std::vector<int>& set, std::vector<std::pair<int, int>>* loads) {
    std::vector<char> in_pass(E, 0);
    for (const int e : set) in_pass[e] = 1;
    loads->clear();
    ++passes;
    for (const int e : set) {
      int s = expert_slot[e];
      if (s >= 0) {
        ++hits;
      } else {
        ++misses;
        for (int c = 0; c < n_slots && s < 0; ++c)
          if (slot_expert[c] < 0) s = c;
        if (s < 0) {
          unsigned long long best = ~0ull;
          for (int c = 0; c < n_slots; ++c) {
            if (in_pass[slot_expert[c]]) continue;
            if (last_use[c] < best) {
              best = last_use[c];
              s = c;
            }
          }
          expert_slot[slot_expert[s]] = -1;
          ++evictions;
        }
        slot_expert[s] = e;
        expert_slot[e] = s;
        loads->push_back({e, s});
      }
      last_use[s] = ++clock;
    }
  }
};

// Copies n16 16-byte units from src (host memory the device can address, read
// over NVLink-C2C) to dst (device memory); several loads in flight per thread.
__global__ void __launch_bounds__(256) k_copy_from_host(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                        size_t n16) {
  pdl_enter();
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_copy_from_host(const void* src, void* dst, size_t bytes, int sms, cudaStream_t s) {
  if (bytes % 16 || (reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) % 16)
    return cudaErrorInvalidValue;
  if (bytes == 0) return cudaSuccess;
  const size_t n16 = bytes / 16;
  const int grid = (int)std::min<size_t>((size_t)std::max(sms, 1) * 8, (n16 + 255) / 256);
  return launch_pdl(k_copy_from_host, dim3(grid), dim3(256), 0, s, static_cast<const uint4*>(src),
                    static_cast<uint4*>(dst), n16);
}

}  // namespace moe

using namespace moe;

struct moe_expert_cache {
  int device = 0;
  int E = 0, H = 0, I = 0, topk = 0, n_slots = 0, max_tokens = 0, max_passes = 1, sms = 0;
  moe_dtype w_dtype = MOE_BF16;
  int copy_mode = MOE_CACHE_COPY_OVERLAP;
  size_t w13_bytes = 0, w2_bytes = 0;  // per expert
  const uint8_t* host_w13 = nullptr;
  const uint8_t* host_w2 = nullptr;
  const float* host_s13 = nullptr;
  const float* host_s2 = nullptr;
  const uint8_t* dev_host_w13 = nullptr;  // device addresses of the host weights (copy kernel), or null
  const uint8_t* dev_host_w2 = nullptr;
  bool registered_w13 = false, registered_w2 = false;
  // device
  uint8_t* pool_w13 = nullptr;
  uint8_t* pool_w2 = nullptr;
  float* pool_s13 = nullptr;
  float* pool_s2 = nullptr;
  float* logits = nullptr;   // [max_tokens][E]
  float* topk_w = nullptr;   // [max_tokens][topk]
  int32_t* ids = nullptr;    // [max_tokens][topk] expert ids
  int32_t* slots = nullptr;  // [max_passes][max_tokens][topk] slot ids per pass (-1: another pass)
  unsigned* ready = nullptr; // [2][n_slots] readiness words of w13 / w2 (version of the slot's contents)
  unsigned* want = nullptr;  // [max_passes][n_slots] versions each pass needs
  // pinned host staging
  int32_t* h_ids = nullptr;
  int32_t* h_slots = nullptr;  // [max_passes][pairs16]
  unsigned* h_want = nullptr;  // [max_passes][slots16]
  const uint8_t* dev_h_slots = nullptr;  // device addresses of the two staging buffers above
  const uint8_t* dev_h_want = nullptr;
  size_t pairs16 = 0, slots16 = 0;       // per-pass strides, rounded up to 16 bytes
  unsigned* h_words = nullptr; // [2][max_passes][n_slots] version words copied after each weight copy
  float* h_s13 = nullptr;      // [n_slots] scale of the expert in each slot (FP8)
  float* h_s2 = nullptr;
  std::vector<unsigned> version;  // [n_slots] host copy of each slot's version
  cudaStream_t copy = nullptr;
  cudaEvent_t copied = nullptr, done = nullptr, ids_in = nullptr, slots_up = nullptr;
  std::vector<cudaEvent_t> pass_done;  // [max_passes]
  bool any_call = false;
  ExpertCacheLru lru;
  std::vector<std::pair<int, int>> loads;
  std::vector<std::vector<int>> groups;
  unsigned long long calls = 0, bytes_h2d = 0;
  std::mutex mu;
};

namespace {

bool is_pinned(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

void release(moe_expert_cache* c) {
  if (!c) return;
  cudaSetDevice(c->device);
  if (c->copy) cudaStreamSynchronize(c->copy);
  cudaFree(c->pool_w13);
  cudaFree(c->pool_w2);
  cudaFree(c->pool_s13);
  cudaFree(c->pool_s2);
  cudaFree(c->logits);
  cudaFree(c->topk_w);
  cudaFree(c->ids);
  cudaFree(c->slots);
  cudaFree(c->ready);
  cudaFree(c->want);
  cudaFreeHost(c->h_ids);
  cudaFreeHost(c->h_slots);
  cudaFreeHost(c->h_want);
  cudaFreeHost(c->h_words);
  cudaFreeHost(c->h_s13);
  cudaFreeHost(c->h_s2);
  if (c->copied) cudaEventDestroy(c->copied);
  if (c->done) cudaEventDestroy(c->done);
  if (c->ids_in) cudaEventDestroy(c->ids_in);
  if (c->slots_up) cudaEventDestroy(c->slots_up);
  for (cudaEvent_t ev : c->pass_done)
    if (ev) cudaEventDestroy(ev);
  if (c->copy) cudaStreamDestroy(c->copy);
  if (c->registered_w13) cudaHostUnregister(const_cast<uint8_t*>(c->host_w13));
  if (c->registered_w2) cudaHostUnregister(const_cast<uint8_t*>(c->host_w2));
  delete c;
}

const uint8_t* device_view(const void* host) {
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host), 0) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<const uint8_t*>(d);
}

}  // namespace

extern "C" {

int moe_cache_create(const void* host_w13, const void* host_w2, const float* host_w13_scale,
                     const float* host_w2_scale, int E, int H, int I, moe_dtype w_dtype, int n_slots, int max_tokens,
                     int topk, moe_expert_cache** cache) {
  if (!cache) return MOE_ERR_ARG;
  *cache = nullptr;
  if (!host_w13 || !host_w2 || E < 1 || E > 1024 || H < 1 || I < 1 || n_slots < topk || n_slots > E ||
      max_tokens < 1 || topk < 1 || topk > E || topk > 32)
    return MOE_ERR_ARG;
  if (w_dtype != MOE_BF16 && w_dtype != MOE_E4M3) return MOE_ERR_UNSUPPORTED;
  if (w_dtype == MOE_E4M3 && (!host_w13_scale || !host_w2_scale)) return MOE_ERR_ARG;
  if (H % 128 || I % 128) return MOE_ERR_UNSUPPORTED;
  moe_expert_cache* c = new (std::nothrow) moe_expert_cache();
  if (!c) return MOE_ERR_CUDA;
  cudaGetDevice(&c->device);
  cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->device);
  c->E = E;
  c->H = H;
  c->I = I;
  c->topk = topk;
  c->n_slots = n_slots;
  c->max_tokens = max_tokens;
  c->w_dtype = w_dtype;
  const long distinct_max = std::min<long>(E, (long)max_tokens * topk);
  c->max_passes = (int)((distinct_max + n_slots - 1) / n_slots);
  const size_t eb = w_dtype == MOE_E4M3 ? 1 : 2;
  c->w13_bytes = (size_t)2 * I * H * eb;
  c->w2_bytes = (size_t)H * I * eb;
  c->host_w13 = static_cast<const uint8_t*>(host_w13);
  c->host_w2 = static_cast<const uint8_t*>(host_w2);
  c->host_s13 = host_w13_scale;
  c->host_s2 = host_w2_scale;
  // asynchronous host -> device copies need page-locked memory
  bool ok = true;
  if (!is_pinned(host_w13)) {
    ok = cudaHostRegister(const_cast<void*>(host_w13), c->w13_bytes * E, cudaHostRegisterDefault) == cudaSuccess;
    c->registered_w13 = ok;
  }
  if (ok && !is_pinned(host_w2)) {
    ok = cudaHostRegister(const_cast<void*>(host_w2), c->w2_bytes * E, cudaHostRegisterDefault) == cudaSuccess;
    c->registered_w2 = ok;
  }
  if (ok) {
    c->dev_host_w13 = device_view(host_w13);
    c->dev_host_w2 = device_view(host_w2);
  }
  const size_t pairs = (size_t)max_tokens * topk;
  const size_t P = (size_t)c->max_passes;
  c->pairs16 = (pairs + 3) / 4 * 4;
  c->slots16 = ((size_t)n_slots + 3) / 4 * 4;
  c->pass_done.assign(P, nullptr);
  ok = ok && cudaMalloc(&c->pool_w13, c->w13_bytes * n_slots) == cudaSuccess &&
       cudaMalloc(&c->pool_w2, c->w2_bytes * n_slots) == cudaSuccess &&
       cudaMalloc(&c->pool_s13, sizeof(float) * n_slots) == cudaSuccess &&
       cudaMalloc(&c->pool_s2, sizeof(float) * n_slots) == cudaSuccess &&
       cudaMalloc(&c->logits, sizeof(float) * (size_t)max_tokens * E) == cudaSuccess &&
       cudaMalloc(&c->topk_w, sizeof(float) * pairs) == cudaSuccess &&
       cudaMalloc(&c->ids, sizeof(int32_t) * pairs) == cudaSuccess &&
       cudaMalloc(&c->slots, sizeof(int32_t) * c->pairs16 * P) == cudaSuccess &&
       cudaMalloc(&c->ready, sizeof(unsigned) * 2 * n_slots) == cudaSuccess &&
       cudaMalloc(&c->want, sizeof(unsigned) * c->slots16 * P) == cudaSuccess &&
       cudaMemset(c->ready, 0, sizeof(unsigned) * 2 * n_slots) == cudaSuccess &&
       cudaMallocHost(&c->h_ids, sizeof(int32_t) * pairs) == cudaSuccess &&
       cudaMallocHost(&c->h_slots, sizeof(int32_t) * c->pairs16 * P) == cudaSuccess &&
       cudaMallocHost(&c->h_want, sizeof(unsigned) * c->slots16 * P) == cudaSuccess &&
       cudaMallocHost(&c->h_words, sizeof(unsigned) * 2 * n_slots * P) == cudaSuccess &&
       cudaMallocHost(&c->h_s13, sizeof(float) * n_slots) == cudaSuccess &&
       cudaMallocHost(&c->h_s2, sizeof(float) * n_slots) == cudaSuccess &&
       cudaStreamCreateWithFlags(&c->copy, cudaStreamNonBlocking) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->copied, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->ids_in, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->slots_up, cudaEventDisableTiming) == cudaSuccess;
  for (size_t i = 0; ok && i < P; ++i)
    ok = cudaEventCreateWithFlags(&c->pass_done[i], cudaEventDisableTiming) == cudaSuccess;
  // the per-pass slot ids and versions go up by the copy kernel (reading the pinned staging
  // buffers directly): copy-engine uploads would queue behind the expert copies
  if (ok) {
    c->dev_h_slots = device_view(c->h_slots);
    c->dev_h_want = device_view(c->h_want);
    ok = c->dev_h_slots && c->dev_h_want;
  }
  if (!ok) {
    cudaGetLastError();
    release(c);
    return MOE_ERR_CUDA;
  }
  for (int sl = 0; sl < n_slots; ++sl) c->h_s13[sl] = c->h_s2[sl] = 1.0f;
  c->version.assign(n_slots, 0u);
  c->lru.init(E, n_slots);
  *cache = c;
  return MOE_OK;
}

int moe_cache_destroy(moe_expert_cache* cache) {
  if (!cache) return MOE_ERR_ARG;
  release(cache);
  return MOE_OK;
}

int moe_cache_set_copy_mode(moe_expert_cache* cache, int mode) {
  if (!cache || mode < MOE_CACHE_COPY_OVERLAP || mode > MOE_CACHE_COPY_KERNEL) return MOE_ERR_ARG;
  if (mode == MOE_CACHE_COPY_KERNEL && (!cache->dev_host_w13 || !cache->dev_host_w2)) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(cache->mu);
  cache->copy_mode = mode;
  return MOE_OK;
}

int moe_cache_workspace_size(const moe_expert_cache* cache, int T, moe_dtype act_dtype, const moe_options* opts,
                             size_t* bytes) {
  if (!cache || !bytes) return MOE_ERR_ARG;
  if (T > cache->max_tokens) return MOE_ERR_ARG;
  moe_options o = opts ? *opts : moe_options{};
  o.single_launch = 2;
  return moe_workspace_size(T, cache->H, cache->I, cache->n_slots, cache->topk, act_dtype, cache->w_dtype, &o, bytes);
}

int moe_cache_stats(const moe_expert_cache* cache, moe_cache_stats_t* stats) {
  if (!cache || !stats) return MOE_ERR_ARG;
  stats->calls = cache->calls;
  stats->hits = cache->lru.hits;
  stats->misses = cache->lru.misses;
  stats->evictions = cache->lru.evictions;
  stats->bytes_h2d = cache->bytes_h2d;
  stats->passes = cache->lru.passes;
  return MOE_OK;
}

int moe_forward_cached(moe_expert_cache* c, const void* hidden, const void* router_w, int T, int renorm,
                       moe_dtype act_dtype, void* out, void* workspace, size_t workspace_bytes,
                       const moe_options* opts, moe_stream_t stream) {
  if (!c) return MOE_ERR_ARG;
  if (T < 0 || T > c->max_tokens) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (opts && (opts->single_launch == 1 || opts->inject_timeout)) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(c->mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != c->device) return MOE_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int n = T * c->topk;
  const size_t pairs = c->pairs16;
  // 1. routing
  int rc = moe_route(hidden, router_w, T, c->H, c->E, c->topk, renorm, act_dtype, c->logits, c->topk_w, c->ids, stream);
  if (rc) return rc;
  // 2. expert ids to the host (the previous call's uploads and copies read the pinned
  // staging buffers: they are done first)
  if (c->any_call && (cudaEventSynchronize(c->slots_up) != cudaSuccess || cudaEventSynchronize(c->copied) != cudaSuccess))
    return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(c->h_ids, c->ids, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaEventRecord(c->ids_in, s) != cudaSuccess || cudaEventSynchronize(c->ids_in) != cudaSuccess)
    return MOE_ERR_CUDA;
  // 3. passes: FP8 needs one pass (its intermediate scale spans every pair of the call)
  rc = c->lru.plan_passes(c->h_ids, n, &c->groups);
  if (rc) return rc;
  if (c->groups.size() > 1 && c->w_dtype == MOE_E4M3) return MOE_ERR_UNSUPPORTED;
  if ((int)c->groups.size() > c->max_passes) return MOE_ERR_ARG;
  moe_options o = opts ? *opts : moe_options{};
  o.single_launch = 2;
  const bool overlap = c->copy_mode == MOE_CACHE_COPY_OVERLAP;
  const size_t eb_scale = sizeof(float) * c->n_slots;
  std::vector<int> expert_pass(c->E, -1);
  for (size_t p = 0; p < c->groups.size(); ++p)
    for (const int e : c->groups[p]) expert_pass[e] = (int)p;
  for (size_t p = 0; p < c->groups.size(); ++p) {
    c->lru.assign_pass(c->groups[p], &c->loads);
    // 4. copies of the missing experts, once the kernels that last read their slots are done
    cudaEvent_t after = p == 0 ? (c->any_call ? c->done : nullptr) : c->pass_done[p - 1];
    if (after && !c->loads.empty() && c->copy_mode != MOE_CACHE_COPY_KERNEL &&
        cudaStreamWaitEvent(c->copy, after, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    for (const auto& ld : c->loads) {
      const int sl = ld.second;
      ++c->version[sl];
      if (c->w_dtype == MOE_E4M3) {
        c->h_s13[sl] = c->host_s13[ld.first];
        c->h_s2[sl] = c->host_s2[ld.first];
      }
    }
    unsigned* words = c->h_words + (size_t)2 * c->n_slots * p;
    if (c->copy_mode == MOE_CACHE_COPY_KERNEL) {
      // copy kernels on the compute stream: ordered after this stream's earlier reads of the slots
      if (c->w_dtype == MOE_E4M3 && !c->loads.empty() &&
          (cudaMemcpyAsync(c->pool_s13, c->h_s13, eb_scale, cudaMemcpyHostToDevice, s) != cudaSuccess ||
           cudaMemcpyAsync(c->pool_s2, c->h_s2, eb_scale, cudaMemcpyHostToDevice, s) != cudaSuccess))
        return MOE_ERR_CUDA;
      for (const auto& ld : c->loads) {
        const int e = ld.first, sl = ld.second;
        if (launch_copy_from_host(c->dev_host_w13 + c->w13_bytes * e, c->pool_w13 + c->w13_bytes * sl, c->w13_bytes,
                                  c->sms, s) != cudaSuccess ||
            launch_copy_from_host(c->dev_host_w2 + c->w2_bytes * e, c->pool_w2 + c->w2_bytes * sl, c->w2_bytes,
                                  c->sms, s) != cudaSuccess)
          return MOE_ERR_CUDA;
      }
    } else if (!c->loads.empty()) {
      if (c->w_dtype == MOE_E4M3 &&
          (cudaMemcpyAsync(c->pool_s13, c->h_s13, eb_scale, cudaMemcpyHostToDevice, c->copy) != cudaSuccess ||
           cudaMemcpyAsync(c->pool_s2, c->h_s2, eb_scale, cudaMemcpyHostToDevice, c->copy) != cudaSuccess))
        return MOE_ERR_CUDA;
      // w13 of every missing expert, each announced by its version word, then w2 likewise:
      // GEMM1 of an expert can start as soon as its w13 has landed
      for (int part = 0; part < 2; ++part) {
        for (size_t i = 0; i < c->loads.size(); ++i) {
          const int e = c->loads[i].first, sl = c->loads[i].second;
          const size_t bytes = part == 0 ? c->w13_bytes : c->w2_bytes;
          uint8_t* dst = (part == 0 ? c->pool_w13 : c->pool_w2) + bytes * sl;
          const uint8_t* src = (part == 0 ? c->host_w13 : c->host_w2) + bytes * e;
          unsigned* word = words + part * c->n_slots + sl;
          *word = c->version[sl];
          if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, c->copy) != cudaSuccess ||
              cudaMemcpyAsync(c->ready + part * c->n_slots + sl, word, sizeof(unsigned), cudaMemcpyHostToDevice,
                              c->copy) != cudaSuccess)
            return MOE_ERR_CUDA;
        }
      }
      if (cudaEventRecord(c->copied, c->copy) != cudaSuccess) return MOE_ERR_CUDA;
      if (!overlap && cudaStreamWaitEvent(s, c->copied, 0) != cudaSuccess) return MOE_ERR_CUDA;
    }
    for (const auto& ld : c->loads) c->bytes_h2d += c->w13_bytes + c->w2_bytes;
    // 5. this pass's slot ids and wanted versions up, then its expert steps
    int32_t* hs = c->h_slots + pairs * p;
    for (int i = 0; i < n; ++i) hs[i] = expert_pass[c->h_ids[i]] == (int)p ? c->lru.expert_slot[c->h_ids[i]] : -1;
    unsigned* hw = c->h_want + c->slots16 * p;
    for (int sl = 0; sl < c->n_slots; ++sl) hw[sl] = c->version[sl];
    int32_t* ds = c->slots + pairs * p;
    unsigned* dw = c->want + c->slots16 * p;
    if (launch_copy_from_host(c->dev_h_slots + sizeof(int32_t) * pairs * p, ds,
                              sizeof(int32_t) * ((size_t)(n + 3) / 4 * 4), c->sms, s) != cudaSuccess ||
        launch_copy_from_host(c->dev_h_want + sizeof(unsigned) * c->slots16 * p, dw, sizeof(unsigned) * c->slots16,
                              c->sms, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    const SlotGate gate = {c->ready, c->ready + c->n_slots, dw};
    const bool last = p + 1 == c->groups.size();
    rc = forward_routed_pass(hidden, c->topk_w, ds, c->pool_w13, c->pool_w2, T, c->H, c->I, c->n_slots, c->topk,
                             act_dtype, c->w_dtype, c->w_dtype == MOE_E4M3 ? c->pool_s13 : nullptr,
                             c->w_dtype == MOE_E4M3 ? c->pool_s2 : nullptr, out, workspace, workspace_bytes, &o, s,
                             true, last, overlap ? &gate : nullptr);
    if (rc) return rc;
    if (cudaEventRecord(c->pass_done[p], s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (cudaEventRecord(c->slots_up, s) != cudaSuccess || cudaEventRecord(c->done, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  c->any_call = true;
  ++c->calls;
  return MOE_OK;
}

int moe_copy_from_host(const void* src_host, void* dst, size_t bytes, moe_stream_t stream) {
  if (!src_host || !dst) return MOE_ERR_ARG;
  if (bytes % 16 || (reinterpret_cast<uintptr_t>(src_host) | reinterpret_cast<uintptr_t>(dst)) % 16)
    return MOE_ERR_ALIGNMENT;
  const uint8_t* src = device_view(src_host);
  if (!src) return MOE_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess)
    return MOE_ERR_CUDA;
  return launch_copy_from_host(src, dst, bytes, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

int moe_cache_lru_plan(int E, int n_slots, int n_calls, int pairs, const int32_t* ids, int32_t* slot_ids,
                       int32_t* loaded_expert, unsigned long long* hits, unsigned long long* misses) {
  if (E < 1 || n_slots < 1 || n_slots > E || n_calls < 0 || pairs < 1 || !ids || !slot_ids || !loaded_expert)
    return MOE_ERR_ARG;
  ExpertCacheLru lru;
  lru.init(E, n_slots);
  std::vector<std::pair<int, int>> loads;
  std::vector<std::vector<int>> groups;
  for (int call = 0; call < n_calls; ++call) {
    const int32_t* cid = ids + (size_t)call * pairs;
    const int rc = lru.plan_passes(cid, pairs, &groups);
    if (rc) return rc;
    int32_t* le = loaded_expert + (size_t)call * n_slots;
    for (int sl = 0; sl < n_slots; ++sl) le[sl] = -1;
    int32_t* so = slot_ids + (size_t)call * pairs;
    for (const auto& g : groups) {
      lru.assign_pass(g, &loads);
      for (const auto& ld : loads) le[ld.second] = ld.first;
      for (int i = 0; i < pairs; ++i)
        if (std::find(g.begin(), g.end(), cid[i]) != g.end()) so[i] = lru.expert_slot[cid[i]];
    }
  }
  if (hits) *hits = lru.hits;
  if (misses) *misses = lru.misses;
  return MOE_OK;
}

}  // extern "C"
