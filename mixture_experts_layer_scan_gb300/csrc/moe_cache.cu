// Expert cache: expert weights resident in host memory, a pool of HBM slots
// holding the recently used experts ("FusedMoE vs MegaMoE" (zwxr.cn), section
// 4: MegaMoE keeps the expert weights in host memory and stages the experts a
// batch needs into GPU memory, loading synchronously when an expert is
// missing).  On a GB300 the host memory is the Grace CPU's, reached over
// NVLink-C2C.
//
// One moe_forward_cached call:
//   1. the router (S1-S2) runs on the GPU into cache-owned buffers;
//   2. the host reads the expert ids back (the call's one host synchronisation);
//   3. the host plans the slots (ExpertCacheLru below): experts already in a
//      slot are hits; missing ones take a free slot or evict the least recently
//      used expert that this call does not need;
//   4. missing experts are copied host -> slot on a copy stream (one
//      cudaMemcpyAsync per weight matrix), after the previous call's kernels
//      are done with the slots they overwrite;
//   5. the ids are rewritten as slot ids and the expert part of the layer
//      (moe_forward_routed over the slot pool) runs once the copies land.
// The prediction of future experts from past routing is not built.
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "moe_internal.h"

namespace moe {

// Slot bookkeeping, host only.  Deterministic: the experts of a call are
// visited in order of first appearance in the id list; a hit refreshes the
// expert's use time; a miss takes the lowest free slot, else evicts the slot
// with the oldest use time among those this call does not need.
struct ExpertCacheLru {
  int E = 0, n_slots = 0;
  std::vector<int> slot_expert;   // [n_slots] expert held, -1 empty
  std::vector<int> expert_slot;   // [E] slot of the expert, -1 absent
  std::vector<unsigned long long> last_use;  // [n_slots]
  unsigned long long clock = 0, hits = 0, misses = 0, evictions = 0;

  void init(int e, int s) {
    E = e;
    n_slots = s;
    slot_expert.assign(s, -1);
    expert_slot.assign(e, -1);
    last_use.assign(s, 0);
  }

  // ids[n] -> slot_ids[n]; loads receives the (expert, slot) pairs to copy.
  int assign(const int32_t* ids, int n, int32_t* slot_ids, std::vector<std::pair<int, int>>* loads) {
    std::vector<int> needed;
    std::vector<char> in_call(E, 0);
    for (int i = 0; i < n; ++i) {
      const int e = ids[i];
      if (e < 0 || e >= E) return MOE_ERR_DEVICE_INDEX;
      if (!in_call[e]) {
        in_call[e] = 1;
        needed.push_back(e);
      }
    }
    if ((int)needed.size() > n_slots) return MOE_ERR_UNSUPPORTED;
    loads->clear();
    for (const int e : needed) {
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
            if (in_call[slot_expert[c]]) continue;
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
    for (int i = 0; i < n; ++i) slot_ids[i] = expert_slot[ids[i]];
    return MOE_OK;
  }
};

}  // namespace moe

using namespace moe;

struct moe_expert_cache {
  int device = 0;
  int E = 0, H = 0, I = 0, topk = 0, n_slots = 0, max_tokens = 0;
  moe_dtype w_dtype = MOE_BF16;
  size_t w13_bytes = 0, w2_bytes = 0;  // per expert
  const uint8_t* host_w13 = nullptr;
  const uint8_t* host_w2 = nullptr;
  const float* host_s13 = nullptr;
  const float* host_s2 = nullptr;
  bool registered_w13 = false, registered_w2 = false;
  // device
  uint8_t* pool_w13 = nullptr;
  uint8_t* pool_w2 = nullptr;
  float* pool_s13 = nullptr;
  float* pool_s2 = nullptr;
  float* logits = nullptr;  // [max_tokens][E]
  float* topk_w = nullptr;  // [max_tokens][topk]
  int32_t* ids = nullptr;   // [max_tokens][topk] expert ids
  int32_t* slots = nullptr; // [max_tokens][topk] slot ids
  // pinned host staging
  int32_t* h_ids = nullptr;
  int32_t* h_slots = nullptr;
  float* h_s13 = nullptr;  // [n_slots] scale of the expert in each slot (FP8)
  float* h_s2 = nullptr;
  cudaStream_t copy = nullptr;
  cudaEvent_t copied = nullptr, done = nullptr, ids_in = nullptr, slots_up = nullptr;
  bool any_call = false;
  ExpertCacheLru lru;
  std::vector<std::pair<int, int>> loads;
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
  cudaFreeHost(c->h_ids);
  cudaFreeHost(c->h_slots);
  cudaFreeHost(c->h_s13);
  cudaFreeHost(c->h_s2);
  if (c->copied) cudaEventDestroy(c->copied);
  if (c->done) cudaEventDestroy(c->done);
  if (c->ids_in) cudaEventDestroy(c->ids_in);
  if (c->slots_up) cudaEventDestroy(c->slots_up);
  if (c->copy) cudaStreamDestroy(c->copy);
  if (c->registered_w13) cudaHostUnregister(const_cast<uint8_t*>(c->host_w13));
  if (c->registered_w2) cudaHostUnregister(const_cast<uint8_t*>(c->host_w2));
  delete c;
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
  c->E = E;
  c->H = H;
  c->I = I;
  c->topk = topk;
  c->n_slots = n_slots;
  c->max_tokens = max_tokens;
  c->w_dtype = w_dtype;
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
  const size_t pairs = (size_t)max_tokens * topk;
  ok = ok && cudaMalloc(&c->pool_w13, c->w13_bytes * n_slots) == cudaSuccess &&
       cudaMalloc(&c->pool_w2, c->w2_bytes * n_slots) == cudaSuccess &&
       cudaMalloc(&c->pool_s13, sizeof(float) * n_slots) == cudaSuccess &&
       cudaMalloc(&c->pool_s2, sizeof(float) * n_slots) == cudaSuccess &&
       cudaMalloc(&c->logits, sizeof(float) * (size_t)max_tokens * E) == cudaSuccess &&
       cudaMalloc(&c->topk_w, sizeof(float) * pairs) == cudaSuccess &&
       cudaMalloc(&c->ids, sizeof(int32_t) * pairs) == cudaSuccess &&
       cudaMalloc(&c->slots, sizeof(int32_t) * pairs) == cudaSuccess &&
       cudaMallocHost(&c->h_ids, sizeof(int32_t) * pairs) == cudaSuccess &&
       cudaMallocHost(&c->h_slots, sizeof(int32_t) * pairs) == cudaSuccess &&
       cudaMallocHost(&c->h_s13, sizeof(float) * n_slots) == cudaSuccess &&
       cudaMallocHost(&c->h_s2, sizeof(float) * n_slots) == cudaSuccess &&
       cudaStreamCreateWithFlags(&c->copy, cudaStreamNonBlocking) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->copied, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->done, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->ids_in, cudaEventDisableTiming) == cudaSuccess &&
       cudaEventCreateWithFlags(&c->slots_up, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    release(c);
    return MOE_ERR_CUDA;
  }
  for (int sl = 0; sl < n_slots; ++sl) c->h_s13[sl] = c->h_s2[sl] = 1.0f;
  c->lru.init(E, n_slots);
  *cache = c;
  return MOE_OK;
}

int moe_cache_destroy(moe_expert_cache* cache) {
  if (!cache) return MOE_ERR_ARG;
  release(cache);
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
  // 1. routing
  int rc = moe_route(hidden, router_w, T, c->H, c->E, c->topk, renorm, act_dtype, c->logits, c->topk_w, c->ids, stream);
  if (rc) return rc;
  // 2. expert ids to the host (the previous call's slot-id upload read h_slots: it is done first)
  if (c->any_call && cudaEventSynchronize(c->slots_up) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyAsync(c->h_ids, c->ids, sizeof(int32_t) * n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaEventRecord(c->ids_in, s) != cudaSuccess || cudaEventSynchronize(c->ids_in) != cudaSuccess)
    return MOE_ERR_CUDA;
  // 3. slot plan
  rc = c->lru.assign(c->h_ids, n, c->h_slots, &c->loads);
  if (rc) return rc;
  // 4. copies of the missing experts, once the previous call no longer reads their slots
  if (c->any_call && cudaStreamWaitEvent(c->copy, c->done, 0) != cudaSuccess) return MOE_ERR_CUDA;
  for (const auto& ld : c->loads) {
    const int e = ld.first, sl = ld.second;
    if (cudaMemcpyAsync(c->pool_w13 + c->w13_bytes * sl, c->host_w13 + c->w13_bytes * e, c->w13_bytes,
                        cudaMemcpyHostToDevice, c->copy) != cudaSuccess ||
        cudaMemcpyAsync(c->pool_w2 + c->w2_bytes * sl, c->host_w2 + c->w2_bytes * e, c->w2_bytes,
                        cudaMemcpyHostToDevice, c->copy) != cudaSuccess)
      return MOE_ERR_CUDA;
    c->bytes_h2d += c->w13_bytes + c->w2_bytes;
    if (c->w_dtype == MOE_E4M3) {
      c->h_s13[sl] = c->host_s13[e];
      c->h_s2[sl] = c->host_s2[e];
    }
  }
  if (c->w_dtype == MOE_E4M3 && !c->loads.empty()) {
    if (cudaMemcpyAsync(c->pool_s13, c->h_s13, sizeof(float) * c->n_slots, cudaMemcpyHostToDevice, c->copy) !=
            cudaSuccess ||
        cudaMemcpyAsync(c->pool_s2, c->h_s2, sizeof(float) * c->n_slots, cudaMemcpyHostToDevice, c->copy) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
  }
  if (cudaEventRecord(c->copied, c->copy) != cudaSuccess || cudaStreamWaitEvent(s, c->copied, 0) != cudaSuccess)
    return MOE_ERR_CUDA;
  // 5. slot ids up, then the expert steps over the slot pool
  if (cudaMemcpyAsync(c->slots, c->h_slots, sizeof(int32_t) * n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaEventRecord(c->slots_up, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_options o = opts ? *opts : moe_options{};
  o.single_launch = 2;
  rc = moe_forward_routed(hidden, c->topk_w, c->slots, c->pool_w13, c->pool_w2, T, c->H, c->I, c->n_slots, c->topk,
                          act_dtype, c->w_dtype, c->w_dtype == MOE_E4M3 ? c->pool_s13 : nullptr,
                          c->w_dtype == MOE_E4M3 ? c->pool_s2 : nullptr, out, workspace, workspace_bytes, &o, stream);
  if (rc) return rc;
  if (cudaEventRecord(c->done, s) != cudaSuccess) return MOE_ERR_CUDA;
  c->any_call = true;
  ++c->calls;
  return MOE_OK;
}

int moe_cache_lru_plan(int E, int n_slots, int n_calls, int pairs, const int32_t* ids, int32_t* slot_ids,
                       int32_t* loaded_expert, unsigned long long* hits, unsigned long long* misses) {
  if (E < 1 || n_slots < 1 || n_slots > E || n_calls < 0 || pairs < 1 || !ids || !slot_ids || !loaded_expert)
    return MOE_ERR_ARG;
  ExpertCacheLru lru;
  lru.init(E, n_slots);
  std::vector<std::pair<int, int>> loads;
  for (int call = 0; call < n_calls; ++call) {
    const int rc = lru.assign(ids + (size_t)call * pairs, pairs, slot_ids + (size_t)call * pairs, &loads);
    if (rc) return rc;
    int32_t* le = loaded_expert + (size_t)call * n_slots;
    for (int sl = 0; sl < n_slots; ++sl) le[sl] = -1;
    for (const auto& ld : loads) le[ld.second] = ld.first;
  }
  if (hits) *hits = lru.hits;
  if (misses) *misses = lru.misses;
  return MOE_OK;
}

}  // extern "C"
