// slot_cache.cu -- residency of expert weights in a bounded set of device
// slots: the host-side logic of the expert tier (moe_tier_* in api.cu).
//
// "Distributed MoE" (tenzro docs), expert-residency paragraph: experts live
// in a byte-bounded LRU tier over a colder one, and before a forward
// dispatches, readahead brings in the experts the routing decision selected.
// "Module expert_store" (ferrox-core docs), design list: a lease pins an
// entry so that it is never evicted while work still reads it, and when the
// experts of a step do not all fit, the request still succeeds (capacity
// pressure costs more transfers, never a wrong answer or a deadlock).
//
// Here a step's experts are assigned slots in passes.  Pass 0 holds every
// expert already resident (hits, pinned first) and as many of the rest as
// fit, each taking a free slot or else the least recently used unpinned one;
// when every slot is pinned by the current pass, a new pass starts and the
// previous pass's pins are dropped (on the device the passes run one after
// another in stream order, so a slot is overwritten only after the previous
// pass's kernels have read it).  Pins last for one assignment; ordering
// against earlier device work is the caller's stream order.
//
// moe_host_alloc / moe_host_free (the tier's host memory) are here too.
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <sys/mman.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <thread>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

SlotCache::SlotCache(int n_slots, int n_experts)
    : slot_expert_(n_slots, -1), expert_slot_(n_experts, -1), stamp_(n_slots, 0),
      pinned_(n_slots, 0) {}

int SlotCache::pick() const {
  int best = -1;
  for (int s = 0; s < n_slots(); ++s) {
    if (pinned_[s]) continue;
    if (slot_expert_[s] < 0) return s;  // a free slot first, lowest index
    if (best < 0 || stamp_[s] < stamp_[best]) best = s;
  }
  return best;
}

bool SlotCache::assign(const int32_t* experts, int n, int32_t* slot, int32_t* load, int32_t* pass,
                       int32_t* n_passes) {
  if (n < 0 || (n > 0 && (!experts || !slot || !load || !pass)) || !n_passes) return false;
  std::vector<char> seen(n_experts(), 0);
  for (int i = 0; i < n; ++i) {
    const int e = experts[i];
    if (e < 0 || e >= n_experts() || seen[e]) return false;
    seen[e] = 1;
  }
  ++clock_;
  ++stats_.steps;
  std::fill(pinned_.begin(), pinned_.end(), 0);
  for (int i = 0; i < n; ++i) {  // hits: no bytes to move, pinned for pass 0
    const int s = expert_slot_[experts[i]];
    pass[i] = -1;
    if (s < 0) continue;
    slot[i] = s;
    load[i] = 0;
    pass[i] = 0;
    pinned_[s] = 1;
    stamp_[s] = clock_;
    ++stats_.hits;
  }
  int cur = 0;
  for (int i = 0; i < n; ++i) {
    if (pass[i] >= 0) continue;
    int s = pick();
    if (s < 0) {  // every slot pinned by this pass: the rest go to the next one
      ++cur;
      ++stats_.extra_passes;
      std::fill(pinned_.begin(), pinned_.end(), 0);
      s = pick();
    }
    const int old = slot_expert_[s];
    if (old >= 0) {
      expert_slot_[old] = -1;
      ++stats_.evictions;
    }
    slot_expert_[s] = experts[i];
    expert_slot_[experts[i]] = s;
    pinned_[s] = 1;
    stamp_[s] = clock_;
    slot[i] = s;
    load[i] = 1;
    pass[i] = cur;
    ++stats_.misses;
  }
  std::fill(pinned_.begin(), pinned_.end(), 0);
  *n_passes = n > 0 ? cur + 1 : 0;
  return true;
}

int SlotCache::resident() const {
  int r = 0;
  for (int e : slot_expert_) r += e >= 0;
  return r;
}

void SlotCache::fill_stats(moe_tier_stats* out) const {
  out->steps = stats_.steps;
  out->hits = stats_.hits;
  out->misses = stats_.misses;
  out->evictions = stats_.evictions;
  out->extra_passes = stats_.extra_passes;
  out->bytes_loaded = 0;
  out->n_slots = n_slots();
  out->resident = resident();
}

}  // namespace moe

namespace {

// Host memory for the tier's colder level.  The device reads host memory
// through its own address translation, and with base pages (64 KB on this
// class of host) a region of tens of GB misses that translation often enough
// to halve host -> device copy bandwidth on first touch; memory backed by
// transparent huge pages does not.  So: align to the huge-page size, ask for
// huge pages, fault every page in (in parallel), then page-lock it.
size_t huge_page_bytes() {
  size_t v = 0;
  if (FILE* f = fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
    unsigned long long x = 0;
    if (fscanf(f, "%llu", &x) == 1) v = (size_t)x;
    fclose(f);
  }
  return v >= 4096 && (v & (v - 1)) == 0 ? v : (size_t)2 << 20;
}

std::mutex g_host_mu;
std::map<void*, size_t> g_host_blocks;

}  // namespace

struct moe_slot_cache {
  moe::SlotCache cache;
  std::mutex mu;
  moe_slot_cache(int s, int e) : cache(s, e) {}
};

extern "C" {

moe_status moe_slot_cache_create(int n_slots, int n_experts, moe_slot_cache** out) {
  if (!out || n_slots < 1 || n_experts < 1 || n_experts > (1 << 20) || n_slots > n_experts)
    return MOE_ERR_INVALID_ARG;
  *out = new moe_slot_cache(n_slots, n_experts);
  return MOE_OK;
}

moe_status moe_slot_cache_destroy(moe_slot_cache* c) {
  delete c;
  return MOE_OK;
}

moe_status moe_slot_cache_assign(moe_slot_cache* c, const int32_t* experts, int n,
                                 int32_t* slot, int32_t* load, int32_t* pass,
                                 int32_t* n_passes) {
  if (!c) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(c->mu);
  return c->cache.assign(experts, n, slot, load, pass, n_passes) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

moe_status moe_slot_cache_slot_of(moe_slot_cache* c, int expert, int32_t* slot) {
  if (!c || !slot || expert < 0 || expert >= c->cache.n_experts()) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(c->mu);
  *slot = c->cache.slot_of(expert);
  return MOE_OK;
}

moe_status moe_slot_cache_get_stats(moe_slot_cache* c, moe_tier_stats* out) {
  if (!c || !out) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(c->mu);
  c->cache.fill_stats(out);
  return MOE_OK;
}

moe_status moe_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const size_t align = huge_page_bytes();
  const size_t size = (bytes + align - 1) / align * align;
  void* p = aligned_alloc(align, size);
  if (!p) return MOE_ERR_CUDA;
  (void)madvise(p, size, MADV_HUGEPAGE);  // advice only: base pages still work
  const unsigned hw = std::thread::hardware_concurrency();
  const size_t n_threads = std::min<size_t>(hw ? hw : 1, std::max<size_t>(1, size / align));
  std::vector<std::thread> pool;
  const size_t per = (size / n_threads + align - 1) / align * align;
  for (size_t i = 0; i < n_threads; ++i) {
    const size_t lo = i * per;
    if (lo >= size) break;
    const size_t len = std::min(per, size - lo);
    pool.emplace_back([p, lo, len] { memset(static_cast<char*>(p) + lo, 0, len); });
  }
  for (auto& t : pool) t.join();
  if (cudaHostRegister(p, size, cudaHostRegisterDefault) != cudaSuccess) {
    (void)cudaGetLastError();
    free(p);
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> g(g_host_mu);
  g_host_blocks[p] = size;
  *out = p;
  return MOE_OK;
}

moe_status moe_host_free(void* p) {
  if (!p) return MOE_OK;
  {
    std::lock_guard<std::mutex> g(g_host_mu);
    auto it = g_host_blocks.find(p);
    if (it == g_host_blocks.end()) return MOE_ERR_INVALID_ARG;
    g_host_blocks.erase(it);
  }
  const cudaError_t e = cudaHostUnregister(p);
  free(p);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
