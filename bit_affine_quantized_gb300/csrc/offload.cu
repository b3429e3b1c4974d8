// Per-layer expert slot cache of the expert offload (page "TurboFieldfare -
// System design", sections "Resource split" and "Load and ownership": every
// opened layer owns 16 expert slots; a hit reuses the slot, a miss takes an
// evictable slot and reads the expert into it; eviction is least frequently
// used with recency as the tie-breaker).  Here the experts live in host
// memory and the slots in device memory.  This file holds the policy (host
// code: which slot each selected expert occupies after a step and which slots
// must be filled) and the kernel that fills slots from device-mapped host
// memory.
//
// Readings (the pages leave these open): an expert's use count starts at 1
// when it enters a slot, grows by 1 at every step that selects it, and is
// dropped with the slot when the expert is evicted; "recency" is the step at
// which a slot's expert was last selected; empty slots are taken first, in
// slot order; the experts selected by the current step are never evicted by
// that step's own misses; remaining ties go to the lower slot index.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "kernels.h"
#include "moe.h"

struct moe_expert_cache {
  int n_layers, n_slots;
  struct Layer {
    std::vector<int32_t> expert;    // [n_slots], -1: empty
    std::vector<uint64_t> count;    // uses since the expert entered the slot
    std::vector<uint64_t> last;     // step of the last use
    uint64_t clock = 0;             // steps seen
    long long hits = 0, misses = 0;
  };
  std::vector<Layer> layers;
};

extern "C" int moe_cache_create(int n_layers, int n_slots, moe_expert_cache **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_layers < 1 || n_slots < 1 || n_slots > MOE_CACHE_MAX_SLOTS) return MOE_ERR_INVALID_ARG;
  moe_expert_cache *c = new (std::nothrow) moe_expert_cache;
  if (!c) return MOE_ERR_CUDA;
  c->n_layers = n_layers;
  c->n_slots = n_slots;
  c->layers.resize(n_layers);
  for (auto &L : c->layers) {
    L.expert.assign(n_slots, -1);
    L.count.assign(n_slots, 0);
    L.last.assign(n_slots, 0);
  }
  *out = c;
  return MOE_OK;
}

extern "C" void moe_cache_destroy(moe_expert_cache *c) { delete c; }

extern "C" int moe_cache_lookup(moe_expert_cache *c, int layer, const int32_t *ids, int n, int32_t *slots,
                                int32_t *load_slots, int32_t *load_ids, int *n_loads) {
  if (!c || !ids || !slots || !n_loads || layer < 0 || layer >= c->n_layers || n < 1) return MOE_ERR_INVALID_ARG;
  moe_expert_cache::Layer &L = c->layers[layer];
  const int S = c->n_slots;
  for (int j = 0; j < n; ++j)
    if (ids[j] < 0) return MOE_ERR_BAD_EXPERT_ID;
  // distinct experts of the step must fit the slots
  int distinct = 0;
  for (int j = 0; j < n; ++j) {
    bool seen = false;
    for (int i = 0; i < j; ++i) seen = seen || ids[i] == ids[j];
    distinct += seen ? 0 : 1;
  }
  if (distinct > S) return MOE_ERR_UNSUPPORTED;
  const uint64_t step = ++L.clock;
  bool pinned[MOE_CACHE_MAX_SLOTS] = {};
  int nl = 0;
  // hits first (a step's own experts are then safe from its misses)
  for (int j = 0; j < n; ++j) {
    slots[j] = -1;
    for (int s = 0; s < S; ++s)
      if (L.expert[s] == ids[j]) {
        slots[j] = s;
        break;
      }
    if (slots[j] < 0) continue;
    const int s = slots[j];
    if (L.last[s] != step) {  // a repeated id counts once per step
      ++L.count[s];
      L.last[s] = step;
      ++L.hits;
    }
    pinned[s] = true;
  }
  // misses in selection order: an empty slot, else the least used, then the least recent
  for (int j = 0; j < n; ++j) {
    if (slots[j] >= 0) continue;
    int dup = -1;
    for (int i = 0; i < j; ++i)
      if (ids[i] == ids[j]) dup = i;
    if (dup >= 0) {  // the same expert twice in one step: one slot, one load
      slots[j] = slots[dup];
      continue;
    }
    int v = -1;
    for (int s = 0; s < S && v < 0; ++s)
      if (L.expert[s] < 0 && !pinned[s]) v = s;
    for (int s = 0; s < S && v < 0; ++s) {
      if (pinned[s]) continue;
      v = s;
      for (int t = s + 1; t < S; ++t) {
        if (pinned[t]) continue;
        if (L.count[t] < L.count[v] || (L.count[t] == L.count[v] && L.last[t] < L.last[v])) v = t;
      }
    }
    if (v < 0) return MOE_ERR_UNSUPPORTED;  // unreachable: distinct <= S
    L.expert[v] = ids[j];
    L.count[v] = 1;
    L.last[v] = step;
    pinned[v] = true;
    slots[j] = v;
    ++L.misses;
    if (load_slots) load_slots[nl] = v;
    if (load_ids) load_ids[nl] = ids[j];
    ++nl;
  }
  *n_loads = nl;
  return MOE_OK;
}

extern "C" int moe_cache_stats(const moe_expert_cache *c, int layer, long long *hits, long long *misses) {
  if (!c || layer < 0 || layer >= c->n_layers) return MOE_ERR_INVALID_ARG;
  if (hits) *hits = c->layers[layer].hits;
  if (misses) *misses = c->layers[layer].misses;
  return MOE_OK;
}

extern "C" int moe_cache_slot_expert(const moe_expert_cache *c, int layer, int slot) {
  if (!c || layer < 0 || layer >= c->n_layers || slot < 0 || slot >= c->n_slots) return -2;
  return c->layers[layer].expert[slot];
}

extern "C" int moe_cache_slots(const moe_expert_cache *c) { return c ? c->n_slots : 0; }

// ------------------------------------------------------------ slot fills
// The missing experts of a step copied into their slots by the GPU itself:
// every block streams one share of one blob from host memory (device-mapped
// pinned memory, read over the host link) into the slot.  GPU-initiated
// reads keep many more requests in flight than the copy engines do.
namespace moe {
namespace {
constexpr int kFillThreads = 256;
constexpr int kFillBlocksPerBlob = 48;

__global__ void __launch_bounds__(kFillThreads) fill_slots_kernel(const FillArgs a) {
  const int i = blockIdx.x / kFillBlocksPerBlob, part = blockIdx.x - i * kFillBlocksPerBlob;
  if (i >= a.n) return;
  const uint4 *src = reinterpret_cast<const uint4 *>(a.src[i]);
  uint4 *dst = reinterpret_cast<uint4 *>(a.dst[i]);
  const size_t n16 = a.bytes / 16, per = (n16 + kFillBlocksPerBlob - 1) / kFillBlocksPerBlob;
  const size_t b0 = (size_t)part * per, b1 = b0 + per < n16 ? b0 + per : n16;
  // four 16-byte loads in flight per thread
  size_t j = b0 + threadIdx.x;
  for (; j + 3 * kFillThreads < b1; j += 4 * kFillThreads) {
    const uint4 v0 = src[j], v1 = src[j + kFillThreads], v2 = src[j + 2 * kFillThreads], v3 = src[j + 3 * kFillThreads];
    dst[j] = v0;
    dst[j + kFillThreads] = v1;
    dst[j + 2 * kFillThreads] = v2;
    dst[j + 3 * kFillThreads] = v3;
  }
  for (; j < b1; j += kFillThreads) dst[j] = src[j];
}
}  // namespace

cudaError_t launch_fill_slots(const FillArgs &a, cudaStream_t st) {
  if (a.n < 1 || a.n > kMaxFill || a.bytes % 16) return cudaErrorInvalidValue;
  fill_slots_kernel<<<a.n * kFillBlocksPerBlob, kFillThreads, 0, st>>>(a);
  return cudaGetLastError();
}
}  // namespace moe
