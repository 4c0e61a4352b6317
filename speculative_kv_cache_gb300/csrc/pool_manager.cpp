// Host-side slot manager of the KV pool (InfiniGen paper-graph summary, section 3.4, "KV Cache
// Pool Management Under Memory Pressure"): per (layer, sequence) pool, fold a step's "used by
// any head" flags into the slots' state and place the next token, the victim chosen by the
// pool's policy -- the counter policy InfiniGen uses, or FIFO / LRU, the two it is compared
// with in Table 2.  Pools are independent, so a whole step's pools are processed in parallel.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <thread>
#include <vector>

#include "../../include/ig.h"
#include "pool_impl.h"

namespace ig {
ig_status fail(ig_status st, const char* fmt, ...);
}

#define IG_REQUIRE(cond, ...)                                   \
  do {                                                          \
    if (!(cond)) return ::ig::fail(IG_ERR_INVALID, __VA_ARGS__); \
  } while (0)

namespace {

// One update of pool pb with a step's flags: counters +1 (8-bit; the whole pool halved when
// one reaches 255) and the LRU time of each used slot.  Both are kept whatever the policy;
// only the victim choice differs.
void fold_use(ig_pool* pool, size_t pb, const uint8_t* used) {
  const int cap = pool->cap;
  uint8_t* cnt = pool->counter.data() + pb * cap;
  uint32_t* last = pool->last_use.data() + pb * cap;
  const uint32_t now = ++pool->clock[pb];
  const int filled = pool->filled[pb];
  bool sat = false;
  for (int s = 0; s < filled; ++s) {
    if (used[s]) {
      if (cnt[s] < 255) ++cnt[s];
      last[s] = now;
    }
    sat |= (cnt[s] == 255);
  }
  if (sat)
    for (int s = 0; s < filled; ++s) cnt[s] >>= 1;
}

// The victim of a full pool; ties go to the oldest insertion, then the lowest slot.
//   counter: the smallest counter;  FIFO: the oldest insertion;  LRU: the oldest last use
//   (an insertion counts as a use at that time).
int victim(const ig_pool* pool, size_t pb) {
  const int cap = pool->cap;
  const uint8_t* cnt = pool->counter.data() + pb * cap;
  const uint32_t* seq = pool->seq.data() + pb * cap;
  const uint32_t* last = pool->last_use.data() + pb * cap;
  int v = 0;
  switch (pool->policy) {
    case IG_POOL_FIFO:
      for (int s = 1; s < cap; ++s)
        if (seq[s] < seq[v]) v = s;
      break;
    case IG_POOL_LRU:
      for (int s = 1; s < cap; ++s)
        if (last[s] < last[v] || (last[s] == last[v] && seq[s] < seq[v])) v = s;
      break;
    default:
      for (int s = 1; s < cap; ++s)
        if (cnt[s] < cnt[v] || (cnt[s] == cnt[v] && seq[s] < seq[v])) v = s;
      break;
  }
  return v;
}

// Places the next token of pool pb: the next free slot while there is one, else the victim.
int place(ig_pool* pool, size_t pb) {
  const int cap = pool->cap;
  int32_t& filled = pool->filled[pb];
  int slot;
  if (filled < cap) {
    slot = filled++;
  } else {
    slot = victim(pool, pb);
    pool->evictions[pb] += 1;
  }
  pool->counter[pb * cap + slot] = 0;
  pool->last_use[pb * cap + slot] = pool->clock[pb];
  pool->seq[pb * cap + slot] = pool->next_seq[pb]++;
  return slot;
}

// Runs f(pb) for pb in [0, n), on several threads when the work is large enough to pay for
// them (each pool is touched by one thread only).
template <class F>
void for_each_pool(size_t n, size_t work_per_pool, F f) {
  const unsigned hw = std::max(1u, std::thread::hardware_concurrency());
  size_t nt = std::min<size_t>({hw, 16, n});
  if (n * work_per_pool < (1u << 17)) nt = 1;
  if (nt <= 1) {
    for (size_t pb = 0; pb < n; ++pb) f(pb);
    return;
  }
  std::vector<std::thread> th;
  th.reserve(nt - 1);
  auto run = [&](size_t t) {
    for (size_t pb = n * t / nt; pb < n * (t + 1) / nt; ++pb) f(pb);
  };
  for (size_t t = 1; t < nt; ++t) th.emplace_back(run, t);
  run(0);
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" ig_status ig_pool_update(ig_pool* pool, int layer, int b, const uint8_t* used) {
  IG_REQUIRE(pool && used, "null argument");
  IG_REQUIRE(layer >= 0 && layer < pool->layers && b >= 0 && b < pool->B, "layer/b out of range");
  fold_use(pool, (size_t)layer * pool->B + b, used);
  return IG_OK;
}

extern "C" ig_status ig_pool_evict(ig_pool* pool, int layer, int b, const uint8_t* used,
                                   int32_t* slot_out, int32_t* filled_out) {
  IG_REQUIRE(pool && slot_out, "null argument");
  IG_REQUIRE(layer >= 0 && layer < pool->layers && b >= 0 && b < pool->B, "layer/b out of range");
  const size_t pb = (size_t)layer * pool->B + b;
  if (used) fold_use(pool, pb, used);
  *slot_out = place(pool, pb);
  if (filled_out) *filled_out = pool->filled[pb];
  return IG_OK;
}

extern "C" ig_status ig_pool_prefill(ig_pool* pool, int n_tokens, int32_t* slots_out) {
  IG_REQUIRE(pool && n_tokens >= 0, "bad argument");
  const size_t npb = (size_t)pool->layers * pool->B;
  for_each_pool(npb, (size_t)n_tokens, [&](size_t pb) {
    for (int t = 0; t < n_tokens; ++t) {
      const int s = place(pool, pb);
      if (pb == 0 && slots_out) slots_out[t] = s;
    }
  });
  return IG_OK;
}

extern "C" ig_status ig_pool_step(ig_pool* pool, const uint8_t* used, int Lcap, int32_t* slots_out) {
  IG_REQUIRE(pool, "null pool");
  IG_REQUIRE(!used || Lcap >= pool->cap, "Lcap must cover the pool capacity");
  const size_t npb = (size_t)pool->layers * pool->B;
  for_each_pool(npb, 2 * (size_t)pool->cap, [&](size_t pb) {
    if (used) fold_use(pool, pb, used + pb * (size_t)Lcap);
    if (slots_out) slots_out[pb] = place(pool, pb);
  });
  return IG_OK;
}

extern "C" ig_status ig_pool_full(const ig_pool* pool, int* any_full) {
  IG_REQUIRE(pool && any_full, "null argument");
  *any_full = 0;
  for (int32_t f : pool->filled)
    if (f >= pool->cap) *any_full = 1;
  return IG_OK;
}

extern "C" ig_status ig_pool_counters(const ig_pool* pool, int layer, int b, uint8_t* out) {
  IG_REQUIRE(pool && out, "null argument");
  IG_REQUIRE(layer >= 0 && layer < pool->layers && b >= 0 && b < pool->B, "layer/b out of range");
  memcpy(out, pool->counter.data() + ((size_t)layer * pool->B + b) * pool->cap, pool->cap);
  return IG_OK;
}

extern "C" ig_status ig_pool_slot_tokens(const ig_pool* pool, int layer, int b, int32_t* out) {
  IG_REQUIRE(pool && out, "null argument");
  IG_REQUIRE(layer >= 0 && layer < pool->layers && b >= 0 && b < pool->B, "layer/b out of range");
  const size_t pb = (size_t)layer * pool->B + b;
  const uint32_t* seq = pool->seq.data() + pb * pool->cap;
  for (int s = 0; s < pool->cap; ++s) out[s] = s < pool->filled[pb] ? (int32_t)seq[s] : -1;
  return IG_OK;
}

extern "C" ig_status ig_pool_evictions(const ig_pool* pool, int layer, int b, int64_t* out) {
  IG_REQUIRE(pool && out, "null argument");
  IG_REQUIRE(layer >= 0 && layer < pool->layers && b >= 0 && b < pool->B, "layer/b out of range");
  *out = pool->evictions[(size_t)layer * pool->B + b];
  return IG_OK;
}
