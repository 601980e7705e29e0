// Host planner (see planner.h).
//
// The plan/run split follows vLLM "vllm.v1.attention.backends.mla.prefill.flashinfer",
// FlashInferPrefillBackend.finalize_attention_metadata: metadata for a batch is built once
// on the host and reused by every layer's run.  Masking follows the same page's two plan
// calls: causal for the new tokens, non-causal for prefix chunks, plus window_left.
#include "planner.h"

#include <algorithm>
#include <climits>
#include <functional>
#include <queue>
#include <utility>

#include "../../include/mla_prefill.h"

namespace mla {

namespace {

// Key range [lo, hi] (inclusive, positions inside the request) that query rows
// [p0, p1] may see.  Empty when hi < lo.
inline void key_span(int64_t p0, int64_t p1, int64_t kv_len, int64_t diag, bool causal,
                     int window_left, int64_t* lo, int64_t* hi) {
  int64_t h = kv_len - 1;
  if (causal) h = std::min(h, p1 + diag);
  int64_t l = 0;
  if (window_left >= 0) l = std::max<int64_t>(0, p0 + diag - window_left);
  *lo = l;
  *hi = h;
}

// Allowed pairs of one request (one head), counted row by row in closed form.
int64_t allowed_pairs(int64_t lq, int64_t lkv, bool causal, int window_left) {
  int64_t total = 0;
  const int64_t diag = lkv - lq;
  for (int64_t i = 0; i < lq; ++i) {
    int64_t lo, hi;
    key_span(i, i, lkv, diag, causal, window_left, &lo, &hi);
    if (hi >= lo) total += hi - lo + 1;
  }
  return total;
}

}  // namespace

int build_plan(const int32_t* qo, const int32_t* kv, int batch, int num_heads, bool causal,
               int window_left, int max_ctas, PlanResult* out, int rows_per_unit) {
  if (!qo || !kv || !out || batch < 0 || num_heads < 1 || max_ctas < 1) return MLA_ERR_INVALID_ARG;
  if (rows_per_unit != kTileM && rows_per_unit != 2 * kTileM) return MLA_ERR_INVALID_ARG;
  if (window_left < -1) return MLA_ERR_INVALID_ARG;
  if (qo[0] != 0 || kv[0] != 0) return MLA_ERR_SHAPE;
  for (int r = 0; r < batch; ++r)
    if (qo[r + 1] < qo[r] || kv[r + 1] < kv[r]) return MLA_ERR_SHAPE;
  // kv tile indices are packed in 16 bits.
  for (int r = 0; r < batch; ++r)
    if ((int64_t)(kv[r + 1] - kv[r]) > (int64_t)kTileN * 65535) return MLA_ERR_UNSUPPORTED;

  struct Group {            // one (request, head): its tiles, and their total cost
    int64_t cost;
    int32_t first, count;   // slice of `pending`
  };
  std::vector<Unit> pending;
  std::vector<int64_t> pending_cost;
  std::vector<Group> groups;
  out->allowed_pairs = 0;
  out->kv_tiles = 0;

  for (int r = 0; r < batch; ++r) {
    const int64_t lq = qo[r + 1] - qo[r];
    const int64_t lkv = kv[r + 1] - kv[r];
    if (lq == 0) continue;
    out->allowed_pairs += allowed_pairs(lq, lkv, causal, window_left);
    const int64_t diag = lkv - lq;
    // Tiles of this request, identical for every head.
    std::vector<std::pair<Unit, int64_t>> tiles;
    for (int64_t p0 = 0; p0 < lq; p0 += rows_per_unit) {
      const int64_t p1 = std::min(lq, p0 + rows_per_unit) - 1;
      int64_t lo, hi;
      key_span(p0, p1, lkv, diag, causal, window_left, &lo, &hi);
      int32_t tlo = 0, thi = 0;   // empty range: the kernel writes O = 0, LSE = -inf
      if (hi >= lo) {
        tlo = (int32_t)(lo / kTileN);
        thi = (int32_t)(hi / kTileN + 1);
      }
      Unit u;
      u.head = 0;
      u.q_row0 = (int32_t)(qo[r] + p0);
      u.q_rows = (int32_t)(p1 - p0 + 1);
      u.q_pos0 = (int32_t)p0;
      u.kv_row0 = kv[r];
      u.kv_len = (int32_t)lkv;
      u.diag = (int32_t)diag;
      u.kv_tiles = tlo | (thi << 16);
      // Cost in half key tiles: two per key tile plus three for the unit's fixed work
      // (Q load, pipeline fill, epilogue), which measures at about 1.5 key tiles.
      tiles.push_back({u, 2 * (int64_t)(thi - tlo) + 3});
    }
    // Longest tiles first inside a group.
    std::stable_sort(tiles.begin(), tiles.end(),
                     [](const auto& a, const auto& b) { return a.second > b.second; });
    int64_t group_cost = 0;
    for (auto& t : tiles) group_cost += t.second;
    for (int h = 0; h < num_heads; ++h) {
      Group g{group_cost, (int32_t)pending.size(), (int32_t)tiles.size()};
      for (auto& t : tiles) {
        Unit u = t.first;
        u.head = h;
        pending.push_back(u);
        pending_cost.push_back(t.second);
        out->kv_tiles += (t.second - 3) / 2;
      }
      groups.push_back(g);
    }
  }

  const int64_t n_units = (int64_t)pending.size();
  const int num_ctas = (int)std::max<int64_t>(1, std::min<int64_t>(max_ctas, n_units));
  // Heaviest (request, head) groups first; ties keep request/head order.
  std::vector<int32_t> order(groups.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = (int32_t)i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return groups[a].cost > groups[b].cost; });

  // Greedy list scheduling: walk the units group by group and give each one to the
  // CTA that is least loaded so far.  Units of one (request, head) therefore start
  // close together in time and share its K/V tiles through L2.
  using Slot = std::pair<int64_t, int32_t>;   // (load, cta)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
  for (int c = 0; c < num_ctas; ++c) heap.push({0, c});
  std::vector<std::vector<int32_t>> per_cta(num_ctas);
  for (int32_t gi : order) {
    const Group& g = groups[gi];
    for (int32_t i = g.first; i < g.first + g.count; ++i) {
      Slot s = heap.top();
      heap.pop();
      per_cta[s.second].push_back(i);
      s.first += pending_cost[i];
      heap.push(s);
    }
  }
  out->units.clear();
  out->units.reserve(n_units);
  out->cta_offsets.assign(num_ctas + 1, 0);
  for (int c = 0; c < num_ctas; ++c) {
    out->cta_offsets[c] = (int32_t)out->units.size();
    for (int32_t i : per_cta[c]) out->units.push_back(pending[i]);
  }
  out->cta_offsets[num_ctas] = (int32_t)out->units.size();
  return MLA_OK;
}

int build_absorbed_units(const int32_t* qo, const int32_t* kv_lens, int batch, int num_heads, bool causal,
                         std::vector<AbsUnit>* out, int64_t* allowed) {
  if (!qo || !kv_lens || !out || !allowed || batch < 0 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (qo[0] != 0) return MLA_ERR_SHAPE;
  for (int r = 0; r < batch; ++r)
    if (qo[r + 1] < qo[r] || kv_lens[r] < 0) return MLA_ERR_SHAPE;
  // Pair indices (row * heads + head) and key positions are 32-bit on the device.
  if ((int64_t)qo[batch] * num_heads > INT32_MAX - 128) return MLA_ERR_UNSUPPORTED;
  out->clear();
  *allowed = 0;
  constexpr int kPairs = 128, kKeys = 64;
  for (int r = 0; r < batch; ++r) {
    const int64_t lq = qo[r + 1] - qo[r], lkv = kv_lens[r];
    if (lq == 0) continue;
    *allowed += allowed_pairs(lq, lkv, causal, -1);
    const int64_t diag = lkv - lq, pairs = lq * num_heads;
    for (int64_t p0 = 0; p0 < pairs; p0 += kPairs) {
      const int64_t np = std::min<int64_t>(kPairs, pairs - p0);
      const int64_t last_pos = (p0 + np - 1) / num_heads;   // position of the run's last row
      int64_t khi = causal ? std::min(lkv, last_pos + diag + 1) : lkv;
      if (khi < 0) khi = 0;
      AbsUnit u;
      u.pair0 = (int32_t)((int64_t)qo[r] * num_heads + p0);
      u.npairs = (int32_t)np;
      u.q_row0 = qo[r];
      u.q_len = (int32_t)lq;
      u.kv_len = (int32_t)lkv;
      u.ntiles = (int32_t)((khi + kKeys - 1) / kKeys);
      u.req = r;
      for (int h = 0; h < 2; ++h) {
        u.half = h;
        out->push_back(u);
      }
    }
  }
  std::stable_sort(out->begin(), out->end(), [](const AbsUnit& a, const AbsUnit& b) { return a.ntiles > b.ntiles; });
  return MLA_OK;
}

}  // namespace mla
