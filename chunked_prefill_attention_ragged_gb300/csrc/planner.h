// Host planner for ragged prefill attention: cuts every (request, head) into
// 128-row query tiles, gives each tile the range of 128-key tiles that hold at
// least one allowed key, and spreads the tiles over a persistent grid.
#pragma once
#include <cstdint>
#include <vector>

namespace mla {

constexpr int kTileM = 128;   // query rows per tile
constexpr int kTileN = 128;   // keys per tile

// One work unit = one query tile of one head.  32 bytes, read by the kernel.
struct Unit {
  int32_t head;
  int32_t q_row0;     // global row of the tile's first query
  int32_t q_rows;     // valid query rows in the tile (1..128)
  int32_t q_pos0;     // position of the first query inside its request
  int32_t kv_row0;    // global row of the request's first key
  int32_t kv_len;     // keys of the request
  int32_t diag;       // kv_len - q_len: query position p sits at key position p + diag
  int32_t kv_tiles;   // kv tile range: lo | hi << 16, tiles [lo, hi) of 128 keys
};
static_assert(sizeof(Unit) == 32, "unit layout");

inline int unit_tile_lo(const Unit& u) { return u.kv_tiles & 0xFFFF; }
inline int unit_tile_hi(const Unit& u) { return (u.kv_tiles >> 16) & 0xFFFF; }

struct PlanResult {
  std::vector<Unit> units;        // execution order, grouped per CTA
  std::vector<int32_t> cta_offsets;  // num_ctas + 1
  int64_t allowed_pairs = 0;      // sum over requests of allowed (query, key) pairs
  int64_t kv_tiles = 0;           // sum over units of (hi - lo)
};

// Returns 0 or a negative MLA_ERR_* code.  Inputs are validated here.  rows_per_unit is
// kTileM (one CTA per unit) or 2 * kTileM (a CTA pair per unit: the two CTAs of a cluster
// take the unit's first and second 128 rows and share its key tiles); max_ctas then
// counts CTA pairs.
int build_plan(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch, int num_heads,
               bool causal, int window_left, int max_ctas, PlanResult* out, int rows_per_unit = kTileM);

// One unit of the absorbed-weight (MQA) prefill: up to 128 consecutive (query row, head)
// pairs of one request and one half of the 512 latent value columns.  32 bytes, read by
// the kernel.
struct AbsUnit {
  int32_t pair0;    // first pair: global query row * num_heads + head
  int32_t npairs;   // pairs in the unit (1..128)
  int32_t q_row0;   // global row of the request's first query
  int32_t q_len;    // queries of the request
  int32_t kv_len;   // keys of the request (its cache positions 0 .. kv_len - 1)
  int32_t ntiles;   // 64-key tiles holding an allowed key of some pair of the unit
  int32_t half;     // value columns [256 half, 256 half + 256)
  int32_t req;      // request (block-table row)
};
static_assert(sizeof(AbsUnit) == 32, "absorbed unit layout");

// Units of the absorbed-weight prefill: for each request r (queries qo[r] .. qo[r+1] - 1,
// the last q_len of its kv_lens[r] cache positions), its (row, head) pairs in runs of 128,
// each run once per value half, with the number of 64-key tiles that hold an allowed key
// of the run's last pair (the one with the most keys); longest first.  *allowed_pairs
// receives the allowed (query, key) pairs summed over requests (one head).  Returns 0 or a
// negative MLA_ERR_* code.
int build_absorbed_units(const int32_t* qo_indptr, const int32_t* kv_lens, int batch, int num_heads, bool causal,
                         std::vector<AbsUnit>* out, int64_t* allowed_pairs);

}  // namespace mla
