// Paged-cache addressing shared by the gather and the paged up-projection.
//
// Slot rule from vLLM "vllm/models/deepseek_v4/sparse_mla.py",
// _build_c128a_topk_metadata_kernel (decode branch): position p of request r lives in
// block block_table[r, p / block_size] at offset p % block_size, flat slot
// block * block_size + offset.  Output row cu[r] + t of a chunk is prefix position
// starts[r] + t of request r ("vllm.v1.attention.backends.mla.prefill.flashinfer":
// chunk i's kv_indptr is chunked_context.cu_seq_lens[i]).
#pragma once
#include <cstdint>

namespace mla {

// Request owning output row `row`: the last r with cu[r] <= row (cu is non-decreasing).
__device__ __forceinline__ int find_request(const int32_t* cu, int batch, int64_t row) {
  int lo = 0, hi = batch;   // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)__ldg(cu + mid) <= row) lo = mid; else hi = mid;
  }
  return lo;
}

// Cache slot of output row `row`; false when the row's block is unknown (a block id
// outside [0, num_blocks), a table slot past max_blocks, or a row past its request).
// With fewer than 32 requests, lane i holds cu[i] in cu_l and starts[i] in st_l and the
// request is found by shuffles (all 32 lanes must call); otherwise by binary search.
struct RowMap {
  const int32_t* cu;
  const int32_t* starts;
  const int32_t* table;
  int batch, max_blocks, block_size;
  int64_t num_blocks;
};

__device__ __forceinline__ bool resolve_slot(const RowMap& m, int64_t row, bool active, int32_t cu_l, int32_t st_l,
                                             int64_t* slot) {
  int r = 0;
  int64_t cu_r = 0, cu_r1 = 0, start_r = 0;
  if (m.batch < 32) {
    for (int i = 1; i < m.batch; ++i) r += __shfl_sync(0xffffffffu, cu_l, i) <= row ? 1 : 0;
    cu_r = __shfl_sync(0xffffffffu, cu_l, r);
    cu_r1 = __shfl_sync(0xffffffffu, cu_l, r + 1);
    start_r = __shfl_sync(0xffffffffu, st_l, r);
  } else if (active) {
    r = find_request(m.cu, m.batch, row);
    cu_r = __ldg(m.cu + r);
    cu_r1 = __ldg(m.cu + r + 1);
    start_r = __ldg(m.starts + r);
  }
  if (!active) return false;
  const int64_t pos = start_r + (row - cu_r);
  const int64_t bi = pos / m.block_size;
  bool ok = row < cu_r1 && pos >= 0 && bi < m.max_blocks;
  const int64_t blk = ok ? (int64_t)__ldg(m.table + (int64_t)r * m.max_blocks + bi) : -1;
  ok = ok && blk >= 0 && blk < m.num_blocks;
  *slot = ok ? blk * m.block_size + (pos - bi * m.block_size) : 0;
  return ok;
}

}  // namespace mla
