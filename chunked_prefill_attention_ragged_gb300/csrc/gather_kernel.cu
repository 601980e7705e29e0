// Paged latent gather: out[cu_seq_lens[r] + t] = cache row of prefix position
// chunk_starts[r] + t of request r.
//
// Slot rule from vLLM "vllm/models/deepseek_v4/sparse_mla.py",
// _build_c128a_topk_metadata_kernel (decode branch): position p of request r lives in
// block block_table[r, p / block_size] at offset p % block_size.  Rows are 16-byte
// vectorised: consecutive threads copy consecutive 16-byte pieces of the output, so
// stores are fully coalesced and each cache row is read as whole 128-byte lines.
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Request owning output row `row`: the last r with cu[r] <= row (cu is non-decreasing).
__device__ __forceinline__ int find_request(const int32_t* cu, int batch, int64_t row) {
  int lo = 0, hi = batch;   // answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)__ldg(cu + mid) <= row) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads)
gather_kernel(const uint4* __restrict__ cache, int64_t num_blocks, int block_size, int vec_per_row,
              const int32_t* __restrict__ block_table, int max_blocks,
              const int32_t* __restrict__ cu, const int32_t* __restrict__ starts, int batch,
              int64_t total_vec, uint4* __restrict__ out, int32_t* status) {
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t base = (int64_t)blockIdx.x * kThreads * kVecPerThread + threadIdx.x; base < total_vec;
       base += stride * kVecPerThread) {
    uint4 v[kVecPerThread];
    int64_t dst[kVecPerThread];
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k) {
      const int64_t idx = base + (int64_t)k * kThreads;
      dst[k] = -1;
      v[k] = make_uint4(0, 0, 0, 0);
      if (idx >= total_vec) continue;
      dst[k] = idx;
      const int64_t row = idx / vec_per_row;
      const int e = (int)(idx - row * vec_per_row);
      const int r = find_request(cu, batch, row);
      const int64_t t = row - __ldg(cu + r);
      const bool in_req = row < __ldg(cu + r + 1);
      const int64_t pos = (int64_t)__ldg(starts + r) + t;
      const int64_t bi = pos / block_size;
      bool ok = in_req && pos >= 0 && bi < max_blocks;
      const int64_t blk = ok ? (int64_t)__ldg(block_table + (int64_t)r * max_blocks + bi) : -1;
      ok = ok && blk >= 0 && blk < num_blocks;
      if (ok) {
        const int64_t slot = blk * block_size + (pos - bi * block_size);
        v[k] = ld_stream(cache + slot * vec_per_row + e);
      } else if (e == 0 && status) {
        atomicOr(status, MLA_DEVSTAT_BAD_INDEX);
      }
    }
#pragma unroll
    for (int k = 0; k < kVecPerThread; ++k)
      if (dst[k] >= 0) out[dst[k]] = v[k];
  }
}

}  // namespace

cudaError_t launch_gather(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                          const int32_t* block_table, int max_blocks_per_req,
                          const int32_t* cu_seq_lens, const int32_t* chunk_starts, int batch,
                          int64_t total_tokens, void* out, int32_t* status, cudaStream_t stream) {
  const int vec_per_row = entry_dim * 2 / 16;
  const int64_t total_vec = total_tokens * vec_per_row;
  if (total_vec == 0) return cudaSuccess;
  const int sms = device_sm_count();
  const int64_t want = (total_vec + (int64_t)kThreads * kVecPerThread - 1) / ((int64_t)kThreads * kVecPerThread);
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
  const int grid = (int)(want < cap ? want : cap);
  gather_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(cache), num_blocks, block_size,
                                               vec_per_row, block_table, max_blocks_per_req, cu_seq_lens,
                                               chunk_starts, batch, total_vec, static_cast<uint4*>(out),
                                               status);
  return cudaGetLastError();
}

}  // namespace mla
