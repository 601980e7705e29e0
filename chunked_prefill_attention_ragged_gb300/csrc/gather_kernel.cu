// Paged latent gather: out[cu_seq_lens[r] + t] = cache row of prefix position
// chunk_starts[r] + t of request r.
//
// Slot rule from vLLM "vllm/models/deepseek_v4/sparse_mla.py",
// _build_c128a_topk_metadata_kernel (decode branch): position p of request r lives in
// block block_table[r, p / block_size] at offset p % block_size.
//
// Main kernel (rows up to 36 KB): one warp per CTA moves a batch of consecutive output
// rows (about 4.5 KB: 4 rows of 576 bf16).  Each lane resolves its row's cache slot and
// starts one bulk copy (cp.async.bulk) of the whole row into shared memory; once all
// have landed, one bulk copy writes the batch, which is contiguous in both shared and
// global memory, back out.  Small batches give many CTAs per SM, so loads of some
// overlap stores of others; measured, this matches a plain device-to-device copy of
// the same bytes (a persistent variant with several batches in flight per CTA, 2 to 6
// stages of 4 to 16 rows, 2 to 16 CTAs per SM, was 3 % to 2x slower on the 75 MB
// all-chunk gather).  Wider rows use the register-vector kernel below.
#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"

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

constexpr int kBulkBatch = 4608;        // bytes per bulk-gather CTA (4 rows of 576 bf16)
constexpr int kBulkMaxRow = 36 * 1024;  // widest row the bulk path takes
constexpr uint64_t kBulkWaitNs = 2000000000ull;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(32)
gather_bulk_kernel(const uint8_t* __restrict__ cache, int64_t num_blocks, int block_size, int row_bytes,
                   int rows_per_cta, const int32_t* __restrict__ block_table, int max_blocks,
                   const int32_t* __restrict__ cu, const int32_t* __restrict__ starts, int batch,
                   int64_t total_rows, uint8_t* __restrict__ out, int32_t* status) {
  extern __shared__ __align__(128) uint8_t rows_smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int lane = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * rows_per_cta;
  const int nrows = total_rows - row0 < rows_per_cta ? (int)(total_rows - row0) : rows_per_cta;
  const uint32_t bar_a = smem_addr(&bar);
  if (lane == 0) {
    mbar_init(bar_a, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  // Resolve this lane's row.  With at most 31 requests the warp loads cu and starts
  // once (lane i holds cu[i] and starts[i]) and finds each row's request by shuffles,
  // which leaves the block-table read as the only dependent load before the copy.
  const int64_t row = row0 + lane;
  bool active = lane < nrows, ok = false;
  int64_t slot = 0;
  int r = 0;
  int64_t cu_r = 0, cu_r1 = 0, start_r = 0;
  if (batch < 32) {
    const int32_t cu_l = lane <= batch ? __ldg(cu + lane) : 0x7fffffff;
    const int32_t st_l = lane < batch ? __ldg(starts + lane) : 0;
    for (int i = 1; i < batch; ++i) r += __shfl_sync(0xffffffffu, cu_l, i) <= row ? 1 : 0;
    cu_r = __shfl_sync(0xffffffffu, cu_l, r);
    cu_r1 = __shfl_sync(0xffffffffu, cu_l, r + 1);
    start_r = __shfl_sync(0xffffffffu, st_l, r);
  } else if (active) {
    r = find_request(cu, batch, row);
    cu_r = __ldg(cu + r);
    cu_r1 = __ldg(cu + r + 1);
    start_r = __ldg(starts + r);
  }
  if (active) {
    const int64_t t = row - cu_r;
    const int64_t pos = start_r + t;
    const int64_t bi = pos / block_size;
    ok = row < cu_r1 && pos >= 0 && bi < max_blocks;
    const int64_t blk = ok ? (int64_t)__ldg(block_table + (int64_t)r * max_blocks + bi) : -1;
    ok = ok && blk >= 0 && blk < num_blocks;
    slot = ok ? blk * block_size + (pos - bi * block_size) : 0;
  }
  const unsigned good = __ballot_sync(0xffffffffu, active && ok);
  if (active && !ok) {   // unknown block: the row is written as zeros and flagged
    uint4* z = reinterpret_cast<uint4*>(rows_smem + (size_t)lane * row_bytes);
    for (int i = 0; i < row_bytes / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
    if (status) atomicOr(status, MLA_DEVSTAT_BAD_INDEX);
  }
  // Generic-proxy zero rows must be visible to the bulk copy that reads them.
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(bar_a, (uint32_t)__popc(good) * (uint32_t)row_bytes);
  __syncwarp();
  if (active && ok)
    bulk_g2s(smem_addr(rows_smem) + (uint32_t)lane * row_bytes, cache + slot * row_bytes, (uint32_t)row_bytes,
             bar_a);
  if (lane == 0) {
    if (mbar_wait_bounded(bar_a, 0, &abort_flag, status, MLA_DEVSTAT_TIMEOUT, kBulkWaitNs))
      bulk_s2g(out + row0 * row_bytes, smem_addr(rows_smem), (uint32_t)nrows * (uint32_t)row_bytes);
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
  const int row_bytes = entry_dim * 2;
  if (row_bytes <= kBulkMaxRow) {
    const int rows_per_cta = max(1, min(32, kBulkBatch / row_bytes));
    const int64_t grid = (total_tokens + rows_per_cta - 1) / rows_per_cta;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    const int smem = rows_per_cta * row_bytes;
    gather_bulk_kernel<<<(unsigned)grid, 32, smem, stream>>>(
        static_cast<const uint8_t*>(cache), num_blocks, block_size, row_bytes, rows_per_cta, block_table,
        max_blocks_per_req, cu_seq_lens, chunk_starts, batch, total_tokens, static_cast<uint8_t*>(out), status);
    return cudaGetLastError();
  }
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
