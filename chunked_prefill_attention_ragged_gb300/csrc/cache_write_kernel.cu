// Paged latent cache write: cache row at flat slot slot_mapping[t] = latent[t], for
// every token whose slot is >= 0 (a negative slot is a padding token).
//
// sglang issue #3849 ("[DeepseekR1] How ragged prefill manage kv_cache?"): ragged
// prefill saves the new tokens' compressed rows (512 latent + 64 rope) in the paged cache
// before attention.  vLLM "vllm/models/deepseek_v4/sparse_mla.py": a token's flat slot is
// block * block_size + offset, and tokens with a negative slot are not valid.
//
// One warp per CTA moves a batch of consecutive tokens (about 4.5 KB: 4 rows of 576 bf16):
// the batch is contiguous in the source, so one bulk copy (cp.async.bulk) brings it into
// shared memory; then each lane whose slot is valid writes its row to the cache with one
// bulk copy.  Slots past the cache are skipped and flagged (MLA_DEVSTAT_BAD_INDEX).
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kBatchBytes = 4608;          // bytes per CTA
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
               : "memory");
}

__global__ void __launch_bounds__(32)
cache_write_kernel(uint8_t* __restrict__ cache, int64_t num_slots, int row_bytes, int rows_per_cta,
                   const uint8_t* __restrict__ latent, const int64_t* __restrict__ slot_mapping,
                   int64_t num_tokens, int32_t* status) {
  extern __shared__ __align__(128) uint8_t rows_smem[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const int lane = threadIdx.x;
  const int64_t row0 = (int64_t)blockIdx.x * rows_per_cta;
  const int nrows = num_tokens - row0 < rows_per_cta ? (int)(num_tokens - row0) : rows_per_cta;
  const uint32_t bar_a = smem_addr(&bar);
  if (lane == 0) {
    mbar_init(bar_a, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  int64_t slot = -1;
  if (lane < nrows) {
    slot = __ldg(slot_mapping + row0 + lane);
    if (slot >= num_slots) {
      if (status) atomicOr(status, MLA_DEVSTAT_BAD_INDEX);
      slot = -1;
    }
  }
  const unsigned write = __ballot_sync(0xffffffffu, slot >= 0);
  if (write == 0) return;   // all padding: nothing to move
  if (lane == 0) {
    const uint32_t bytes = (uint32_t)nrows * (uint32_t)row_bytes;
    mbar_arrive_expect_tx(bar_a, bytes);
    bulk_g2s(smem_addr(rows_smem), latent + row0 * row_bytes, bytes, bar_a);
  }
  // Every writing lane sees the batch land itself before reading it out.
  const bool landed = slot >= 0 && mbar_wait_bounded(bar_a, 0, &abort_flag, status,
                                                     MLA_DEVSTAT_TIMEOUT, kWaitNs);
  if (landed) {
    bulk_s2g(cache + slot * row_bytes, smem_addr(rows_smem) + (uint32_t)lane * row_bytes, (uint32_t)row_bytes);
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  // Lanes that wrote nothing must not leave the copy into shared memory outstanding.
  if (lane == 0 && !(slot >= 0)) mbar_wait_bounded(bar_a, 0, &abort_flag, status, MLA_DEVSTAT_TIMEOUT, kWaitNs);
}

}  // namespace

cudaError_t launch_cache_write(void* cache, int64_t num_slots, int entry_dim, const void* latent,
                               const int64_t* slot_mapping, int64_t num_tokens, int32_t* status,
                               cudaStream_t stream) {
  const int row_bytes = entry_dim * 2;
  if (num_tokens == 0) return cudaSuccess;
  const int rows_per_cta = max(1, min(32, kBatchBytes / row_bytes));
  const int64_t grid = (num_tokens + rows_per_cta - 1) / rows_per_cta;
  if (grid > 0x7fffffff) return cudaErrorInvalidValue;
  const int smem = rows_per_cta * row_bytes;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(cache_write_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  cache_write_kernel<<<(unsigned)grid, 32, smem, stream>>>(static_cast<uint8_t*>(cache), num_slots, row_bytes,
                                                            rows_per_cta, static_cast<const uint8_t*>(latent),
                                                            slot_mapping, num_tokens, status);
  return cudaGetLastError();
}

}  // namespace mla
