// Declarations shared between the C-ABI layer and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "../../include/mla_prefill.h"
#include "planner.h"

namespace mla {

// ---- prefill attention -------------------------------------------------------
struct PrefillParams {
  const Unit* units;          // work list, grouped per CTA
  const int32_t* cta_offsets; // [grid + 1]
  int* status;                // device status word (MLA_DEVSTAT_* bits)
  __nv_bfloat16* o;           // [total_q, H, 128]
  float* lse;                 // [total_q, H] or null (never null when merge is set)
  int merge;                  // o/lse hold a partial state on entry: write its LSE merge
                              // with this attention instead of the attention alone
  int num_heads;
  int o_align32;              // o is 32-byte aligned: the epilogue uses 32-byte stores
  int causal;
  int window_left;
  int has_cap;
  float scale_log2;           // sm_scale * log2(e)            (no soft cap)
  float cap_log2;             // logits_soft_cap * log2(e)     (soft cap)
  float x_to_cap;             // sm_scale / logits_soft_cap    (soft cap)
};

int prefill_smem_bytes();
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, int num_ctas, cudaStream_t stream);

// ---- tensor maps (tma.cpp) ---------------------------------------------------
// bf16 tensor of rank 2 or 3 (dims innermost first, strides in bytes for dims 1..),
// 128-byte swizzle, zero fill out of bounds.  Returns 0 or MLA_ERR_*.
int make_tensor_map_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides_bytes, const uint32_t* box);

// ---- gather / up-projection / merge -----------------------------------------
cudaError_t launch_gather(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                          const int32_t* block_table, int max_blocks_per_req,
                          const int32_t* cu_seq_lens, const int32_t* chunk_starts, int batch,
                          int64_t total_tokens, void* out, int32_t* status, cudaStream_t stream);

cudaError_t launch_cache_write(void* cache, int64_t num_slots, int entry_dim, const void* latent,
                               const int64_t* slot_mapping, int64_t num_tokens, int32_t* status,
                               cudaStream_t stream);

int up_proj_smem_bytes();
cudaError_t launch_up_proj(const CUtensorMap& ta, const CUtensorMap& tb, const void* latent,
                           int64_t num_tokens, int num_heads, void* k_out, void* v_out,
                           int32_t* status, cudaStream_t stream);

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                         void* o_out, float* lse_out, int64_t rows, int num_heads, int head_dim,
                         cudaStream_t stream);

int device_sm_count();

}  // namespace mla
