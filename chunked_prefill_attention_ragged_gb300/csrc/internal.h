// Declarations shared between the C-ABI layer and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <mutex>

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
  float cap_ex2_scale;        // 2 * log2(e) * sm_scale / logits_soft_cap: e^(2y) = 2^(x * this)
  uint64_t wait_limit_ns;     // a pipeline wait gives up after this long (default 2 s)
  int force_timeout;          // test mode: one wait that nothing satisfies (see below)
  int shared_rope;            // K's RoPE columns come from one [kv rows, 64] tensor (map tm_r)
  int pair;                   // units of 256 rows run by CTA pairs (clusters of two); the K
                              // and rope maps then have 64-row boxes
};

// Time-out test mode.  When the environment variable MLA_TEST_FORCE_TIMEOUT_NS holds a
// value in 1 .. 2e9 at plan time, the plan's runs make one pipeline wait on a barrier
// that nothing arrives on, with that value as every wait's limit: the wait gives up,
// the kernel records MLA_DEVSTAT_TIMEOUT, drains its own copies and MMAs, frees TMEM
// and returns.  Nothing faults or hangs; it lets tests drive the time-out path.
// Returns 0 when the mode is off, else the limit in ns.
uint64_t forced_timeout_ns();
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // the normal limit of a pipeline wait

int prefill_smem_bytes();
// tr: the shared RoPE tensor's map when p.shared_rope is set (any valid map otherwise).
// num_slots: CTAs, or CTA pairs when p.pair is set (the plan's cta_offsets has num_slots + 1
// entries).
cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tr, const PrefillParams& p, int num_slots, cudaStream_t stream);

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

cudaError_t launch_gather_fp8(const void* cache, int64_t num_blocks, int block_size, const int32_t* block_table,
                              int max_blocks_per_req, const int32_t* cu_seq_lens, const int32_t* chunk_starts,
                              int batch, int64_t total_tokens, void* out, int32_t* status, cudaStream_t stream);

cudaError_t launch_cache_write(void* cache, int64_t num_slots, int entry_dim, const void* latent,
                               const int64_t* slot_mapping, int64_t num_tokens, int32_t* status,
                               cudaStream_t stream);

int up_proj_smem_bytes();
cudaError_t launch_up_proj(const CUtensorMap& ta, const CUtensorMap& tb, const void* latent,
                           int64_t num_tokens, int num_heads, void* k_out, void* v_out,
                           int32_t* status, cudaStream_t stream);

cudaError_t launch_up_proj_paged(const CUtensorMap& ta, const CUtensorMap& tb, const void* cache, int64_t num_blocks,
                                 int block_size, const int32_t* block_table, int max_blocks_per_req,
                                 const int32_t* cu_seq_lens, const int32_t* chunk_starts, int batch,
                                 int64_t total_tokens, int num_heads, void* k_out, void* v_out, void* rope_out,
                                 int32_t* status, cudaStream_t stream);

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                         void* o_out, float* lse_out, int64_t rows, int num_heads, int head_dim,
                         cudaStream_t stream);

int device_sm_count();


struct AbsorbedParams {
  const AbsUnit* units;
  const int32_t* block_table;   // [batch, max_blocks]
  int max_blocks, block_size;
  int64_t num_blocks;
  int32_t oob_row;              // a row coordinate past the cache: the copy fills it with zeros
  int piece_rows;               // rows of one tile load of the block map (0: gather4 only)
  int grouped;                  // 64-row pieces by runs of panels (the three-dimensional map)
  __nv_bfloat16* o;             // [total_q, H, 512]
  float* lse;                   // [total_q, H] or null
  int* status;
  int num_heads, causal, has_cap, force_timeout;
  float scale_log2, cap_log2, cap_ex2_scale;
  uint64_t wait_limit_ns;
};

// The absorbed prefill kernel, one CTA per unit.  tq: q_abs as [total_q * H, 576] rows, box
// {64, 128}; tc: the cache as [num_blocks * block_size, 576] rows, box {64, 1} (gather4);
// tb: the same rows with box {64, piece_rows} (any valid map when piece_rows is 0); t4: the
// rows as {64 columns, rows, 9 column groups} (strides 1152 and 128 bytes), box {64, 64, 4}
// (any valid map when grouped is 0).
cudaError_t launch_absorbed(const CUtensorMap& tq, const CUtensorMap& tc, const CUtensorMap& tb,
                            const CUtensorMap& t4, const AbsorbedParams& p, int num_units, cudaStream_t stream);

// MLA_PLAN_CTA_PAIRS: 1 when "1" (plan prefills on CTA pairs), 0 when "0", -1 otherwise.
int cta_pair_mode();

// How many clusters of two prefill CTAs the current device runs at once (0 on error).
int prefill_max_pairs();

// Runs a set-up step (kernel attributes, symbol lookups) once per device, from any
// number of host threads: the first caller on a device runs it under a lock, later
// callers see the recorded success.  A failed step is retried by the next call.
class PerDeviceOnce {
 public:
  static constexpr int kMaxDevices = 64;
  template <class F>
  cudaError_t run(F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mutex_);
    if (done_[dev]) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess) done_[dev] = true;
    return e;
  }

 private:
  std::mutex mutex_;
  bool done_[kMaxDevices] = {};
};

}  // namespace mla
