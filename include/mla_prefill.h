/*
 * mla_prefill.h -- C ABI of the GB300 (sm_103a) MLA ragged prefill library.
 *
 * The operations follow these pages:
 *   [vLLM-FI]  vLLM API docs, "vllm.v1.attention.backends.mla.prefill.flashinfer":
 *              FlashInferPrefillBackend.finalize_attention_metadata (plan of a
 *              causal ragged problem over the new tokens and of one non-causal
 *              problem per prefix chunk, with head_dim_qk = 128 NoPE + 64 RoPE,
 *              head_dim_vo = 128, explicit sm_scale, window_left,
 *              logits_soft_cap) and FlashInferPrefillImpl.run_prefill_new_tokens /
 *              run_prefill_context_chunk (run(q, k, v, return_lse) -> O, LSE with
 *              LSE laid out (q_len, num_heads)).
 *   [sglang]   sglang issue #3849, "[DeepseekR1] How ragged prefill manage
 *              kv_cache?": prefill attention is MHA with 192-dim Q/K and 128-dim V
 *              while the cache keeps 512 latent + 64 rope per token.
 *   [TVM]      Apache TVM PR #17674, "[KVCache] PagedKVCache refactor, FlashInfer
 *              JIT and MLA integration": sm_scale is always passed explicitly.
 *   [vLLM-V4]  vLLM "vllm/models/deepseek_v4/sparse_mla.py",
 *              _build_c128a_topk_metadata_kernel (decode branch): the paged
 *              slot rule block_table[r, pos / block_size] * block_size +
 *              pos % block_size.
 *
 * Conventions for every entry point:
 *   - Return value: MLA_OK (0) or a negative MLA_ERR_* code; nothing aborts,
 *     throws or prints.  mla_error_string() names a code.
 *   - Tensors are caller-owned, contiguous, row-major device memory (bf16 as
 *     raw 16-bit storage, fp32 LSE).  Device pointers must be 16-byte aligned
 *     (MLA_ERR_INVALID_ARG otherwise).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device work is enqueued asynchronously on it; argument
 *     checks happen on the host before anything is enqueued, so an error
 *     return means nothing was launched.
 *   - Only the plan call allocates (its own device workspace).  The run,
 *     gather, up-projection and merge calls allocate nothing.
 *   - Device-side problems (a block id outside the cache, a pipeline wait
 *     that timed out) never fault the GPU: the kernel skips the access,
 *     records a flag in a status word and returns.
 */
#ifndef MLA_PREFILL_H_
#define MLA_PREFILL_H_

#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MLA_OK                  0
#define MLA_ERR_INVALID_ARG    -1   /* null/misaligned pointer, bad scalar   */
#define MLA_ERR_SHAPE          -2   /* indptr not monotone, sizes disagree   */
#define MLA_ERR_UNSUPPORTED    -3   /* head dims other than 192/128, etc.    */
#define MLA_ERR_CUDA           -4   /* a CUDA runtime/driver call failed     */
#define MLA_ERR_DEVICE_TIMEOUT -5   /* a kernel pipeline wait gave up        */
#define MLA_ERR_DEVICE_BOUNDS  -6   /* a kernel met an out-of-range index    */

/* bits a kernel may set in a device status word */
#define MLA_DEVSTAT_TIMEOUT    0x1
#define MLA_DEVSTAT_BAD_INDEX  0x2

/* Name of a status code ("ok", "invalid argument", ...).  Never NULL. */
MLA_API const char* mla_error_string(int status);

/* ABI version, currently 1. */
MLA_API int mla_abi_version(void);

/* ======================================================================
 * Ragged prefill attention: plan once per batch, run once per layer.
 * [vLLM-FI] finalize_attention_metadata / run_prefill_*; [TVM] sm_scale.
 * ====================================================================== */
typedef struct mla_plan* mla_plan_t;

/*
 * Plan a ragged prefill problem.
 *   qo_indptr, kv_indptr : HOST int32 arrays of batch+1 prefix sums
 *       (qo_indptr[0] = kv_indptr[0] = 0, non-decreasing).  Request r owns
 *       query rows [qo_indptr[r], qo_indptr[r+1]) and key rows
 *       [kv_indptr[r], kv_indptr[r+1]).
 *   num_heads            : query heads = KV heads (MHA), >= 1.
 *   head_dim_qk          : must be 192 (128 NoPE + 64 RoPE), else MLA_ERR_UNSUPPORTED.
 *   head_dim_vo          : must be 128, else MLA_ERR_UNSUPPORTED.
 *   causal               : nonzero = causal, aligned bottom-right (query row i
 *       of a request sits at key position i + Lkv - Lq).
 *   sm_scale             : logits are sm_scale * q.k (finite and > 0, required).
 *   window_left          : -1 = none; w >= 0 keeps keys with position
 *       >= i + Lkv - Lq - w.  Values below -1 are invalid.
 *   logits_soft_cap      : <= 0 = none; c > 0 replaces a logit x by
 *       c * tanh(x / c) (after sm_scale).
 *   stream               : the plan's work list is uploaded asynchronously
 *       on this stream; runs on other streams must be ordered after it.
 * On success *out owns a device workspace (work list + status word) until
 * mla_plan_destroy.  Rows that see no key produce O = 0 and LSE = -inf.
 * A kernel pipeline wait gives up after 2 s (status MLA_ERR_DEVICE_TIMEOUT).  Test
 * mode: if the environment variable MLA_TEST_FORCE_TIMEOUT_NS holds a value in
 * 1 .. 2000000000 when the plan is made, its runs make one wait that nothing
 * satisfies, with that limit, so that tests can drive the time-out path (the kernel
 * gives up, records MLA_DEVSTAT_TIMEOUT, releases its resources and returns).
 */
MLA_API int mla_prefill_plan(mla_plan_t* out, const int32_t* qo_indptr, const int32_t* kv_indptr,
                     int batch, int num_heads, int head_dim_qk, int head_dim_vo, int causal,
                     float sm_scale, int window_left, float logits_soft_cap, void* stream);

/*
 * Run a planned problem ("NHD" ragged layout).
 *   q   : bf16 [qo_indptr[batch], num_heads, 192]
 *   k   : bf16 [kv_indptr[batch], num_heads, 192]
 *   v   : bf16 [kv_indptr[batch], num_heads, 128]
 *   o   : bf16 [qo_indptr[batch], num_heads, 128]            (written)
 *   lse : fp32 [qo_indptr[batch], num_heads], natural log, or NULL to skip.
 * Allocates nothing and does not synchronise; safe to capture in a CUDA
 * graph.  Kernel-side failures are reported by mla_prefill_status.
 */
MLA_API int mla_prefill_run(mla_plan_t plan, const void* q, const void* k, const void* v, void* o,
                    float* lse, void* stream);

/*
 * Run a planned problem and merge its result into a partial state, in one
 * kernel: the chunked-prefix step of [vLLM-FI] (run_prefill_context_chunk
 * returns LSE so that chunk results merge with the new tokens' result).
 * Same arguments, layout and checks as mla_prefill_run, except:
 *   o   : bf16 [qo_indptr[batch], num_heads, 128], read and written: on entry a
 *         partial attention output over other keys, on return the merge
 *   lse : fp32 [qo_indptr[batch], num_heads], natural log, read and written;
 *         required (NULL gives MLA_ERR_INVALID_ARG)
 * With (O_a, la) the entry state and (O_b, lb) this attention, every row gets
 * the mla_merge_state result: O = (e^{la-m} O_a + e^{lb-m} O_b) / (e^{la-m} +
 * e^{lb-m}), LSE = m + ln(...), m = max(la, lb).  A side with LSE = -inf
 * contributes nothing (its O is not read): rows that see no key here keep
 * their entry state, and rows with LSE = -inf on both sides get O = 0.  O_b is
 * rounded to bf16 before the merge, as it would be if it were written out and
 * merged by mla_merge_state.
 */
MLA_API int mla_prefill_run_merge(mla_plan_t plan, const void* q, const void* k, const void* v, void* o,
                                  float* lse, void* stream);

/*
 * Run a planned problem with K given in two parts: the per-head NoPE columns and ONE RoPE
 * row per key shared by every head.  [sglang]: the cache keeps a single 64-dim rope per
 * token, so after decompression K = [K_nope(h) || rope] repeats the same 64 values in
 * every head; [vLLM-FI]: the latent cache has one KV head.  Reading the rope once per key
 * instead of once per (key, head) saves the decompression 20 % of its output and the
 * attention a third of its K bytes.  Same result, bit for bit, as mla_prefill_run /
 * mla_prefill_run_merge on the concatenated K.
 *   k_nope      : bf16 [kv_indptr[batch], num_heads, 128]
 *   k_rope      : bf16, row t (key t) at k_rope + t * rope_stride, 64 values; rope_stride
 *                 (elements) >= 64 and a multiple of 8, k_rope 16-byte aligned.  E.g. the
 *                 rope columns of a gathered latent [T, 576]: k_rope = latent + 512,
 *                 rope_stride = 576.
 *   merge       : 0 = write O/LSE (as mla_prefill_run), 1 = merge into o/lse (as
 *                 mla_prefill_run_merge; lse required)
 * Other arguments as for mla_prefill_run.
 */
MLA_API int mla_prefill_run_shared_rope(mla_plan_t plan, const void* q, const void* k_nope, const void* k_rope,
                                        int64_t rope_stride, const void* v, void* o, float* lse, int merge,
                                        void* stream);

/*
 * Read and clear the plan's device status word (a blocking device-to-host
 * copy; call after the run's stream has completed).  Returns MLA_OK,
 * MLA_ERR_DEVICE_TIMEOUT or MLA_ERR_CUDA.
 */
MLA_API int mla_prefill_status(mla_plan_t plan);

/*
 * Release the plan and its workspace.  Does not synchronise: the workspace goes back
 * to the device's stream-ordered memory pool once the plan's last use has completed
 * (the plan upload, and the last run enqueued on a stream that was not being
 * captured).  A plan whose run was captured into a CUDA graph must outlive every
 * launch of that graph.  NULL is a no-op.
 */
MLA_API int mla_plan_destroy(mla_plan_t plan);

/* Plan facts: which = 0 work units, 1 CTAs launched (CTA pairs when 6 is 1), 2 total
 * query rows, 3 total key rows, 4 allowed (query, key) pairs summed over requests (one
 * head), 5 KV tiles summed over units, 6 whether units of 256 query rows run on clusters
 * of two CTAs (1) or units of 128 rows on single CTAs (0).  Single CTAs unless the
 * environment variable MLA_PLAN_CTA_PAIRS is "1" when the plan is made. */
MLA_API int mla_plan_query(mla_plan_t plan, int which, int64_t* value);

/*
 * Host-only planner (no CUDA call), for inspection and tests.  Same
 * arguments as mla_prefill_plan plus `num_ctas` (the persistent grid).
 * Writes at most `capacity` units as 8 int32 each:
 *   {head, q_row0, q_rows, q_pos0, kv_row0, kv_len, diag, kv_tile_lo | kv_tile_hi << 16}
 * in execution order, and cta_offsets[num_ctas+1] (CTA c runs units
 * [cta_offsets[c], cta_offsets[c+1])).  *num_units receives the count even
 * when capacity is too small (then MLA_ERR_SHAPE is returned).  With
 * MLA_PLAN_CTA_PAIRS = "1" units are 256 query rows (q_rows up to 256) and num_ctas
 * counts CTA pairs, as mla_prefill_plan then plans.
 */
MLA_API int mla_plan_units_host(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch,
                        int num_heads, int causal, int window_left, int num_ctas,
                        int32_t* units, int64_t capacity, int32_t* cta_offsets,
                        int64_t* num_units);

/* ======================================================================
 * Paged latent gather.  [vLLM-V4] slot rule; [sglang] 512 latent + 64 rope
 * per cache row; [vLLM-FI] chunk i's kv_indptr = chunked_context.cu_seq_lens[i].
 * ====================================================================== */
/*
 *   cache        : bf16 [num_blocks, block_size, entry_dim] (entry_dim % 8 == 0; 576 for MLA)
 *   block_table  : DEVICE int32 [batch, max_blocks_per_req]
 *   cu_seq_lens  : DEVICE int32 [batch+1], this chunk's kv_indptr
 *   chunk_starts : DEVICE int32 [batch], first prefix position of the chunk per request
 *   total_tokens : host copy of cu_seq_lens[batch] (rows of `out`)
 *   out          : bf16 [total_tokens, entry_dim]; row cu_seq_lens[r] + t is
 *                  position chunk_starts[r] + t of request r
 *   status       : DEVICE int32 word or NULL; MLA_DEVSTAT_BAD_INDEX is OR-ed in when a
 *                  row's block id is outside [0, num_blocks) or its table slot is past
 *                  max_blocks_per_req (that row is written as zeros).
 * Bit-exact copy; allocates nothing.
 */
MLA_API int mla_gather_latent(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                      const int32_t* block_table, int max_blocks_per_req,
                      const int32_t* cu_seq_lens, const int32_t* chunk_starts, int batch,
                      int64_t total_tokens, void* out, int32_t* status, void* stream);

/* ======================================================================
 * Paged gather of an fp8 latent cache, dequantized.  [vLLM-V4] cache dtype
 * fp8_ds_mla: an fp8 NoPE part, 128 bytes of bf16 RoPE and 8 scale bytes per
 * token; here for [sglang]'s 512 latent + 64 rope.
 * ====================================================================== */
/*
 *   cache        : uint8 [num_blocks, block_size, entry_bytes], entry_bytes must be 648
 *                  (MLA_ERR_UNSUPPORTED otherwise): bytes [0, 512) the latent as float8
 *                  e4m3 (no infinities; 0x7F/0xFF are NaN), [512, 640) the rope as 64 bf16,
 *                  [640, 648) scale bytes, scale g = 2^(byte_g - 127) covering latent
 *                  values [64 g, 64 g + 64) (byte 255 is NaN).  8-byte aligned.
 *   block_table, max_blocks_per_req, cu_seq_lens, chunk_starts, batch, total_tokens,
 *   status       : as for mla_gather_latent.
 *   out          : bf16 [total_tokens, 576]: value i < 512 is e4m3(byte_i) * scale_(i/64)
 *                  rounded to bf16 (round to nearest even; exact unless below bf16's
 *                  normal range or above its largest value), values 512 .. 575 the rope
 *                  bits copied.  Rows whose block is unknown are zeros (flagged).
 * Allocates nothing.
 */
MLA_API int mla_gather_latent_fp8(const void* cache, int64_t num_blocks, int block_size, int entry_bytes,
                                  const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                                  const int32_t* chunk_starts, int batch, int64_t total_tokens, void* out,
                                  int32_t* status, void* stream);

/* ======================================================================
 * Paged latent cache write.  [sglang] ragged prefill saves the new tokens'
 * compressed rows (512 latent + 64 rope) in the cache before attention;
 * [vLLM-V4] a token's flat slot is block * block_size + offset, and a
 * negative slot marks a padding token.
 * ====================================================================== */
/*
 *   cache        : bf16 [num_blocks, block_size, entry_dim] (entry_dim % 8 == 0, at most
 *                  102400; 576 for MLA), written in place
 *   latent       : bf16 [num_tokens, entry_dim], the new tokens' rows
 *   slot_mapping : DEVICE int64 [num_tokens]; row t goes to flat slot slot_mapping[t]
 *                  (block = slot / block_size, offset = slot % block_size); a negative
 *                  slot writes nothing; a slot >= num_blocks * block_size writes nothing
 *                  and ORs MLA_DEVSTAT_BAD_INDEX into status
 *   status       : DEVICE int32 word or NULL
 * Bit-exact copy; allocates nothing.  If two tokens name the same slot, the row left
 * there is one of theirs (unspecified which).  Pointers: cache and latent 16-byte
 * aligned, slot_mapping 8-byte aligned.
 */
MLA_API int mla_cache_write(void* cache, int64_t num_blocks, int block_size, int entry_dim,
                            const void* latent, const int64_t* slot_mapping, int64_t num_tokens,
                            int32_t* status, void* stream);

/* ======================================================================
 * Latent up-projection.  [sglang] 512 latent + 64 rope -> MHA K (192) / V (128).
 * ====================================================================== */
/*
 *   latent : bf16 [num_tokens, 576] (512 latent then 64 rope), e.g. gather output
 *   w_kvb  : bf16 [512, num_heads * 256]; columns h*256 + [0,128) give head h's
 *            K_nope, h*256 + [128,256) its V
 *   k_out  : bf16 [num_tokens, num_heads, 192] = [latent[:, :512] @ W_knope(h) || rope]
 *   v_out  : bf16 [num_tokens, num_heads, 128] = latent[:, :512] @ W_v(h)
 *   status : DEVICE int32 word or NULL; MLA_DEVSTAT_TIMEOUT is OR-ed in if a pipeline
 *            wait of the kernel gave up (outputs are then incomplete).
 * fp32 accumulation on tensor cores, one rounding to bf16.  Allocates nothing.
 */
MLA_API int mla_up_proj(const void* latent, const void* w_kvb, int64_t num_tokens, int num_heads,
                void* k_out, void* v_out, int32_t* status, void* stream);

/* ======================================================================
 * Paged up-projection: gather + up-projection in one kernel.  [sglang] asks
 * whether the compressed kv is decompressed every time; this decompresses a
 * prefix chunk straight out of the paged cache ([vLLM-V4] slot rule), without
 * a gathered latent buffer.
 * ====================================================================== */
/*
 * Same result, bit for bit, as mla_gather_latent into a [total_tokens, 576]
 * buffer followed by mla_up_proj on it:
 *   cache        : bf16 [num_blocks, block_size, entry_dim]; entry_dim must be 576
 *                  (MLA_ERR_UNSUPPORTED otherwise); num_blocks * block_size < 2^31 - 1
 *   block_table, max_blocks_per_req, cu_seq_lens, chunk_starts, batch, total_tokens :
 *                  as for mla_gather_latent (DEVICE int32 tables; chunk row
 *                  cu_seq_lens[r] + t is prefix position chunk_starts[r] + t of request r)
 *   w_kvb        : bf16 [512, num_heads * 256], as for mla_up_proj
 *   k_out, v_out : bf16 [total_tokens, num_heads, 192] / [total_tokens, num_heads, 128]
 *   status       : DEVICE int32 word or NULL; MLA_DEVSTAT_BAD_INDEX is OR-ed in when a
 *                  row's block is unknown (that row's latent is taken as zeros, so its
 *                  K_nope, V and rope are zero); MLA_DEVSTAT_TIMEOUT as for mla_up_proj.
 * Allocates nothing.
 */
MLA_API int mla_up_proj_paged(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                              const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                              const int32_t* chunk_starts, int batch, int64_t total_tokens, const void* w_kvb,
                              int num_heads, void* k_out, void* v_out, int32_t* status, void* stream);

/*
 * mla_up_proj_paged with K in the two parts mla_prefill_run_shared_rope takes:
 *   k_nope_out : bf16 [total_tokens, num_heads, 128] = the K_nope of mla_up_proj_paged's K
 *   rope_out   : bf16 [total_tokens, 64] = each row's rope (K's last 64 columns, the same in
 *                every head), written once per token; 16-byte aligned, required
 *   v_out      : as for mla_up_proj_paged
 * Bit-identical to the corresponding parts of mla_up_proj_paged's output.
 */
MLA_API int mla_up_proj_paged_split(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                                    const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                                    const int32_t* chunk_starts, int batch, int64_t total_tokens, const void* w_kvb,
                                    int num_heads, void* k_nope_out, void* v_out, void* rope_out, int32_t* status,
                                    void* stream);

/* ======================================================================
 * Absorbed-weight paged prefill.  [sglang] prefill with a cached prefix runs
 * forward_absorb: every head attends to the compressed cache rows themselves
 * (multi-query attention, one KV head: Dqk = 576 = 512 latent + 64 rope, Dv =
 * 512), with W_UK folded into the query; [TVM] sm_scale is explicit because
 * absorption changes the effective head dim; [vLLM-V4] slot rule for the
 * cache positions.
 * ====================================================================== */
/*
 * Plan (host work list + device workspace) for a batch:
 *   qo_indptr : HOST int32 [batch+1], new query rows per request (qo[0] = 0)
 *   kv_lens   : HOST int32 [batch], keys per request: its cache positions
 *               0 .. kv_lens[r]-1 (the new tokens' rows must already be in the
 *               cache); query row i of a request of q_len rows sits at position
 *               kv_len - q_len + i (bottom-right causal alignment; rows with no
 *               allowed key get O = 0, LSE = -inf)
 *   block_size: cache block size (any value >= 1)
 *   causal, sm_scale (> 0), logits_soft_cap (<= 0: none) as for mla_prefill_plan
 * The plan object is an mla_plan_t: mla_prefill_status, mla_plan_query and
 * mla_plan_destroy apply to it; mla_prefill_run and its variants reject it
 * (MLA_ERR_INVALID_ARG), as mla_absorbed_run rejects an MHA plan.
 */
MLA_API int mla_absorbed_plan(mla_plan_t* out, const int32_t* qo_indptr, const int32_t* kv_lens, int batch,
                              int num_heads, int block_size, int causal, float sm_scale, float logits_soft_cap,
                              void* stream);

/*
 *   q_abs      : bf16 [total_q, num_heads, 576] (W_UK(h) q_nope(h) || q_rope(h))
 *   cache      : bf16 [num_blocks, block_size, 576] (512 latent + 64 rope per slot)
 *   block_table: DEVICE int32 [batch, max_blocks_per_req]; max_blocks_per_req must
 *                cover the longest request (MLA_ERR_SHAPE otherwise)
 *   o_lat      : bf16 [total_q, num_heads, 512] (O_lat; the MHA output of head h
 *                is O_lat(h) W_UV(h))
 *   lse        : fp32 [total_q, num_heads] natural-log LSE, or NULL
 * A block id outside [0, num_blocks) reads as a zero row and sets
 * MLA_DEVSTAT_BAD_INDEX in the plan's status word (mla_prefill_status then
 * returns MLA_ERR_DEVICE_BOUNDS).  Allocates nothing.
 */
MLA_API int mla_absorbed_run(mla_plan_t plan, const void* q_abs, const void* cache, int64_t num_blocks,
                             const int32_t* block_table, int max_blocks_per_req, void* o_lat, float* lse,
                             void* stream);

/* ======================================================================
 * LSE merge of two partial attention states.  [vLLM-FI]
 * run_prefill_context_chunk always returns LSE so chunk results can merge.
 * ====================================================================== */
/*
 *   o_a, o_b : bf16 [rows, num_heads, head_dim]; lse_a, lse_b : fp32 [rows, num_heads]
 *   o_out    : bf16 [rows, num_heads, head_dim]; lse_out : fp32 [rows, num_heads] or NULL
 *   head_dim : a power of two in [8, 256] (128 for MLA)
 * O = (e^{la-m} Oa + e^{lb-m} Ob) / (e^{la-m} + e^{lb-m}), LSE = m + ln(...), m = max(la, lb);
 * a side with LSE = -inf contributes nothing; both -inf gives O = 0, LSE = -inf.
 * o_out may alias o_a (and lse_out lse_a): in-place accumulation is supported.
 */
MLA_API int mla_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                    void* o_out, float* lse_out, int64_t rows, int num_heads, int head_dim,
                    void* stream);

/* ======================================================================
 * Allocation-free prefill (the pages have no counterpart; this exists for
 * callers that cannot allocate device memory).
 * ====================================================================== */
/*
 * Plan and run one ragged prefill in a single call without allocating device
 * memory.  For callers that cannot call cudaMalloc: a serving engine whose
 * memory pool already owns the device's HBM, a host that forbids allocation
 * after start-up, or code that must not risk the synchronisation an
 * allocation or free can bring.  Arguments are those of mla_prefill_plan
 * followed by those of mla_prefill_run (same meaning, layout and checks),
 * plus:
 *   status : DEVICE int32 word or NULL.  When given, kernel-side problems are
 *            OR-ed into it (MLA_DEVSTAT_*; the caller clears it); when NULL
 *            they go to a word inside the library's scratch array that each
 *            call clears and nobody reads.
 * The work list lives in a fixed device array compiled into the library
 * (about 2 MiB, held by every GPU that loads the library until exit).  Limit:
 * at most 65536 work units, i.e. sum over requests of ceil(Lq / 128) times
 * num_heads; larger problems return MLA_ERR_UNSUPPORTED before any device
 * work.  The first call on a device looks the array's address up (once per
 * device).  Every call reuses the same
 * array, so calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller.  Planning happens on
 * the host at every call.
 */
MLA_API int mla_prefill_run_noalloc(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch,
                                    int num_heads, int head_dim_qk, int head_dim_vo, int causal,
                                    float sm_scale, int window_left, float logits_soft_cap,
                                    const void* q, const void* k, const void* v, void* o, float* lse,
                                    int32_t* status, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif
#endif /* MLA_PREFILL_H_ */
