// C ABI of the library (declared in include/mla_prefill.h): argument checks, the
// plan object and its device workspace, tensor maps, kernel launches.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "internal.h"

using namespace mla;

struct mla_plan {
  int device = 0;
  int batch = 0, num_heads = 0, causal = 0, window_left = -1;
  float sm_scale = 0.f, soft_cap = 0.f;
  uint64_t forced_timeout_ns = 0;   // test mode (see forced_timeout_ns())
  int64_t total_q = 0, total_kv = 0;
  PlanResult plan;
  int num_ctas = 0;              // CTAs, or CTA pairs when pair is set
  int pair = 0;                  // units of 256 rows, each run by a cluster of two CTAs
  int kind = 0;                  // 0: MHA prefill (mla_prefill_plan); 1: absorbed (mla_absorbed_plan)
  int block_size = 0, max_kv_blocks = 0;   // absorbed: cache block size, blocks the longest request needs
  std::vector<AbsUnit> aunits;   // absorbed: the work units (one CTA each)
  void* workspace = nullptr;     // units | cta offsets | status word (stream-ordered allocation)
  cudaEvent_t last_use = nullptr;  // recorded after the upload and after every uncaptured run
  Unit* d_units = nullptr;       // MHA units, or the absorbed units (AbsUnit, same size)
  int32_t* d_offsets = nullptr;
  int* d_status = nullptr;
};

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// A non-blocking stream per device on which destroyed plans hand their workspace back,
// in stream order after their last use, so that freeing never waits for the device.
cudaStream_t release_stream(cudaError_t* err) {
  static cudaStream_t streams[PerDeviceOnce::kMaxDevices] = {};
  static PerDeviceOnce created;
  *err = created.run([] {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return cudaStreamCreateWithFlags(&streams[dev], cudaStreamNonBlocking);
  });
  int dev = 0;
  if (*err == cudaSuccess) *err = cudaGetDevice(&dev);
  return *err == cudaSuccess ? streams[dev] : nullptr;
}

bool stream_capturing(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &st) != cudaSuccess) return true;   // unknown: do not record
  return st != cudaStreamCaptureStatusNone;
}

void free_plan_storage(mla_plan* p) {
  if (p->last_use) cudaEventDestroy(p->last_use);
  delete p;
}

// The plan's device workspace (stream-ordered): work units, CTA offsets, status word; the
// uploads are ordered on `s` and recorded as the plan's first use.  Frees the plan on error.
int upload_plan(mla_plan* p, const void* units, size_t unit_bytes, const int32_t* offsets, size_t num_offsets,
                cudaStream_t s) {
  const size_t units_bytes = round_up(std::max<size_t>(1, unit_bytes), 256);
  const size_t offs_bytes = round_up(std::max<size_t>(1, num_offsets) * sizeof(int32_t), 256);
  if (cudaEventCreateWithFlags(&p->last_use, cudaEventDisableTiming) != cudaSuccess) {
    p->last_use = nullptr;
    free_plan_storage(p);
    return MLA_ERR_CUDA;
  }
  if (cudaMallocAsync(&p->workspace, units_bytes + offs_bytes + 256, s) != cudaSuccess) {
    free_plan_storage(p);
    return MLA_ERR_CUDA;
  }
  char* ws = static_cast<char*>(p->workspace);
  p->d_units = reinterpret_cast<Unit*>(ws);
  p->d_offsets = reinterpret_cast<int32_t*>(ws + units_bytes);
  p->d_status = reinterpret_cast<int*>(ws + units_bytes + offs_bytes);
  cudaError_t e = cudaSuccess;
  if (unit_bytes) e = cudaMemcpyAsync(p->d_units, units, unit_bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess && num_offsets)
    e = cudaMemcpyAsync(p->d_offsets, offsets, num_offsets * sizeof(int32_t), cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(p->d_status, 0, sizeof(int), s);
  if (e == cudaSuccess) e = cudaEventRecord(p->last_use, s);
  if (e != cudaSuccess) {
    cudaStreamSynchronize(s);
    cudaFreeAsync(p->workspace, s);
    free_plan_storage(p);
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

}  // namespace

extern "C" {

const char* mla_error_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_SHAPE: return "inconsistent shapes or indptr";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "device index out of range";
    default: return "unknown status";
  }
}

int mla_abi_version(void) { return 1; }

int mla_plan_units_host(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch, int num_heads,
                        int causal, int window_left, int num_ctas, int32_t* units, int64_t capacity,
                        int32_t* cta_offsets, int64_t* num_units) {
  if (!num_units || !cta_offsets || (capacity > 0 && !units) || num_ctas < 1) return MLA_ERR_INVALID_ARG;
  PlanResult pr;
  const int rows = cta_pair_mode() == 1 ? 2 * kTileM : kTileM;
  const int rc = build_plan(qo_indptr, kv_indptr, batch, num_heads, causal != 0, window_left, num_ctas, &pr, rows);
  if (rc != MLA_OK) return rc;
  *num_units = (int64_t)pr.units.size();
  if ((int64_t)pr.units.size() > capacity) return MLA_ERR_SHAPE;
  if (!pr.units.empty()) std::memcpy(units, pr.units.data(), pr.units.size() * sizeof(Unit));
  const int used = (int)pr.cta_offsets.size() - 1;
  for (int c = 0; c <= num_ctas; ++c)
    cta_offsets[c] = c <= used ? pr.cta_offsets[c] : (int32_t)pr.units.size();
  return MLA_OK;
}

int mla_prefill_plan(mla_plan_t* out, const int32_t* qo_indptr, const int32_t* kv_indptr, int batch,
                     int num_heads, int head_dim_qk, int head_dim_vo, int causal, float sm_scale,
                     int window_left, float logits_soft_cap, void* stream) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!qo_indptr || !kv_indptr || batch < 0 || num_heads < 1 || num_heads > 65535) return MLA_ERR_INVALID_ARG;
  if (head_dim_qk != 192 || head_dim_vo != 128) return MLA_ERR_UNSUPPORTED;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f) || !std::isfinite(logits_soft_cap) || window_left < -1)
    return MLA_ERR_INVALID_ARG;
  // Shape checks first (host only), so a bad call never touches the device.
  {
    PlanResult probe;
    const int rc = build_plan(qo_indptr, kv_indptr, batch, num_heads, causal != 0, window_left, 1, &probe);
    if (rc != MLA_OK) return rc;
  }
  const int sms = device_sm_count();
  if (sms <= 0) return MLA_ERR_CUDA;

  mla_plan* p = new (std::nothrow) mla_plan();
  if (!p) return MLA_ERR_CUDA;
  int rc = build_plan(qo_indptr, kv_indptr, batch, num_heads, causal != 0, window_left, sms, &p->plan);
  if (rc != MLA_OK) { delete p; return rc; }
  // CTA pairs only on request: on every batch shape measured they ran 3-10% slower than
  // single CTAs (the pair relieves shared-memory bandwidth, but its tiles wait on the same
  // softmax-to-MMA chain and its causal units carry more masked tiles).
  if (cta_pair_mode() == 1) {
    const int max_pairs = prefill_max_pairs();
    if (max_pairs < 1) { delete p; return MLA_ERR_CUDA; }
    rc = build_plan(qo_indptr, kv_indptr, batch, num_heads, causal != 0, window_left, max_pairs, &p->plan,
                    2 * kTileM);
    if (rc != MLA_OK) { delete p; return rc; }
    p->pair = 1;
  }
  cudaGetDevice(&p->device);
  p->batch = batch;
  p->num_heads = num_heads;
  p->causal = causal != 0;
  p->window_left = window_left;
  p->sm_scale = sm_scale;
  p->soft_cap = logits_soft_cap > 0.f ? logits_soft_cap : 0.f;
  p->forced_timeout_ns = forced_timeout_ns();
  p->total_q = qo_indptr[batch];
  p->total_kv = kv_indptr[batch];
  p->num_ctas = (int)p->plan.cta_offsets.size() - 1;

  const int rc2 = upload_plan(p, p->plan.units.data(), p->plan.units.size() * sizeof(Unit), p->plan.cta_offsets.data(),
                              p->plan.cta_offsets.size(), as_stream(stream));
  if (rc2 != MLA_OK) return rc2;
  *out = p;
  return MLA_OK;
}

// k_rope == nullptr: K is [kv rows, H, 192].  Otherwise K is given as k = K_nope [kv rows,
// H, 128] and k_rope = the one RoPE row per key, rope_stride elements apart, shared by all
// heads.
static int prefill_run_impl(mla_plan_t p, const void* q, const void* k, const void* k_rope, int64_t rope_stride,
                            const void* v, void* o, float* lse, int merge, void* stream) {
  if (!p || p->kind != 0) return MLA_ERR_INVALID_ARG;
  if (merge && !lse) return MLA_ERR_INVALID_ARG;
  if (p->plan.units.empty()) return MLA_OK;   // no query rows
  if (!q || !o || !aligned16(q) || !aligned16(o) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (p->total_kv > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return MLA_ERR_INVALID_ARG;
  const bool shared_rope = k_rope != nullptr;
  if (shared_rope && (!aligned16(k_rope) || rope_stride < 64 || rope_stride % 8 != 0)) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return MLA_ERR_INVALID_ARG;

  // With no key rows at all no K/V tile is ever loaded; the maps still need a valid base.
  const void* kb = p->total_kv > 0 ? k : q;
  const void* vb = p->total_kv > 0 ? v : q;
  const uint64_t H = (uint64_t)p->num_heads;
  const uint64_t kv_rows = p->total_kv > 0 ? (uint64_t)p->total_kv : 1;
  CUtensorMap tq, tk, tv, tr;
  const uint32_t box[3] = {64, 1, 128};
  // A CTA of a pair loads 64 keys of each K tile.
  const uint32_t krows = p->pair ? 64 : 128;
  const uint32_t kbox[3] = {64, 1, krows};
  {
    const uint64_t dims[3] = {192, H, (uint64_t)p->total_q};
    const uint64_t strides[2] = {192 * 2, H * 192 * 2};
    if (make_tensor_map_bf16(&tq, q, 3, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  {
    const uint64_t kd = shared_rope ? 128 : 192;
    const uint64_t dims[3] = {kd, H, kv_rows};
    const uint64_t strides[2] = {kd * 2, H * kd * 2};
    if (make_tensor_map_bf16(&tk, kb, 3, dims, strides, kbox) != MLA_OK) return MLA_ERR_CUDA;
  }
  if (shared_rope && p->total_kv > 0) {
    const uint64_t dims[2] = {64, kv_rows};
    const uint64_t strides[1] = {(uint64_t)rope_stride * 2};
    const uint32_t rbox[2] = {64, krows};
    if (make_tensor_map_bf16(&tr, k_rope, 2, dims, strides, rbox) != MLA_OK) return MLA_ERR_CUDA;
  } else {
    tr = tk;
  }
  {
    const uint64_t dims[3] = {128, H, kv_rows};
    const uint64_t strides[2] = {128 * 2, H * 128 * 2};
    if (make_tensor_map_bf16(&tv, vb, 3, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  PrefillParams prm;
  prm.units = p->d_units;
  prm.cta_offsets = p->d_offsets;
  prm.status = p->d_status;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  prm.lse = lse;
  prm.merge = merge;
  prm.num_heads = p->num_heads;
  prm.causal = p->causal;
  prm.window_left = p->window_left;
  const float LOG2E = 1.4426950408889634f;
  prm.has_cap = p->soft_cap > 0.f;
  prm.scale_log2 = p->sm_scale * LOG2E;
  prm.cap_log2 = prm.has_cap ? p->soft_cap * LOG2E : 0.f;
  prm.x_to_cap = prm.has_cap ? p->sm_scale / p->soft_cap : 0.f;
  prm.cap_ex2_scale = 2.f * LOG2E * prm.x_to_cap;
  prm.force_timeout = p->forced_timeout_ns != 0;
  prm.wait_limit_ns = prm.force_timeout ? p->forced_timeout_ns : kWaitLimitNs;
  prm.shared_rope = shared_rope && p->total_kv > 0;
  prm.pair = p->pair;
  const cudaStream_t s = as_stream(stream);
  if (launch_prefill(tq, tk, tv, tr, prm, p->num_ctas, s) != cudaSuccess) return MLA_ERR_CUDA;
  // Remember the last use for mla_plan_destroy.  A run captured into a graph is not
  // recorded: the plan must then outlive every launch of that graph.
  if (!stream_capturing(s) && cudaEventRecord(p->last_use, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_prefill_run(mla_plan_t p, const void* q, const void* k, const void* v, void* o, float* lse,
                    void* stream) {
  return prefill_run_impl(p, q, k, nullptr, 0, v, o, lse, 0, stream);
}

int mla_prefill_run_merge(mla_plan_t p, const void* q, const void* k, const void* v, void* o, float* lse,
                          void* stream) {
  return prefill_run_impl(p, q, k, nullptr, 0, v, o, lse, 1, stream);
}

int mla_prefill_run_shared_rope(mla_plan_t p, const void* q, const void* k_nope, const void* k_rope,
                                int64_t rope_stride, const void* v, void* o, float* lse, int merge, void* stream) {
  if (!k_rope && p && p->total_kv > 0) return MLA_ERR_INVALID_ARG;
  return prefill_run_impl(p, q, k_nope, k_rope, rope_stride, v, o, lse, merge != 0, stream);
}

int mla_prefill_status(mla_plan_t p) {
  if (!p) return MLA_ERR_INVALID_ARG;
  int word = 0;
  if (cudaMemcpy(&word, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (word != 0 && cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
  if (word & MLA_DEVSTAT_TIMEOUT) return MLA_ERR_DEVICE_TIMEOUT;
  if (word & MLA_DEVSTAT_BAD_INDEX) return MLA_ERR_DEVICE_BOUNDS;
  return MLA_OK;
}

int mla_plan_destroy(mla_plan_t p) {
  if (!p) return MLA_OK;
  int rc = MLA_OK;
  if (p->workspace) {
    // Free in stream order after the plan's last recorded use, on a library stream of the
    // plan's device: neither the host nor other streams wait.
    int cur = 0;
    const bool have_cur = cudaGetDevice(&cur) == cudaSuccess;
    if (!have_cur || cur != p->device) {
      if (cudaSetDevice(p->device) != cudaSuccess) rc = MLA_ERR_CUDA;
    }
    cudaError_t e = cudaSuccess;
    cudaStream_t rs = rc == MLA_OK ? release_stream(&e) : nullptr;
    if (rc == MLA_OK && e == cudaSuccess) e = cudaStreamWaitEvent(rs, p->last_use, 0);
    if (rc == MLA_OK && e == cudaSuccess) e = cudaFreeAsync(p->workspace, rs);
    if (e != cudaSuccess) rc = MLA_ERR_CUDA;
    if (have_cur && cur != p->device) cudaSetDevice(cur);
  }
  free_plan_storage(p);
  return rc;
}

int mla_absorbed_plan(mla_plan_t* out, const int32_t* qo_indptr, const int32_t* kv_lens, int batch, int num_heads,
                      int block_size, int causal, float sm_scale, float logits_soft_cap, void* stream) {
  if (!out) return MLA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!qo_indptr || !kv_lens || batch < 0 || num_heads < 1 || num_heads > 65535 || block_size < 1)
    return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f) || !std::isfinite(logits_soft_cap)) return MLA_ERR_INVALID_ARG;
  std::vector<AbsUnit> units;
  int64_t allowed = 0;
  const int rc = build_absorbed_units(qo_indptr, kv_lens, batch, num_heads, causal != 0, &units, &allowed);
  if (rc != MLA_OK) return rc;
  int max_kv_blocks = 0;
  for (int r = 0; r < batch; ++r)
    max_kv_blocks = std::max(max_kv_blocks, (int)(((int64_t)kv_lens[r] + block_size - 1) / block_size));
  mla_plan* p = new (std::nothrow) mla_plan();
  if (!p) return MLA_ERR_CUDA;
  cudaGetDevice(&p->device);
  p->kind = 1;
  p->batch = batch;
  p->num_heads = num_heads;
  p->causal = causal != 0;
  p->sm_scale = sm_scale;
  p->soft_cap = logits_soft_cap > 0.f ? logits_soft_cap : 0.f;
  p->forced_timeout_ns = forced_timeout_ns();
  p->total_q = qo_indptr[batch];
  p->block_size = block_size;
  p->max_kv_blocks = max_kv_blocks;
  p->plan.allowed_pairs = allowed;
  for (const AbsUnit& u : units) p->plan.kv_tiles += u.ntiles;
  p->aunits = std::move(units);
  p->num_ctas = (int)p->aunits.size();
  const int rc2 = upload_plan(p, p->aunits.data(), p->aunits.size() * sizeof(AbsUnit), nullptr, 0, as_stream(stream));
  if (rc2 != MLA_OK) return rc2;
  *out = p;
  return MLA_OK;
}

int mla_absorbed_run(mla_plan_t p, const void* q_abs, const void* cache, int64_t num_blocks,
                     const int32_t* block_table, int max_blocks_per_req, void* o_lat, float* lse, void* stream) {
  if (!p || p->kind != 1 || num_blocks < 0 || max_blocks_per_req < 0) return MLA_ERR_INVALID_ARG;
  if (p->aunits.empty()) return MLA_OK;   // no query rows
  if (max_blocks_per_req < p->max_kv_blocks) return MLA_ERR_SHAPE;
  // Slots are TMA row coordinates (int32), and one past the last slot marks a missing row.
  if (num_blocks * (int64_t)p->block_size >= 0x7fffffff) return MLA_ERR_UNSUPPORTED;
  if (!q_abs || !o_lat || !aligned16(q_abs) || !aligned16(o_lat) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return MLA_ERR_INVALID_ARG;
  const bool any_keys = p->max_kv_blocks > 0;
  if (any_keys && (!cache || !block_table || !aligned16(cache) || num_blocks < 1)) return MLA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return MLA_ERR_INVALID_ARG;
  CUtensorMap tq, tc;
  {
    const uint64_t dims[2] = {576, (uint64_t)p->total_q * (uint64_t)p->num_heads};
    const uint64_t strides[1] = {576 * 2};
    const uint32_t box[2] = {64, 128};
    if (make_tensor_map_bf16(&tq, q_abs, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  {
    // With no key at all no cache row is ever fetched; the map still needs a valid base.
    const uint64_t slots = any_keys ? (uint64_t)num_blocks * (uint64_t)p->block_size : 1;
    const uint64_t dims[2] = {576, slots};
    const uint64_t strides[1] = {576 * 2};
    const uint32_t box[2] = {64, 1};   // one row high: rows are fetched four at a time by gather4
    if (make_tensor_map_bf16(&tc, any_keys ? cache : q_abs, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  // Whole 64-key tiles by tile loads of block pieces: a block size that is a multiple of 64
  // (one 64-row piece) or 8, 16 or 32 (64 / block_size pieces, each a whole block; 8 rows
  // keep each piece on the 128-byte swizzle's 1024-byte period).
  const int bs = p->block_size;
  const int piece_rows = (bs % 64 == 0) ? 64 : ((bs % 8 == 0 && 64 % bs == 0) ? bs : 0);
  CUtensorMap tb = tc;
  if (any_keys && piece_rows > 0) {
    const uint64_t dims[2] = {576, (uint64_t)num_blocks * (uint64_t)bs};
    const uint64_t strides[1] = {576 * 2};
    const uint32_t box[2] = {64, (uint32_t)piece_rows};
    if (make_tensor_map_bf16(&tb, cache, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  // 64-row pieces of several adjacent 64-column panels in one copy: the rows seen as
  // {64 columns, rows, 9 groups of 64 columns}.  Without such a map, one copy per panel.
  CUtensorMap t4 = tc;
  int grouped = 0;
  if (any_keys && piece_rows == 64) {
    const uint64_t dims[3] = {64, (uint64_t)num_blocks * (uint64_t)bs, 9};
    const uint64_t strides[2] = {576 * 2, 64 * 2};
    const uint32_t box[3] = {64, 64, 4};
    grouped = make_tensor_map_bf16(&t4, cache, 3, dims, strides, box) == MLA_OK ? 1 : 0;
    if (!grouped) t4 = tc;
  }
  AbsorbedParams prm;
  prm.units = reinterpret_cast<const AbsUnit*>(p->d_units);
  prm.block_table = block_table;
  prm.max_blocks = max_blocks_per_req;
  prm.block_size = p->block_size;
  prm.num_blocks = any_keys ? num_blocks : 0;
  prm.oob_row = any_keys ? (int32_t)(num_blocks * p->block_size) : 1;
  prm.piece_rows = any_keys ? piece_rows : 0;
  prm.grouped = grouped;
  prm.o = static_cast<__nv_bfloat16*>(o_lat);
  prm.lse = lse;
  prm.status = p->d_status;
  prm.num_heads = p->num_heads;
  prm.causal = p->causal;
  const float LOG2E = 1.4426950408889634f;
  prm.has_cap = p->soft_cap > 0.f;
  prm.scale_log2 = p->sm_scale * LOG2E;
  prm.cap_log2 = prm.has_cap ? p->soft_cap * LOG2E : 0.f;
  prm.cap_ex2_scale = prm.has_cap ? 2.f * LOG2E * p->sm_scale / p->soft_cap : 0.f;
  prm.force_timeout = p->forced_timeout_ns != 0;
  prm.wait_limit_ns = prm.force_timeout ? p->forced_timeout_ns : kWaitLimitNs;
  const cudaStream_t s = as_stream(stream);
  if (launch_absorbed(tq, tc, tb, t4, prm, (int)p->aunits.size(), s) != cudaSuccess) return MLA_ERR_CUDA;
  if (!stream_capturing(s) && cudaEventRecord(p->last_use, s) != cudaSuccess) return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_plan_query(mla_plan_t p, int which, int64_t* value) {
  if (!p || !value) return MLA_ERR_INVALID_ARG;
  switch (which) {
    case 0: *value = p->kind ? (int64_t)p->aunits.size() : (int64_t)p->plan.units.size(); break;
    case 1: *value = p->num_ctas; break;
    case 2: *value = p->total_q; break;
    case 3: *value = p->total_kv; break;
    case 4: *value = p->plan.allowed_pairs; break;
    case 5: *value = p->plan.kv_tiles; break;
    case 6: *value = p->pair; break;
    default: return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

int mla_gather_latent(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                      const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                      const int32_t* chunk_starts, int batch, int64_t total_tokens, void* out,
                      int32_t* status, void* stream) {
  if (total_tokens < 0 || batch < 0 || num_blocks < 0 || block_size < 1 || entry_dim < 8 ||
      entry_dim % 8 != 0 || max_blocks_per_req < 0)
    return MLA_ERR_INVALID_ARG;
  if (total_tokens == 0) return MLA_OK;
  if (batch == 0) return MLA_ERR_SHAPE;
  if (!cache || !block_table || !cu_seq_lens || !chunk_starts || !out || !aligned16(cache) || !aligned16(out))
    return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(status) & 3u) != 0) return MLA_ERR_INVALID_ARG;
  return launch_gather(cache, num_blocks, block_size, entry_dim, block_table, max_blocks_per_req,
                       cu_seq_lens, chunk_starts, batch, total_tokens, out, status,
                       as_stream(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_gather_latent_fp8(const void* cache, int64_t num_blocks, int block_size, int entry_bytes,
                          const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                          const int32_t* chunk_starts, int batch, int64_t total_tokens, void* out, int32_t* status,
                          void* stream) {
  if (total_tokens < 0 || batch < 0 || num_blocks < 0 || block_size < 1 || max_blocks_per_req < 0)
    return MLA_ERR_INVALID_ARG;
  if (entry_bytes != 648) return MLA_ERR_UNSUPPORTED;
  if (total_tokens == 0) return MLA_OK;
  if (batch == 0) return MLA_ERR_SHAPE;
  if (!cache || !block_table || !cu_seq_lens || !chunk_starts || !out || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(cache) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return MLA_ERR_INVALID_ARG;
  return launch_gather_fp8(cache, num_blocks, block_size, block_table, max_blocks_per_req, cu_seq_lens,
                           chunk_starts, batch, total_tokens, out, status, as_stream(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_cache_write(void* cache, int64_t num_blocks, int block_size, int entry_dim, const void* latent,
                    const int64_t* slot_mapping, int64_t num_tokens, int32_t* status, void* stream) {
  if (num_tokens < 0 || num_blocks < 0 || block_size < 1 || entry_dim < 8 || entry_dim % 8 != 0)
    return MLA_ERR_INVALID_ARG;
  if ((int64_t)entry_dim * 2 > 200 * 1024) return MLA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MLA_OK;
  if (!cache || !latent || !slot_mapping || !aligned16(cache) || !aligned16(latent) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0 || (reinterpret_cast<uintptr_t>(status) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  return launch_cache_write(cache, num_blocks * (int64_t)block_size, entry_dim, latent, slot_mapping, num_tokens,
                            status, as_stream(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_up_proj(const void* latent, const void* w_kvb, int64_t num_tokens, int num_heads, void* k_out,
                void* v_out, int32_t* status, void* stream) {
  if (num_tokens < 0 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (num_tokens > (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
  if (!latent || !w_kvb || !k_out || !v_out || !aligned16(latent) || !aligned16(w_kvb) ||
      !aligned16(k_out) || !aligned16(v_out))
    return MLA_ERR_INVALID_ARG;
  if (((num_tokens + 127) / 128) * (int64_t)num_heads > 0x7fffffff) return MLA_ERR_UNSUPPORTED;
  CUtensorMap ta, tb;
  {
    const uint64_t dims[2] = {576, (uint64_t)num_tokens};
    const uint64_t strides[1] = {576 * 2};
    const uint32_t box[2] = {64, 128};
    if (make_tensor_map_bf16(&ta, latent, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  {
    const uint64_t n = (uint64_t)num_heads * 256;
    const uint64_t dims[2] = {n, 512};
    const uint64_t strides[1] = {n * 2};
    const uint32_t box[2] = {64, 64};
    if (make_tensor_map_bf16(&tb, w_kvb, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  return launch_up_proj(ta, tb, latent, num_tokens, num_heads, k_out, v_out, status, as_stream(stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

static int up_proj_paged_impl(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                              const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                              const int32_t* chunk_starts, int batch, int64_t total_tokens, const void* w_kvb,
                              int num_heads, void* k_out, void* v_out, void* rope_out, int32_t* status,
                              void* stream) {
  if (total_tokens < 0 || batch < 0 || num_blocks < 0 || block_size < 1 || max_blocks_per_req < 0 ||
      num_heads < 1)
    return MLA_ERR_INVALID_ARG;
  if (entry_dim != 576) return MLA_ERR_UNSUPPORTED;
  if (total_tokens == 0) return MLA_OK;
  if (batch == 0) return MLA_ERR_SHAPE;
  // Slots are TMA row coordinates (int32), and one past the last slot marks a missing row.
  if (num_blocks * (int64_t)block_size >= 0x7fffffff || total_tokens > (int64_t)1 << 31) return MLA_ERR_UNSUPPORTED;
  if (((total_tokens + 127) / 128) * (int64_t)num_heads > 0x7fffffff) return MLA_ERR_UNSUPPORTED;
  if (!cache || !block_table || !cu_seq_lens || !chunk_starts || !w_kvb || !k_out || !v_out || !aligned16(cache) ||
      !aligned16(w_kvb) || !aligned16(k_out) || !aligned16(v_out) || (reinterpret_cast<uintptr_t>(status) & 3u))
    return MLA_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  {
    const uint64_t slots = (uint64_t)num_blocks * (uint64_t)block_size;
    const uint64_t dims[2] = {576, slots > 0 ? slots : 1};
    const uint64_t strides[1] = {576 * 2};
    const uint32_t box[2] = {64, 1};   // one row high: rows are fetched four at a time by gather4
    if (make_tensor_map_bf16(&ta, cache, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  {
    const uint64_t n = (uint64_t)num_heads * 256;
    const uint64_t dims[2] = {n, 512};
    const uint64_t strides[1] = {n * 2};
    const uint32_t box[2] = {64, 64};
    if (make_tensor_map_bf16(&tb, w_kvb, 2, dims, strides, box) != MLA_OK) return MLA_ERR_CUDA;
  }
  if (rope_out && !aligned16(rope_out)) return MLA_ERR_INVALID_ARG;
  return launch_up_proj_paged(ta, tb, cache, num_blocks, block_size, block_table, max_blocks_per_req, cu_seq_lens,
                              chunk_starts, batch, total_tokens, num_heads, k_out, v_out, rope_out, status,
                              as_stream(stream)) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_up_proj_paged(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                      const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                      const int32_t* chunk_starts, int batch, int64_t total_tokens, const void* w_kvb, int num_heads,
                      void* k_out, void* v_out, int32_t* status, void* stream) {
  return up_proj_paged_impl(cache, num_blocks, block_size, entry_dim, block_table, max_blocks_per_req, cu_seq_lens,
                            chunk_starts, batch, total_tokens, w_kvb, num_heads, k_out, v_out, nullptr, status,
                            stream);
}

int mla_up_proj_paged_split(const void* cache, int64_t num_blocks, int block_size, int entry_dim,
                            const int32_t* block_table, int max_blocks_per_req, const int32_t* cu_seq_lens,
                            const int32_t* chunk_starts, int batch, int64_t total_tokens, const void* w_kvb,
                            int num_heads, void* k_nope_out, void* v_out, void* rope_out, int32_t* status,
                            void* stream) {
  if (!rope_out && total_tokens > 0) return MLA_ERR_INVALID_ARG;
  return up_proj_paged_impl(cache, num_blocks, block_size, entry_dim, block_table, max_blocks_per_req, cu_seq_lens,
                            chunk_starts, batch, total_tokens, w_kvb, num_heads, k_nope_out, v_out, rope_out, status,
                            stream);
}

int mla_merge_state(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b, void* o_out,
                    float* lse_out, int64_t rows, int num_heads, int head_dim, void* stream) {
  if (rows < 0 || num_heads < 1) return MLA_ERR_INVALID_ARG;
  if (head_dim < 8 || head_dim > 256 || (head_dim & (head_dim - 1)) != 0) return MLA_ERR_UNSUPPORTED;
  if (rows == 0) return MLA_OK;
  if (!o_a || !o_b || !lse_a || !lse_b || !o_out || !aligned16(o_a) || !aligned16(o_b) || !aligned16(o_out))
    return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse_a) | reinterpret_cast<uintptr_t>(lse_b) |
       reinterpret_cast<uintptr_t>(lse_out)) & 3u)
    return MLA_ERR_INVALID_ARG;
  return launch_merge(o_a, lse_a, o_b, lse_b, o_out, lse_out, rows, num_heads, head_dim, as_stream(stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // extern "C"
