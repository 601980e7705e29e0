// Allocation-free ragged prefill: mla_prefill_run_noalloc.
//
// Some callers cannot call cudaMalloc: code running inside a pre-sized memory pool
// that owns every byte of the device (serving engines reserve almost all HBM for the KV
// cache at start-up), hosts that forbid allocation after initialisation, and callers
// that must not trigger the device synchronisation an allocation or free can imply.
// mla_prefill_plan allocates its work list on the device, so those callers get this
// entry point instead: it plans on the host each call and puts the work list, the
// per-CTA offsets and the status word into one file-scope device array that lives as
// long as the library is loaded, then launches the same prefill kernel.
//
// The scratch array (g_noalloc_scratch) is part of the module image, so every GPU that
// loads this library holds it (about 2 MiB) until the process exits.  Its address is
// looked up once per device (a host-side symbol lookup), on the first call made with that
// device current.  All calls share the array and it keeps the last
// call's contents, so calls that overlap on the GPU (different streams, or several host
// threads) race on it and must be ordered by the caller.
#include <cmath>
#include <mutex>
#include <vector>

#include "internal.h"

namespace mla {
namespace {

constexpr int64_t kNoAllocMaxUnits = 65536;   // 128-row query tiles x heads
constexpr int kNoAllocMaxCtas = 1023;
constexpr size_t kUnitsBytes = (size_t)kNoAllocMaxUnits * sizeof(Unit);            // 2 MiB
constexpr size_t kOffsetsBytes = (size_t)(kNoAllocMaxCtas + 1) * sizeof(int32_t);   // 4 KiB
constexpr size_t kStatusOffset = kUnitsBytes + kOffsetsBytes;
constexpr size_t kScratchBytes = kStatusOffset + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (host-side symbol lookup,
// once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MLA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" MLA_API int mla_prefill_run_noalloc(const int32_t* qo_indptr, const int32_t* kv_indptr, int batch,
                                               int num_heads, int head_dim_qk, int head_dim_vo, int causal,
                                               float sm_scale, int window_left, float logits_soft_cap,
                                               const void* q, const void* k, const void* v, void* o, float* lse,
                                               int32_t* status, void* stream) {
  if (!qo_indptr || !kv_indptr || batch < 0 || num_heads < 1 || num_heads > 65535) return MLA_ERR_INVALID_ARG;
  if (head_dim_qk != 192 || head_dim_vo != 128) return MLA_ERR_UNSUPPORTED;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f) || !std::isfinite(logits_soft_cap) || window_left < -1)
    return MLA_ERR_INVALID_ARG;
  {
    PlanResult probe;   // host-only shape checks and the unit count, before any CUDA call
    const int rc = build_plan(qo_indptr, kv_indptr, batch, num_heads, causal != 0, window_left, 1, &probe);
    if (rc != MLA_OK) return rc;
    if ((int64_t)probe.units.size() > kNoAllocMaxUnits) return MLA_ERR_UNSUPPORTED;   // scratch too small
    if (probe.units.empty()) return MLA_OK;
  }
  const int64_t total_q = qo_indptr[batch], total_kv = kv_indptr[batch];
  if (!q || !o || !aligned16(q) || !aligned16(o) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) ||
      (status && (reinterpret_cast<uintptr_t>(status) & 3u)))
    return MLA_ERR_INVALID_ARG;
  if (total_kv > 0 && (!k || !v || !aligned16(k) || !aligned16(v))) return MLA_ERR_INVALID_ARG;

  const int sms = device_sm_count();
  if (sms <= 0) return MLA_ERR_CUDA;
  PlanResult plan;
  int rc = build_plan(qo_indptr, kv_indptr, batch, num_heads, causal != 0, window_left,
                      sms < kNoAllocMaxCtas ? sms : kNoAllocMaxCtas, &plan);
  if (rc != MLA_OK) return rc;
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != MLA_OK) return rc;
  char* base = static_cast<char*>(scratch);
  Unit* d_units = reinterpret_cast<Unit*>(base);
  int32_t* d_offsets = reinterpret_cast<int32_t*>(base + kUnitsBytes);
  int* d_status = status ? status : reinterpret_cast<int*>(base + kStatusOffset);

  // Pageable host sources: each copy has been staged when cudaMemcpyAsync returns.
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(d_units, plan.units.data(), plan.units.size() * sizeof(Unit), cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyAsync(d_offsets, plan.cta_offsets.data(), plan.cta_offsets.size() * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (!status && cudaMemsetAsync(d_status, 0, sizeof(int), s) != cudaSuccess) return MLA_ERR_CUDA;

  const void* kb = total_kv > 0 ? k : q;
  const void* vb = total_kv > 0 ? v : q;
  const uint64_t H = (uint64_t)num_heads;
  const uint64_t kv_rows = total_kv > 0 ? (uint64_t)total_kv : 1;
  const uint32_t box[3] = {64, 1, 128};
  CUtensorMap tq, tk, tv;
  const uint64_t qd[3] = {192, H, (uint64_t)total_q}, kd[3] = {192, H, kv_rows}, vd[3] = {128, H, kv_rows};
  const uint64_t qks[2] = {192 * 2, H * 192 * 2}, vs[2] = {128 * 2, H * 128 * 2};
  if (make_tensor_map_bf16(&tq, q, 3, qd, qks, box) != MLA_OK || make_tensor_map_bf16(&tk, kb, 3, kd, qks, box) != MLA_OK ||
      make_tensor_map_bf16(&tv, vb, 3, vd, vs, box) != MLA_OK)
    return MLA_ERR_CUDA;

  PrefillParams prm;
  prm.merge = 0;
  prm.units = d_units;
  prm.cta_offsets = d_offsets;
  prm.status = d_status;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.o_align32 = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
  prm.lse = lse;
  prm.num_heads = num_heads;
  prm.causal = causal != 0;
  prm.window_left = window_left;
  const float LOG2E = 1.4426950408889634f;
  const float cap = logits_soft_cap > 0.f ? logits_soft_cap : 0.f;
  prm.has_cap = cap > 0.f;
  prm.scale_log2 = sm_scale * LOG2E;
  prm.cap_log2 = prm.has_cap ? cap * LOG2E : 0.f;
  prm.x_to_cap = prm.has_cap ? sm_scale / cap : 0.f;
  prm.cap_ex2_scale = 2.f * LOG2E * prm.x_to_cap;
  prm.force_timeout = 0;
  prm.shared_rope = 0;
  prm.pair = 0;
  prm.wait_limit_ns = kWaitLimitNs;
  const int num_ctas = (int)plan.cta_offsets.size() - 1;
  return launch_prefill(tq, tk, tv, tk, prm, num_ctas, s) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
