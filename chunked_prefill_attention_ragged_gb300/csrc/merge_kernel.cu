// LSE merge of two partial attention states, per (row, head):
//   m = max(la, lb), wa = 2^((la - m) log2 e), wb = 2^((lb - m) log2 e)
//   O = (wa Oa + wb Ob) / (wa + wb),  LSE = m + ln(wa + wb)
// A side with LSE = -inf has weight 0; both -inf gives O = 0, LSE = -inf.
//
// Needed because vLLM "vllm.v1.attention.backends.mla.prefill.flashinfer",
// run_prefill_context_chunk, returns each prefix chunk's LSE so the chunk outputs can be
// combined with the new-token output.  Memory bound: each group of head_dim/8 lanes of
// one warp owns one (row, head) and moves it with 16-byte loads and stores, so a warp
// streams 512 contiguous bytes of each input per step.
#include "internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;

// Streaming 16-byte load.  The read-only (non-coherent) path is legal only for data no
// thread of the kernel writes, so the first input takes the coherent path when the
// outputs alias it (in-place merge).
template <bool kReadOnly>
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  if constexpr (kReadOnly)
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
  else
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
  return v;
}

__device__ __forceinline__ float2 unpack(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t pack(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// log2(vec) lanes per (row, head); vec = head_dim / 8 <= 32.  kInPlace: o_out/lse_out may
// alias o_a/lse_a, so those are read through coherent loads.
template <bool kInPlace>
__global__ void __launch_bounds__(kThreads)
merge_kernel(const uint4* oa, const float* la, const uint4* ob, const float* lb, uint4* oo, float* lo,
             int64_t n_rh, int vec_shift) {
  const int vec = 1 << vec_shift;
  const int64_t groups_per_step = (int64_t)gridDim.x * kThreads >> vec_shift;
  const int64_t g0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> vec_shift;
  const int e = threadIdx.x & (vec - 1);
  const float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
  // Iterate so that every lane of a warp takes the same number of steps (keeps
  // __syncwarp legal).
  const int64_t steps = (n_rh + groups_per_step - 1) / groups_per_step;
  for (int64_t s = 0; s < steps; ++s) {
    const int64_t rh = g0 + s * groups_per_step;
    const bool live = rh < n_rh;
    float a = 0.f, b = 0.f;
    uint4 va = make_uint4(0, 0, 0, 0), vb = va;
    if (live) {
      a = kInPlace ? la[rh] : __ldg(la + rh);
      b = __ldg(lb + rh);
      va = ld_stream<!kInPlace>(oa + (rh << vec_shift) + e);
      vb = ld_stream<true>(ob + (rh << vec_shift) + e);
    }
    // Every lane of the group has read la/lb and its slice before any lane writes
    // (outputs may alias the first input).
    __syncwarp();
    if (!live) continue;
    const float m = fmaxf(a, b);
    const bool empty = !(m > -__int_as_float(0x7f800000));   // both -inf
    float wa = 0.f, wb = 0.f, tot = 1.f;
    if (!empty) {
      wa = exp2f((a - m) * LOG2E);
      wb = exp2f((b - m) * LOG2E);
      tot = wa + wb;
      const float inv = 1.f / tot;
      wa *= inv;
      wb *= inv;
    }
    const uint32_t ia[4] = {va.x, va.y, va.z, va.w}, ib[4] = {vb.x, vb.y, vb.z, vb.w};
    uint32_t res[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = unpack(ia[k]), y = unpack(ib[k]);
      res[k] = pack(wa * x.x + wb * y.x, wa * x.y + wb * y.y);
    }
    oo[(rh << vec_shift) + e] = make_uint4(res[0], res[1], res[2], res[3]);
    if (lo && e == 0) lo[rh] = empty ? -__int_as_float(0x7f800000) : m + log2f(tot) * LN2;
  }
}

}  // namespace

cudaError_t launch_merge(const void* o_a, const float* lse_a, const void* o_b, const float* lse_b,
                         void* o_out, float* lse_out, int64_t rows, int num_heads, int head_dim,
                         cudaStream_t stream) {
  const int64_t n_rh = rows * num_heads;
  if (n_rh == 0) return cudaSuccess;
  int vec_shift = 0;
  while ((8 << vec_shift) < head_dim) ++vec_shift;
  const int sms = device_sm_count();
  const int64_t groups_per_block = kThreads >> vec_shift;
  const int64_t want = (n_rh + groups_per_block - 1) / groups_per_block;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 16;
  const int grid = (int)(want < cap ? want : cap);
  const bool in_place = o_out == o_a || (lse_out != nullptr && lse_out == lse_a);
  auto kernel = in_place ? merge_kernel<true> : merge_kernel<false>;
  kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(o_a), lse_a, static_cast<const uint4*>(o_b),
                                        lse_b, static_cast<uint4*>(o_out), lse_out, n_rh, vec_shift);
  return cudaGetLastError();
}

}  // namespace mla
