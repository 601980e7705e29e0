// Latent up-projection on tcgen05 tensor cores:
//   kv[t, h*256 + d] = sum_c latent[t, c] * W[c, h*256 + d]      (c < 512)
//   K[t, h, 0:128] = kv[t, h*256 + 0:128],  K[t, h, 128:192] = latent[t, 512:576]
//   V[t, h, 0:128] = kv[t, h*256 + 128:256]
// sglang issue #3849 ("[DeepseekR1] How ragged prefill manage kv_cache?"): the cache
// keeps 512 latent + 64 rope per token while prefill attention runs as MHA with
// 192-dim K and 128-dim V; this kernel is that decompression, with the rope copy fused
// into the epilogue so K and V are written once, in their final layout.
//
// Persistent kernel, one CTA per SM, output tile = 128 tokens x one head (N = 256):
//   warp 0     TMA producer: latent panel [128 x 64] (K-major) and W panel
//              [64 x 256] (N-major) per 64-wide slice of the 512 reduction, 4-stage ring.
//   warp 1     MMA issuer: tcgen05.mma M=128 N=256 K=16 into one of two TMEM
//              accumulators (512 columns), so the epilogue of tile i overlaps the
//              MMAs of tile i+1.
//   warps 2-5  epilogue: one thread per token row reads its accumulator row, rounds to
//              bf16 and writes K_nope, V and the rope copy.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "tmem_wide.cuh"

namespace mla {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, KDIM = 512, KBLOCKS = KDIM / BK;
constexpr int NS = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_PANEL = BK * 64 * 2;          // 8 KB: 64 k-rows x 64 n
constexpr int B_BYTES = 4 * B_PANEL;          // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + NS * A_BYTES;
constexpr int OFF_BAR = OFF_B + NS * B_BYTES;
enum Bar { FULL = 0, EMPTY = 4, AFULL = 8, AEMPTY = 10, FIN = 12, NBAR = 13 };
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false, true);
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;

struct Ctx {
  uint32_t sbase;
  volatile int* abort_flag;
  int* status;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8 * i; }
  __device__ bool wait(int b, uint32_t parity) const {
    return mbar_wait_bounded(bar(b), parity, abort_flag, status, MLA_DEVSTAT_TIMEOUT, WAIT_LIMIT_NS);
  }
  __device__ void drain(int b, uint32_t parity) const {
    int dummy = 0;
    mbar_wait_bounded(bar(b), parity, &dummy, status, MLA_DEVSTAT_TIMEOUT, DRAIN_LIMIT_NS);
  }
};

struct UpParams {
  const __nv_bfloat16* latent;
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int* status;
  int64_t num_tokens;
  int num_heads;
  int num_tiles;
};

__global__ void __launch_bounds__(NTHREADS, 1)
up_proj_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const UpParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(smem + OFF_MISC + 4);
  Ctx c{smem_addr(smem), abort_flag, p.status};
  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(c.bar(i), 1);
    mbar_init(c.bar(AEMPTY + 0), 128);
    mbar_init(c.bar(AEMPTY + 1), 128);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
      const int m0 = (tile / p.num_heads) * BM, h = tile % p.num_heads;
      for (int kb = 0; kb < KBLOCKS; ++kb, ++it) {
        const int s = it % NS;
        const uint32_t use = it / NS;
        if (use > 0 && !c.wait(EMPTY + s, (use - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(c.bar(FULL + s), A_BYTES + B_BYTES);
        tma_load_2d(c.sbase + OFF_A + s * A_BYTES, &tm_a, c.bar(FULL + s), kb * BK, m0);
        for (int i = 0; i < 4; ++i)
          tma_load_2d(c.sbase + OFF_B + s * B_BYTES + i * B_PANEL, &tm_b, c.bar(FULL + s),
                      h * BN + i * 64, kb * BK);
      }
    }
    for (int s = 0; s < NS; ++s)
      if (it > s) c.drain(FULL + s, ((it - 1 - s) / NS) & 1);
  } else if (warp == 1 && lane == 0) {
    int it = 0, acc = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++acc) {
      const int a = acc & 1;
      if (acc >= 2 && !c.wait(AEMPTY + a, ((acc >> 1) - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      for (int kb = 0; kb < KBLOCKS; ++kb, ++it) {
        const int s = it % NS;
        if (!c.wait(FULL + s, (it / NS) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(c.sbase + OFF_A + s * A_BYTES + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(c.sbase + OFF_B + s * B_BYTES + kk * 16 * 128, B_PANEL, 1024);
          mma_ss(tmem + a * BN, ad, bd, IDESC, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(c.bar(EMPTY + s));
      }
      if (ok) tc_commit(c.bar(AFULL + a));
    }
    tc_commit(c.bar(FIN));
    c.drain(FIN, 0);
  } else if (warp >= 2) {
    const int quad = warp & 3, row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    int acc = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++acc) {
      const int a = acc & 1;
      if (!__all_sync(0xffffffffu, c.wait(AFULL + a, (acc >> 1) & 1))) break;
      tc_fence_after();
      const int64_t t = (int64_t)(tile / p.num_heads) * BM + row;
      const int h = tile % p.num_heads;
      const bool live = t < p.num_tokens;
      const int64_t kr = (t * p.num_heads + h) * 192, vr = (t * p.num_heads + h) * 128;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[64];
        tmem_ld64_sync(lane_addr + a * BN + ch * 64, r);
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(ch < 2 ? p.k + kr + ch * 64 : p.v + vr + (ch - 2) * 64);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]), __uint_as_float(r[8 * i + 1]));
            w.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]), __uint_as_float(r[8 * i + 3]));
            w.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]), __uint_as_float(r[8 * i + 5]));
            w.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]), __uint_as_float(r[8 * i + 7]));
            dst[i] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(c.bar(AEMPTY + a));
      if (live) {
        const uint4* src = reinterpret_cast<const uint4*>(p.latent + t * 576 + 512);
        uint4* dst = reinterpret_cast<uint4*>(p.k + kr + 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = __ldg(src + i);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int up_proj_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_up_proj(const CUtensorMap& ta, const CUtensorMap& tb, const void* latent,
                           int64_t num_tokens, int num_heads, void* k_out, void* v_out,
                           int32_t* status, cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(up_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  UpParams p;
  p.latent = static_cast<const __nv_bfloat16*>(latent);
  p.k = static_cast<__nv_bfloat16*>(k_out);
  p.v = static_cast<__nv_bfloat16*>(v_out);
  p.status = status;
  p.num_tokens = num_tokens;
  p.num_heads = num_heads;
  const int64_t m_tiles = (num_tokens + BM - 1) / BM;
  p.num_tiles = (int)(m_tiles * num_heads);
  if (p.num_tiles == 0) return cudaSuccess;
  const int sms = device_sm_count();
  const int grid = p.num_tiles < sms ? p.num_tiles : (sms > 0 ? sms : 148);
  up_proj_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace mla
