// Paged gather of fp8 latent cache entries, dequantized to bf16 rows of 576.
//
// Entry layout (vLLM "vllm/models/deepseek_v4/sparse_mla.py", cache dtype fp8_ds_mla:
// fp8 NoPE part, then 128 bytes of bf16 RoPE, then 8 scale bytes; here for the 512 + 64
// rows of sglang issue #3849): bytes [0, 512) latent as float8 e4m3, [512, 640) rope as
// 64 bf16, [640, 648) one power-of-two scale byte (2^(b - 127)) per 64 latent values.
// Output row t = [e4m3(x_i) * scale_(i / 64) rounded to bf16 for i < 512 | rope]; rows
// are addressed by the paged slot rule (block_table[r, pos / block_size] * block_size +
// pos % block_size).
//
// Memory bound (648 bytes read, 1152 written per token).  One warp per row at a time:
// lane l converts latent values 8 l .. 8 l + 7 and 256 + 8 l .. 256 + 8 l + 7 (scale
// groups l / 8 and 4 + l / 8) with the hardware e4m3x2 -> f16x2 conversion (exact), one
// fp32 multiply by the scale (exact: a 4-bit significand times a power of two) and one
// rounding to bf16, so that each warp-wide load reads 256 contiguous bytes and each
// warp-wide store writes 512; lanes 0-15 copy the rope.  The grid is exactly one wave of
// resident warps (grid-stride over rows, two rows in flight per warp): with one row batch
// per warp and as many warps as batches, the second, partial wave of a 75 MB gather left
// most SMs idle.
#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kEntry = 648;
constexpr int kRowsPerWarp = 2;
constexpr int kBlocksPerSm = 6;   // 48 warps per SM, every one resident from the start
constexpr int kThreads = 256;

__device__ __forceinline__ uint2 ld_nc_u2(const uint8_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// 2^(b - 127) as an fp32 bit pattern: b = 0 is the subnormal 2^-127, b = 255 is NaN.
__device__ __forceinline__ float ue8m0_scale(uint32_t b) {
  const uint32_t bits = b == 0 ? 0x00400000u : (b == 255 ? 0x7FC00000u : b << 23);
  return __uint_as_float(bits);
}

// Two e4m3 values (low byte first) scaled and rounded to one bf16x2 word.
__device__ __forceinline__ uint32_t dequant2(uint32_t two_fp8, float scale) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_fp8));
  float lo, hi;
  asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi) : "r"(h2));
  float xl, xh;
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(xl) : "f"(lo), "f"(scale));
  asm("mul.rn.f32 %0, %1, %2;" : "=f"(xh) : "f"(hi), "f"(scale));
  return pack_bf16x2(xl, xh);
}

__global__ void __launch_bounds__(kThreads, kBlocksPerSm)
gather_fp8_kernel(const uint8_t* __restrict__ cache, RowMap m, int64_t total_rows, uint8_t* __restrict__ out,
                  int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;
  const int32_t cu_l = m.batch < 32 && lane <= m.batch ? __ldg(m.cu + lane) : 0x7fffffff;
  const int32_t st_l = m.batch < 32 && lane < m.batch ? __ldg(m.starts + lane) : 0;
  for (int64_t base = warp * kRowsPerWarp; base < total_rows; base += nwarps * kRowsPerWarp) {
    uint2 lat[kRowsPerWarp][2], rope[kRowsPerWarp], sc[kRowsPerWarp];
    bool have[kRowsPerWarp];
#pragma unroll
    for (int u = 0; u < kRowsPerWarp; ++u) {
      const int64_t row = base + u;
      const bool active = row < total_rows;
      int64_t slot = 0;
      have[u] = resolve_slot(m, row, active, cu_l, st_l, &slot);   // the same row in every lane
      if (active && !have[u] && lane == 0 && status) atomicOr(status, MLA_DEVSTAT_BAD_INDEX);
      lat[u][0] = lat[u][1] = rope[u] = sc[u] = make_uint2(0, 0);
      if (have[u]) {
        const uint8_t* src = cache + slot * kEntry;
        lat[u][0] = ld_nc_u2(src + lane * 8);
        lat[u][1] = ld_nc_u2(src + 256 + lane * 8);
        sc[u] = ld_nc_u2(src + 640);
        if (lane < 16) rope[u] = ld_nc_u2(src + 512 + lane * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPerWarp; ++u) {
      const int64_t row = base + u;
      if (row >= total_rows) break;
      uint8_t* dst = out + row * (576 * 2);
      uint32_t w[8];
      if (have[u]) {
        // values 8 lane ..: group lane / 8 (scale bytes 0-3); 256 + 8 lane ..: group 4 + lane / 8
        const int sh = 8 * (lane >> 3);
        const float s0 = ue8m0_scale((sc[u].x >> sh) & 0xFFu), s1 = ue8m0_scale((sc[u].y >> sh) & 0xFFu);
        const uint32_t src[4] = {lat[u][0].x, lat[u][0].y, lat[u][1].x, lat[u][1].y};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float sq = q < 2 ? s0 : s1;
          w[2 * q] = dequant2(src[q] & 0xFFFFu, sq);
          w[2 * q + 1] = dequant2(src[q] >> 16, sq);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) w[q] = 0;
      }
      reinterpret_cast<uint4*>(dst)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
      reinterpret_cast<uint4*>(dst + 512)[lane] = make_uint4(w[4], w[5], w[6], w[7]);
      if (lane < 16) *reinterpret_cast<uint2*>(dst + 1024 + lane * 8) = rope[u];
    }
  }
}

}  // namespace

cudaError_t launch_gather_fp8(const void* cache, int64_t num_blocks, int block_size, const int32_t* block_table,
                              int max_blocks_per_req, const int32_t* cu_seq_lens, const int32_t* chunk_starts,
                              int batch, int64_t total_tokens, void* out, int32_t* status, cudaStream_t stream) {
  if (total_tokens == 0) return cudaSuccess;
  const int sms = device_sm_count();
  const int64_t warps_needed = (total_tokens + kRowsPerWarp - 1) / kRowsPerWarp;
  const int64_t blocks_needed = (warps_needed + kThreads / 32 - 1) / (kThreads / 32);
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * kBlocksPerSm;
  const int grid = (int)(blocks_needed < cap ? blocks_needed : cap);
  RowMap m{cu_seq_lens, chunk_starts, block_table, batch, max_blocks_per_req, block_size, num_blocks};
  gather_fp8_kernel<<<grid, kThreads, 0, stream>>>(static_cast<const uint8_t*>(cache), m, total_tokens,
                                                   static_cast<uint8_t*>(out), status);
  return cudaGetLastError();
}

}  // namespace mla
