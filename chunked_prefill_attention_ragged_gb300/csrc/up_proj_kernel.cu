// Latent up-projection on tcgen05 tensor cores:
//   kv[t, h*256 + d] = sum_c latent[t, c] * W[c, h*256 + d]      (c < 512)
//   K[t, h, 0:128] = kv[t, h*256 + 0:128],  K[t, h, 128:192] = latent[t, 512:576]
//   V[t, h, 0:128] = kv[t, h*256 + 128:256]
// sglang issue #3849 ("[DeepseekR1] How ragged prefill manage kv_cache?"): the cache
// keeps 512 latent + 64 rope per token while prefill attention runs as MHA with
// 192-dim K and 128-dim V; this kernel is that decompression, with the rope copy fused
// into the epilogue so K and V are written once, in their final layout.
//
// Persistent kernel, one CTA per SM, output tile = 128 tokens x one head (N = 256).
// Each CTA takes a contiguous range of tiles ordered (token block, head) with the head
// fastest, so the 128-token latent tile (A, 128 x 512, 128 KB) stays in shared memory
// while the CTA walks through heads; only W's 512 x 256 slice of each head (B, 256 KB)
// streams.  Per tile that is 256 KB of operand traffic for 4096 cycles of MMA instead
// of 384 KB, below what L2 delivers to one SM.
//   warp 0     TMA producer: the latent tile when the token block changes (8 K-major
//              panels of 128 x 64), and W's slice as [64 x 256] blocks (4 N-major
//              panels of 64 x 64) through a 3-stage ring, marked evict-last in L2 (the
//              K/V output is stored evict-first), so W is read from HBM about once.
//   warp 1     MMA issuer: tcgen05.mma M=128 N=256 K=16 into one of two TMEM
//              accumulators (512 columns), so the epilogue of tile i overlaps the
//              MMAs of tile i+1.
//   warps 2-5  epilogue: one thread per token row reads its accumulator row, rounds to
//              bf16 and writes K_nope, V and the rope copy (read once per token block)
//              with 32-byte stores when the outputs allow it.
#include <cuda_bf16.h>

#include "internal.h"
#include "paged.cuh"
#include "ptx.cuh"
#include "tmem_wide.cuh"

namespace mla {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, KDIM = 512, KBLOCKS = KDIM / BK;
constexpr int NS = 3;
constexpr int A_PANEL = BM * BK * 2;          // 16 KB: 128 token rows x 64 latent columns
constexpr int A_BYTES = KBLOCKS * A_PANEL;    // 128 KB: the whole 128 x 512 latent tile
constexpr int B_PANEL = BK * 64 * 2;          // 8 KB: 64 k-rows x 64 n
constexpr int B_BYTES = 4 * B_PANEL;          // 32 KB
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + A_BYTES;
constexpr int OFF_BAR = OFF_B + NS * B_BYTES;
enum Bar { FULL = 0, EMPTY = 3, AFULL = 6, AEMPTY = 8, LF = 10, LE = 11, FIN = 12, NBAR = 13 };
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
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
  const __nv_bfloat16* latent;   // [num_tokens, 576]; paged: the cache [num_slots, 576]
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int* status;
  int64_t num_tokens;
  int num_heads;
  int num_tiles;
  int out_align32;   // k and v 32-byte aligned: 32-byte stores
  // split form: k holds K_nope [T, H, 128] only and rope_out [T, 64] the one RoPE row per
  // token that every head's K shares (written once, by the tile of head 0)
  __nv_bfloat16* rope_out;
  int split_rope;
  // paged form: token row t of the output is the cache row of the chunk's row t
  RowMap rows;
  int32_t oob_row;   // a row coordinate past the cache: the TMA fills it with zeros
};

// Cache slot of chunk row `row` for the paged form (all 32 lanes of the warp call; rows
// past the chunk or with an unknown block give `p.oob_row` and, for rows inside the
// chunk, flag MLA_DEVSTAT_BAD_INDEX).
__device__ __forceinline__ int32_t paged_row(const UpParams& p, int64_t row, int32_t cu_l, int32_t st_l) {
  const bool active = row < p.num_tokens;
  int64_t slot = 0;
  const bool ok = resolve_slot(p.rows, row, active, cu_l, st_l, &slot);
  if (active && !ok && p.status) atomicOr(p.status, MLA_DEVSTAT_BAD_INDEX);
  return ok ? (int32_t)slot : p.oob_row;
}

__device__ __forceinline__ void tile_range(int num_tiles, int& beg, int& end) {
  beg = (int)((int64_t)blockIdx.x * num_tiles / gridDim.x);
  end = (int)((int64_t)(blockIdx.x + 1) * num_tiles / gridDim.x);
}

// kPaged: the latent rows come straight out of the paged cache (tm_a maps the cache as
// [num_slots, 576] rows; each token block's 128 rows are fetched four at a time by
// tile::gather4 copies), so no gathered latent buffer is needed.
template <bool kPaged>
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
  int tbeg, tend;
  tile_range(p.num_tiles, tbeg, tend);
  const int H = p.num_heads;

  if (warp == 0) {
    // Producer warp.  Lane 0 waits and issues W's slices; in the paged form every lane
    // resolves four latent rows and issues their gather copies.
    int it = 0, a_loads = 0;
    bool ok = true;
    // W (32 MB for 128 heads) is read by every token block: keep it in L2 while the
    // much larger K/V output streams through.
    const uint64_t w_policy = l2_policy_evict_last();
    int32_t cu_l = 0, st_l = 0;
    if constexpr (kPaged) {
      cu_l = p.rows.batch < 32 && lane <= p.rows.batch ? __ldg(p.rows.cu + lane) : 0x7fffffff;
      st_l = p.rows.batch < 32 && lane < p.rows.batch ? __ldg(p.rows.starts + lane) : 0;
    }
    for (int tile = tbeg; tile < tend && ok; ++tile) {
      const int m = tile / H, h = tile % H;
      if (tile == tbeg || h == 0) {   // new token block: reload the latent tile
        int free = 1;
        if (lane == 0 && a_loads > 0) free = c.wait(LE, (a_loads - 1) & 1);
        if (!__shfl_sync(0xffffffffu, free, 0)) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(c.bar(LF), A_BYTES);
        __syncwarp();
        if constexpr (kPaged) {
          // Lane l fetches token rows 4l .. 4l+3 of the block: one gather per 64-column panel.
          int32_t r4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) r4[j] = paged_row(p, (int64_t)m * BM + 4 * lane + j, cu_l, st_l);
          for (int kb = 0; kb < KBLOCKS; ++kb)
            tma_gather4(c.sbase + OFF_A + kb * A_PANEL + lane * 4 * 128, &tm_a, c.bar(LF), kb * BK, r4[0], r4[1],
                        r4[2], r4[3]);
        } else if (lane == 0) {
          for (int kb = 0; kb < KBLOCKS; ++kb)
            tma_load_2d(c.sbase + OFF_A + kb * A_PANEL, &tm_a, c.bar(LF), kb * BK, m * BM);
        }
        ++a_loads;
      }
      int went = 1;
      if (lane == 0) {
        for (int kb = 0; kb < KBLOCKS; ++kb, ++it) {
          const int s = it % NS;
          const uint32_t use = it / NS;
          if (use > 0 && !c.wait(EMPTY + s, (use - 1) & 1)) { went = 0; break; }
          mbar_arrive_expect_tx(c.bar(FULL + s), B_BYTES);
          for (int i = 0; i < 4; ++i)
            tma_load_2d_hint(c.sbase + OFF_B + s * B_BYTES + i * B_PANEL, &tm_b, c.bar(FULL + s),
                             h * BN + i * 64, kb * BK, w_policy);
        }
      }
      ok = __shfl_sync(0xffffffffu, went, 0) != 0;
    }
    if (lane == 0) {
      if (a_loads > 0) c.drain(LF, (a_loads - 1) & 1);
      for (int s = 0; s < NS; ++s)
        if (it > s) c.drain(FULL + s, ((it - 1 - s) / NS) & 1);
    }
  } else if (warp == 1 && lane == 0) {
    int it = 0, acc = 0, a_loads = 0;
    bool ok = true;
    const uint64_t a_desc0 = sdesc_sw128(c.sbase + OFF_A, 16, 1024);
    const uint64_t b_desc0 = sdesc_sw128(c.sbase + OFF_B, B_PANEL, 1024);
    for (int tile = tbeg; tile < tend && ok; ++tile, ++acc) {
      const int h = tile % H;
      if (tile == tbeg || h == 0) {
        if (!c.wait(LF, a_loads & 1)) { ok = false; break; }
        ++a_loads;
      }
      const int a = acc & 1;
      if (acc >= 2 && !c.wait(AEMPTY + a, ((acc >> 1) - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      for (int kb = 0; kb < KBLOCKS; ++kb, ++it) {
        const int s = it % NS;
        if (!c.wait(FULL + s, (it / NS) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = a_desc0 + (uint64_t)(kb * A_PANEL >> 4);
        const uint64_t bd = b_desc0 + (uint64_t)(s * B_BYTES >> 4);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_ss(tmem + a * BN, ad + (uint64_t)(kk * 32 >> 4), bd + (uint64_t)(kk * 16 * 128 >> 4), IDESC,
                 (kb > 0 || kk > 0) ? 1u : 0u);
        tc_commit(c.bar(EMPTY + s));
      }
      if (!ok) break;
      tc_commit(c.bar(AFULL + a));
      // The latent tile is free once the last head of its token block (in this CTA's
      // range) has been multiplied.
      if (tile + 1 == tend || h == H - 1) tc_commit(c.bar(LE));
    }
    tc_commit(c.bar(FIN));
    c.drain(FIN, 0);
  } else if (warp >= 2) {
    const int quad = warp & 3, row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    int acc = 0;
    uint4 rope[8];
    const uint64_t out_policy = l2_policy_evict_first();   // K/V are written once here
    int32_t cu_l = 0, st_l = 0;
    if constexpr (kPaged) {
      cu_l = p.rows.batch < 32 && lane <= p.rows.batch ? __ldg(p.rows.cu + lane) : 0x7fffffff;
      st_l = p.rows.batch < 32 && lane < p.rows.batch ? __ldg(p.rows.starts + lane) : 0;
    }
    for (int tile = tbeg; tile < tend; ++tile, ++acc) {
      const int a = acc & 1;
      const int64_t t = (int64_t)(tile / H) * BM + row;
      const int h = tile % H;
      const bool live = t < p.num_tokens;
      if (tile == tbeg || h == 0) {   // rope part of this token, the same for every head
        int64_t src_row = t;
        bool have = live;
        if constexpr (kPaged) {
          int64_t slot = 0;
          have = resolve_slot(p.rows, t, live, cu_l, st_l, &slot);   // warp-wide call
          src_row = slot;
        }
        if (have) {
          const uint4* src = reinterpret_cast<const uint4*>(p.latent + src_row * 576 + 512);
#pragma unroll
          for (int i = 0; i < 8; ++i) rope[i] = __ldg(src + i);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) rope[i] = make_uint4(0, 0, 0, 0);   // unknown block: zeros
        }
      }
      if (!__all_sync(0xffffffffu, c.wait(AFULL + a, (acc >> 1) & 1))) break;
      tc_fence_after();
      const int64_t kr = (t * H + h) * (p.split_rope ? 128 : 192), vr = (t * H + h) * 128;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t r[64];
        tmem_ld64_sync(lane_addr + a * BN + ch * 64, r);
        if (live) {
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
          char* dst = reinterpret_cast<char*>(ch < 2 ? p.k + kr + ch * 64 : p.v + vr + (ch - 2) * 64);
          if (p.out_align32) {
#pragma unroll
            for (int q = 0; q < 4; ++q) st_global_v8_hint(dst + q * 32, w + 8 * q, out_policy);
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(c.bar(AEMPTY + a));
      if (live && (!p.split_rope || h == 0)) {
        uint4* dst = reinterpret_cast<uint4*>(p.split_rope ? p.rope_out + t * 64 : p.k + kr + 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = rope[i];
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

template <bool kPaged>
static cudaError_t launch_up_proj_t(const CUtensorMap& ta, const CUtensorMap& tb, UpParams& p, cudaStream_t stream) {
  static PerDeviceOnce configured;
  cudaError_t e = configured.run([] {
    return cudaFuncSetAttribute(up_proj_kernel<kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  const int64_t m_tiles = (p.num_tokens + BM - 1) / BM;
  p.num_tiles = (int)(m_tiles * p.num_heads);
  if (p.num_tiles == 0) return cudaSuccess;
  const int sms = device_sm_count();
  const int grid = p.num_tiles < sms ? p.num_tiles : (sms > 0 ? sms : 148);
  up_proj_kernel<kPaged><<<grid, NTHREADS, SMEM_BYTES, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

static UpParams up_params(const void* latent, int64_t num_tokens, int num_heads, void* k_out, void* v_out,
                          int32_t* status) {
  UpParams p{};
  p.latent = static_cast<const __nv_bfloat16*>(latent);
  p.k = static_cast<__nv_bfloat16*>(k_out);
  p.v = static_cast<__nv_bfloat16*>(v_out);
  p.status = status;
  p.num_tokens = num_tokens;
  p.num_heads = num_heads;
  p.out_align32 = ((reinterpret_cast<uintptr_t>(k_out) | reinterpret_cast<uintptr_t>(v_out)) & 31u) == 0;
  return p;
}

cudaError_t launch_up_proj(const CUtensorMap& ta, const CUtensorMap& tb, const void* latent,
                           int64_t num_tokens, int num_heads, void* k_out, void* v_out,
                           int32_t* status, cudaStream_t stream) {
  UpParams p = up_params(latent, num_tokens, num_heads, k_out, v_out, status);
  return launch_up_proj_t<false>(ta, tb, p, stream);
}

cudaError_t launch_up_proj_paged(const CUtensorMap& ta, const CUtensorMap& tb, const void* cache, int64_t num_blocks,
                                 int block_size, const int32_t* block_table, int max_blocks_per_req,
                                 const int32_t* cu_seq_lens, const int32_t* chunk_starts, int batch,
                                 int64_t total_tokens, int num_heads, void* k_out, void* v_out, void* rope_out,
                                 int32_t* status, cudaStream_t stream) {
  UpParams p = up_params(cache, total_tokens, num_heads, k_out, v_out, status);
  p.rope_out = static_cast<__nv_bfloat16*>(rope_out);
  p.split_rope = rope_out != nullptr;
  if (p.split_rope) p.out_align32 = p.out_align32 && (reinterpret_cast<uintptr_t>(rope_out) & 31u) == 0;
  p.rows = RowMap{cu_seq_lens, chunk_starts, block_table, batch, max_blocks_per_req, block_size, num_blocks};
  p.oob_row = (int32_t)(num_blocks * block_size);
  return launch_up_proj_t<true>(ta, tb, p, stream);
}

}  // namespace mla
