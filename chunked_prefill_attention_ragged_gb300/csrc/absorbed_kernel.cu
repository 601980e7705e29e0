// Absorbed-weight MLA prefill: multi-query attention of every head over the compressed
// latent cache rows, O_lat = softmax(sm_scale * q_abs . c^T) c[:, :512] and the per-row LSE.
//
// What is computed follows sglang issue #3849 ("[DeepseekR1] How ragged prefill manage
// kv_cache?"): prefill with a cached prefix runs forward_absorb, attention over the cache
// rows (512 latent + 64 rope per token, one KV head shared by all heads) with W_UK folded
// into the query; Apache TVM PR #17674: under absorption sm_scale is passed explicitly.
// The keys of request r are its cache positions 0 .. kv_len - 1, found through the block
// table by the slot rule of vLLM "vllm/models/deepseek_v4/sparse_mla.py"
// (_build_c128a_topk_metadata_kernel, decode branch); its queries are the last q_len of
// them (bottom-right causal alignment, as in the MHA prefill).
//
// Design.  A unit is 128 consecutive (query row, head) pairs of one request (all heads of
// a row share its keys and its causal limit) and one half of the 512 value columns: a
// 128 x 512 fp32 accumulator would take all 512 TMEM columns, so each CTA keeps O for 256
// of them (256 columns) beside two S buffers of 64 keys, and S = q_abs . K^T (576 deep) is
// computed once per half.  Shared memory holds the unit's Q tile (128 x 576 bf16, nine
// 64-column panels, 144 KB) and one 64-key tile of cache rows in nine 8 KB panel slots
// (72 KB); V is the tile's own first 512 columns, so the four panels of this CTA's value
// half serve S = Q K^T and then P V.  Per tile t the MMA issuer runs P(t - 1) V(t - 1)
// first (which frees the value panels for tile t's loads, so they travel while the next
// products run), then S(t)'s products over the five panels outside the value half (loaded
// long before; their slots refill for tile t + 1 at once), then over the value panels.
//   warps 0, 3 producers (warp 0: the Q tile and the five panels outside the value half,
//              warp 3: the four value panels), each panel group behind one barrier.  A
//              tile inside kv_len comes by tile copies: one per run of adjacent panels
//              when the block size is a multiple of 64, one per panel and block when it
//              is 8, 16 or 32; otherwise (a request's last tile, other block sizes) by
//              tile::gather4 copies, lanes 0-15 fetching keys 4l .. 4l+3 by slot (rows
//              past kv_len or in an unknown block read as zeros)
//   warp 1     MMA issuer (one thread): S = Q K^T (M 128, N 64) into S[t % 2];
//              O += P V (M 128, N 256) with P from TMEM
//   warp 2     TMEM allocation
//   warps 4-7  softmax, one thread per pair: online softmax in base 2, O in TMEM rescaled
//              only when a row's max grows by more than 2^8; at the end O / l -> bf16 and
//              the natural-log LSE
// Every wait is bounded: on time-out the CTA records MLA_DEVSTAT_TIMEOUT, drains its own
// copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "tmem_wide.cuh"

namespace mla {
namespace {

constexpr int AM = 128;                 // (row, head) pairs per unit
constexpr int AN = 64;                  // keys per tile
constexpr int NP = 9;                   // 64-column panels of 576
constexpr int Q_PANEL = AM * 128;       // 16 KB
constexpr int K_PANEL = AN * 128;       // 8 KB
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + NP * Q_PANEL;
constexpr int OFF_BAR = OFF_K + NP * K_PANEL;
enum ABar {
  QF = 0,             // Q tile landed
  KF = 1,             // [panel group] this tile's panels landed (group 0: the five panels
                      // outside the value half; group 1: the value half's four)
  KE = KF + 2,        // [panel group] the group's last product done: its slots may refill
  SF = KE + 2,        // [S buffer] S = Q K^T done
  SE = SF + 2,        // [S buffer] P V done reading its P
  PR = SE + 2,        // [S buffer] P written by all four softmax warps
  OD = PR + 2,        // [tile parity] O += P V done
  FIN = OD + 2,       // every MMA drained before TMEM is released
  NEVER,              // nothing arrives here: the time-out test mode waits on it
  NBAR
};
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM = OFF_MISC + 16 + 1024;   // + slack for 1024-byte alignment
static_assert(SMEM <= 227 * 1024, "shared memory budget");
constexpr int NTHREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0;                  // 256 columns: this CTA's value half
__device__ __forceinline__ constexpr uint32_t TM_S(int b) { return 256u + (uint32_t)b * 64u; }
constexpr uint32_t IDESC_QK = idesc_bf16_f32(AM, AN, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16_f32(AM, 256, false, true);
constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;
constexpr float RESCALE_THRESHOLD = 8.0f;

// Issue order of a tile's panels: the five outside the value half, then its four.
__device__ __forceinline__ int panel_order(int i, int half) {
  const int v0 = 4 * half;   // first value panel
  if (i < 5) return i < v0 ? i : i + 4;   // half 0: 4..8; half 1: 0..3, 8
  return v0 + (i - 5);
}

struct ACtx {
  uint32_t sbase;
  volatile int* abort_flag;
  int* status;
  uint64_t wait_limit_ns;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BAR + 8 * i; }
  __device__ bool wait(int b, uint32_t parity) const {
    return mbar_wait_bounded(bar(b), parity, abort_flag, status, MLA_DEVSTAT_TIMEOUT, wait_limit_ns);
  }
  __device__ void drain(int b, uint32_t parity) const {
    int dummy = 0;
    mbar_wait_bounded(bar(b), parity, &dummy, status, MLA_DEVSTAT_TIMEOUT, DRAIN_LIMIT_NS);
  }
};

__device__ __forceinline__ AbsUnit load_aunit(const AbsUnit* units, int i) {
  const int4* q = reinterpret_cast<const int4*>(units + i);
  const int4 a = __ldg(q), b = __ldg(q + 1);
  AbsUnit u;
  u.pair0 = a.x; u.npairs = a.y; u.q_row0 = a.z; u.q_len = a.w;
  u.kv_len = b.x; u.ntiles = b.y; u.half = b.z; u.req = b.w;
  return u;
}

// Cache row of key position `key` of the unit's request; past kv_len, or in a block that
// the table does not name, the row past the cache (read as zeros), the latter flagged.
__device__ __forceinline__ int32_t key_row(const AbsorbedParams& p, const AbsUnit& u, int key) {
  if (key >= u.kv_len) return p.oob_row;
  const int bi = key / p.block_size;
  const int32_t blk = bi < p.max_blocks ? __ldg(p.block_table + (int64_t)u.req * p.max_blocks + bi) : -1;
  if (blk < 0 || (int64_t)blk >= p.num_blocks) {
    if (p.status) atomicOr(p.status, MLA_DEVSTAT_BAD_INDEX);
    return p.oob_row;
  }
  return (int32_t)((int64_t)blk * p.block_size + (key - bi * p.block_size));
}

// ------------------------------------------------------------------ producers (warps 0, 3)
// Panel group g of every tile (and, for group 0, the Q tile): warp 0 loads the five panels
// outside the value half, warp 3 the four value panels, so that tile t + 1's first panels
// load as soon as S(t) has used their slots, without waiting behind tile t's value panels
// (which wait for P(t - 1) V).  A whole tile inside kv_len with 64-row block pieces takes
// one copy per run of adjacent panels (a three-dimensional map over the cache rows: 64
// columns, rows, nine 64-column groups).
__device__ void run_producer(const ACtx& c, const AbsorbedParams& p, const AbsUnit& u, const CUtensorMap* tq,
                             const CUtensorMap* tc, const CUtensorMap* tb, const CUtensorMap* t4, int g) {
  const int lane = threadIdx.x & 31;
  const int h = u.half;
  const int i0 = g == 0 ? 0 : 5, i1 = g == 0 ? 5 : NP;
  if (g == 0 && lane == 0) {
    mbar_arrive_expect_tx(c.bar(QF), NP * Q_PANEL);
    for (int i = 0; i < NP; ++i) tma_load_2d(c.sbase + OFF_Q + i * Q_PANEL, tq, c.bar(QF), i * 64, u.pair0);
  }
  bool ok = true;
  int issued = 0;   // tiles requested
  const int pieces = p.piece_rows > 0 ? AN / p.piece_rows : 0;
  for (int t = 0; t < u.ntiles && ok; ++t) {
    // Whole tile inside the request and block pieces available: tile loads, lane k
    // holding piece k's row.  Rows are looked up once per tile, for all the panels.
    const bool by_block = pieces > 0 && (t + 1) * AN <= u.kv_len;
    int32_t r4[4] = {0, 0, 0, 0};
    int32_t piece_row = 0;
    if (by_block) {
      if (lane < pieces) piece_row = key_row(p, u, t * AN + lane * p.piece_rows);
    } else if (lane < 16) {
#pragma unroll
      for (int j = 0; j < 4; ++j) r4[j] = key_row(p, u, t * AN + 4 * lane + j);
    }
    int free = 1;
    if (lane == 0 && t > 0) free = c.wait(KE + g, (t - 1) & 1);
    if (!__shfl_sync(0xffffffffu, free, 0)) { ok = false; break; }
    if (lane == 0) mbar_arrive_expect_tx(c.bar(KF + g), (i1 - i0) * K_PANEL);
    __syncwarp();
    if (by_block && p.grouped) {
      // Runs of adjacent panels: value half [4h, 4h+4); outside it, half 0: [4, 8) and 8,
      // half 1: [0, 4) and 8.
      if (lane == 0) {
        const uint32_t bar = c.bar(KF + g);
        if (g == 1) {
          tma_load_3d(c.sbase + OFF_K + 4 * h * K_PANEL, t4, bar, 0, piece_row, 4 * h);
        } else {
          const int run0 = h == 0 ? 4 : 0;
          tma_load_3d(c.sbase + OFF_K + run0 * K_PANEL, t4, bar, 0, piece_row, run0);
          tma_load_2d(c.sbase + OFF_K + 8 * K_PANEL, tb, bar, 8 * 64, piece_row);
        }
      }
    } else {
      for (int i = i0; i < i1; ++i) {
        const int pnl = panel_order(i, h);
        if (by_block) {
          if (lane < pieces)
            tma_load_2d(c.sbase + OFF_K + pnl * K_PANEL + lane * p.piece_rows * 128, tb, c.bar(KF + g), pnl * 64,
                        piece_row);
        } else if (lane < 16) {
          tma_gather4(c.sbase + OFF_K + pnl * K_PANEL + lane * 4 * 128, tc, c.bar(KF + g), pnl * 64, r4[0], r4[1],
                      r4[2], r4[3]);
        }
      }
    }
    ++issued;
  }
  // Let every copy started here land before the CTA can exit.
  if (lane == 0) {
    if (g == 0) c.drain(QF, 0);
    if (issued > 0) c.drain(KF + g, (issued - 1) & 1);
  }
}

// ------------------------------------------------------------------ MMA issuer (warp 1)
__device__ void run_mma(const ACtx& c, const AbsorbedParams& p, const AbsUnit& u, uint32_t tmem) {
  const int n = u.ntiles, h = u.half;
  bool ok = true;
  if (p.force_timeout) ok = c.wait(NEVER, 0);
  if (ok && n > 0) ok = c.wait(QF, 0);
  const uint64_t q_desc = sdesc_sw128(c.sbase + OFF_Q, 16, 1024);
  const uint64_t k_desc = sdesc_sw128(c.sbase + OFF_K, 16, 1024);
  const uint64_t v_desc = sdesc_sw128(c.sbase + OFF_K + 4 * h * K_PANEL, K_PANEL, 1024);
  auto s_products = [&](int t, int g) {   // S(t) += Q K^T over panel group g (0: i = 0..4, 1: i = 5..8)
    if (!c.wait(KF + g, t & 1)) return false;
    tc_fence_after();
    for (int i = g == 0 ? 0 : 5; i < (g == 0 ? 5 : NP); ++i) {
      const int pnl = panel_order(i, h);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t qo = (uint64_t)((pnl * Q_PANEL + kk * 32) >> 4);
        const uint64_t ko = (uint64_t)((pnl * K_PANEL + kk * 32) >> 4);
        mma_ss(tmem + TM_S(t & 1), q_desc + qo, k_desc + ko, IDESC_QK, (i > 0 || kk > 0) ? 1u : 0u);
      }
    }
    if (g == 0) tc_commit(c.bar(KE + 0));   // the panels outside the value half: free after S
    return true;
  };
  for (int t = 0; t <= n && ok; ++t) {
    if (t >= 1) {
      const int v = t - 1, pb = v & 1;
      if (!c.wait(PR + pb, (v >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < AN / 16; ++kk)
        mma_ts(tmem + TM_O, tmem + TM_S(pb) + kk * 8, v_desc + (uint64_t)(kk * 16 * 128 >> 4), IDESC_PV,
               (v > 0 || kk > 0) ? 1u : 0u);
      tc_commit(c.bar(KE + 1));   // the value panels: free after P V
      tc_commit(c.bar(SE + pb));
      tc_commit(c.bar(OD + pb));
    }
    if (t < n) {
      // S(t) overwrites the buffer that held P(t - 2): P(t - 2) V must be done.
      if (t >= 2 && !c.wait(SE + (t & 1), ((t - 2) >> 1) & 1)) { ok = false; break; }
      if (!s_products(t, 0)) { ok = false; break; }
      if (!s_products(t, 1)) { ok = false; break; }
      tc_commit(c.bar(SF + (t & 1)));
    }
  }
  tc_commit(c.bar(FIN));
  c.drain(FIN, 0);
}

// ------------------------------------------------------------------ softmax (warps 4-7)
__device__ void run_softmax(const ACtx& c, const AbsorbedParams& p, const AbsUnit& u, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = (warp - 4) * 32 + lane;   // TMEM lane = pair of the unit
  const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const float NEG_INF = -__int_as_float(0x7f800000);
  const int64_t pair = (int64_t)u.pair0 + i;
  const bool live = i < u.npairs;
  const int pos = (int)(pair / p.num_heads) - u.q_row0;   // query position inside the request
  const int diag = u.kv_len - u.q_len;
  const int khi = p.causal ? min(u.kv_len, pos + diag + 1) : u.kv_len;   // allowed keys [0, khi)
  __nv_bfloat16* orow = p.o + pair * 512 + u.half * 256;
  const int n = u.ntiles;
  if (n == 0) {   // no key at all: O = 0, LSE = -inf
    if (live) {
      uint4* d = reinterpret_cast<uint4*>(orow);
#pragma unroll
      for (int k = 0; k < 32; ++k) d[k] = make_uint4(0, 0, 0, 0);
      if (p.lse && u.half == 0) p.lse[pair] = NEG_INF;
    }
    return;
  }
  const float sc = p.has_cap ? 1.f : p.scale_log2;
  const float2 sc2 = make_float2(sc, sc);
  float m_used = NEG_INF, l = 0.f;
  bool ok = true;
  for (int t = 0; t < n; ++t) {
    const int sb = t & 1;
    if (!__all_sync(0xffffffffu, c.wait(SF + sb, (t >> 1) & 1))) { ok = false; break; }
    tc_fence_after();
    float sv[64];
    tmem_ld64_sync(lane_addr + TM_S(sb), reinterpret_cast<uint32_t*>(sv));
    if (p.has_cap) {
      // c * tanh(sm_scale * x / c) in log2 units, from tanh(y) = 1 - 2 / (e^(2y) + 1).
      const float2 k2 = make_float2(p.cap_ex2_scale, p.cap_ex2_scale);
      const float2 one = make_float2(1.f, 1.f);
      const float2 m2c = make_float2(-2.f * p.cap_log2, -2.f * p.cap_log2);
      const float2 c2 = make_float2(p.cap_log2, p.cap_log2);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float2 a = fmul2(make_float2(sv[2 * k], sv[2 * k + 1]), k2);
        const float2 d = fadd2(make_float2(ex2_approx(a.x), ex2_approx(a.y)), one);
        const float2 r = ffma2(make_float2(rcp_approx(d.x), rcp_approx(d.y)), m2c, c2);
        sv[2 * k] = r.x;
        sv[2 * k + 1] = r.y;
      }
    }
    const int c_hi = khi - t * AN;
    if (c_hi < AN) {
#pragma unroll
      for (int k = 0; k < 64; ++k)
        if (k >= c_hi) sv[k] = NEG_INF;
    }
    float mx[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      mx[k] = fmax3(fmax3(sv[8 * k], sv[8 * k + 1], sv[8 * k + 2]), fmax3(sv[8 * k + 3], sv[8 * k + 4], sv[8 * k + 5]),
                    fmaxf(sv[8 * k + 6], sv[8 * k + 7]));
    const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sc;
    float m_new = m_used;
    bool rescale = false;
    if (t == 0) {
      m_new = mt;
    } else if (mt > m_used + RESCALE_THRESHOLD) {
      m_new = mt;
      rescale = true;
    }
    const float msub = (m_new == NEG_INF) ? 0.f : m_new;
    const float2 neg_m = make_float2(-msub, -msub);
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    uint32_t pr[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float2 a = ffma2(make_float2(sv[2 * k], sv[2 * k + 1]), sc2, neg_m);
      const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
      acc[k & 3] = fadd2(acc[k & 3], e);
      pr[k] = pack_bf16x2(e.x, e.y);
    }
    const float2 s01 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
    const float sum = s01.x + s01.y;
    tmem_st32_sync(lane_addr + TM_S(sb), pr);   // P over the front of its S
    float alpha = 1.f;
    // tcgen05.ld/st are warp-collective: the whole warp rescales (alpha = 1 for rows that
    // keep their max), after P(t - 1) V has landed in O.
    if (t > 0 && __any_sync(0xffffffffu, rescale)) {
      const int pv = t - 1;
      if (!__all_sync(0xffffffffu, c.wait(OD + (pv & 1), (pv >> 1) & 1))) { ok = false; break; }
      tc_fence_after();
      if (rescale) alpha = ex2_approx(m_used - m_new);
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        float ov[64];
        tmem_ld64_sync(lane_addr + TM_O + q * 64, reinterpret_cast<uint32_t*>(ov));
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float2 r = fmul2(make_float2(ov[2 * k], ov[2 * k + 1]), a2);
          ov[2 * k] = r.x;
          ov[2 * k + 1] = r.y;
        }
        tmem_st64_sync(lane_addr + TM_O + q * 64, reinterpret_cast<uint32_t*>(ov));
      }
    }
    l = l * alpha + sum;
    m_used = m_new;
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(PR + sb));
  }
  if (!ok) return;
  // The unit's last product.  Its parity wait is exact: P(n - 3) V completed before S(n - 1)
  // could be computed (S(n - 1) reuses P(n - 3)'s buffer), and no later product exists.
  const int last = n - 1;
  if (!__all_sync(0xffffffffu, c.wait(OD + (last & 1), (last >> 1) & 1))) return;
  tc_fence_after();
  const bool empty = !(l > 0.f);
  const float inv = empty ? 0.f : 1.f / l;
  const float2 inv2 = make_float2(inv, inv);
#pragma unroll 1
  for (int q = 0; q < 4; ++q) {
    float ov[64];
    tmem_ld64_sync(lane_addr + TM_O + q * 64, reinterpret_cast<uint32_t*>(ov));
    uint32_t w[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const float2 r = fmul2(make_float2(ov[2 * k], ov[2 * k + 1]), inv2);
      w[k] = pack_bf16x2(r.x, r.y);
    }
    if (live) {
      uint4* d = reinterpret_cast<uint4*>(orow + q * 64);
#pragma unroll
      for (int k = 0; k < 8; ++k) d[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
    }
  }
  if (live && p.lse && u.half == 0) {
    float lg;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l));
    p.lse[pair] = empty ? NEG_INF : (m_used + lg) * 0.6931471805599453f;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
absorbed_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_c,
                const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_4,
                const AbsorbedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* abort_flag = reinterpret_cast<int*>(smem + OFF_MISC + 4);
  ACtx c{smem_addr(smem), abort_flag, p.status, p.wait_limit_ns};
  const AbsUnit u = load_aunit(p.units, blockIdx.x);
  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(c.bar(i), 1);
    for (int i = 0; i < 2; ++i) mbar_init(c.bar(PR + i), 4);   // one arrival per softmax warp
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_c);
    if (p.piece_rows > 0) tma_prefetch_desc(&tm_b);
    if (p.grouped) tma_prefetch_desc(&tm_4);
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 0) {
    if (u.ntiles > 0) run_producer(c, p, u, &tm_q, &tm_c, &tm_b, &tm_4, 0);
  } else if (warp == 3) {
    if (u.ntiles > 0) run_producer(c, p, u, &tm_q, &tm_c, &tm_b, &tm_4, 1);
  } else if (warp == 1) {
    if (lane == 0) run_mma(c, p, u, tmem);
  } else if (warp >= 4) {
    run_softmax(c, p, u, tmem);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) {
    __syncwarp();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_absorbed(const CUtensorMap& tq, const CUtensorMap& tc, const CUtensorMap& tb,
                            const CUtensorMap& t4, const AbsorbedParams& p, int num_units, cudaStream_t stream) {
  static PerDeviceOnce configured;
  const cudaError_t e = configured.run(
      [] { return cudaFuncSetAttribute(absorbed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM); });
  if (e != cudaSuccess) return e;
  absorbed_kernel<<<num_units, NTHREADS, SMEM, stream>>>(tq, tc, tb, t4, p);
  return cudaGetLastError();
}

}  // namespace mla
