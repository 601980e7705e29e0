// Ragged MLA prefill attention for sm_103a: O = softmax(sm_scale * Q K^T) V and the
// per-row LSE, for query/key head dim 192 (128 NoPE + 64 RoPE) and value dim 128.
//
// What is computed follows vLLM "vllm.v1.attention.backends.mla.prefill.flashinfer"
// (FlashInferPrefillBackend.finalize_attention_metadata: ragged qo/kv indptr, MHA,
// causal for new tokens / non-causal for prefix chunks, sm_scale, window_left,
// logits_soft_cap; FlashInferPrefillImpl.run_prefill_*: O and LSE per (row, head)).
//
// Design (persistent, one CTA per SM, four warpgroups, registers moved between them with
// setmaxnreg).  A work unit is 128 query rows of one head (kPair = false), or 256 rows of
// one head run by the two CTAs of a cluster (kPair): each CTA owns 128 of the rows, and
// the pair's tensor-core products (tcgen05 cta_group::2, M = 256) read each K and V tile
// half from either CTA, so every CTA loads half of the K/V bytes and its rings hold four
// stages instead of two.  Plans use the pair instances only when asked to: on every
// batch shape measured they ran 3-10% slower than single CTAs.
//   warps 0, 2  TMA producers: warp 0 loads the Q tile once per unit and K tiles of 128
//               keys (a CTA of a pair: its 64 of them), warp 2 V tiles (a CTA of a pair:
//               its 64 of the 128 value columns).
//   warps 1, 3  MMA issuers (one thread each; in a pair only in the even CTA): warp 1
//               issues S = Q K^T into one of three TMEM S buffers (both operands from
//               shared memory), so S runs up to two tiles ahead of the softmax; warp 3
//               issues O += P V with P read from TMEM.  In the odd CTA of a pair these
//               warps forward its own Q/K and V arrivals to the even CTA's barriers.
//   warps 4-11  softmax: two threads per query row (= one TMEM lane), each owning 64
//               of the tile's 128 key columns and 64 of O's 128 columns.  Online
//               softmax in base 2; O in TMEM is rescaled only when the running max
//               grows by more than 2^8, so most tiles need no correction pass.  At the
//               end of a unit they only publish each row's sum and max and go on.
//   warps 12-15 epilogue: read O from TMEM once the unit's last P V is done, release
//               it for the next unit's first P V, then normalise, write O (bf16) and
//               the natural-log LSE (fp32), off the softmax warps' critical path.  In
//               the merging instance (kMerge) they instead merge the result into the
//               partial (O, LSE) state already in memory: the chunk step of chunked
//               prefill, where run_prefill_context_chunk's LSE serves that merge.
// TMEM: S buffers 0-2 (128 columns each; P overwrites the front of its S as bf16), O.
// Every pipeline wait is bounded: on time-out the CTA records MLA_DEVSTAT_TIMEOUT,
// drains its own copies and MMAs, frees TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "tmem_wide.cuh"

namespace mla {
namespace {

constexpr int BM = kTileM;    // 128 query rows per CTA
constexpr int BN = kTileN;    // 128 keys per tile
constexpr int PANEL = 128 * 64 * 2;   // one 128-row x 64-element bf16 panel, 128B swizzle
constexpr int Q_PANELS = 3, K_PANELS = 3;
constexpr int NSB = 3;   // S buffers in TMEM

// Shared-memory layout.  One CTA per unit: K and V tiles of 128 keys, two stages each.  A
// CTA pair per unit: each CTA holds 64 keys of every K tile and 64 of the 128 value
// columns of every V tile, four stages each.
template <bool kPair>
struct Lay {
  static constexpr int KROWS = kPair ? 64 : 128;                 // keys of a K tile held here
  static constexpr int KPANEL = KROWS * 64 * 2;                   // one 64-column K panel
  static constexpr int V_PANELS = kPair ? 1 : 2;                  // 64-column V panels held here
  static constexpr int NK = kPair ? 4 : 2, NV = kPair ? 4 : 2;   // stages
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_PANELS * PANEL;
  static constexpr int OFF_V = OFF_K + NK * K_PANELS * KPANEL;
  static constexpr int OFF_BAR = OFF_V + NV * V_PANELS * PANEL;
};
constexpr int MAX_STAGES = 4;
enum Bar {
  QF = 0, QE = 1,       // Q landed (in a pair's even CTA: both CTAs' Q) / released
  KF = 2,               // [stage] K tile landed (a pair's even CTA: both halves)
  KE = KF + MAX_STAGES, // [stage] K tile released
  VF = KE + MAX_STAGES, // [stage] V tile landed (a pair's even CTA: both halves)
  VE = VF + MAX_STAGES, // [stage] V tile released
  SF = VE + MAX_STAGES, // [S buffer] S = Q K^T done
  SE = SF + NSB,        // [S buffer] P V done reading P: S may be overwritten
  OD = SE + NSB,        // [tile parity] O += P V done
  FINQ = OD + 2,        // all MMAs of the S issuer drained before TMEM is released
  FINP,                 // the same for the P V issuer
  PR,                   // [S buffer][half row] P written by that half's four softmax warps
                        // (of both CTAs of a pair): keys 0-63 / 64-127 of the tile
  LR = PR + 2 * NSB,    // [unit parity] row sums and max of a unit published
  LFR = LR + 2,         // [unit parity] the epilogue has read them
  OFR = LFR + 2,        // the epilogue (of both CTAs of a pair) has read O: the next
                        // unit's first P V may overwrite it
  NEVER,                // nothing arrives here: the time-out test mode waits on it
  NBAR
};
// Parity waits: a wait for phase f of a barrier is exact only while phase f - 1 has
// completed and phase f + 1 cannot have.  O-done is split by tile parity so that the
// softmax (which waits for product g - 1 only when tile g rescales O) and the epilogue
// (which waits for a unit's last two products) both meet that: products complete in
// order, P(g - 3) V has completed whenever S(g) exists, and P(g + 1) V needs a P (or the
// epilogue's release of O) not yet given.
// Exchange area: per (tile parity, half, row) an 8-byte word (half-row max, tile) for the
// max exchange between the two halves of a row, then per unit parity both halves' row
// sums and the row max: 4096 + 3 x 2 x 128 x 4 bytes.
constexpr int XCHG_WORDS = 2 * 2 * 128;   // (max, tile) words
constexpr int XCHG_BYTES = XCHG_WORDS * 8 + 6 * 128 * 4;
template <bool kPair>
struct Off {
  static constexpr int XCHG = Lay<kPair>::OFF_BAR + NBAR * 8;
  static constexpr int MISC = XCHG + XCHG_BYTES;
  static constexpr int SMEM = MISC + 16 + 1024;   // + slack for 1024-byte alignment
};
static_assert(Off<false>::SMEM <= 227 * 1024 && Off<true>::SMEM <= 227 * 1024, "shared memory budget");

constexpr int NTHREADS = 512;   // 4 warpgroups: control, softmax x 2, epilogue
// Registers per thread: launched at 65536 / 512 = 128; the control and epilogue
// warpgroups give some up and the two softmax warpgroups take them (counts at which
// ptxas reports no spills; the merging epilogue needs a few more).
constexpr int LAUNCH_REGS = 128;
template <bool kMerge>
struct RegSplit {
  static constexpr int ctrl = kMerge ? 96 : 88, softmax = kMerge ? 152 : 160, epi = kMerge ? 112 : 104;
  static_assert(4 * 32 * (ctrl + 2 * softmax + epi) <= 4 * 32 * 4 * LAUNCH_REGS,
                "register split exceeds the launch allocation");
};
constexpr uint32_t TMEM_COLS = 512;
__device__ __forceinline__ constexpr uint32_t TM_S(int b) { return (uint32_t)b * 128u; }
constexpr uint32_t TM_O = 384;

// M = 128 rows per CTA, or 256 over a pair; N = 128 keys (S) or 128 value columns (P V).
template <bool kPair>
struct Idesc {
  static constexpr uint32_t QK = idesc_bf16_f32(kPair ? 256 : BM, BN, false, false);
  static constexpr uint32_t PV = idesc_bf16_f32(kPair ? 256 : BM, 128, false, true);
};

constexpr uint64_t DRAIN_LIMIT_NS = 200000000ull;    // 0.2 s: own copies and MMAs after an abort
constexpr float RESCALE_THRESHOLD = 8.0f;             // log2 units

template <bool kPair>
struct Ctx {
  uint32_t sbase;
  volatile int* abort_flag;
  int* status;
  uint64_t wait_limit_ns;
  uint32_t rank;   // the CTA's rank in its pair (0 without pairs)
  __device__ uint32_t bar(int i) const { return sbase + Lay<kPair>::OFF_BAR + 8 * i; }
  __device__ bool wait(int b, uint32_t parity) const {
    return mbar_wait_bounded(bar(b), parity, abort_flag, status, MLA_DEVSTAT_TIMEOUT, wait_limit_ns);
  }
  // For barriers that threads of the other CTA of a pair arrive on (the even CTA's Q/K/V
  // landed, P written and O read barriers): acquire at cluster scope.
  __device__ bool wait_pair(int b, uint32_t parity) const {
    return mbar_wait_bounded(bar(b), parity, abort_flag, status, MLA_DEVSTAT_TIMEOUT, wait_limit_ns, kPair);
  }
  __device__ void drain(int b, uint32_t parity) const {
    int dummy = 0;
    mbar_wait_bounded(bar(b), parity, &dummy, status, MLA_DEVSTAT_TIMEOUT, DRAIN_LIMIT_NS, kPair);
  }
  // Arrive on barrier b of the even CTA of the pair (this CTA's own without pairs).
  __device__ void arrive_leader(int b) const {
    if (kPair && rank != 0)
      mbar_arrive_remote(mapa_shared(bar(b), 0));
    else
      mbar_arrive(bar(b));
  }
  // Commit this thread's tensor-core work to barrier b of this CTA, or of both CTAs of a pair.
  __device__ void commit(int b) const {
    if constexpr (kPair) tc_commit_pair(bar(b)); else tc_commit(bar(b));
  }
  __device__ void commit_both(int b) const {
    if constexpr (kPair) {
      tc_commit_pair(bar(b));
      tc_commit_pair(mapa_shared(bar(b), 1));
    } else {
      tc_commit(bar(b));
    }
  }
};

__device__ __forceinline__ Unit load_unit(const Unit* units, int i) {
  const int4* p = reinterpret_cast<const int4*>(units + i);
  int4 a = __ldg(p), b = __ldg(p + 1);
  Unit u;
  u.head = a.x; u.q_row0 = a.y; u.q_rows = a.z; u.q_pos0 = a.w;
  u.kv_row0 = b.x; u.kv_len = b.y; u.diag = b.z; u.kv_tiles = b.w;
  return u;
}

// The unit's query rows that this CTA owns: all of them without pairs (at most 128); in a
// pair the first 128 for the even CTA and the rest (possibly none) for the odd one.
template <bool kPair>
__device__ __forceinline__ Unit own_rows(Unit u, uint32_t rank) {
  if constexpr (kPair) {
    if (rank != 0) {
      u.q_row0 += BM;
      u.q_pos0 += BM;
      u.q_rows = u.q_rows > BM ? u.q_rows - BM : 0;
    } else if (u.q_rows > BM) {
      u.q_rows = BM;
    }
  }
  return u;
}

// ------------------------------------------------------------------ producers
// Two producer threads, so that a K load never queues behind a V load waiting for its
// stage: warp 0 loads Q (once per unit) and K tiles, warp 2 loads V tiles.  A K stage
// frees when its S = Q K^T is done, a V stage when its P V is done.  In a pair each CTA
// loads its own Q rows, its half of the K tile's keys and its half of V's columns.
template <bool kPair>
__device__ void run_producer_qk(const Ctx<kPair>& c, const PrefillParams& p, const CUtensorMap* tq,
                                const CUtensorMap* tk, const CUtensorMap* tr, int ubeg, int uend) {
  using L = Lay<kPair>;
  int q_g = 0, k_g = 0;   // loads issued so far (Q tiles, K tiles)
  bool ok = true;
  for (int ui = ubeg; ui < uend && ok; ++ui) {
    const Unit u = load_unit(p.units, ui);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    if (hi <= lo) continue;
    if (q_g > 0 && !c.wait(QE, (q_g - 1) & 1)) { ok = false; break; }
    mbar_arrive_expect_tx(c.bar(QF), Q_PANELS * PANEL);
    const int q_row = u.q_row0 + (kPair ? BM * (int)c.rank : 0);
    for (int i = 0; i < Q_PANELS; ++i)
      tma_load_3d(c.sbase + L::OFF_Q + i * PANEL, tq, c.bar(QF), i * 64, u.head, q_row);
    ++q_g;
    for (int t = lo; t < hi; ++t) {
      const int row = u.kv_row0 + t * BN + (kPair ? L::KROWS * (int)c.rank : 0);
      const int s = k_g % L::NK;
      const uint32_t use = k_g / L::NK;
      if (use > 0 && !c.wait(KE + s, (use - 1) & 1)) { ok = false; break; }
      mbar_arrive_expect_tx(c.bar(KF + s), K_PANELS * L::KPANEL);
      // Panels 0-1 are K's NoPE columns; panel 2 its RoPE columns, which with a shared
      // rope come from the one [tokens, 64] rope tensor that every head uses.
      for (int i = 0; i < K_PANELS; ++i) {
        const uint32_t dst = c.sbase + L::OFF_K + (s * K_PANELS + i) * L::KPANEL;
        if (p.shared_rope && i == K_PANELS - 1)
          tma_load_2d(dst, tr, c.bar(KF + s), 0, row);
        else
          tma_load_3d(dst, tk, c.bar(KF + s), i * 64, u.head, row);
      }
      ++k_g;
    }
  }
  // Let every copy this thread started land before the CTA can exit: wait for the
  // last phase issued on each barrier (already complete on the normal path).
  if (q_g > 0) c.drain(QF, (q_g - 1) & 1);
  for (int s = 0; s < L::NK; ++s)
    if (k_g > s) c.drain(KF + s, (((k_g - 1 - s) / L::NK)) & 1);
}

template <bool kPair>
__device__ void run_producer_v(const Ctx<kPair>& c, const PrefillParams& p, const CUtensorMap* tv, int ubeg,
                               int uend) {
  using L = Lay<kPair>;
  int v_g = 0;
  bool ok = true;
  for (int ui = ubeg; ui < uend && ok; ++ui) {
    const Unit u = load_unit(p.units, ui);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    for (int t = lo; t < hi; ++t) {
      const int row = u.kv_row0 + t * BN;
      const int s = v_g % L::NV;
      const uint32_t use = v_g / L::NV;
      if (use > 0 && !c.wait(VE + s, (use - 1) & 1)) { ok = false; break; }
      mbar_arrive_expect_tx(c.bar(VF + s), L::V_PANELS * PANEL);
      for (int i = 0; i < L::V_PANELS; ++i)
        tma_load_3d(c.sbase + L::OFF_V + (s * L::V_PANELS + i) * PANEL, tv, c.bar(VF + s),
                    kPair ? 64 * (int)c.rank : i * 64, u.head, row);
      ++v_g;
    }
  }
  for (int s = 0; s < L::NV; ++s)
    if (v_g > s) c.drain(VF + s, (((v_g - 1 - s) / L::NV)) & 1);
}

// The odd CTA of a pair: once its own Q / K half / V half of a tile has landed, tell the
// even CTA, whose MMA issuers wait for both CTAs' halves on their own barriers.
__device__ void run_forward_qk(const Ctx<true>& c, const PrefillParams& p, int ubeg, int uend) {
  using L = Lay<true>;
  int q_g = 0, k_g = 0;
  for (int ui = ubeg; ui < uend; ++ui) {
    const Unit u = load_unit(p.units, ui);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    if (hi <= lo) continue;
    if (!c.wait(QF, q_g & 1)) return;
    mbar_arrive_remote(mapa_shared(c.bar(QF), 0));
    ++q_g;
    for (int t = lo; t < hi; ++t, ++k_g) {
      const int s = k_g % L::NK;
      if (!c.wait(KF + s, (k_g / L::NK) & 1)) return;
      mbar_arrive_remote(mapa_shared(c.bar(KF + s), 0));
    }
  }
}

__device__ void run_forward_v(const Ctx<true>& c, const PrefillParams& p, int ubeg, int uend) {
  using L = Lay<true>;
  int v_g = 0;
  for (int ui = ubeg; ui < uend; ++ui) {
    const Unit u = load_unit(p.units, ui);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    for (int t = lo; t < hi; ++t, ++v_g) {
      const int s = v_g % L::NV;
      if (!c.wait(VF + s, (v_g / L::NV) & 1)) return;
      mbar_arrive_remote(mapa_shared(c.bar(VF + s), 0));
    }
  }
}

// ------------------------------------------------------------------ MMA issuer
// Two MMA issuers.  A tcgen05.mma issue returns only once the tensor pipe takes the
// instruction, so every wait of an issuing thread leaves the pipe idle unless another
// thread has products queued: warp 1 issues S = Q K^T, warp 3 issues O += P V, and
// each one's waits hide behind the other's products.  S of tile g + 3 reuses the S
// buffer whose P the product of tile g reads, which the SE barrier orders.  In a pair
// the even CTA issues for both, and commits the barriers of both CTAs.
template <bool kPair>
__device__ void run_mma_qk(const Ctx<kPair>& c, const PrefillParams& p, uint32_t tmem, int ubeg, int uend) {
  using L = Lay<kPair>;
  int q_g = 0, kv_g = 0;
  bool ok = true;
  const uint64_t q_desc = sdesc_sw128(c.sbase + L::OFF_Q, 16, 1024);
  const uint64_t k_desc0 = sdesc_sw128(c.sbase + L::OFF_K, 16, 1024);
  // Time-out test mode: phase 0 of NEVER never completes, so this wait gives up after
  // the plan's limit and the whole CTA takes its abort path.
  if (p.force_timeout) ok = c.wait(NEVER, 0);
  for (int ui = ubeg; ui < uend && ok; ++ui) {
    const Unit u = load_unit(p.units, ui);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    const int n = hi - lo;
    if (n <= 0) continue;
    if (!c.wait_pair(QF, q_g & 1)) { ok = false; break; }
    ++q_g;
    for (int j = 0; j < n && ok; ++j) {
      const int g = kv_g + j, s = g % L::NK, b = g % NSB;
      if (!c.wait_pair(KF + s, (g / L::NK) & 1)) { ok = false; break; }
      if (g >= NSB && !c.wait(SE + b, ((g - NSB) / NSB) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint64_t kd = k_desc0 + (uint64_t)(s * K_PANELS * L::KPANEL >> 4);
#pragma unroll
      for (int kk = 0; kk < 192 / 16; ++kk) {
        const uint64_t q_off = (uint64_t)(((kk >> 2) * PANEL + (kk & 3) * 32) >> 4);
        const uint64_t k_off = (uint64_t)(((kk >> 2) * L::KPANEL + (kk & 3) * 32) >> 4);
        if constexpr (kPair)
          mma_ss_pair(tmem + TM_S(b), q_desc + q_off, kd + k_off, Idesc<kPair>::QK, kk > 0 ? 1u : 0u);
        else
          mma_ss(tmem + TM_S(b), q_desc + q_off, kd + k_off, Idesc<kPair>::QK, kk > 0 ? 1u : 0u);
      }
      c.commit_both(SF + b);
      c.commit_both(KE + s);
      if (j == n - 1) c.commit_both(QE);
    }
    kv_g += n;
  }
  // Every MMA issued by this thread must finish before TMEM is released.
  c.commit(FINQ);
  c.drain(FINQ, 0);
}

template <bool kPair>
__device__ void run_mma_pv(const Ctx<kPair>& c, const PrefillParams& p, uint32_t tmem, int ubeg, int uend) {
  using L = Lay<kPair>;
  int g = 0, k = 0;   // tiles and non-empty units so far
  bool ok = true;
  const uint64_t v_desc0 = sdesc_sw128(c.sbase + L::OFF_V, PANEL, 1024);
  for (int ui = ubeg; ui < uend && ok; ++ui) {
    const Unit u = load_unit(p.units, ui);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    const int n = hi - lo;
    if (n <= 0) continue;
    // The first product of a unit overwrites O: the epilogue must have read the
    // previous unit's O out of TMEM.
    if (k > 0 && !c.wait_pair(OFR, (k - 1) & 1)) { ok = false; break; }
    ++k;
    for (int j = 0; j < n; ++j, ++g) {
      // Tiles are counted alike for S buffers and V stages (both advance once per tile).
      const int b = g % NSB, s = g % L::NV;
      // V lands tiles ahead; P is the input that arrives last, so it is waited for last,
      // one half row at a time: keys 0-63 (P columns 0-31) as soon as that half's softmax
      // warps have written them, keys 64-127 after the other half's.
      if (!c.wait_pair(VF + s, (g / L::NV) & 1)) { ok = false; break; }
      const uint64_t vd = v_desc0 + (uint64_t)(s * L::V_PANELS * PANEL >> 4);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        if (kk % (BN / 32) == 0) {
          if (!c.wait_pair(PR + 2 * b + kk / (BN / 32), (g / NSB) & 1)) { ok = false; break; }
          tc_fence_after();
        }
        if constexpr (kPair)
          mma_ts_pair(tmem + TM_O, tmem + TM_S(b) + kk * 8, vd + (uint64_t)(kk * 16 * 128 >> 4), Idesc<kPair>::PV,
                      (j > 0 || kk > 0) ? 1u : 0u);
        else
          mma_ts(tmem + TM_O, tmem + TM_S(b) + kk * 8, vd + (uint64_t)(kk * 16 * 128 >> 4), Idesc<kPair>::PV,
                 (j > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      c.commit_both(VE + s);
      c.commit(SE + b);
      c.commit_both(OD + (g & 1));
    }
  }
  c.commit(FINP);
  c.drain(FINP, 0);
}

// ------------------------------------------------------------------ softmax
// Publish this half's row max for tile `tile` and read the other half's: one 8-byte
// shared-memory word per half, polled (a bounded spin, as every wait here) until it names
// the tile.  Cheaper than a 256-arrival barrier on the softmax's critical path.
template <bool kPair>
__device__ __forceinline__ bool exchange_max(const Ctx<kPair>& c, uint32_t mine, uint32_t theirs, float m,
                                             int tile, float* other) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(mine), "r"(__float_as_uint(m)), "r"((uint32_t)tile)
               : "memory");
  uint32_t v0, v1;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    asm volatile("ld.volatile.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(theirs) : "memory");
    if (v1 == (uint32_t)tile) break;
    if ((it & 63) == 63) {
      if (*c.abort_flag) return false;
      if (global_timer_ns() - t0 > c.wait_limit_ns) {
        *c.abort_flag = 1;
        atomicOr(c.status, MLA_DEVSTAT_TIMEOUT);
        return false;
      }
    }
  }
  *other = __uint_as_float(v0);
  return true;
}

// Two threads per query row: warps 4-7 own key columns 0-63 of every tile, warps 8-11
// columns 64-127 (a warp may only touch TMEM lanes 32*(warp%4)..+31, so both halves cover
// all 128 rows).  The halves agree on the row max through shared memory once per tile;
// at the end of a unit each publishes its row sum (and half 0 the row max) for the
// epilogue warps.  Every exchange sits behind an mbarrier or a bounded spin, so every
// wait can give up.
template <bool kMerge, bool kPair>
__device__ void run_softmax(const Ctx<kPair>& c, const PrefillParams& p, uint32_t tmem, float* xchg,
                            int ubeg, int uend) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;                 // TMEM lanes this warp may touch
  const int half = (warp - 4) >> 2;          // 0: key columns 0-63, 1: 64-127
  const int row = quad * 32 + lane;
  const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
  const uint32_t xword = smem_addr(xchg);    // [2 parity][2 half][128 rows] of (max, tile)
  float* xlm = xchg + 2 * XCHG_WORDS;        // [2 unit parity][sum half 0, sum half 1, max][128 rows]
  int s_g = 0, k = 0;                        // tiles and non-empty units so far
  bool ok = true;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float2 sc2 = make_float2(p.has_cap ? 1.f : p.scale_log2, p.has_cap ? 1.f : p.scale_log2);
  for (int ui = ubeg; ui < uend && ok; ++ui) {
    const Unit u = own_rows<kPair>(load_unit(p.units, ui), c.rank);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    const int n = hi - lo;
    const int qpos = u.q_pos0 + row;
    if (n <= 0) {
      // No allowed key: O = 0, LSE = -inf.  Merged into a partial state that leaves the
      // state as it is, except that a state at LSE = -inf (no key on either side) gets
      // O = 0 whatever its O held.
      const size_t orow = (size_t)(u.q_row0 + row) * p.num_heads + u.head;
      if (row < u.q_rows && (!kMerge || p.lse[orow] == NEG_INF)) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + orow * 128 + half * 64);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
        if (!kMerge && p.lse && half == 0) p.lse[orow] = NEG_INF;
      }
      continue;
    }
    // Per-row key window inside the request: allowed positions [klo, khi).
    const int khi = p.causal ? min(u.kv_len, qpos + u.diag + 1) : u.kv_len;
    const int klo = p.window_left >= 0 ? max(0, qpos + u.diag - p.window_left) : 0;
    float m_used = NEG_INF, l = 0.f;          // running max (log2 units) and this half's sum
    for (int j = 0; j < n; ++j) {
      const int sg = s_g + j, b = sg % NSB, xb = sg & 1;
      if (!__all_sync(0xffffffffu, c.wait(SF + b, (sg / NSB) & 1))) { ok = false; break; }
      tc_fence_after();
      float sv[64];
      tmem_ld64_sync(lane_addr + TM_S(b) + half * 64, reinterpret_cast<uint32_t*>(sv));
      if (p.has_cap) {
        // Soft cap c * tanh(sm_scale * x / c), in log2 units afterwards, from the identity
        // tanh(y) = 1 - 2 / (e^(2y) + 1): one ex2 and one reciprocal on the SFU per logit
        // (an overflowing e^(2y) gives 1, an underflowing one -1).
        const float2 k2 = make_float2(p.cap_ex2_scale, p.cap_ex2_scale);
        const float2 one = make_float2(1.f, 1.f);
        const float2 m2c = make_float2(-2.f * p.cap_log2, -2.f * p.cap_log2);
        const float2 c2 = make_float2(p.cap_log2, p.cap_log2);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float2 a = fmul2(make_float2(sv[2 * i], sv[2 * i + 1]), k2);
          const float2 d = fadd2(make_float2(ex2_approx(a.x), ex2_approx(a.y)), one);
          const float2 r = ffma2(make_float2(rcp_approx(d.x), rcp_approx(d.y)), m2c, c2);
          sv[2 * i] = r.x;
          sv[2 * i + 1] = r.y;
        }
      }
      const int kp0 = (lo + j) * BN + half * 64;
      const int c_hi = khi - kp0, c_lo = klo - kp0;
      if (c_hi < 64 || c_lo > 0) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i >= c_hi || i < c_lo) sv[i] = NEG_INF;
      }
      // Row max of this half (raw logits: sm_scale > 0 keeps the order), then of the row.
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        mx[k] = fmax3(fmax3(sv[8 * k], sv[8 * k + 1], sv[8 * k + 2]), fmax3(sv[8 * k + 3], sv[8 * k + 4], sv[8 * k + 5]),
                      fmaxf(sv[8 * k + 6], sv[8 * k + 7]));
      float m_half = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      // The other half's max: each half stores (max, tile) in one 8-byte word and polls
      // the other's word until it carries this tile (a word per tile parity, so a half
      // one tile ahead cannot overwrite what its partner has yet to read).
      float m_other;
      if (!__all_sync(0xffffffffu,
                      exchange_max(c, xword + (uint32_t)((xb * 2 + half) * 128 + row) * 8,
                                   xword + (uint32_t)((xb * 2 + (half ^ 1)) * 128 + row) * 8, m_half, sg, &m_other)))
        { ok = false; break; }
      const float m_raw = fmaxf(m_half, m_other);
      const float mt = m_raw * sc2.x;       // tile max in log2 units (-inf stays -inf)
      float m_new = m_used;
      bool rescale = false;
      if (j == 0) {
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
      for (int i = 0; i < 32; ++i) {
        const float2 a = ffma2(make_float2(sv[2 * i], sv[2 * i + 1]), sc2, neg_m);
        const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
        acc[i & 3] = fadd2(acc[i & 3], e);
        pr[i] = pack_bf16x2(e.x, e.y);
      }
      const float2 s01 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
      const float sum = s01.x + s01.y;
      tmem_st32_sync(lane_addr + TM_S(b) + half * 32, pr);
      float alpha = 1.f;
      // tcgen05.ld/st are warp-collective (.sync.aligned): the whole warp rescales its 32
      // rows together, rows that keep their max with alpha = 1.  A warp none of whose rows
      // rescale does not touch O and need not wait for the previous product: products
      // accumulate in issue order, so P_j V_j may queue behind P_{j-1} V_{j-1}.
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O must hold P_{j-1} V_{j-1} before it may be rescaled (tiles and products are
        // counted alike: that product is tile sg - 1).
        const int pg = sg - 1;
        if (!__all_sync(0xffffffffu, c.wait(OD + (pg & 1), (pg >> 1) & 1))) { ok = false; break; }
        tc_fence_after();
        if (rescale) alpha = ex2_approx(m_used - m_new);
        {
          float ov[64];
          tmem_ld64_sync(lane_addr + TM_O + half * 64, reinterpret_cast<uint32_t*>(ov));
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float2 r = fmul2(make_float2(ov[2 * i], ov[2 * i + 1]), a2);
            ov[2 * i] = r.x;
            ov[2 * i + 1] = r.y;
          }
          tmem_st64_sync(lane_addr + TM_O + half * 64, reinterpret_cast<uint32_t*>(ov));
        }
      }
      l = l * alpha + sum;
      m_used = m_new;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) c.arrive_leader(PR + 2 * b + half);
    }
    if (!ok) break;
    // Hand the unit to the epilogue warps: this half's row sum and the row max.  The
    // slot of this unit's parity is free once the epilogue has read unit k - 2.
    const int slot = k & 1;
    if (k >= 2 && !__all_sync(0xffffffffu, c.wait(LFR + slot, ((k >> 1) - 1) & 1))) { ok = false; break; }
    xlm[(slot * 3 + half) * 128 + row] = l;
    if (half == 0) xlm[(slot * 3 + 2) * 128 + row] = m_used;
    mbar_arrive(c.bar(LR + slot));
    ++k;
    s_g += n;
  }
}

// ------------------------------------------------------------------ register split
// Whole warpgroups (4 consecutive warps) change their per-thread register count.
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------ epilogue
// 64 columns of O, scaled by 1/l and rounded to bf16: w[q] = columns 16q .. 16q+15.
__device__ __forceinline__ void load_scaled_half(uint32_t lane_addr, float inv, uint32_t (&w)[4][8]) {
  const float2 inv2 = make_float2(inv, inv);
#pragma unroll
  for (int hq = 0; hq < 2; ++hq) {   // 32 columns at a time keeps the peak register count low
    float ov[32];
    tmem_ld32_sync(lane_addr + hq * 32, reinterpret_cast<uint32_t*>(ov));
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 x = fmul2(make_float2(ov[16 * q + 2 * e], ov[16 * q + 2 * e + 1]), inv2);
        w[2 * hq + q][e] = pack_bf16x2(x.x, x.y);
      }
  }
}

// w (bf16 pairs of 64 columns) += a * the 64 bf16 columns at src (16-byte aligned), in
// fp32, rounded back to bf16.
__device__ __forceinline__ void merge_old(const char* src, float a, uint32_t (&w)[4][8]) {
  const float2 a2 = make_float2(a, a);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + q * 32);
    const uint4 x = s4[0], y = s4[1];
    const uint32_t old[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 o = make_float2(__uint_as_float(old[e] << 16), __uint_as_float(old[e] & 0xffff0000u));
      const float2 n = make_float2(__uint_as_float(w[q][e] << 16), __uint_as_float(w[q][e] & 0xffff0000u));
      const float2 r = ffma2(o, a2, n);
      w[q][e] = pack_bf16x2(r.x, r.y);
    }
  }
}

// 64 columns of a row of O: 128 contiguous bytes, four 32-byte stores or eight 16-byte ones.
__device__ __forceinline__ void store_half(char* dst, int align32, const uint32_t (&w)[4][8]) {
  if (align32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) st_global_v8(dst + q * 32, w[q]);
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      reinterpret_cast<uint4*>(dst + q * 32)[0] = make_uint4(w[q][0], w[q][1], w[q][2], w[q][3]);
      reinterpret_cast<uint4*>(dst + q * 32)[1] = make_uint4(w[q][4], w[q][5], w[q][6], w[q][7]);
    }
  }
}

// One row of O: 256 contiguous bytes, eight 32-byte stores (whole sectors), or sixteen
// 16-byte stores when O is only 16-byte aligned.
__device__ __forceinline__ void store_row(char* dst, int align32, const uint32_t (&w0)[4][8],
                                          const uint32_t (&w1)[4][8]) {
  if (align32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      st_global_v8(dst + q * 32, w0[q]);
      st_global_v8(dst + 128 + q * 32, w1[q]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      reinterpret_cast<uint4*>(dst + q * 32)[0] = make_uint4(w0[q][0], w0[q][1], w0[q][2], w0[q][3]);
      reinterpret_cast<uint4*>(dst + q * 32)[1] = make_uint4(w0[q][4], w0[q][5], w0[q][6], w0[q][7]);
      reinterpret_cast<uint4*>(dst + 128 + q * 32)[0] = make_uint4(w1[q][0], w1[q][1], w1[q][2], w1[q][3]);
      reinterpret_cast<uint4*>(dst + 128 + q * 32)[1] = make_uint4(w1[q][4], w1[q][5], w1[q][6], w1[q][7]);
    }
  }
}

// Warps 12-15, one per TMEM lane quadrant, one thread per query row and all 128 columns
// of O.  Per unit: wait for the softmax's row sums and max, then for the unit's last
// P V; read O, release it to the P V issuer, and store.  The stores are row per thread
// (eight 32-byte stores of 256 contiguous bytes): off the softmax's critical path, a
// shuffle exchange that would coalesce them costs more issue slots than it saves.
template <bool kMerge, bool kPair>
__device__ void run_epilogue(const Ctx<kPair>& c, const PrefillParams& p, uint32_t tmem, const float* xchg,
                             int ubeg, int uend) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
  const float* xlm = xchg + 2 * XCHG_WORDS;
  const float NEG_INF = -__int_as_float(0x7f800000);
  int g = 0, k = 0;   // tiles and non-empty units so far
  for (int ui = ubeg; ui < uend; ++ui) {
    const Unit u = own_rows<kPair>(load_unit(p.units, ui), c.rank);
    const int lo = u.kv_tiles & 0xFFFF, hi = (u.kv_tiles >> 16) & 0xFFFF;
    const int n = hi - lo;
    if (n <= 0) continue;
    const int slot = k & 1;
    if (!__all_sync(0xffffffffu, c.wait(LR + slot, (k >> 1) & 1))) break;
    const float l_row = xlm[(slot * 3 + 0) * 128 + row] + xlm[(slot * 3 + 1) * 128 + row];
    const float m_row = xlm[(slot * 3 + 2) * 128 + row];
    mbar_arrive(c.bar(LFR + slot));
    // The unit's last product.  A parity wait on it is exact only once the product before
    // it on the same barrier (tile gl - 2) has completed: for n = 1 this warp waited for
    // tile gl - 1 (the previous unit's last product); for n > 1 it waits for tile gl - 1
    // first (whose own predecessor, tile gl - 3, has completed: S of tile gl exists).
    // Products complete in order, so gl - 1 done means gl - 2 done.
    const int gl = g + n - 1;
    if (n > 1 && !__all_sync(0xffffffffu, c.wait(OD + ((gl - 1) & 1), ((gl - 1) >> 1) & 1))) break;
    if (!__all_sync(0xffffffffu, c.wait(OD + (gl & 1), (gl >> 1) & 1))) break;
    tc_fence_after();
    const bool live = row < u.q_rows;
    const bool empty = !(l_row > 0.f);
    if constexpr (!kMerge) {
      const float inv = empty ? 0.f : 1.f / l_row;
      uint32_t w0[4][8], w1[4][8];
      load_scaled_half(lane_addr + TM_O, inv, w0);
      load_scaled_half(lane_addr + TM_O + 64, inv, w1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) c.arrive_leader(OFR);
      // (The row address is formed twice on purpose: holding it across the stores
      // costs registers this warpgroup does not have.)
      if (live)
        store_row(reinterpret_cast<char*>(p.o + ((size_t)(u.q_row0 + row) * p.num_heads + u.head) * 128),
                  p.o_align32, w0, w1);
      if (p.lse && live) {
        float lg;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l_row));
        p.lse[(size_t)(u.q_row0 + row) * p.num_heads + u.head] = empty ? NEG_INF : (m_row + lg) * 0.6931471805599453f;
      }
    } else {
      // Merge with the entry state (O_a, la): O = a * O_a + b * acc, LSE = lse2_out
      // (log2 units), the weights taken in base 2 from both LSEs.
      float a = 0.f, b = 0.f, lse2_out = NEG_INF;
      if (live) {
        float lg;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(l_row));
        const float lse2_new = empty ? NEG_INF : m_row + lg;
        const float lse2_old = p.lse[(size_t)(u.q_row0 + row) * p.num_heads + u.head] * 1.4426950408889634f;
        const float mx = fmaxf(lse2_old, lse2_new);   // -inf only if both sides are empty
        if (mx != NEG_INF) {
          const float w_old = ex2_approx(lse2_old - mx), w_new = ex2_approx(lse2_new - mx);
          const float sum = w_old + w_new, inv_sum = 1.f / sum;
          float ls;
          asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(ls) : "f"(sum));
          a = w_old * inv_sum;
          b = empty ? 0.f : w_new * inv_sum / l_row;
          lse2_out = mx + ls;
        }
      }
      uint32_t w0[4][8], w1[4][8];
      load_scaled_half(lane_addr + TM_O, b, w0);
      load_scaled_half(lane_addr + TM_O + 64, b, w1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) c.arrive_leader(OFR);
      if (live) {
        // A side with LSE = -inf gets weight 0 and its O is never read.  One half at a
        // time, merged then stored (the barrier keeps the second half's loads below the
        // first half's stores, which bounds the registers in use).
        char* dst = reinterpret_cast<char*>(p.o + ((size_t)(u.q_row0 + row) * p.num_heads + u.head) * 128);
        if (a != 0.f) merge_old(dst, a, w0);
        store_half(dst, p.o_align32, w0);
        asm volatile("" ::: "memory");
        if (a != 0.f) merge_old(dst + 128, a, w1);
        store_half(dst + 128, p.o_align32, w1);
      }
      if (live)
        p.lse[(size_t)(u.q_row0 + row) * p.num_heads + u.head] =
            lse2_out == NEG_INF ? NEG_INF : lse2_out * 0.6931471805599453f;
    }
    g += n;
    ++k;
  }
}

// kMerge: o/lse hold a partial state that the epilogue merges this attention into.
// kPair: launched as clusters of two CTAs, unit lists indexed by cluster.
template <bool kMerge, bool kPair>
__global__ void __launch_bounds__(NTHREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_r,
               const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Off<kPair>::MISC);
  int* abort_flag = reinterpret_cast<int*>(smem + Off<kPair>::MISC + 4);
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  Ctx<kPair> c{smem_addr(smem), abort_flag, p.status, p.wait_limit_ns, rank};

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(c.bar(i), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(c.bar(LR + i), 256);
      mbar_init(c.bar(LFR + i), 128);  // every epilogue thread
    }
    // One arrival per softmax warp / epilogue warp, of both CTAs in a pair's even CTA.
    const int both = kPair && rank == 0 ? 2 : 1;
    for (int i = 0; i < 2 * NSB; ++i) mbar_init(c.bar(PR + i), 4 * both);
    mbar_init(c.bar(OFR), 4 * both);
    if (kPair && rank == 0) {   // own load (with its bytes) + the odd CTA's forwarded arrival
      mbar_init(c.bar(QF), 2);
      for (int s = 0; s < Lay<kPair>::NK; ++s) mbar_init(c.bar(KF + s), 2);
      for (int s = 0; s < Lay<kPair>::NV; ++s) mbar_init(c.bar(VF + s), 2);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  {   // exchange words: no tile yet
    uint32_t* words = reinterpret_cast<uint32_t*>(smem + Off<kPair>::XCHG);
    for (int i = threadIdx.x; i < XCHG_WORDS; i += NTHREADS) words[2 * i + 1] = 0xffffffffu;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (p.shared_rope) tma_prefetch_desc(&tm_r);
  }
  if (warp == 1) {
    if constexpr (kPair) {   // one warp of each CTA of the pair, together
      tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int slot_idx = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ubeg = p.cta_offsets[slot_idx], uend = p.cta_offsets[slot_idx + 1];

  float* xchg = reinterpret_cast<float*>(smem + Off<kPair>::XCHG);
  if (warp < 4) {
    setmaxnreg_dec<RegSplit<kMerge>::ctrl>();
    if (lane == 0) {
      const bool issuer = !kPair || rank == 0;
      if (warp == 0) {
        run_producer_qk<kPair>(c, p, &tm_q, &tm_k, &tm_r, ubeg, uend);
      } else if (warp == 2) {
        run_producer_v<kPair>(c, p, &tm_v, ubeg, uend);
      } else if (issuer) {
        if (warp == 1) run_mma_qk<kPair>(c, p, tmem, ubeg, uend);
        else run_mma_pv<kPair>(c, p, tmem, ubeg, uend);
      } else if constexpr (kPair) {
        if (warp == 1) run_forward_qk(c, p, ubeg, uend);
        else run_forward_v(c, p, ubeg, uend);
      }
    }
  } else if (warp < 12) {
    setmaxnreg_inc<RegSplit<kMerge>::softmax>();
    run_softmax<kMerge, kPair>(c, p, tmem, xchg, ubeg, uend);
  } else {
    setmaxnreg_dec<RegSplit<kMerge>::epi>();
    run_epilogue<kMerge, kPair>(c, p, tmem, xchg, ubeg, uend);
  }
  tc_fence_before();
  __syncthreads();
  // In a pair, neither CTA leaves (freeing its shared memory and TMEM) while the even
  // CTA's products may still read or write the other's.
  if constexpr (kPair) cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if constexpr (kPair) tmem_dealloc_pair(tmem, TMEM_COLS); else tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int prefill_smem_bytes() { return Off<false>::SMEM; }

template <bool kMerge, bool kPair>
static cudaError_t configure_prefill() {
  cudaError_t r = cudaFuncSetAttribute(prefill_kernel<kMerge, kPair>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Off<kPair>::SMEM);
  if (r != cudaSuccess) return r;
  // The warpgroups' setmaxnreg split assumes every thread starts with LAUNCH_REGS
  // registers; with fewer, the softmax warpgroups' increase could never be granted.
  cudaFuncAttributes attr;
  r = cudaFuncGetAttributes(&attr, prefill_kernel<kMerge, kPair>);
  if (r != cudaSuccess) return r;
  return attr.numRegs == LAUNCH_REGS ? cudaSuccess : cudaErrorInvalidConfiguration;
}

static cudaLaunchConfig_t pair_config(cudaLaunchAttribute* attr, int num_pairs, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_pairs, 1, 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = Off<true>::SMEM;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

int prefill_max_pairs() {
  static PerDeviceOnce configured;
  if (configured.run([] { return configure_prefill<false, true>(); }) != cudaSuccess) return 0;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = pair_config(attr, 1, nullptr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, prefill_kernel<false, true>, &cfg) != cudaSuccess) return 0;
  return n;
}

template <bool kMerge, bool kPair>
static cudaError_t launch_prefill_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const CUtensorMap& tr, const PrefillParams& p, int num_slots,
                                    cudaStream_t stream) {
  static PerDeviceOnce configured;
  cudaError_t e = configured.run([] { return configure_prefill<kMerge, kPair>(); });
  if (e != cudaSuccess) return e;
  if constexpr (kPair) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config(attr, num_slots, stream);
    return cudaLaunchKernelEx(&cfg, prefill_kernel<kMerge, true>, tq, tk, tv, tr, p);
  } else {
    prefill_kernel<kMerge, false><<<num_slots, NTHREADS, Off<false>::SMEM, stream>>>(tq, tk, tv, tr, p);
    return cudaGetLastError();
  }
}

cudaError_t launch_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tr, const PrefillParams& p, int num_slots, cudaStream_t stream) {
  if (p.pair)
    return p.merge ? launch_prefill_t<true, true>(tq, tk, tv, tr, p, num_slots, stream)
                   : launch_prefill_t<false, true>(tq, tk, tv, tr, p, num_slots, stream);
  return p.merge ? launch_prefill_t<true, false>(tq, tk, tv, tr, p, num_slots, stream)
                 : launch_prefill_t<false, false>(tq, tk, tv, tr, p, num_slots, stream);
}

}  // namespace mla
