"""Seeded synthetic inputs for MLA ragged prefill.

This module only draws numbers and lays them out; it holds none of the
attention, gather, up-projection or merge arithmetic.  Both the CUDA path
(through ``chunked_prefill_attention_ragged_gb300``) and the fp64 oracle
(under ``oracle/``) are fed from here, so they see identical bits.

Shapes follow DeepSeek-R1 MLA as described by sglang issue #3849
("[DeepseekR1] How ragged prefill manage kv_cache?": query/key head dim 192 =
128 NoPE + 64 RoPE, value/output head dim 128, a compressed cache row of
512 latent + 64 rope) and by the vLLM page
``vllm.v1.attention.backends.mla.prefill.flashinfer``
(``FlashInferPrefillBackend.finalize_attention_metadata``: ragged
``qo_indptr``/``kv_indptr``, as many KV heads as query heads, a one-head
latent cache).

Recipe (stated once, used everywhere):
  * ``numpy.random.default_rng(1000 + workload index)``;
  * draw order: lengths, then Q, K, V, then (prefix workload only) the latent
    cache, the block permutation and the up-projection weight;
  * values drawn as float32 standard normals (weights scaled by 512**-0.5)
    and rounded to bfloat16 with round-to-nearest-even on the host, so every
    consumer sees the same bits.

bfloat16 tensors are carried as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

DQK = 192          # 128 NoPE + 64 RoPE
DQK_NOPE = 128
DQK_ROPE = 64
DV = 128
KV_LORA_RANK = 512
LATENT_DIM = KV_LORA_RANK + DQK_ROPE   # 576 = one cache row
DEFAULT_SM_SCALE = DQK ** -0.5


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as uint16.  Inputs here are finite normals,
    so no NaN handling is needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def _normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return to_bf16_bits(x)


def indptr_from_lengths(lengths) -> np.ndarray:
    """Exclusive prefix sum of per-request lengths, int32 [B+1]."""
    lengths = np.asarray(lengths, dtype=np.int64)
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=out[1:])
    assert out[-1] < 2**31
    return out.astype(np.int32)


@dataclass
class RaggedBatch:
    """One ragged prefill problem in the "NHD" layout.

    q: [sum(q_lens), H, 192], k: [sum(kv_lens), H, 192], v: [sum(kv_lens), H, 128],
    all bfloat16 bit patterns.
    """
    name: str
    q_lens: np.ndarray
    kv_lens: np.ndarray
    num_heads: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    causal: bool = True
    sm_scale: float = DEFAULT_SM_SCALE
    window_left: int = -1
    logits_soft_cap: float = 0.0

    @property
    def qo_indptr(self) -> np.ndarray:
        return indptr_from_lengths(self.q_lens)

    @property
    def kv_indptr(self) -> np.ndarray:
        return indptr_from_lengths(self.kv_lens)

    @property
    def batch(self) -> int:
        return len(self.q_lens)


def random_ragged(seed: int, q_lens, kv_lens=None, num_heads: int = 4, *,
                  dqk: int = DQK, dv: int = DV, causal: bool = True,
                  sm_scale: float = DEFAULT_SM_SCALE, window_left: int = -1,
                  logits_soft_cap: float = 0.0, name: str = "random",
                  rng: np.random.Generator | None = None) -> RaggedBatch:
    """Draw Q, K, V for the given lengths (kv_lens defaults to q_lens)."""
    rng = np.random.default_rng(seed) if rng is None else rng
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens = q_lens.copy() if kv_lens is None else np.asarray(kv_lens, dtype=np.int64)
    tq, tk = int(q_lens.sum()), int(kv_lens.sum())
    q = _normal_bf16(rng, (tq, num_heads, dqk))
    k = _normal_bf16(rng, (tk, num_heads, dqk))
    v = _normal_bf16(rng, (tk, num_heads, dv))
    return RaggedBatch(name, q_lens, kv_lens, num_heads, q, k, v, causal,
                       float(sm_scale), int(window_left), float(logits_soft_cap))


# --------------------------------------------------------------------------
# The five workloads.  Index i uses seed 1000 + i.
# --------------------------------------------------------------------------

WORKLOAD_NAMES = (
    "tiny_ragged_causal",            # 0
    "deepseek_ragged_8x_u512_4096_h128",   # 1
    "chunked_prefix_4x2048_p8192",   # 2
    "long_single_32768_h128",        # 3
    "many_short_256_geo200_h16",     # 4
)


def workload_lengths(index: int, rng: np.random.Generator) -> np.ndarray:
    """First draw of each workload: the per-request new-token lengths."""
    if index == 0:
        return np.array([17, 40], dtype=np.int64)
    if index == 1:
        return rng.integers(512, 4097, size=8).astype(np.int64)
    if index == 2:
        return np.full(4, 2048, dtype=np.int64)
    if index == 3:
        return np.array([32768], dtype=np.int64)
    if index == 4:
        return np.clip(rng.geometric(1.0 / 200.0, size=256), 1, 1024).astype(np.int64)
    raise ValueError(index)


WORKLOAD_HEADS = {0: 4, 1: 128, 2: 128, 3: 128, 4: 16}


def make_workload(index: int, logits_soft_cap: float = 0.0) -> RaggedBatch:
    """Ragged batch of workload ``index`` (0, 1, 3, 4; for 2 see make_chunked_prefix).

    Workload 4 has two variants that share inputs: no soft cap and a cap of 30.
    """
    if index == 2:
        return make_chunked_prefix().new
    rng = np.random.default_rng(1000 + index)
    lens = workload_lengths(index, rng)
    name = WORKLOAD_NAMES[index] + (f"_cap{logits_soft_cap:g}" if logits_soft_cap > 0 else "")
    return random_ragged(0, lens, lens, WORKLOAD_HEADS[index], causal=True,
                         logits_soft_cap=logits_soft_cap, name=name, rng=rng)


@dataclass
class ChunkLayout:
    """How a per-request prefix is cut into chunks.

    For chunk c: ``cu_seq_lens[c]`` is that chunk's kv_indptr [B+1] and
    ``chunk_starts[c][r]`` is the first prefix position of request r in it.
    """
    cu_seq_lens: np.ndarray     # int32 [num_chunks, B+1]
    chunk_starts: np.ndarray    # int32 [num_chunks, B]

    @property
    def num_chunks(self) -> int:
        return self.cu_seq_lens.shape[0]


def chunk_layout(prefix_lens, chunk_tokens: int) -> ChunkLayout:
    """Cut each request's prefix into pieces of ``chunk_tokens`` positions.

    Chunk c holds positions [c*chunk_tokens, min((c+1)*chunk_tokens, P_r)) of
    request r (empty if P_r <= c*chunk_tokens).
    """
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    n = int(max(1, -(-int(prefix_lens.max(initial=0)) // chunk_tokens)))
    cu = np.zeros((n, len(prefix_lens) + 1), dtype=np.int32)
    st = np.zeros((n, len(prefix_lens)), dtype=np.int32)
    for c in range(n):
        start = c * chunk_tokens
        piece = np.clip(prefix_lens - start, 0, chunk_tokens)
        st[c] = np.minimum(start, prefix_lens)
        cu[c] = indptr_from_lengths(piece)
    return ChunkLayout(cu, st)


@dataclass
class ChunkedPrefixBatch:
    """New tokens attending to themselves (causal) and to a cached prefix.

    cache: [num_blocks, block_size, 576] bf16 bits (512 latent then 64 rope),
    block_table: int32 [B, max_blocks_per_req], w_kvb: [512, H*256] bf16 bits.
    """
    new: RaggedBatch
    prefix_lens: np.ndarray
    cache: np.ndarray
    block_table: np.ndarray
    w_kvb: np.ndarray
    block_size: int
    chunk_tokens: int
    layout: ChunkLayout = field(init=False)

    def __post_init__(self):
        self.layout = chunk_layout(self.prefix_lens, self.chunk_tokens)


def random_chunked_prefix(seed: int, new_lens, prefix_lens, num_heads: int, *,
                          num_blocks: int, block_size: int = 64, chunk_tokens: int = 4096,
                          name: str = "chunked", rng: np.random.Generator | None = None,
                          logits_soft_cap: float = 0.0, window_left: int = -1) -> ChunkedPrefixBatch:
    """Draw a chunked-prefix problem.

    The block table is the first sum(ceil(P_r/block_size)) entries of a random
    permutation of all blocks, handed out request by request; unused cache
    blocks are filled too, so a wrong block index reads visible garbage.
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    new = random_ragged(0, new_lens, new_lens, num_heads, causal=True, name=name, rng=rng,
                        logits_soft_cap=logits_soft_cap, window_left=window_left)
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    cache = _normal_bf16(rng, (num_blocks, block_size, LATENT_DIM))
    perm = rng.permutation(num_blocks).astype(np.int32)
    per_req = [-(-int(p) // block_size) for p in prefix_lens]
    max_blocks = max(1, max(per_req))
    assert sum(per_req) <= num_blocks
    table = np.full((len(prefix_lens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for r, nb in enumerate(per_req):
        table[r, :nb] = perm[pos:pos + nb]
        pos += nb
    w = _normal_bf16(rng, (KV_LORA_RANK, num_heads * (DQK_NOPE + DV)), scale=KV_LORA_RANK ** -0.5)
    return ChunkedPrefixBatch(new, prefix_lens, cache, table, w, block_size, chunk_tokens)


def random_fp8_cache(rng: np.random.Generator, num_blocks: int, block_size: int,
                     scale_exp=(119, 130), code_exp=None) -> np.ndarray:
    """A paged cache of fp8 latent entries, uint8 [num_blocks, block_size, 648]: 512 random
    float8 e4m3 codes (NaN codes 0x7F/0xFF excluded), 64 bf16 N(0,1) rope values (128 bytes)
    and 8 scale exponent bytes drawn uniformly from ``scale_exp`` (inclusive).

    ``code_exp=(lo, hi)`` restricts the codes' 4-bit exponent field to lo..hi (random sign
    and mantissa), e.g. (4, 8) for magnitudes between 1/8 and 3.75, so that the latent
    has a realistic spread when the scale is 1."""
    n = num_blocks * block_size
    if code_exp is None:
        codes = rng.integers(0, 254, size=(n, 512), dtype=np.uint16)
        codes = np.where(codes >= 0x7F, codes + 1, codes).astype(np.uint8)      # skip 0x7F; 0xFF is never drawn
    else:
        sign = rng.integers(0, 2, size=(n, 512), dtype=np.uint16) << 7
        expo = rng.integers(code_exp[0], min(code_exp[1], 14) + 1, size=(n, 512), dtype=np.uint16) << 3
        mant = rng.integers(0, 8, size=(n, 512), dtype=np.uint16)
        codes = (sign | expo | mant).astype(np.uint8)
    rope = _normal_bf16(rng, (n, 64)).view(np.uint8).reshape(n, 128)
    scales = rng.integers(scale_exp[0], scale_exp[1] + 1, size=(n, 8)).astype(np.uint8)
    return np.concatenate([codes, rope, scales], axis=1).reshape(num_blocks, block_size, 648)


def make_chunked_prefix() -> ChunkedPrefixBatch:
    """Workload 2: 4 requests x (2048 new + 8192 cached), 128 heads, 4096-token chunks."""
    rng = np.random.default_rng(1002)
    lens = workload_lengths(2, rng)
    return random_chunked_prefix(0, lens, np.full(4, 8192), WORKLOAD_HEADS[2], num_blocks=1024,
                                 block_size=64, chunk_tokens=4096, name=WORKLOAD_NAMES[2], rng=rng)


@dataclass
class AbsorbedBatch:
    """Absorbed-weight prefill inputs: request r has q_lens[r] new query rows, the last of
    its kv_lens[r] positions in the paged latent cache.

    q_abs: [sum q_lens, H, 576] bf16 bits (the absorbed query W_UK(h) q_nope(h) || q_rope(h),
    drawn directly), cache: [num_blocks, block_size, 576] bf16 bits, block_table: int32
    [B, max blocks] (unused entries -1)."""
    name: str
    q_lens: np.ndarray
    kv_lens: np.ndarray
    num_heads: int
    block_size: int
    causal: bool
    sm_scale: float
    logits_soft_cap: float
    q_abs: np.ndarray
    cache: np.ndarray
    block_table: np.ndarray
    qo_indptr: np.ndarray = field(init=False)

    def __post_init__(self):
        self.qo_indptr = indptr_from_lengths(self.q_lens)

    @property
    def batch(self) -> int:
        return len(self.q_lens)


def random_absorbed(seed: int, q_lens, kv_lens, num_heads: int, *, block_size: int = 64,
                    num_blocks: int | None = None, causal: bool = True, logits_soft_cap: float = 0.0,
                    sm_scale: float = DEFAULT_SM_SCALE, name: str = "absorbed") -> AbsorbedBatch:
    """Draw an absorbed-weight prefill problem (same recipe: N(0,1) rounded to bf16).

    The block table is the first sum(ceil(kv_len/block_size)) entries of a random
    permutation of the cache blocks, handed out request by request; the cache is filled
    everywhere, so a wrong block index reads visible values.  The softmax scale is the MHA
    one (192^-0.5) unless given."""
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    per_req = [-(-int(k) // block_size) for k in kv_lens]
    if num_blocks is None:
        num_blocks = max(1, sum(per_req) + 3)
    assert sum(per_req) <= num_blocks
    q_abs = _normal_bf16(rng, (int(q_lens.sum()), num_heads, LATENT_DIM))
    cache = _normal_bf16(rng, (num_blocks, block_size, LATENT_DIM))
    perm = rng.permutation(num_blocks).astype(np.int32)
    table = np.full((len(q_lens), max(1, max(per_req, default=1))), -1, dtype=np.int32)
    pos = 0
    for r, nb in enumerate(per_req):
        table[r, :nb] = perm[pos:pos + nb]
        pos += nb
    return AbsorbedBatch(name, q_lens, kv_lens, num_heads, block_size, causal, float(sm_scale),
                         float(logits_soft_cap), q_abs, cache, table)
