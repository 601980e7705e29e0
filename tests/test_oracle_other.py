"""Pins for the gather, up-projection, merge, bf16 and chunked-pipeline oracles (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import (bf16_bits_to_f64, chunked_prefill_attention, gather_latent, merge_state,
                    ragged_attention, round_f64_to_bf16, slot_of, up_project)

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 helpers
def test_bf16_roundtrip_and_ties():
    assert round_f64_to_bf16(np.array([1.0 + 2.0**-8]))[0] == 1.0                 # tie -> even
    assert round_f64_to_bf16(np.array([1.0 + 3 * 2.0**-8]))[0] == 1.0 + 2.0**-6   # tie -> even (up)
    assert round_f64_to_bf16(np.array([1.0 + 2.0**-8 + 2.0**-30]))[0] == 1.0 + 2.0**-7
    assert round_f64_to_bf16(np.array([-3.0]))[0] == -3.0
    bits = np.arange(0, 0x7F80, 7, dtype=np.uint16)          # finite positive patterns
    vals = bf16_bits_to_f64(bits)
    np.testing.assert_array_equal(round_f64_to_bf16(vals), vals)


def test_bf16_rounding_agrees_with_generator():
    # The generator rounds float32 -> bf16; the oracle rounds float64 -> bf16.
    # On float32 inputs both are the same round-to-nearest-even.
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32)
    np.testing.assert_array_equal(bf16_bits_to_f64(wl.to_bf16_bits(x)), round_f64_to_bf16(x.astype(np.float64)))


# ---------------------------------------------------------------- gather
def _gather_fixture():
    g = json.load(open(os.path.join(GOLD, "gather_hand_case.json")))
    nb, bs, e = g["num_blocks"], g["block_size"], g["entry_dim"]
    slots = np.arange(nb * bs)
    cache = (10 * slots[:, None] + np.arange(e)[None, :]).reshape(nb, bs, e).astype(np.int64)
    return g, cache


def test_gather_hand_case():
    g, cache = _gather_fixture()
    table = np.array(g["block_table"], dtype=np.int32)
    for ch in g["chunks"]:
        out = gather_latent(cache, table, np.array(ch["cu_seq_lens"]), np.array(ch["chunk_starts"]))
        expect = 10 * np.array(ch["slots"])[:, None] + np.arange(g["entry_dim"])[None, :]
        np.testing.assert_array_equal(out, expect)


def test_gather_hand_case_matches_chunk_layout():
    g, _ = _gather_fixture()
    lay = wl.chunk_layout(g["prefix_lens"], 2)
    assert lay.num_chunks == len(g["chunks"])
    for c, ch in enumerate(g["chunks"]):
        np.testing.assert_array_equal(lay.cu_seq_lens[c], ch["cu_seq_lens"])
        np.testing.assert_array_equal(lay.chunk_starts[c], ch["chunk_starts"])


def test_gather_brute_force_random_tables():
    # A second formulation: build the full per-request position list, map each
    # position through the table with vectorised integer ops, then index.
    for seed in range(4):
        rng = np.random.default_rng(seed)
        nb, bs, e = 37, int(rng.choice([1, 4, 16, 64])), 9
        prefix = rng.integers(0, 5 * bs, size=3)
        need = [-(-int(p) // bs) for p in prefix]
        perm = rng.permutation(nb)
        table = np.full((3, max(1, max(need))), -1, dtype=np.int32)
        off = 0
        for r, n in enumerate(need):
            table[r, :n] = perm[off:off + n]; off += n
        cache = rng.integers(0, 2**16, size=(nb, bs, e)).astype(np.uint16)
        lay = wl.chunk_layout(prefix, int(rng.integers(1, 3 * bs + 1)))
        for c in range(lay.num_chunks):
            out = gather_latent(cache, table, lay.cu_seq_lens[c], lay.chunk_starts[c])
            rows = []
            for r in range(3):
                n = lay.cu_seq_lens[c, r + 1] - lay.cu_seq_lens[c, r]
                pos = lay.chunk_starts[c, r] + np.arange(n)
                blk = table[r, pos // bs]
                rows.append(cache[blk, pos % bs])
            np.testing.assert_array_equal(out, np.concatenate(rows) if rows else out)
            for r in range(3):
                for t in range(lay.cu_seq_lens[c, r + 1] - lay.cu_seq_lens[c, r]):
                    s = slot_of(table, r, int(lay.chunk_starts[c, r]) + t, bs)
                    assert 0 <= s < nb * bs


# ---------------------------------------------------------------- up-projection
def test_up_proj_triple_loop():
    rng = np.random.default_rng(1)
    T, H = 2, 2
    lat = wl.to_bf16_bits(rng.standard_normal((T, 576)).astype(np.float32))
    w = wl.to_bf16_bits((rng.standard_normal((512, H * 256)) * 0.05).astype(np.float32))
    k, v = up_project(lat, w, H)
    L, W = bf16_bits_to_f64(lat).tolist(), bf16_bits_to_f64(w).tolist()
    for t in range(T):
        for h in range(H):
            for d in range(256):
                acc = math.fsum(L[t][c] * W[c][h * 256 + d] for c in range(512))
                got = k[t, h, d] if d < 128 else v[t, h, d - 128]
                assert abs(got - acc) < 1e-12
            for d in range(64):
                assert k[t, h, 128 + d] == L[t][512 + d]


def test_up_proj_column_layout_one_hot():
    # W[c, n] = 1 iff c == n: head h's K_nope[d] = latent[h*256 + d], V[d] = latent[h*256 + 128 + d].
    H = 2
    w = np.zeros((512, H * 256), dtype=np.float32)
    w[np.arange(512), np.arange(512)] = 1.0
    lat = wl.to_bf16_bits(np.random.default_rng(2).standard_normal((5, 576)).astype(np.float32))
    k, v = up_project(lat, wl.to_bf16_bits(w), H)
    x = bf16_bits_to_f64(lat)
    for h in range(H):
        np.testing.assert_array_equal(k[:, h, :128], x[:, h * 256:h * 256 + 128])
        np.testing.assert_array_equal(v[:, h, :], x[:, h * 256 + 128:h * 256 + 256])
        np.testing.assert_array_equal(k[:, h, 128:], x[:, 512:576])


# ---------------------------------------------------------------- merge
def test_merge_closed_forms():
    oa = np.array([[[1.0, 2.0]]]); ob = np.array([[[3.0, -2.0]]])
    o, l = merge_state(oa, np.array([[0.7]]), ob, np.array([[0.7]]))        # equal weights
    np.testing.assert_allclose(o, [[[2.0, 0.0]]], atol=1e-15)
    assert abs(l[0, 0] - (0.7 + math.log(2))) < 1e-15
    o, l = merge_state(oa, np.array([[math.log(3)]]), ob, np.array([[0.0]]))  # weights 3:1
    np.testing.assert_allclose(o, [[[1.5, 1.0]]], atol=1e-15)
    assert abs(l[0, 0] - math.log(4)) < 1e-15
    o, l = merge_state(oa, np.array([[-np.inf]]), ob, np.array([[5.0]]))     # empty side
    np.testing.assert_array_equal(o, ob); assert l[0, 0] == 5.0
    o, l = merge_state(oa, np.array([[2.0]]), ob, np.array([[-np.inf]]))
    np.testing.assert_array_equal(o, oa); assert l[0, 0] == 2.0
    o, l = merge_state(oa, np.array([[-np.inf]]), ob, np.array([[-np.inf]]))  # both empty
    np.testing.assert_array_equal(o, 0 * oa); assert l[0, 0] == -np.inf


def test_merge_large_lse_is_stable():
    o, l = merge_state(np.ones((1, 1, 2)), np.array([[1000.0]]), np.zeros((1, 1, 2)), np.array([[999.0]]))
    w = 1 / (1 + math.exp(-1))
    np.testing.assert_allclose(o, [[[w, w]]], atol=1e-14)
    assert abs(l[0, 0] - (1000 + math.log1p(math.exp(-1)))) < 1e-12


# ---------------------------------------------------------------- chunked pipeline
def _tiny_chunked(seed=4, cap=0.0):
    return wl.random_chunked_prefix(seed, [5, 12], [7, 20], 2, num_blocks=16, block_size=4,
                                    chunk_tokens=8, logits_soft_cap=cap)


@pytest.mark.parametrize("cap", [0.0, 3.0])
def test_chunked_equals_chunk_then_merge(cap):
    """Unchunked reference == causal new-token part merged with every non-causal prefix chunk."""
    cb = _tiny_chunked(cap=cap)
    b = cb.new
    ref_o, ref_l = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                             cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale,
                                             logits_soft_cap=cap, kv_as_bf16=False)
    o, l = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=True,
                            sm_scale=b.sm_scale, logits_soft_cap=cap)
    lay = cb.layout
    assert lay.num_chunks == 3
    for c in range(lay.num_chunks):
        lat = gather_latent(cb.cache, cb.block_table, lay.cu_seq_lens[c], lay.chunk_starts[c])
        kc, vc = up_project(lat, cb.w_kvb, b.num_heads)
        oc, lc = ragged_attention(b.q, kc, vc, b.qo_indptr, lay.cu_seq_lens[c], causal=False,
                                  sm_scale=b.sm_scale, logits_soft_cap=cap)
        o, l = merge_state(o, l, oc, lc)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


def test_chunked_zero_prefix_is_plain_causal():
    cb = wl.random_chunked_prefix(8, [6, 3], [0, 0], 2, num_blocks=4, block_size=4, chunk_tokens=8)
    b = cb.new
    o0, l0 = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                       cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale)
    o1, l1 = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=True, sm_scale=b.sm_scale)
    np.testing.assert_allclose(o0, o1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l0, l1, rtol=0, atol=1e-13)


def test_chunked_rows_and_heads_subset():
    cb = _tiny_chunked()
    b = cb.new
    full_o, full_l = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                               cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale)
    rows = [np.array([0, 4]), np.array([3, 11])]
    o, l = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                     cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale, rows=rows, heads=[1])
    idx = [0, 4, 5 + 3, 5 + 11]
    np.testing.assert_array_equal(o[:, 0], full_o[idx, 1])
    np.testing.assert_array_equal(l[:, 0], full_l[idx, 1])
