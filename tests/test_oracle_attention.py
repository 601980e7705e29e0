"""Pins for the fp64 attention oracle (CPU only).

The pages print no numeric example, so the oracle is pinned by
  * hand-derived closed forms (tests/golden/attention_hand_cases.json),
  * an independent pure-Python brute force on tiny inputs,
  * invariants that hold for softmax attention whatever the data.
"""
import json
import math
import os

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import allowed_mask, attend_request, bf16_bits_to_f64, merge_state, ragged_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attention_hand_cases.json")


def _f(x):
    return -math.inf if x == "-inf" else float(x)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_cases(case):
    q = np.array(case["q"], dtype=np.float64)[:, None, :]
    k = np.array(case["k"], dtype=np.float64)[:, None, :]
    v = np.array(case["v"], dtype=np.float64)[:, None, :]
    o, lse = attend_request(q, k, v, causal=case["causal"], sm_scale=case["sm_scale"],
                            window_left=case["window_left"], logits_soft_cap=case["cap"])
    np.testing.assert_allclose(o[:, 0, :], np.array(case["o"], dtype=np.float64), rtol=0, atol=1e-13)
    exp_lse = np.array([_f(x) for x in case["lse"]])
    assert np.array_equal(np.isinf(lse[:, 0]), np.isinf(exp_lse))
    fin = np.isfinite(exp_lse)
    np.testing.assert_allclose(lse[fin, 0], exp_lse[fin], rtol=0, atol=1e-13)


def _brute(q, k, v, causal, scale, window, cap, dv):
    """Per-element loops with math.fsum; a separate formulation of the same definition."""
    lq, lkv = len(q), len(k)
    out_o, out_l = [], []
    for i in range(lq):
        pos = i + lkv - lq
        logits = []
        for j in range(lkv):
            if causal and j > pos:
                continue
            if window >= 0 and j < pos - window:
                continue
            x = scale * math.fsum(a * b for a, b in zip(q[i], k[j]))
            logits.append((j, cap * math.tanh(x / cap) if cap > 0 else x))
        if not logits:
            out_o.append([0.0] * dv)
            out_l.append(-math.inf)
            continue
        top = max(s for _, s in logits)
        lse = top + math.log(math.fsum(math.exp(s - top) for _, s in logits))
        out_o.append([math.fsum(math.exp(s - lse) * v[j][e] for j, s in logits) for e in range(dv)])
        out_l.append(lse)
    return np.array(out_o).reshape(lq, dv), np.array(out_l)


BRUTE_CASES = [
    # (q_lens, kv_lens, heads, causal, window, cap, dqk, dv)
    ([3, 9, 1], None, 2, True, -1, 0.0, 192, 128),
    ([5, 2], [7, 9], 2, True, -1, 0.0, 16, 8),
    ([5, 2], [7, 9], 1, False, -1, 0.0, 16, 8),
    ([9], None, 2, True, 2, 0.0, 16, 8),
    ([4, 6], [4, 8], 1, True, 1, 5.0, 16, 8),
    ([6], [3], 1, True, -1, 0.0, 8, 4),        # Lkv < Lq: leading rows see nothing
    ([0, 4], [3, 4], 1, False, -1, 30.0, 8, 4),  # an empty request
    ([2], [0], 1, False, -1, 0.0, 8, 4),       # no keys at all
]


@pytest.mark.parametrize("qlens,kvlens,heads,causal,window,cap,dqk,dv", BRUTE_CASES)
def test_brute_force_tiny(qlens, kvlens, heads, causal, window, cap, dqk, dv):
    b = wl.random_ragged(7, qlens, kvlens, heads, dqk=dqk, dv=dv, causal=causal,
                         window_left=window, logits_soft_cap=cap, sm_scale=0.37)
    o, lse = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=causal,
                              sm_scale=0.37, window_left=window, logits_soft_cap=cap)
    qo, kv = b.qo_indptr, b.kv_indptr
    q, k, v = bf16_bits_to_f64(b.q), bf16_bits_to_f64(b.k), bf16_bits_to_f64(b.v)
    for r in range(b.batch):
        for h in range(heads):
            bo, bl = _brute(q[qo[r]:qo[r + 1], h].tolist(), k[kv[r]:kv[r + 1], h].tolist(),
                            v[kv[r]:kv[r + 1], h].tolist(), causal, 0.37, window, cap, dv)
            np.testing.assert_allclose(o[qo[r]:qo[r + 1], h], bo, rtol=0, atol=1e-12)
            got = lse[qo[r]:qo[r + 1], h]
            assert np.array_equal(np.isinf(got), np.isinf(bl))
            np.testing.assert_allclose(got[np.isfinite(bl)], bl[np.isfinite(bl)], rtol=0, atol=1e-12)


def _small(seed=3, lens=(17, 40, 5), heads=3, **kw):
    return wl.random_ragged(seed, list(lens), None, heads, **kw)


def _run(b, **over):
    args = dict(causal=b.causal, sm_scale=b.sm_scale, window_left=b.window_left,
                logits_soft_cap=b.logits_soft_cap)
    args.update(over)
    return ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, **args)


def test_first_causal_row_is_v0():
    b = _small()
    o, lse = _run(b)
    q, k, v = (bf16_bits_to_f64(x) for x in (b.q, b.k, b.v))
    for r in range(b.batch):
        s = b.qo_indptr[r]
        np.testing.assert_array_equal(o[s], v[s])
        np.testing.assert_allclose(lse[s], b.sm_scale * np.einsum("hd,hd->h", q[s], k[s]),
                                   rtol=0, atol=1e-13)


def test_constant_v_gives_constant_o():
    b = _small()
    c = wl.to_bf16_bits(np.random.default_rng(1).standard_normal(128).astype(np.float32))
    b.v[:] = c[None, None, :]
    o, _ = _run(b)
    np.testing.assert_allclose(o, np.broadcast_to(bf16_bits_to_f64(c), o.shape), rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one():
    # With V = identity rows, O is the probability row itself.
    lq = lkv = 12
    rng = np.random.default_rng(5)
    q = rng.standard_normal((lq, 1, 24))
    k = rng.standard_normal((lkv, 1, 24))
    v = np.eye(lkv)[:, None, :]
    for causal, window in ((True, -1), (False, -1), (True, 3)):
        o, _ = attend_request(q, k, v, causal=causal, sm_scale=0.5, window_left=window)
        p = o[:, 0, :]
        assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
        assert np.all(p[~allowed_mask(lq, lkv, causal, window)] == 0.0)


def test_lse_bounds():
    b = _small(heads=2)
    o, lse = _run(b)
    q, k = bf16_bits_to_f64(b.q), bf16_bits_to_f64(b.k)
    for r in range(b.batch):
        for i in range(b.q_lens[r]):
            row = b.qo_indptr[r] + i
            ks = k[b.kv_indptr[r]:b.kv_indptr[r] + i + 1]
            s = b.sm_scale * np.einsum("jhd,hd->hj", ks, q[row])
            top = s.max(axis=1)
            assert np.all(lse[row] >= top - 1e-12)
            assert np.all(lse[row] <= top + math.log(i + 1) + 1e-12)


def test_huge_cap_equals_no_cap():
    b = _small()
    o0, l0 = _run(b)
    o1, l1 = _run(b, logits_soft_cap=1e7)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-9)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-9)


def test_cap_bounds_logits():
    b = _small(sm_scale=50.0)
    _, lse = _run(b, logits_soft_cap=2.0, sm_scale=50.0)
    for r in range(b.batch):
        for i in range(b.q_lens[r]):
            assert lse[b.qo_indptr[r] + i].max() <= 2.0 + math.log(i + 1) + 1e-12


def test_wide_window_equals_no_window():
    b = _small()
    o0, l0 = _run(b)
    o1, l1 = _run(b, window_left=int(b.kv_lens.max()))
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(l1, l0)


def test_window_zero_is_diagonal():
    b = _small()
    o, lse = _run(b, window_left=0)
    q, k, v = (bf16_bits_to_f64(x) for x in (b.q, b.k, b.v))
    np.testing.assert_array_equal(o, v)      # Lq == Lkv, so row i sees key i only
    np.testing.assert_allclose(lse, b.sm_scale * np.einsum("thd,thd->th", q, k), rtol=0, atol=1e-12)


def test_noncausal_key_permutation_invariance():
    b = _small(causal=False)
    o0, l0 = _run(b)
    rng = np.random.default_rng(9)
    for r in range(b.batch):
        s, e = b.kv_indptr[r], b.kv_indptr[r + 1]
        perm = s + rng.permutation(e - s)
        b.k[s:e] = b.k[perm]
        b.v[s:e] = b.v[perm]
    o1, l1 = _run(b)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def test_ragged_isolation():
    b = _small()
    o, lse = _run(b)
    for r in range(b.batch):
        qs, qe = b.qo_indptr[r], b.qo_indptr[r + 1]
        ks, ke = b.kv_indptr[r], b.kv_indptr[r + 1]
        o1, l1 = attend_request(b.q[qs:qe], b.k[ks:ke], b.v[ks:ke], causal=True, sm_scale=b.sm_scale)
        np.testing.assert_array_equal(o1, o[qs:qe])
        np.testing.assert_array_equal(l1, lse[qs:qe])


def test_single_token():
    b = wl.random_ragged(11, [1], None, 2)
    o, lse = _run(b)
    q, k, v = (bf16_bits_to_f64(x) for x in (b.q, b.k, b.v))
    np.testing.assert_array_equal(o[0], v[0])
    np.testing.assert_allclose(lse[0], b.sm_scale * np.einsum("hd,hd->h", q[0], k[0]), rtol=0, atol=1e-13)


def test_zero_q_is_uniform():
    b = _small()
    b.q[:] = 0
    o, lse = _run(b)
    v = bf16_bits_to_f64(b.v)
    for r in range(b.batch):
        for i in range(b.q_lens[r]):
            row = b.qo_indptr[r] + i
            keys = v[b.kv_indptr[r]:b.kv_indptr[r] + i + 1]
            np.testing.assert_allclose(o[row], keys.mean(axis=0), rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[row], math.log(i + 1), rtol=0, atol=1e-13)


def test_split_merge_equals_unsplit():
    """Non-causal attention over keys A u B == merge(attn over A, attn over B)."""
    rng = np.random.default_rng(21)
    b = wl.random_ragged(13, [7, 30], [40, 25], 2, causal=False)
    o_full, l_full = _run(b)
    for trial in range(4):
        cuts = [b.kv_indptr[r] + (int(rng.integers(0, b.kv_lens[r] + 1)) if trial else 0)
                for r in range(b.batch)]
        parts = []
        for piece in range(2):
            ks, vs, lens = [], [], []
            for r in range(b.batch):
                s, e, cut = b.kv_indptr[r], b.kv_indptr[r + 1], cuts[r]
                sl = slice(s, cut) if piece == 0 else slice(cut, e)
                ks.append(b.k[sl]); vs.append(b.v[sl]); lens.append(sl.stop - sl.start)
            parts.append(ragged_attention(b.q, np.concatenate(ks), np.concatenate(vs), b.qo_indptr,
                                          wl.indptr_from_lengths(lens), causal=False,
                                          sm_scale=b.sm_scale))
        o, l = merge_state(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
        np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, l_full, rtol=0, atol=1e-12)


def test_masks_match_definition_counts():
    # Causal Lq=Lkv=L has L(L+1)/2 allowed pairs; window w keeps min(i+1, w+1) per row.
    for L in (1, 5, 130):
        assert allowed_mask(L, L, True, -1).sum() == L * (L + 1) // 2
        assert allowed_mask(L, L, False, -1).sum() == L * L
        for w in (0, 3, 200):
            assert allowed_mask(L, L, True, w).sum() == sum(min(i + 1, w + 1) for i in range(L))
