"""Prefill on CTA pairs (units of 256 query rows, one cluster of two CTAs each, tensor-core
products issued for both) against the oracle, and against the single-CTA plan bit for bit.

The planning mode is forced per plan with MLA_PLAN_CTA_PAIRS (read when a plan is made)."""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import chunked_prefill_attention, ragged_attention
from gpu_util import (Guarded, bits_of, check_attention, f64_of_bf16, oracle_parallel, sample_rows, to_dev,
                      to_dev_bf16)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def plan_in_mode(monkeypatch, pairs: bool, b: wl.RaggedBatch):
    import chunked_prefill_attention_ragged_gb300 as mla
    monkeypatch.setenv("MLA_PLAN_CTA_PAIRS", "1" if pairs else "0")
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)
    monkeypatch.delenv("MLA_PLAN_CTA_PAIRS")
    assert plan.cta_pairs == pairs
    return plan


def run_mode(monkeypatch, pairs: bool, b: wl.RaggedBatch, dev=None):
    plan = plan_in_mode(monkeypatch, pairs, b)
    q, k, v = dev if dev is not None else (to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v))
    rows = b.q.shape[0]
    g_o = Guarded((rows, b.num_heads, 128), torch.bfloat16)
    g_l = Guarded((rows, b.num_heads), torch.float32)
    o, lse = plan.run(q, k, v, o=g_o.tensor, lse=g_l.tensor)
    torch.cuda.synchronize()
    assert plan.status() == 0
    g_o.check("O")
    g_l.check("LSE")
    return (q, k, v), o, lse


def oracle(b: wl.RaggedBatch):
    return ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=b.causal, sm_scale=b.sm_scale,
                            window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)


CASES = [
    # name, q_lens, kv_lens, heads, causal, window, cap
    ("tile_edges", [1, 127, 128, 129, 255, 256, 257], None, 2, True, -1, 0.0),
    ("pair_edges", [383, 384, 385, 511, 512, 513], None, 2, True, -1, 0.0),
    ("prefix_longer_kv", [130, 7, 300], [700, 300, 301], 2, True, -1, 0.0),
    ("fewer_keys_than_queries", [300, 200], [100, 50], 2, True, -1, 0.0),
    ("noncausal_ragged", [300, 1, 77, 256], [1000, 129, 5, 3], 2, False, -1, 0.0),
    ("empty_requests", [0, 45, 0, 130, 260], [0, 45, 9, 130, 0], 2, False, -1, 0.0),
    ("window_100", [520, 130], None, 2, True, 100, 0.0),
    ("window_0", [300], None, 1, True, 0, 0.0),
    ("softcap_30", [260, 33], None, 2, True, -1, 30.0),
    ("ring_wrap_noncausal", [600, 40], [2000, 1500], 2, False, -1, 0.0),
    ("prefix_window", [520], [1000], 2, True, 200, 0.0),
]


@pytest.mark.parametrize("name,qlens,kvlens,heads,causal,window,cap", CASES, ids=[c[0] for c in CASES])
def test_pairs_match_oracle_and_single(monkeypatch, name, qlens, kvlens, heads, causal, window, cap):
    b = wl.random_ragged(300 + [c[0] for c in CASES].index(name), qlens, kvlens, heads, causal=causal,
                         window_left=window, logits_soft_cap=cap)
    dev, o2, l2 = run_mode(monkeypatch, True, b)
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o2), l2.double().cpu().numpy(), o_ref, lse_ref, f"pairs {name}")
    _, o1, l1 = run_mode(monkeypatch, False, b, dev)
    # Per row the two modes take the same products and the same softmax steps (a pair's
    # extra, fully masked key tiles add exact zeros), so they agree bit for bit.
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def test_pairs_workload1_full(monkeypatch):
    """The DeepSeek-shaped batch on CTA pairs: every row of every head against the oracle."""
    b = wl.make_workload(1)
    _, o, lse = run_mode(monkeypatch, True, b)
    ob = bits_of(o)
    for r in range(b.batch):
        np.testing.assert_array_equal(ob[b.qo_indptr[r]], b.v[b.kv_indptr[r]])
    o_ref, lse_ref = oracle_parallel(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "workload1 pairs")


def test_pairs_workload3_sampled(monkeypatch):
    b = wl.make_workload(3)
    _, o, lse = run_mode(monkeypatch, True, b)
    rows = sample_rows(b.q_lens, n_random=256, every_tile=2, seed=13)
    o_ref, lse_ref = oracle_parallel(b, rows=rows)
    idx = torch.from_numpy(np.concatenate([b.qo_indptr[r] + rows[r] for r in range(b.batch)])).cuda()
    check_attention(f64_of_bf16(o[idx]), lse[idx].double().cpu().numpy(), o_ref, lse_ref, "workload3 pairs")


@pytest.mark.parametrize("merge", [False, True])
def test_pairs_shared_rope_and_merge(monkeypatch, merge):
    """Shared-rope K (64-row rope boxes on a pair) and the merging epilogue on pairs give
    what the single-CTA plan gives, bit for bit."""
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(391, [300, 77, 1, 256], [700, 129, 5, 300], 4, causal=False)
    rng = np.random.default_rng(392)
    t = b.k.shape[0]
    rope = wl.to_bf16_bits(rng.standard_normal((t, 64)).astype(np.float32))
    b.k[:, :, 128:] = rope[:, None, :]
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    k_nope = k[:, :, :128].contiguous()
    k_rope = to_dev_bf16(rope)
    rows = b.q.shape[0]
    o0 = torch.randn(rows, 4, 128, device="cuda").to(torch.bfloat16)
    l0 = torch.randn(rows, 4, device="cuda")
    l0[::7] = float("-inf")
    outs = []
    for pairs in (False, True):
        plan = plan_in_mode(monkeypatch, pairs, b)
        g_o, g_l = Guarded((rows, 4, 128), torch.bfloat16), Guarded((rows, 4), torch.float32)
        g_o.tensor.copy_(o0)
        g_l.tensor.copy_(l0)
        o, l = mla.mla_prefill_run_shared_rope(plan, q, k_nope, k_rope, v, g_o.tensor, g_l.tensor, merge=merge)
        torch.cuda.synchronize()
        assert plan.status() == 0
        g_o.check("O")
        g_l.check("LSE")
        outs.append((o.clone(), l.clone()))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    if not merge:
        o_ref, lse_ref = oracle(b)
        check_attention(f64_of_bf16(outs[1][0]), outs[1][1].double().cpu().numpy(), o_ref, lse_ref, "pairs rope")


def test_pairs_chunked_pipeline(monkeypatch):
    """The whole chunked-prefix pipeline with every attention plan on CTA pairs."""
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    cb = wl.random_chunked_prefix(321, [260, 5, 130], [300, 0, 1000], 4, num_blocks=64, block_size=64,
                                  chunk_tokens=256)
    b = cb.new
    monkeypatch.setenv("MLA_PLAN_CTA_PAIRS", "1")
    pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                          sm_scale=b.sm_scale)
    monkeypatch.delenv("MLA_PLAN_CTA_PAIRS")
    assert pipe.main.cta_pairs and all(p.cta_pairs for p in pipe.chunks)
    o, lse = pipe.run(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev_bf16(cb.cache),
                      to_dev(cb.block_table), to_dev_bf16(cb.w_kvb))
    torch.cuda.synchronize()
    pipe.check_status()
    o_ref, lse_ref = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                               cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "pairs pipeline")


@pytest.mark.parametrize("merge", [False, True])
def test_pairs_forced_timeout(monkeypatch, merge):
    """The time-out test mode on a pair plan: every CTA of both clusters gives up, the status
    word says so, and the context stays usable."""
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(77, [300, 129], None, 2)
    monkeypatch.setenv("MLA_TEST_FORCE_TIMEOUT_NS", "20000000")
    plan = plan_in_mode(monkeypatch, True, b)
    monkeypatch.delenv("MLA_TEST_FORCE_TIMEOUT_NS")
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    rows = b.q.shape[0]
    o = torch.zeros(rows, 2, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(rows, 2, device="cuda")
    if merge:
        plan.run_merge(q, k, v, o, lse)
    else:
        plan.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    with pytest.raises(mla.MlaError):
        plan.status()
    good = plan_in_mode(monkeypatch, True, b)
    o2, l2 = good.run(q, k, v)
    torch.cuda.synchronize()
    assert good.status() == 0
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o2), l2.double().cpu().numpy(), o_ref, lse_ref, "after time-out")
