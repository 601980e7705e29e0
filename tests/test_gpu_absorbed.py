"""GPU parity of the absorbed-weight prefill (multi-query attention of every head over the
paged latent cache rows, Dqk 576 / Dv 512) against the fp64 oracle."""
import os

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import absorbed_attention, gather_latent
from gpu_util import Guarded, check_attention, f64_of_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def kv_of_requests(b: wl.AbsorbedBatch):
    """Every request's cache rows in position order (the oracle's gather), and their indptr."""
    cu = wl.indptr_from_lengths(b.kv_lens)
    rows = gather_latent(b.cache, b.block_table, cu, np.zeros(b.batch, dtype=np.int32))
    return rows, cu


def oracle(b: wl.AbsorbedBatch, rows=None):
    """rows: per request, the query rows to compute (None: all)."""
    kv, cu = kv_of_requests(b)
    outs, lses = [], []
    for r in range(b.batch):
        q = b.q_abs[b.qo_indptr[r]:b.qo_indptr[r + 1]]
        o, lse = absorbed_attention(q, kv[cu[r]:cu[r + 1]], causal=b.causal, sm_scale=b.sm_scale,
                                    logits_soft_cap=b.logits_soft_cap, rows=None if rows is None else rows[r])
        outs.append(o)
        lses.append(lse)
    return np.concatenate(outs), np.concatenate(lses)


def run_gpu(b: wl.AbsorbedBatch, expect_status=0):
    import chunked_prefill_attention_ragged_gb300 as mla
    plan = mla.mla_absorbed_plan(b.qo_indptr, b.kv_lens, b.num_heads, b.block_size, causal=b.causal,
                                 sm_scale=b.sm_scale, logits_soft_cap=b.logits_soft_cap)
    q, cache, table = to_dev_bf16(b.q_abs), to_dev_bf16(b.cache), to_dev(b.block_table)
    t = b.q_abs.shape[0]
    g_o = Guarded((t, b.num_heads, 512), torch.bfloat16)
    g_l = Guarded((t, b.num_heads), torch.float32)
    o, lse = plan.run(q, cache, table, o=g_o.tensor, lse=g_l.tensor)
    torch.cuda.synchronize()
    if expect_status == 0:
        assert plan.status() == 0
    g_o.check("O_lat")
    g_l.check("LSE")
    return plan, (q, cache, table), o, lse


CASES = [
    # name, q_lens, kv_lens, heads, block_size, causal, cap
    ("basic", [17, 40], [17, 100], 16, 64, True, 0.0),
    ("block_16", [70, 130], [200, 130], 8, 16, True, 0.0),
    ("block_1", [5, 9], [40, 9], 4, 1, True, 0.0),
    ("block_48", [33], [250], 8, 48, True, 0.0),
    ("noncausal", [33, 1], [300, 64], 16, 32, False, 0.0),
    ("kv_shorter_than_q", [50], [20], 4, 64, True, 0.0),
    ("empty_and_zero_kv", [0, 10, 7], [5, 10, 0], 4, 64, True, 0.0),
    ("zero_kv_noncausal", [6, 3], [0, 65], 4, 64, False, 0.0),
    ("heads_128", [3, 2], [130, 300], 128, 64, True, 0.0),
    ("heads_48_rows_span_tiles", [37], [500], 48, 64, True, 0.0),
    ("softcap_30", [40], [200], 16, 64, True, 30.0),
    ("tile_edges", [1, 64, 65], [64, 128, 129], 2, 64, True, 0.0),
]


@pytest.mark.parametrize("name,q_lens,kv_lens,heads,bs,causal,cap", CASES, ids=[c[0] for c in CASES])
def test_absorbed_small_cases_full(name, q_lens, kv_lens, heads, bs, causal, cap):
    b = wl.random_absorbed(500 + [c[0] for c in CASES].index(name), q_lens, kv_lens, heads, block_size=bs,
                           causal=causal, logits_soft_cap=cap)
    _, _, o, lse = run_gpu(b)
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, name)


def test_absorbed_first_causal_row_is_first_latent_row():
    """A causal request with q_len = kv_len: its first row sees key 0 alone, so every head's
    O_lat is that cache row's first 512 values, bit for bit."""
    b = wl.random_absorbed(531, [40, 90], [40, 90], 16, block_size=16)
    _, _, o, _ = run_gpu(b)
    kv, cu = kv_of_requests(b)
    ob = o.view(torch.int16).cpu().numpy().view(np.uint16)
    for r in range(b.batch):
        np.testing.assert_array_equal(ob[b.qo_indptr[r]], np.broadcast_to(kv[cu[r], :512], (16, 512)))


def test_absorbed_prefix_sampled():
    """A prefix-sized case (2 requests of 256 new rows over 2304 and 1280 cache positions,
    128 heads): first 2, last 2, every 64-row step +-1 and 32 random rows, every head."""
    b = wl.random_absorbed(532, [256, 256], [2304, 1280], 128, block_size=64)
    _, _, o, lse = run_gpu(b)
    rng = np.random.default_rng(533)
    rows = []
    for lq in b.q_lens:
        s = {0, 1, int(lq) - 2, int(lq) - 1}
        for t in range(64, int(lq), 64):
            s.update({t - 1, t, t + 1})
        s.update(int(x) for x in rng.choice(int(lq), size=32, replace=False))
        rows.append(np.array(sorted(x for x in s if 0 <= x < lq)))
    o_ref, lse_ref = oracle(b, rows)
    idx = torch.from_numpy(np.concatenate([b.qo_indptr[r] + rows[r] for r in range(b.batch)])).cuda()
    check_attention(f64_of_bf16(o[idx]), lse[idx].double().cpu().numpy(), o_ref, lse_ref, "absorbed prefix")


def test_absorbed_bench_shape_sampled():
    """The benchmarked shape, planned and launched as the benchmark does (4 requests of 2048
    new rows, each the last of 10240 cache positions, 128 heads, 64-slot blocks out of 1024):
    per request the first 2 and last 2 rows, every 64-row tile boundary +-1 and 32 seeded
    random rows, on four heads."""
    b = wl.random_absorbed(1200, [2048] * 4, [10240] * 4, 128, block_size=64, num_blocks=1024)
    _, _, o, lse = run_gpu(b)
    kv, cu = kv_of_requests(b)
    heads = [0, 37, 90, 127]
    rng = np.random.default_rng(1202)
    for r in range(b.batch):
        lq = int(b.q_lens[r])
        s = {0, 1, lq - 2, lq - 1}
        for t in range(64, lq, 64):
            s.update({t - 1, t, t + 1})
        s.update(int(x) for x in rng.choice(lq, size=32, replace=False))
        rows = np.array(sorted(s))
        q = b.q_abs[b.qo_indptr[r]:b.qo_indptr[r + 1]][:, heads]
        o_ref, lse_ref = absorbed_attention(q, kv[cu[r]:cu[r + 1]], causal=True, sm_scale=b.sm_scale, rows=rows)
        idx = torch.from_numpy(b.qo_indptr[r] + rows).cuda()
        hs = torch.tensor(heads).cuda()
        check_attention(f64_of_bf16(o[idx][:, hs]), lse[idx][:, hs].double().cpu().numpy(), o_ref, lse_ref,
                        f"absorbed bench shape, request {r}")


def test_absorbed_repeat_runs_bitwise_identical():
    b = wl.random_absorbed(534, [130, 7], [300, 7], 16, block_size=32)
    plan, (q, cache, table), o1, l1 = run_gpu(b)
    o2, l2 = plan.run(q, cache, table)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def test_absorbed_bad_block_is_flagged_and_read_as_zeros():
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_absorbed(535, [20], [150], 4, block_size=64, causal=False)
    b.block_table[0, 1] = 10 ** 6                      # positions 64..127 name no block
    plan, _, o, lse = run_gpu(b, expect_status=-1)
    with pytest.raises(mla.MlaError) as err:
        plan.status()
    assert err.value.code == -6                        # MLA_ERR_DEVICE_BOUNDS
    # The oracle's view of the same thing: those positions hold zero rows.
    good = wl.random_absorbed(535, [20], [150], 4, block_size=64, causal=False)
    good.cache = np.concatenate([good.cache, np.zeros((1,) + good.cache.shape[1:], dtype=np.uint16)])
    good.block_table[0, 1] = good.cache.shape[0] - 1
    o_ref, lse_ref = oracle(good)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "bad block")


def test_absorbed_forced_timeout_then_normal_run(monkeypatch):
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_absorbed(536, [30], [200], 8, block_size=64)
    monkeypatch.setenv("MLA_TEST_FORCE_TIMEOUT_NS", "20000000")
    bad = mla.mla_absorbed_plan(b.qo_indptr, b.kv_lens, 8, 64, causal=True, sm_scale=b.sm_scale)
    monkeypatch.delenv("MLA_TEST_FORCE_TIMEOUT_NS")
    q, cache, table = to_dev_bf16(b.q_abs), to_dev_bf16(b.cache), to_dev(b.block_table)
    bad.run(q, cache, table)
    torch.cuda.synchronize()
    with pytest.raises(mla.MlaError) as err:
        bad.status()
    assert err.value.code == -5
    _, _, o, lse = run_gpu(b)
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "after time-out")


def test_absorbed_and_mha_plans_reject_each_other():
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_absorbed(537, [8], [8], 2, block_size=16)
    ap = mla.mla_absorbed_plan(b.qo_indptr, b.kv_lens, 2, 16, sm_scale=b.sm_scale)
    q = torch.zeros(8, 2, 192, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(8, 2, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(8, 2, 128, dtype=torch.bfloat16, device="cuda")
    lib = mla.library()
    import ctypes
    vp = lambda t: ctypes.c_void_p(t.data_ptr())
    assert lib.mla_prefill_run(ap.handle, vp(q), vp(q), vp(v), vp(o), None, None) == -1
    mp = mla.mla_prefill_plan(b.qo_indptr, b.qo_indptr, 2, causal=True, sm_scale=0.1)
    assert lib.mla_absorbed_run(mp.handle, vp(q), vp(q), 1, vp(q), 1, vp(o), None, None) == -1
    assert ap.num_units == 2 and ap.allowed_pairs == 8 * 9 // 2
