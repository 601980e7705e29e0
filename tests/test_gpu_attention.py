"""GPU parity of the ragged prefill attention kernel against the fp64 oracle."""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import bf16_bits_to_f64, ragged_attention
from gpu_util import Guarded, bits_of, check_attention, f64_of_bf16, oracle_parallel, sample_rows, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def run_gpu(b: wl.RaggedBatch, return_lse=True):
    """Plan and run through the binding, into outputs wrapped in guard bands that must
    come back untouched."""
    import chunked_prefill_attention_ragged_gb300 as mla
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    rows = b.q.shape[0]
    g_o = Guarded((rows, b.num_heads, 128), torch.bfloat16)
    g_l = Guarded((rows, b.num_heads), torch.float32) if return_lse else None
    o, lse = plan.run(q, k, v, o=g_o.tensor, lse=None if g_l is None else g_l.tensor, return_lse=return_lse)
    torch.cuda.synchronize()
    assert plan.status() == 0
    g_o.check("O")
    if g_l is not None:
        g_l.check("LSE")
    return plan, (q, k, v), o, lse


def assert_first_rows_are_v0(b: wl.RaggedBatch, o):
    """Row 0 of a causal request with Lq = Lkv sees key 0 alone, so its O is V[0] bit for bit."""
    ob = bits_of(o)
    for r in range(b.batch):
        if b.q_lens[r] > 0 and b.q_lens[r] == b.kv_lens[r]:
            np.testing.assert_array_equal(ob[b.qo_indptr[r]], b.v[b.kv_indptr[r]])


def oracle(b: wl.RaggedBatch, rows=None, heads=None):
    return ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=b.causal, sm_scale=b.sm_scale,
                            window_left=b.window_left, logits_soft_cap=b.logits_soft_cap, rows=rows, heads=heads)


SMALL = [
    # name, q_lens, kv_lens, heads, causal, window, cap
    ("tiny_workload", [17, 40], None, 4, True, -1, 0.0),
    ("tile_edges", [1, 127, 128, 129, 255, 256, 257], None, 2, True, -1, 0.0),
    ("prefix_longer_kv", [130, 7], [700, 300], 2, True, -1, 0.0),
    ("fewer_keys_than_queries", [300, 200], [100, 50], 2, True, -1, 0.0),
    ("noncausal_ragged", [300, 1, 77], [1000, 129, 5], 2, False, -1, 0.0),
    ("empty_requests", [0, 45, 0, 130], [0, 45, 9, 130], 2, True, -1, 0.0),
    ("noncausal_no_keys", [33, 20], [0, 64], 2, False, -1, 0.0),
    ("window_100", [520, 130], None, 2, True, 100, 0.0),
    ("window_0", [200], None, 1, True, 0, 0.0),
    ("softcap_30", [260, 33], None, 2, True, -1, 30.0),
    ("softcap_noncausal", [100], [300], 2, False, -1, 5.0),
    ("block_edges", [383, 384, 385, 511, 512, 513], None, 2, True, -1, 0.0),
    ("ring_wrap_noncausal", [300, 40], [2000, 1500], 2, False, -1, 0.0),
    ("window_300_long", [1500], None, 1, True, 300, 0.0),
    ("prefix_window", [260], [1000], 2, True, 200, 0.0),
]


@pytest.mark.parametrize("name,qlens,kvlens,heads,causal,window,cap", SMALL, ids=[c[0] for c in SMALL])
def test_small_cases_full(name, qlens, kvlens, heads, causal, window, cap):
    b = wl.random_ragged(100 + [c[0] for c in SMALL].index(name), qlens, kvlens, heads, causal=causal, window_left=window,
                         logits_soft_cap=cap)
    _, _, o, lse = run_gpu(b)
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, name)


def test_workload0_and_first_row_exact():
    b = wl.make_workload(0)
    _, _, o, lse = run_gpu(b)
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "workload0")
    assert_first_rows_are_v0(b, o)


def test_constant_v_and_lse_optional():
    b = wl.random_ragged(5, [300, 129], None, 2)
    c = wl.to_bf16_bits(np.random.default_rng(2).standard_normal(128).astype(np.float32))
    b.v[:] = c[None, None, :]
    _, _, o, lse = run_gpu(b, return_lse=False)
    assert lse is None
    np.testing.assert_allclose(f64_of_bf16(o), np.broadcast_to(bf16_bits_to_f64(c), o.shape), rtol=0, atol=1e-2)


def test_output_alignment_paths_agree():
    # A 32-byte aligned O takes 32-byte stores, a 16-byte aligned one 16-byte stores.
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(31, [300, 129], None, 4)
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=True, sm_scale=b.sm_scale)
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    rows = b.q.shape[0]
    o32, lse32 = plan.run(q, k, v)
    buf = torch.zeros(rows * 4 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    o16 = buf[8:].view(rows, 4, 128)
    assert o16.data_ptr() % 32 == 16
    plan.run(q, k, v, o=o16, lse=torch.empty_like(lse32))
    torch.cuda.synchronize()
    assert torch.equal(o32.view(torch.int16), o16.view(torch.int16))


def test_repeat_runs_bitwise_identical():
    b = wl.random_ragged(9, [700, 260, 3], None, 4)
    plan, (q, k, v), o1, l1 = run_gpu(b)
    o2, l2 = plan.run(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(l1, l2)


def _trend_batch(q_lens, kv_lens, heads, causal, slope, seed):
    """Q and K share a common direction whose weight in K changes by `slope` logits per key
    (natural units) along each request, plus noise: with slope > 0 a row's running max
    grows by ~slope * 128 per key tile, far past the 2^8 rescale threshold, so the O
    rescale runs on every tile; with slope < 0 the first tile holds the max throughout."""
    rng = np.random.default_rng(seed)
    b = wl.random_ragged(seed, q_lens, kv_lens, heads, causal=causal, name="trend")
    q = 1.0 + 0.3 * rng.standard_normal(b.q.shape)
    k = 0.3 * rng.standard_normal(b.k.shape)
    per_key = slope / (b.sm_scale * 192.0)          # logit change per key for q ~ ones
    for r in range(b.batch):
        lo, hi = int(b.kv_indptr[r]), int(b.kv_indptr[r + 1])
        pos = np.arange(hi - lo, dtype=np.float64)
        w = per_key * (pos if slope > 0 else pos - (hi - lo))
        k[lo:hi] += w[:, None, None]
    b.q = wl.to_bf16_bits(q.astype(np.float32))
    b.k = wl.to_bf16_bits(k.astype(np.float32))
    return b


@pytest.mark.parametrize("q_lens,kv_lens,causal,slope", [
    ([520, 300], None, True, 0.06),
    ([520, 300], None, True, -0.06),
    ([200, 70], [900, 260], False, 0.05),
    ([130], [700], True, 0.2),
], ids=["causal_rising", "causal_falling", "noncausal_rising", "prefix_steep"])
def test_running_max_rescale_paths(q_lens, kv_lens, causal, slope):
    b = _trend_batch(q_lens, kv_lens, 2, causal, slope, seed=len(q_lens) + int(abs(slope) * 100))
    _, _, o, lse = run_gpu(b)
    o_ref, lse_ref = oracle(b)
    # The logits really do span many rescale thresholds.
    assert np.nanmax(lse_ref) - np.nanmin(lse_ref) > 12.0
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, f"trend {slope}")


@pytest.mark.parametrize("cap", [0.0, 30.0])
def test_workload4_many_short_full(cap):
    b = wl.make_workload(4, logits_soft_cap=cap)
    _, _, o, lse = run_gpu(b)
    o_ref, lse_ref = oracle(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, f"workload4 cap={cap}")
    assert_first_rows_are_v0(b, o)


def test_workload1_full():
    """The DeepSeek-shaped batch (8 requests, 128 heads): every row of every head against
    the oracle, computed over (request, head) pieces in a spawned process pool."""
    b = wl.make_workload(1)
    _, _, o, lse = run_gpu(b)
    assert_first_rows_are_v0(b, o)
    o_ref, lse_ref = oracle_parallel(b)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "workload1")


def test_workload3_long_sampled():
    """1 x 32768 tokens, all 128 heads, on a row sample: first 2, last 2, every 128-row
    tile boundary +-1 and 512 seeded random rows."""
    b = wl.make_workload(3)
    _, _, o, lse = run_gpu(b)
    assert_first_rows_are_v0(b, o)
    rows = sample_rows(b.q_lens, n_random=512, every_tile=1, seed=3)
    o_ref, lse_ref = oracle_parallel(b, rows=rows)
    idx = torch.from_numpy(np.concatenate([b.qo_indptr[r] + rows[r] for r in range(b.batch)])).cuda()
    check_attention(f64_of_bf16(o[idx]), lse[idx].double().cpu().numpy(), o_ref, lse_ref, "workload3")


@pytest.mark.parametrize("merge", [False, True])
@pytest.mark.parametrize("strided", [False, True])
def test_shared_rope_equals_full_k(merge, strided):
    """K given as per-head K_nope plus one rope row per key (the same in every head) gives
    bit for bit what the concatenated K [T, H, 192] gives; the rope may be a strided view
    (the rope columns of a [T, 576] latent)."""
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(91, [300, 77, 1], [700, 129, 5], 4, causal=False)
    rng = np.random.default_rng(92)
    t = b.k.shape[0]
    rope = wl.to_bf16_bits(rng.standard_normal((t, 64)).astype(np.float32))
    b.k[:, :, 128:] = rope[:, None, :]                      # the full K carries the rope in every head
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, 4, causal=False, sm_scale=b.sm_scale)
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    k_nope = k[:, :, :128].contiguous()
    if strided:
        lat = torch.zeros(t, 576, dtype=torch.bfloat16, device="cuda")
        lat[:, 512:] = to_dev_bf16(rope)
        k_rope = lat[:, 512:]
    else:
        k_rope = to_dev_bf16(rope)
    rows = b.q.shape[0]
    o0 = torch.randn(rows, 4, 128, device="cuda").to(torch.bfloat16)
    l0 = torch.randn(rows, 4, device="cuda")
    if merge:
        o_ref, l_ref = plan.run_merge(q, k, v, o0.clone(), l0.clone())
        g_o, g_l = Guarded((rows, 4, 128), torch.bfloat16), Guarded((rows, 4), torch.float32)
        g_o.tensor.copy_(o0)
        g_l.tensor.copy_(l0)
        o, l = mla.mla_prefill_run_shared_rope(plan, q, k_nope, k_rope, v, g_o.tensor, g_l.tensor, merge=True)
    else:
        o_ref, l_ref = plan.run(q, k, v)
        g_o, g_l = Guarded((rows, 4, 128), torch.bfloat16), Guarded((rows, 4), torch.float32)
        o, l = mla.mla_prefill_run_shared_rope(plan, q, k_nope, k_rope, v, g_o.tensor, g_l.tensor)
    torch.cuda.synchronize()
    assert plan.status() == 0
    g_o.check("shared-rope O")
    g_l.check("shared-rope LSE")
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(l, l_ref)
    if not merge:
        o_or, l_or = oracle(b)
        check_attention(f64_of_bf16(o), l.double().cpu().numpy(), o_or, l_or, "shared rope")
