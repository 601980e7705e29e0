"""GPU parity of the full chunked-prefix pipeline (gather -> up-proj -> chunk attention -> merge)."""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import chunked_prefill_attention
from gpu_util import check_attention, f64_of_bf16, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def run_pipeline(cb: wl.ChunkedPrefixBatch, fuse_merge=True):
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    b = cb.new
    pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                          sm_scale=b.sm_scale, logits_soft_cap=b.logits_soft_cap, fuse_merge=fuse_merge)
    o, lse = pipe.run(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev_bf16(cb.cache),
                      to_dev(cb.block_table), to_dev_bf16(cb.w_kvb))
    torch.cuda.synchronize()
    pipe.check_status()
    return o, lse


@pytest.mark.parametrize("cap,fuse", [(0.0, True), (30.0, True), (0.0, False)])
def test_small_chunked_full(cap, fuse):
    cb = wl.random_chunked_prefix(21, [130, 5, 260], [300, 0, 1000], 4, num_blocks=64, block_size=64,
                                  chunk_tokens=256, logits_soft_cap=cap)
    o, lse = run_pipeline(cb, fuse_merge=fuse)
    b = cb.new
    o_ref, lse_ref = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                               cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale,
                                               logits_soft_cap=cap)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "small chunked")


def test_workload2_sampled():
    cb = wl.make_chunked_prefix()
    o, lse = run_pipeline(cb)
    b = cb.new
    rows = sample_rows(b.q_lens, n_random=16, every_tile=4, seed=2)
    heads = [0, 127]
    o_ref, lse_ref = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table,
                                               cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale, rows=rows,
                                               heads=heads)
    idx = torch.from_numpy(np.concatenate([b.qo_indptr[r] + rows[r] for r in range(b.batch)])).cuda()
    check_attention(f64_of_bf16(o[idx][:, heads]), lse[idx][:, heads].double().cpu().numpy(), o_ref, lse_ref,
                    "workload2")


def test_all_chunk_gather_matches_oracle_per_chunk():
    # The pipeline gathers every chunk's latent rows with one launch; chunk c's rows must
    # equal the oracle's gather of that chunk alone, bit for bit.
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    from oracle import gather_latent
    cb = wl.random_chunked_prefix(41, [30, 5, 17], [300, 1, 129], 2, num_blocks=40, block_size=16,
                                  chunk_tokens=100)
    b = cb.new
    pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                          sm_scale=b.sm_scale)
    table = torch.from_numpy(cb.block_table).cuda()
    lat = pipe.gather_all(to_dev_bf16(cb.cache), table)
    torch.cuda.synchronize()
    pipe.check_status()
    got = lat.view(torch.int16).cpu().numpy().view(np.uint16)
    for c in range(cb.layout.num_chunks):
        ref = gather_latent(cb.cache, cb.block_table, cb.layout.cu_seq_lens[c], cb.layout.chunk_starts[c])
        np.testing.assert_array_equal(got[pipe.row0[c]:pipe.row0[c + 1]], ref)


@pytest.mark.parametrize("causal", [False, True])
def test_run_merge_matches_oracle_merge(causal):
    """mla_prefill_run_merge on an entry state with live rows, rows at LSE = -inf (their O
    is NaN: it must never be read) and rows this attention gives no key, against the
    oracle's merge of the entry state with the oracle attention."""
    import chunked_prefill_attention_ragged_gb300 as mla
    from oracle import merge_state, ragged_attention
    q_lens, kv_lens = [130, 40, 0, 77], [300, 0, 12, 260]
    b = wl.random_ragged(57, q_lens, kv_lens, 3, causal=causal)
    rng = np.random.default_rng(58)
    rows = int(b.qo_indptr[-1])
    o_a = wl.to_bf16_bits(rng.standard_normal((rows, 3, 128)).astype(np.float32))
    lse_a = (rng.standard_normal((rows, 3)) * 3.0).astype(np.float32)
    dead = rng.random((rows, 3)) < 0.25
    lse_a[dead] = -np.inf
    o_a_dev = to_dev_bf16(o_a)
    o_a_dev[torch.from_numpy(dead).cuda()] = float("nan")
    lse_dev = torch.from_numpy(lse_a.copy()).cuda()
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, 3, causal=causal, sm_scale=b.sm_scale)
    o, lse = plan.run_merge(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v), o_a_dev, lse_dev)
    torch.cuda.synchronize()
    assert plan.status() == 0
    o_b, lse_b = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=causal, sm_scale=b.sm_scale)
    o_ref, lse_ref = merge_state(np.where(dead[..., None], 0, o_a).astype(np.uint16), lse_a, o_b, lse_b)
    assert not bool(torch.isnan(o).any())
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, f"run_merge causal={causal}")


def test_run_merge_requires_lse():
    """The merge entry point reads the entry LSE: a NULL lse is rejected on the host."""
    import ctypes
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(59, [40], [90], 2, causal=False)
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, 2, causal=False, sm_scale=b.sm_scale)
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    o = torch.zeros(40, 2, 128, dtype=torch.bfloat16, device="cuda")
    vp = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = mla.library().mla_prefill_run_merge(plan.handle, vp(q), vp(k), vp(v), vp(o), None, None)
    assert rc == -1
    with pytest.raises(ValueError):
        plan.run_merge(q, k, v, o, None)
