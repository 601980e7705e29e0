"""GPU parity of the full chunked-prefix pipeline (gather -> up-proj -> chunk attention -> merge)."""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import chunked_prefill_attention
from gpu_util import Guarded, check_attention, chunked_oracle_parallel, f64_of_bf16, sample_rows, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def run_pipeline(cb: wl.ChunkedPrefixBatch, fuse_merge=True):
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    b = cb.new
    pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                          sm_scale=b.sm_scale, logits_soft_cap=b.logits_soft_cap, fuse_merge=fuse_merge)
    rows = b.q.shape[0]
    g_o = Guarded((rows, b.num_heads, 128), torch.bfloat16)
    g_l = Guarded((rows, b.num_heads), torch.float32)
    o, lse = pipe.run(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev_bf16(cb.cache),
                      to_dev(cb.block_table), to_dev_bf16(cb.w_kvb), o=g_o.tensor, lse=g_l.tensor)
    torch.cuda.synchronize()
    pipe.check_status()
    g_o.check("pipeline O")
    g_l.check("pipeline LSE")
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
    """4 x (2048 new + 8192 cached), all 128 heads, on a row sample: first 2, last 2, every
    128-row tile boundary +-1 and 512 seeded random rows per request."""
    cb = wl.make_chunked_prefix()
    o, lse = run_pipeline(cb)
    b = cb.new
    rows = sample_rows(b.q_lens, n_random=512, every_tile=1, seed=2)
    o_ref, lse_ref = chunked_oracle_parallel(cb, rows)
    idx = torch.from_numpy(np.concatenate([b.qo_indptr[r] + rows[r] for r in range(b.batch)])).cuda()
    check_attention(f64_of_bf16(o[idx]), lse[idx].double().cpu().numpy(), o_ref, lse_ref, "workload2")


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


def test_small_chunked_fp8_cache_full():
    """The pipeline over an fp8 latent cache (dequantizing gather -> up-projection -> chunk
    attention merged into the new tokens' state) against the unchunked oracle over the
    oracle's dequantization of the same cache."""
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    from oracle import dequant_fp8_entries
    cb = wl.random_chunked_prefix(23, [130, 5, 260], [300, 0, 1000], 4, num_blocks=64, block_size=64,
                                  chunk_tokens=256)
    cache8 = wl.random_fp8_cache(np.random.default_rng(24), 64, 64, scale_exp=(126, 127), code_exp=(4, 8))
    b = cb.new
    pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                          sm_scale=b.sm_scale, cache_fp8=True)
    o, lse = pipe.run(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev(cache8), to_dev(cb.block_table),
                      to_dev_bf16(cb.w_kvb))
    torch.cuda.synchronize()
    pipe.check_status()
    cache_bf16 = dequant_fp8_entries(cache8.reshape(-1, 648)).reshape(64, 64, 576)
    o_ref, lse_ref = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cache_bf16, cb.block_table,
                                               cb.prefix_lens, cb.w_kvb, sm_scale=b.sm_scale)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "fp8 cache pipeline")


@pytest.mark.parametrize("paged", [True, False])
def test_small_chunked_paged_and_gathered_agree(paged):
    """The pipeline with the paged up-projection and with gather + up-projection: both
    against the oracle (and equal to each other bit for bit, same kernels downstream)."""
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    cb = wl.random_chunked_prefix(25, [77, 200], [500, 129], 3, num_blocks=16, block_size=64, chunk_tokens=192)
    b = cb.new
    outs = []
    for pg in (True, False):
        pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                              sm_scale=b.sm_scale, paged_up_proj=pg)
        o, lse = pipe.run(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v), to_dev_bf16(cb.cache),
                          to_dev(cb.block_table), to_dev_bf16(cb.w_kvb))
        torch.cuda.synchronize()
        pipe.check_status()
        outs.append((o, lse))
    assert torch.equal(outs[0][0].view(torch.int16), outs[1][0].view(torch.int16))
    assert torch.equal(outs[0][1], outs[1][1])
    o, lse = outs[0 if paged else 1]
    o_ref, lse_ref = chunked_prefill_attention(b.q, b.k, b.v, b.qo_indptr, cb.cache, cb.block_table, cb.prefix_lens,
                                               cb.w_kvb, sm_scale=b.sm_scale)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, f"paged={paged}")
