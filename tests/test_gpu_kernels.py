"""GPU parity of the gather, up-projection and merge kernels against the oracle."""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import bf16_bits_to_f64, cache_write, gather_latent, merge_state, round_f64_to_bf16, up_project
from gpu_util import Guarded, bits_of, f64_of_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _mla():
    import chunked_prefill_attention_ragged_gb300 as mla
    return mla


# ------------------------------------------------------------------ gather
def test_gather_workload2_bit_exact():
    mla = _mla()
    cb = wl.make_chunked_prefix()
    cache = to_dev_bf16(cb.cache)
    table = to_dev(cb.block_table)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c in range(cb.layout.num_chunks):
        cu, st = cb.layout.cu_seq_lens[c], cb.layout.chunk_starts[c]
        g = Guarded((int(cu[-1]), 576), torch.bfloat16)
        out = mla.mla_gather_latent(cache, table, to_dev(cu), to_dev(st), int(cu[-1]), out=g.tensor, status=status)
        torch.cuda.synchronize()
        g.check("gather")
        np.testing.assert_array_equal(bits_of(out), gather_latent(cb.cache, cb.block_table, cu, st))
    assert int(status.item()) == 0


@pytest.mark.parametrize("block_size,chunk", [(1, 3), (16, 40), (64, 100), (64, 4096)])
def test_gather_random_tables(block_size, chunk):
    mla = _mla()
    cb = wl.random_chunked_prefix(block_size + chunk, [3, 3, 3], [0, 1000, 333], 1,
                                  num_blocks=(2000 // block_size) + 8, block_size=block_size, chunk_tokens=chunk)
    cache, table = to_dev_bf16(cb.cache), to_dev(cb.block_table)
    for c in range(cb.layout.num_chunks):
        cu, st = cb.layout.cu_seq_lens[c], cb.layout.chunk_starts[c]
        g = Guarded((int(cu[-1]), 576), torch.bfloat16)
        out = mla.mla_gather_latent(cache, table, to_dev(cu), to_dev(st), int(cu[-1]), out=g.tensor)
        torch.cuda.synchronize()
        g.check("gather")
        np.testing.assert_array_equal(bits_of(out), gather_latent(cb.cache, cb.block_table, cu, st))


def test_gather_bad_block_id_flags_and_zeroes():
    mla = _mla()
    cb = wl.random_chunked_prefix(4, [2, 2], [70, 70], 1, num_blocks=4, block_size=64, chunk_tokens=128)
    table = cb.block_table.copy()
    table[1, 1] = 99                     # outside the cache
    cu, st = cb.layout.cu_seq_lens[0], cb.layout.chunk_starts[0]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mla.mla_gather_latent(to_dev_bf16(cb.cache), to_dev(table), to_dev(cu), to_dev(st), int(cu[-1]),
                                status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    got = bits_of(out)
    good = table.copy()
    good[1, 1] = cb.block_table[1, 1]
    ref = gather_latent(cb.cache, good, cu, st)
    bad_rows = np.arange(cu[1] + 64, cu[2])     # request 1, positions 64..69
    np.testing.assert_array_equal(got[bad_rows], 0)
    keep = np.setdiff1d(np.arange(cu[-1]), bad_rows)
    np.testing.assert_array_equal(got[keep], ref[keep])


@pytest.mark.parametrize("entry_dim", [8, 72, 18432, 18440])
def test_gather_row_widths(entry_dim):
    # 16-byte rows up to 36 KB go through the bulk-copy kernel (one or several rows per
    # CTA, partial last batch); wider rows take the register-vector kernel.
    mla = _mla()
    rng = np.random.default_rng(entry_dim)
    num_blocks, block_size = 7, 4
    cache = rng.integers(0, 1 << 16, size=(num_blocks, block_size, entry_dim), dtype=np.uint16)
    table = rng.permutation(num_blocks)[:6].reshape(2, 3).astype(np.int32)
    cu = np.array([0, 9, 19], dtype=np.int32)
    st = np.array([1, 0], dtype=np.int32)
    g = Guarded((int(cu[-1]), entry_dim), torch.bfloat16)
    out = mla.mla_gather_latent(to_dev_bf16(cache), to_dev(table), to_dev(cu), to_dev(st), int(cu[-1]), out=g.tensor)
    torch.cuda.synchronize()
    g.check("gather")
    np.testing.assert_array_equal(bits_of(out), gather_latent(cache, table, cu, st))


# ------------------------------------------------------------------ cache write
def _slots(rng, n_tokens, num_slots, pad=0):
    s = rng.permutation(num_slots)[:n_tokens].astype(np.int64)
    if pad:
        s[rng.choice(n_tokens, pad, replace=False)] = -1
    return s


@pytest.mark.parametrize("entry_dim,tokens,pad", [(576, 301, 17), (576, 1, 0), (8, 64, 5), (72, 33, 33),
                                                  (18440, 7, 2), (32768, 5, 1)])
def test_cache_write_bit_exact(entry_dim, tokens, pad):
    # One or several rows per CTA (ragged last batch), padding slots, rows wider than the
    # 48 KB default shared-memory limit.
    mla = _mla()
    rng = np.random.default_rng(entry_dim + tokens)
    nb, bs = 40, 8
    cache = rng.integers(0, 1 << 16, size=(nb, bs, entry_dim), dtype=np.uint16)
    lat = rng.integers(0, 1 << 16, size=(tokens, entry_dim), dtype=np.uint16)
    slots = _slots(rng, tokens, nb * bs, pad)
    g = Guarded((nb, bs, entry_dim), torch.bfloat16)
    d_cache = g.tensor
    d_cache.copy_(to_dev_bf16(cache))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_write(d_cache, to_dev_bf16(lat), to_dev(slots), status=status)
    torch.cuda.synchronize()
    g.check("cache write")
    assert int(status.item()) == 0
    np.testing.assert_array_equal(bits_of(d_cache), cache_write(cache, lat, slots))


def test_cache_write_bad_slot_is_flagged_and_skipped():
    mla = _mla()
    rng = np.random.default_rng(9)
    cache = rng.integers(0, 1 << 16, size=(4, 16, 576), dtype=np.uint16)
    lat = rng.integers(0, 1 << 16, size=(6, 576), dtype=np.uint16)
    slots = np.array([3, 64, 10, 1000, -5, 63], dtype=np.int64)   # 64 and 1000 are past the cache
    g = Guarded((4, 16, 576), torch.bfloat16)
    d_cache = g.tensor
    d_cache.copy_(to_dev_bf16(cache))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_write(d_cache, to_dev_bf16(lat), to_dev(slots), status=status)
    torch.cuda.synchronize()
    g.check("cache write with bad slots")
    assert int(status.item()) & 2
    keep = slots.copy()
    keep[(keep >= 64)] = -1
    np.testing.assert_array_equal(bits_of(d_cache), cache_write(cache, lat, keep))


def test_cache_write_then_gather_round_trip():
    # New positions written through the slot rule come back out of the gather unchanged.
    mla = _mla()
    rng = np.random.default_rng(5)
    nb, bs = 16, 16
    cache = rng.integers(0, 1 << 16, size=(nb, bs, 576), dtype=np.uint16)
    table = rng.permutation(nb)[:12].reshape(2, 6).astype(np.int32)   # 96 positions per request
    starts, lens = [70, 33], [25, 40]
    slots = np.array([int(table[r, p // bs]) * bs + p % bs for r in range(2)
                      for p in range(starts[r], starts[r] + lens[r])], dtype=np.int64)
    lat = rng.integers(0, 1 << 16, size=(len(slots), 576), dtype=np.uint16)
    d_cache = to_dev_bf16(cache)
    mla.mla_cache_write(d_cache, to_dev_bf16(lat), to_dev(slots))
    cu = wl.indptr_from_lengths(lens)
    back = mla.mla_gather_latent(d_cache, to_dev(table), to_dev(cu), to_dev(np.array(starts, dtype=np.int32)),
                                 int(cu[-1]))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits_of(back), lat)


# ------------------------------------------------------------------ up-projection
def _check_up_proj(lat, w, heads, k, v):
    """Element-wise: one bf16 rounding of a value that fp32 accumulation may have moved by
    at most 512 * 2^-23 * sum|latent * W|; the rope part is a bit-exact copy."""
    k_ref, v_ref = up_project(lat, w, heads)
    a = np.abs(bf16_bits_to_f64(lat[:, :512]))
    wa = np.abs(bf16_bits_to_f64(w))
    mag = (a @ wa).reshape(lat.shape[0], heads, 256)
    acc_bound = 512 * 2.0 ** -23 * mag
    kg, vg = f64_of_bf16(k), f64_of_bf16(v)
    np.testing.assert_array_equal(kg[:, :, 128:], k_ref[:, :, 128:])
    for got, ref, bound, what in ((kg[:, :, :128], k_ref[:, :, :128], acc_bound[..., :128], "K_nope"),
                                  (vg, v_ref, acc_bound[..., 128:], "V")):
        rref = round_f64_to_bf16(ref)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
        err = np.abs(got - ref)
        worst = np.max(err / (ulp + bound))
        assert worst <= 1.0, f"{what}: error {worst:.3f} x (ulp + accumulation bound)"
        assert np.mean(got != rref) < 0.02, f"{what}: {np.mean(got != rref):.4f} differ from exact rounding"


@pytest.mark.parametrize("tokens,heads,out_offset", [(300, 4, 0), (128, 1, 0), (1, 2, 0), (1000, 16, 0),
                                                     (300, 4, 8), (77, 3, 8), (2048, 128, 0), (1100, 37, 0)])
def test_up_proj_matches_rounded_oracle(tokens, heads, out_offset):
    """out_offset = 8 elements puts K and V 16 but not 32 bytes into their buffers (16-byte
    stores).  2048 x 128 heads is 2048 tiles, over 13 per CTA: every CTA's range crosses
    token blocks (the latent tile reloaded in mid-range) and reuses both TMEM
    accumulators; 1100 x 37 gives ranges that start and end inside a token block."""
    mla = _mla()
    rng = np.random.default_rng(tokens + heads)
    lat = wl.to_bf16_bits(rng.standard_normal((tokens, 576)).astype(np.float32))
    w = wl.to_bf16_bits((rng.standard_normal((512, heads * 256)) * 512 ** -0.5).astype(np.float32))
    g_k = Guarded((out_offset + tokens * heads * 192,), torch.bfloat16, fill=float("nan"))
    g_v = Guarded((out_offset + tokens * heads * 128,), torch.bfloat16, fill=float("nan"))
    k_out = g_k.tensor[out_offset:].view(tokens, heads, 192)
    v_out = g_v.tensor[out_offset:].view(tokens, heads, 128)
    k, v = mla.mla_up_proj(to_dev_bf16(lat), to_dev_bf16(w), heads, k_out=k_out, v_out=v_out)
    torch.cuda.synchronize()
    g_k.check("up-projection K")
    g_v.check("up-projection V")
    assert bool(torch.isnan(g_k.tensor[:out_offset]).all()) and bool(torch.isnan(g_v.tensor[:out_offset]).all())
    _check_up_proj(lat, w, heads, k, v)


# ------------------------------------------------------------------ merge
def _merge_inputs(rows, heads, seed, dim=128):
    rng = np.random.default_rng(seed)
    oa = wl.to_bf16_bits(rng.standard_normal((rows, heads, dim)).astype(np.float32))
    ob = wl.to_bf16_bits(rng.standard_normal((rows, heads, dim)).astype(np.float32))
    la = (rng.standard_normal((rows, heads)) * 4).astype(np.float32)
    lb = (rng.standard_normal((rows, heads)) * 4).astype(np.float32)
    la[::7, 0] = -np.inf
    lb[::5, -1] = -np.inf
    la[3, :] = -np.inf
    lb[3, :] = -np.inf
    la[4, :] = 80.0
    lb[4, :] = -80.0
    return oa, la, ob, lb


@pytest.mark.parametrize("rows,heads,dim", [(1000, 8, 128), (37, 128, 128), (64, 3, 64), (5, 2, 256)])
def test_merge_matches_oracle(rows, heads, dim):
    mla = _mla()
    oa, la, ob, lb = _merge_inputs(rows, heads, rows, dim)
    g_o, g_l = Guarded((rows, heads, dim), torch.bfloat16), Guarded((rows, heads), torch.float32)
    o, l = mla.mla_merge_state(to_dev_bf16(oa), to_dev(la), to_dev_bf16(ob), to_dev(lb), g_o.tensor, g_l.tensor)
    torch.cuda.synchronize()
    g_o.check("merge O")
    g_l.check("merge LSE")
    o_ref, l_ref = merge_state(oa, la.astype(np.float64), ob, lb.astype(np.float64))
    og = f64_of_bf16(o)
    assert np.abs(og - o_ref).max() <= 2.0 ** -8 * np.abs(o_ref).max() + 1e-6
    lg = l.double().cpu().numpy()
    assert np.array_equal(np.isneginf(lg), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(lg[fin] - l_ref[fin]).max() <= 1e-5 * max(1.0, np.abs(l_ref[fin]).max())
    # one side empty: the other side is copied bit for bit
    only_b = np.isneginf(la) & np.isfinite(lb)
    np.testing.assert_array_equal(bits_of(o)[only_b], ob[only_b])


def test_merge_in_place():
    mla = _mla()
    oa, la, ob, lb = _merge_inputs(500, 16, 11)
    ta, tla = to_dev_bf16(oa), to_dev(la)
    o_sep, l_sep = mla.mla_merge_state(ta.clone(), tla.clone(), to_dev_bf16(ob), to_dev(lb))
    mla.mla_merge_state(ta, tla, to_dev_bf16(ob), to_dev(lb), ta, tla)
    torch.cuda.synchronize()
    assert torch.equal(ta.view(torch.int16), o_sep.view(torch.int16))
    assert torch.equal(tla, l_sep)


# ------------------------------------------------------------------ paged up-projection
def test_up_proj_paged_bit_identical_to_gather_then_up_proj_workload2():
    """Both chunks of the chunked-prefix workload (16384 rows x 128 heads each): the fused
    kernel equals the gather followed by the up-projection, bit for bit."""
    mla = _mla()
    cb = wl.make_chunked_prefix()
    cache, table, w = to_dev_bf16(cb.cache), to_dev(cb.block_table), to_dev_bf16(cb.w_kvb)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    H = cb.new.num_heads
    for c in range(cb.layout.num_chunks):
        cu, st = to_dev(cb.layout.cu_seq_lens[c]), to_dev(cb.layout.chunk_starts[c])
        t = int(cb.layout.cu_seq_lens[c][-1])
        lat = mla.mla_gather_latent(cache, table, cu, st, t, status=status)
        k_ref, v_ref = mla.mla_up_proj(lat, w, H, status=status)
        g_k, g_v = Guarded((t, H, 192), torch.bfloat16), Guarded((t, H, 128), torch.bfloat16)
        k, v = mla.mla_up_proj_paged(cache, table, cu, st, t, w, H, g_k.tensor, g_v.tensor, status=status)
        torch.cuda.synchronize()
        g_k.check("paged K")
        g_v.check("paged V")
        assert int(status.item()) == 0
        assert torch.equal(k.view(torch.int16), k_ref.view(torch.int16)), f"chunk {c}: K differs"
        assert torch.equal(v.view(torch.int16), v_ref.view(torch.int16)), f"chunk {c}: V differs"
        del lat, k_ref, v_ref, k, v, g_k, g_v


@pytest.mark.parametrize("n_req,block_size,chunk,heads", [(3, 64, 300, 4), (3, 16, 100, 2), (40, 1, 37, 2),
                                                         (5, 64, 4096, 3)])
def test_up_proj_paged_matches_oracle(n_req, block_size, chunk, heads):
    """Random tables and ragged chunk layouts (rows of a token block from several requests,
    chunk starts not aligned to blocks, more than 31 requests), against the oracle's
    gather followed by its up-projection, element-wise."""
    mla = _mla()
    rng = np.random.default_rng(n_req * 1000 + block_size)
    prefix = rng.integers(0, 700, size=n_req)
    prefix[0] = 0
    nb = int(sum(-(-int(p) // block_size) for p in prefix)) + 5
    cb = wl.random_chunked_prefix(int(rng.integers(1 << 30)), [1] * n_req, prefix, heads, num_blocks=nb,
                                  block_size=block_size, chunk_tokens=chunk)
    cache, table, w = to_dev_bf16(cb.cache), to_dev(cb.block_table), to_dev_bf16(cb.w_kvb)
    for c in range(cb.layout.num_chunks):
        cu, st = cb.layout.cu_seq_lens[c], cb.layout.chunk_starts[c]
        t = int(cu[-1])
        if t == 0:
            continue
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        k, v = mla.mla_up_proj_paged(cache, table, to_dev(cu), to_dev(st), t, w, heads, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        lat = gather_latent(cb.cache, cb.block_table, cu, st)
        _check_up_proj(lat, cb.w_kvb, heads, k, v)


def test_up_proj_paged_bad_block_gives_zero_rows_and_flag():
    mla = _mla()
    cb = wl.random_chunked_prefix(6, [1, 1], [150, 130], 2, num_blocks=8, block_size=64, chunk_tokens=256)
    table = cb.block_table.copy()
    table[1, 1] = 99                     # outside the cache: request 1, positions 64..127
    cu, st = cb.layout.cu_seq_lens[0], cb.layout.chunk_starts[0]
    t = int(cu[-1])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    k, v = mla.mla_up_proj_paged(to_dev_bf16(cb.cache), to_dev(table), to_dev(cu), to_dev(st), t,
                                 to_dev_bf16(cb.w_kvb), 2, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2
    bad = np.arange(cu[1] + 64, cu[1] + 128)
    kb, vb = bits_of(k), bits_of(v)
    assert not kb[bad].any() and not vb[bad].any()
    good = np.setdiff1d(np.arange(t), bad)
    lat = gather_latent(cb.cache, cb.block_table, cu, st)
    k_ref, v_ref = up_project(lat, cb.w_kvb, 2)
    np.testing.assert_array_equal(f64_of_bf16(k)[good][:, :, 128:], k_ref[good][:, :, 128:])
    assert np.abs(f64_of_bf16(v)[good] - v_ref[good]).max() < 0.05


# ------------------------------------------------------------------ fp8 latent cache
def _fp8_gather(mla, cache, table, cu, st, status=None):
    t = int(cu[-1])
    g = Guarded((t, 576), torch.bfloat16)
    out = mla.mla_gather_latent_fp8(to_dev(cache), to_dev(table), to_dev(cu), to_dev(st), t, out=g.tensor,
                                    status=status)
    torch.cuda.synchronize()
    g.check("fp8 gather")
    return bits_of(out)


@pytest.mark.parametrize("n_req,block_size,chunk", [(4, 64, 4096), (3, 16, 100), (40, 1, 37), (5, 64, 333)])
def test_gather_fp8_bit_exact(n_req, block_size, chunk):
    from oracle import gather_latent_fp8
    mla = _mla()
    rng = np.random.default_rng(n_req * 7 + block_size)
    prefix = rng.integers(1, 900, size=n_req)
    nb = int(sum(-(-int(p) // block_size) for p in prefix)) + 3
    cache = wl.random_fp8_cache(rng, nb, block_size)
    perm = rng.permutation(nb).astype(np.int32)
    per = [-(-int(p) // block_size) for p in prefix]
    table = np.full((n_req, max(per)), -1, dtype=np.int32)
    pos = 0
    for r, k in enumerate(per):
        table[r, :k] = perm[pos:pos + k]
        pos += k
    lay = wl.chunk_layout(prefix, chunk)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for c in range(lay.num_chunks):
        cu, st = lay.cu_seq_lens[c], lay.chunk_starts[c]
        if cu[-1] == 0:
            continue
        got = _fp8_gather(mla, cache, table, cu, st, status)
        np.testing.assert_array_equal(got, gather_latent_fp8(cache, table, cu, st))
    assert int(status.item()) == 0


def test_gather_fp8_extreme_scales_and_nan_codes():
    """Scales at the ends of the range (bf16 subnormal results, overflow to infinity), NaN
    fp8 codes and NaN scales: every finite result bit-exact, NaN exactly where the oracle
    has NaN."""
    from oracle import gather_latent_fp8
    mla = _mla()
    rng = np.random.default_rng(77)
    cache = wl.random_fp8_cache(rng, 8, 16, scale_exp=(0, 6))
    cache[4:] = wl.random_fp8_cache(rng, 4, 16, scale_exp=(245, 254))
    flat = cache.reshape(-1, 648)
    flat[::7, 5] = 0x7F            # NaN codes
    flat[::11, 300] = 0xFF
    flat[3, 641] = 0xFF            # a NaN scale
    table = np.arange(8, dtype=np.int32).reshape(2, 4)
    cu = np.array([0, 64, 128], dtype=np.int32)
    st = np.array([0, 0], dtype=np.int32)
    got = _fp8_gather(mla, cache, table, cu, st)
    ref = gather_latent_fp8(cache, table, cu, st)
    g_nan = (got & 0x7FFF) > 0x7F80
    r_nan = (ref & 0x7FFF) > 0x7F80
    np.testing.assert_array_equal(g_nan, r_nan)
    np.testing.assert_array_equal(got[~r_nan], ref[~r_nan])
    assert r_nan.any() and (ref == 0x7F80).any() and ((ref & 0x7F80) == 0).any()   # NaN, inf, subnormal/zero seen


def test_gather_fp8_bad_block_flags_and_zeroes():
    from oracle import gather_latent_fp8
    mla = _mla()
    rng = np.random.default_rng(78)
    cache = wl.random_fp8_cache(rng, 4, 64)
    table = np.array([[0, 1], [2, 99]], dtype=np.int32)
    cu = np.array([0, 70, 140], dtype=np.int32)
    st = np.array([0, 0], dtype=np.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _fp8_gather(mla, cache, table, cu, st, status)
    assert int(status.item()) & 2
    bad = np.arange(70 + 64, 140)
    assert not got[bad].any()
    good_table = np.array([[0, 1], [2, 3]], dtype=np.int32)
    keep = np.setdiff1d(np.arange(140), bad)
    np.testing.assert_array_equal(got[keep], gather_latent_fp8(cache, good_table, cu, st)[keep])


def test_up_proj_paged_split_matches_paged():
    """The split form writes K_nope, V and one rope row per token: bit-identical to the
    corresponding parts of the paged up-projection's K [T, H, 192] and V."""
    mla = _mla()
    cb = wl.random_chunked_prefix(93, [1, 1, 1], [700, 129, 1000], 3, num_blocks=40, block_size=64,
                                  chunk_tokens=512)
    cache, table, w = to_dev_bf16(cb.cache), to_dev(cb.block_table), to_dev_bf16(cb.w_kvb)
    for c in range(cb.layout.num_chunks):
        cu, st = to_dev(cb.layout.cu_seq_lens[c]), to_dev(cb.layout.chunk_starts[c])
        t = int(cb.layout.cu_seq_lens[c][-1])
        k, v = mla.mla_up_proj_paged(cache, table, cu, st, t, w, 3)
        g_k, g_v, g_r = (Guarded((t, 3, 128), torch.bfloat16), Guarded((t, 3, 128), torch.bfloat16),
                         Guarded((t, 64), torch.bfloat16))
        kn, v2, rope = mla.mla_up_proj_paged_split(cache, table, cu, st, t, w, 3, g_k.tensor, g_v.tensor, g_r.tensor)
        torch.cuda.synchronize()
        for g, what in ((g_k, "K_nope"), (g_v, "V"), (g_r, "rope")):
            g.check(what)
        assert torch.equal(kn.view(torch.int16), k[:, :, :128].contiguous().view(torch.int16))
        assert torch.equal(v2.view(torch.int16), v.view(torch.int16))
        assert torch.equal(rope.view(torch.int16), k[:, 0, 128:].contiguous().view(torch.int16))
        lat = gather_latent(cb.cache, cb.block_table, cb.layout.cu_seq_lens[c], cb.layout.chunk_starts[c])
        np.testing.assert_array_equal(bits_of(rope), lat[:, 512:])
