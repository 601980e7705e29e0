"""GPU parity of the gather, up-projection and merge kernels against the oracle."""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import bf16_bits_to_f64, cache_write, gather_latent, merge_state, round_f64_to_bf16, up_project
from gpu_util import bits_of, f64_of_bf16, to_dev, to_dev_bf16

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
        out = mla.mla_gather_latent(cache, table, to_dev(cu), to_dev(st), int(cu[-1]), status=status)
        torch.cuda.synchronize()
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
        out = mla.mla_gather_latent(cache, table, to_dev(cu), to_dev(st), int(cu[-1]))
        torch.cuda.synchronize()
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
    out = mla.mla_gather_latent(to_dev_bf16(cache), to_dev(table), to_dev(cu), to_dev(st), int(cu[-1]))
    torch.cuda.synchronize()
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
    d_cache = to_dev_bf16(cache)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_write(d_cache, to_dev_bf16(lat), to_dev(slots), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(bits_of(d_cache), cache_write(cache, lat, slots))


def test_cache_write_bad_slot_is_flagged_and_skipped():
    mla = _mla()
    rng = np.random.default_rng(9)
    cache = rng.integers(0, 1 << 16, size=(4, 16, 576), dtype=np.uint16)
    lat = rng.integers(0, 1 << 16, size=(6, 576), dtype=np.uint16)
    slots = np.array([3, 64, 10, 1000, -5, 63], dtype=np.int64)   # 64 and 1000 are past the cache
    d_cache = to_dev_bf16(cache)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_cache_write(d_cache, to_dev_bf16(lat), to_dev(slots), status=status)
    torch.cuda.synchronize()
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
@pytest.mark.parametrize("tokens,heads,out_offset", [(300, 4, 0), (128, 1, 0), (1, 2, 0), (1000, 16, 0),
                                                     (300, 4, 8), (77, 3, 8)])
def test_up_proj_matches_rounded_oracle(tokens, heads, out_offset):
    """out_offset = 8 elements puts K and V 16 but not 32 bytes into their buffers (16-byte stores)."""
    mla = _mla()
    rng = np.random.default_rng(tokens + heads)
    lat = wl.to_bf16_bits(rng.standard_normal((tokens, 576)).astype(np.float32))
    w = wl.to_bf16_bits((rng.standard_normal((512, heads * 256)) * 512 ** -0.5).astype(np.float32))
    k_buf = torch.full((out_offset + tokens * heads * 192,), float("nan"), dtype=torch.bfloat16, device="cuda")
    v_buf = torch.full((out_offset + tokens * heads * 128,), float("nan"), dtype=torch.bfloat16, device="cuda")
    k_out = k_buf[out_offset:].view(tokens, heads, 192)
    v_out = v_buf[out_offset:].view(tokens, heads, 128)
    k, v = mla.mla_up_proj(to_dev_bf16(lat), to_dev_bf16(w), heads, k_out=k_out, v_out=v_out)
    torch.cuda.synchronize()
    assert bool(torch.isnan(k_buf[:out_offset]).all()) and bool(torch.isnan(v_buf[:out_offset]).all())
    k_ref, v_ref = up_project(lat, w, heads)
    # Worst-case fp32 accumulation error of a 512-term dot product, per output element.
    a = np.abs(bf16_bits_to_f64(lat[:, :512]))
    wa = np.abs(bf16_bits_to_f64(w)).reshape(512, heads, 256)
    mag = np.einsum("tc,chd->thd", a, wa)
    acc_bound = 512 * 2.0 ** -23 * mag
    kg, vg = f64_of_bf16(k), f64_of_bf16(v)
    # rope part is a copy: bit-exact
    np.testing.assert_array_equal(kg[:, :, 128:], k_ref[:, :, 128:])
    for got, ref, bound, what in ((kg[:, :, :128], k_ref[:, :, :128], acc_bound[..., :128], "K_nope"),
                                  (vg, v_ref, acc_bound[..., 128:], "V")):
        rref = round_f64_to_bf16(ref)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
        # one bf16 rounding of a value that fp32 accumulation may have moved by `bound`
        err = np.abs(got - ref)
        worst = np.max(err / (ulp + bound))
        assert worst <= 1.0, f"{what}: error {worst:.3f} x (ulp + accumulation bound)"
        assert np.mean(got != rref) < 0.02, f"{what}: {np.mean(got != rref):.4f} differ from exact rounding"


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
    o, l = mla.mla_merge_state(to_dev_bf16(oa), to_dev(la), to_dev_bf16(ob), to_dev(lb))
    torch.cuda.synchronize()
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
