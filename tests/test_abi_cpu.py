"""C-ABI checks that need no GPU: exports, error codes, host validation, planner coverage."""
import ctypes
import os
import re

import numpy as np
import pytest

import chunked_prefill_attention_ragged_gb300 as mla
from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import allowed_mask

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "mla_prefill.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]*?\b(mla_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = mla.library()
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mla.EXPORTED)
    assert lib.mla_abi_version() == 1


def test_error_strings():
    for code in (0, -1, -2, -3, -4, -5, -6, 99):
        assert isinstance(mla.error_string(code), str) and mla.error_string(code)


def _plan_rc(qo, kv, heads=4, dqk=192, dv=128, causal=1, scale=0.1, window=-1, cap=0.0, batch=None):
    lib = mla.library()
    qo = np.asarray(qo, np.int32)
    kv = np.asarray(kv, np.int32)
    h = ctypes.c_void_p()
    b = len(qo) - 1 if batch is None else batch
    p32 = ctypes.POINTER(ctypes.c_int32)
    return lib.mla_prefill_plan(ctypes.byref(h), qo.ctypes.data_as(p32), kv.ctypes.data_as(p32), b, heads, dqk, dv,
                                causal, scale, window, cap, None)


def test_plan_rejects_bad_arguments_without_touching_the_device():
    assert _plan_rc([0, 5], [0, 5], dqk=128) == -3
    assert _plan_rc([0, 5], [0, 5], dv=64) == -3
    assert _plan_rc([0, 5, 3], [0, 5, 9]) == -2          # qo not monotone
    assert _plan_rc([1, 5], [0, 5]) == -2                 # qo[0] != 0
    assert _plan_rc([0, 5], [0, 5], heads=0) == -1
    assert _plan_rc([0, 5], [0, 5], window=-2) == -1
    assert _plan_rc([0, 5], [0, 5], scale=float("nan")) == -1
    assert _plan_rc([0, 5], [0, 5], scale=0.0) == -1
    assert _plan_rc([0, 5], [0, 5], scale=-0.5) == -1
    assert _plan_rc([0, 5], [0, 5], cap=float("inf")) == -1
    assert _plan_rc([0, 5], [0, 5], batch=-1) == -1


def test_entry_points_reject_null_and_misaligned():
    lib = mla.library()
    assert lib.mla_prefill_run(None, None, None, None, None, None, None) == -1
    assert lib.mla_prefill_run_merge(None, None, None, None, None, None, None) == -1
    assert lib.mla_prefill_status(None) == -1
    assert lib.mla_plan_destroy(None) == 0
    assert lib.mla_merge_state(None, None, None, None, None, None, 4, 2, 128, None) == -1
    assert lib.mla_merge_state(None, None, None, None, None, None, 4, 2, 96, None) == -3
    assert lib.mla_merge_state(None, None, None, None, None, None, 0, 2, 128, None) == 0
    assert lib.mla_gather_latent(None, 4, 64, 576, None, 1, None, None, 1, 0, None, None, None) == 0
    assert lib.mla_gather_latent(None, 4, 64, 576, None, 1, None, None, 1, 8, None, None, None) == -1
    assert lib.mla_gather_latent(None, 4, 64, 572, None, 1, None, None, 1, 8, None, None, None) == -1
    assert lib.mla_up_proj(None, None, 0, 4, None, None, None, None) == 0
    assert lib.mla_up_proj(None, None, 8, 4, None, None, None, None) == -1
    assert lib.mla_up_proj(16, 16, 8, 4, 16, 24, None, None) == -1   # misaligned v_out
    # cache write: shapes first, then pointers; nothing reaches the device
    assert lib.mla_cache_write(None, 4, 64, 576, None, None, 0, None, None) == 0
    assert lib.mla_cache_write(None, 4, 64, 572, None, None, 8, None, None) == -1
    assert lib.mla_cache_write(None, 4, 0, 576, None, None, 8, None, None) == -1
    assert lib.mla_cache_write(None, 4, 64, 110000, None, None, 8, None, None) == -3
    assert lib.mla_cache_write(None, 4, 64, 576, None, None, 8, None, None) == -1
    assert lib.mla_cache_write(16, 4, 64, 576, 32, 12, 8, None, None) == -1   # misaligned slot_mapping


def _coverage(units, qo, kv, heads, causal, window, rows=128):
    """For every (head, request, row, key): how many units cover it, and unit validity
    (units of `rows` query rows)."""
    B = len(qo) - 1
    cover = {}
    for u in units:
        h, q_row0, q_rows, q_pos0, kv_row0, kv_len, diag, tiles = (int(x) for x in u)
        lo, hi = tiles & 0xFFFF, tiles >> 16
        r = int(np.searchsorted(qo, q_row0, side="right") - 1)
        assert qo[r] + q_pos0 == q_row0 and kv_row0 == kv[r] and kv_len == kv[r + 1] - kv[r]
        lq = qo[r + 1] - qo[r]
        assert diag == kv_len - lq and 1 <= q_rows <= rows and q_pos0 + q_rows <= lq and q_pos0 % rows == 0
        m = allowed_mask(lq, kv_len, causal, window, np.arange(q_pos0, q_pos0 + q_rows))
        for t in range(lo, hi):   # no kv tile in the range is fully masked
            assert m[:, t * 128:(t + 1) * 128].any()
        key = (h, r, q_pos0)
        assert key not in cover
        cover[key] = (lo, hi, m)
    for h in range(heads):
        for r in range(B):
            lq = qo[r + 1] - qo[r]
            lkv = kv[r + 1] - kv[r]
            full = allowed_mask(lq, lkv, causal, window)
            for p0 in range(0, lq, rows):
                lo, hi, m = cover.pop((h, r, p0))
                # every allowed key of these rows lies inside the unit's tile range
                allowed_cols = np.nonzero(full[p0:p0 + rows].any(axis=0))[0]
                if allowed_cols.size:
                    assert allowed_cols.min() >= lo * 128 and allowed_cols.max() < hi * 128
                else:
                    assert lo == hi
    assert not cover


PLAN_CASES = [
    ([17, 40], None, 4, True, -1),
    ([1, 128, 129, 255, 256, 300], None, 2, True, -1),
    ([300, 5], [700, 5], 2, True, -1),       # prefix before the queries
    ([300, 200], [100, 50], 1, True, -1),    # fewer keys than queries: empty leading rows
    ([300, 0, 77], [1000, 10, 0], 2, False, -1),
    ([520, 130], None, 2, True, 100),        # sliding window
    ([400], [900], 1, True, 0),
]


@pytest.mark.parametrize("qlens,kvlens,heads,causal,window", PLAN_CASES)
def test_planner_covers_every_allowed_pair_once(qlens, kvlens, heads, causal, window):
    qo = wl.indptr_from_lengths(qlens)
    kv = wl.indptr_from_lengths(kvlens if kvlens is not None else qlens)
    for ctas in (1, 3, 152):
        units, offs = mla.mla_plan_units_host(qo, kv, heads, causal, window, ctas)
        assert offs[0] == 0 and offs[-1] == len(units) and np.all(np.diff(offs) >= 0)
        _coverage(units, qo, kv, heads, causal, window)


@pytest.mark.parametrize("qlens,kvlens,heads,causal,window", PLAN_CASES)
def test_pair_planner_covers_every_allowed_pair_once(monkeypatch, qlens, kvlens, heads, causal, window):
    """With MLA_PLAN_CTA_PAIRS=1 units are 256 rows (one per CTA pair), same coverage rules."""
    monkeypatch.setenv("MLA_PLAN_CTA_PAIRS", "1")
    qo = wl.indptr_from_lengths(qlens)
    kv = wl.indptr_from_lengths(kvlens if kvlens is not None else qlens)
    for pairs in (1, 3, 76):
        units, offs = mla.mla_plan_units_host(qo, kv, heads, causal, window, pairs)
        assert offs[0] == 0 and offs[-1] == len(units) and np.all(np.diff(offs) >= 0)
        _coverage(units, qo, kv, heads, causal, window, rows=256)


def test_planner_balance_on_long_causal_request():
    qo = wl.indptr_from_lengths([32768])
    units, offs = mla.mla_plan_units_host(qo, qo, 128, True, -1, 152)
    tiles = (units[:, 7] >> 16) - (units[:, 7] & 0xFFFF)
    cost = 2 * tiles + 3                              # the planner's cost model (half key tiles)
    load = np.array([cost[offs[c]:offs[c + 1]].sum() for c in range(152)])
    assert load.sum() == cost.sum()
    assert load.max() <= load.mean() * 1.02 + cost.max()   # within one unit of perfect balance
    # total tiles: 128 heads x sum_{i=1..256} i
    assert tiles.sum() == 128 * 256 * 257 // 2


def test_planner_units_grouped_by_request_head_early():
    # The first wave of work (one unit per CTA) should come from few (request, head) groups.
    qlens = [4096, 2048, 1024, 512]
    qo = wl.indptr_from_lengths(qlens)
    units, offs = mla.mla_plan_units_host(qo, qo, 16, True, -1, 152)
    first = units[offs[:-1]]
    groups = {(int(u[0]), int(np.searchsorted(qo, u[1], side="right") - 1)) for u in first}
    assert len(groups) <= 8


def test_bindings_check_shapes_before_any_call():
    """The Python wrappers reject outputs of the wrong size before the library sees a
    pointer (the C side gets raw pointers and would write past a short buffer)."""
    import torch
    from chunked_prefill_attention_ragged_gb300 import _binding
    qo = np.array([0, 40, 60], dtype=np.int32)
    bf = torch.bfloat16
    q, k, v = torch.zeros(60, 4, 192, dtype=bf), torch.zeros(60, 4, 192, dtype=bf), torch.zeros(60, 4, 128, dtype=bf)
    with pytest.raises(ValueError):   # O one row short
        _binding.mla_prefill_run_noalloc(qo, qo, 4, q, k, v, torch.zeros(59, 4, 128, dtype=bf), sm_scale=0.1)
    with pytest.raises(ValueError):   # LSE of the wrong shape
        _binding.mla_prefill_run_noalloc(qo, qo, 4, q, k, v, torch.zeros(60, 4, 128, dtype=bf),
                                         torch.zeros(60, 3), sm_scale=0.1)
    with pytest.raises(ValueError):   # kv_indptr shorter than qo_indptr
        _binding.mla_prefill_run_noalloc(qo, qo[:2], 4, q, k, v, torch.zeros(60, 4, 128, dtype=bf), sm_scale=0.1)
    with pytest.raises(ValueError):   # V with the wrong head dim
        _binding.mla_prefill_run_noalloc(qo, qo, 4, q, k, torch.zeros(60, 4, 192, dtype=bf),
                                         torch.zeros(60, 4, 128, dtype=bf), sm_scale=0.1)
    oa = torch.zeros(10, 2, 128, dtype=bf)
    la = torch.zeros(10, 2)
    with pytest.raises(ValueError):   # merge: o_b smaller than o_a
        _binding.mla_merge_state(oa, la, torch.zeros(9, 2, 128, dtype=bf), la)
    with pytest.raises(ValueError):   # merge: lse_b of the wrong shape
        _binding.mla_merge_state(oa, la, oa, torch.zeros(10, 3))


def test_new_entry_points_reject_bad_arguments_on_the_host():
    """Argument checks of the paged, split, shared-rope and fp8 entry points: nothing is
    launched (no GPU is needed to see the codes)."""
    lib = mla.library()
    # paged up-projection: only 576-wide entries; empty chunk is a no-op; null pointers rejected
    assert lib.mla_up_proj_paged(None, 4, 64, 512, None, 1, None, None, 1, 8, None, 4, None, None, None, None) == -3
    assert lib.mla_up_proj_paged(None, 4, 64, 576, None, 1, None, None, 1, 0, None, 4, None, None, None, None) == 0
    assert lib.mla_up_proj_paged(None, 4, 64, 576, None, 1, None, None, 1, 8, None, 4, None, None, None, None) == -1
    assert lib.mla_up_proj_paged(None, 4, 64, 576, None, 1, None, None, 0, 8, None, 4, None, None, None, None) == -2
    # slots must fit a 32-bit TMA row coordinate
    assert lib.mla_up_proj_paged(None, 1 << 26, 64, 576, None, 1, None, None, 1, 8, None, 4, None, None, None,
                                 None) == -3
    # split form: the rope output is required
    assert lib.mla_up_proj_paged_split(None, 4, 64, 576, None, 1, None, None, 1, 8, None, 4, None, None, None, None,
                                       None) == -1
    # fp8 gather: only 648-byte entries; misaligned output rejected
    assert lib.mla_gather_latent_fp8(None, 4, 64, 656, None, 1, None, None, 1, 8, None, None, None) == -3
    assert lib.mla_gather_latent_fp8(None, 4, 64, 648, None, 1, None, None, 1, 0, None, None, None) == 0
    assert lib.mla_gather_latent_fp8(8, 4, 64, 648, 16, 1, 16, 16, 1, 8, 24, None, None) == -1
    # shared-rope run: a null plan is rejected
    assert lib.mla_prefill_run_shared_rope(None, None, None, None, 64, None, None, None, 0, None) == -1


def test_shared_rope_binding_checks_shapes():
    import torch
    from chunked_prefill_attention_ragged_gb300 import _binding

    class FakePlan:   # only the fields the wrapper reads before any library call
        num_heads, total_q, total_kv, handle = 2, 10, 20, None
    bf = torch.bfloat16
    q, kn, v = torch.zeros(10, 2, 192, dtype=bf), torch.zeros(20, 2, 128, dtype=bf), torch.zeros(20, 2, 128, dtype=bf)
    with pytest.raises(ValueError):   # rope of the wrong width
        _binding.mla_prefill_run_shared_rope(FakePlan(), q, kn, torch.zeros(20, 32, dtype=bf), v)
    with pytest.raises(ValueError):   # K_nope with the rope still attached
        _binding.mla_prefill_run_shared_rope(FakePlan(), q, torch.zeros(20, 2, 192, dtype=bf),
                                             torch.zeros(20, 64, dtype=bf), v)
    with pytest.raises(ValueError):   # merge without the partial state
        _binding.mla_prefill_run_shared_rope(FakePlan(), q, kn, torch.zeros(20, 64, dtype=bf), v, merge=True)


def test_absorbed_entry_points_check_arguments_on_the_host():
    """Bad arguments to the absorbed-weight plan and run are refused before anything
    touches the device (no GPU here)."""
    import ctypes
    lib = mla.library()
    qo = np.array([0, 4, 9], dtype=np.int32)
    kl = np.array([10, 9], dtype=np.int32)
    P32 = ctypes.POINTER(ctypes.c_int32)
    h = ctypes.c_void_p()

    def plan(qo_, kl_, batch, heads, bs, scale, cap=0.0):
        return lib.mla_absorbed_plan(ctypes.byref(h), qo_.ctypes.data_as(P32), kl_.ctypes.data_as(P32), batch,
                                     heads, bs, 1, scale, cap, None)

    assert plan(qo, kl, 2, 4, 0, 0.1) == -1                  # block size 0
    assert plan(qo, kl, 2, 0, 64, 0.1) == -1                 # no heads
    assert plan(qo, kl, 2, 4, 64, 0.0) == -1                 # sm_scale must be > 0
    assert plan(qo, kl, 2, 4, 64, float("nan")) == -1
    assert plan(np.array([1, 4, 9], dtype=np.int32), kl, 2, 4, 64, 0.1) == -2    # qo_indptr[0] != 0
    assert plan(np.array([0, 4, 3], dtype=np.int32), kl, 2, 4, 64, 0.1) == -2    # not monotone
    assert plan(qo, np.array([10, -1], dtype=np.int32), 2, 4, 64, 0.1) == -2     # negative kv length
    assert lib.mla_absorbed_run(None, None, None, 0, None, 0, None, None, None) == -1
    with pytest.raises(ValueError):
        mla.mla_absorbed_plan(qo, kl, 4, 64)                  # sm_scale is required
    with pytest.raises(ValueError):
        mla.mla_absorbed_plan(qo, kl[:1], 4, 64, sm_scale=0.1)   # kv_lens must be [batch]
