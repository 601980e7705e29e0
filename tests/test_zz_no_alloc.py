"""The allocation-free prefill entry point (GPU).

mla_prefill_run_noalloc is for callers that cannot allocate device memory (a serving
engine whose memory pool already owns the GPU, a host that forbids allocation after
start-up).  It keeps its work list in a fixed array inside the library instead of a
plan-owned workspace.  These tests call it through the C ABI and compare it with the
allocating entry points (mla_prefill_plan + mla_prefill_run), which run the same kernel
on the same plan, so the outputs must be bit-identical, on several calls in a row (later
calls also show that the shared array is rewritten correctly); the first call is also
compared with the fp64 oracle.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import ragged_attention
from gpu_util import check_attention, f64_of_bf16, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

P32 = ctypes.POINTER(ctypes.c_int32)


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, b, q, k, v, o, lse, status):
    qo = np.ascontiguousarray(b.qo_indptr, dtype=np.int32)
    kv = np.ascontiguousarray(b.kv_indptr, dtype=np.int32)
    return lib.mla_prefill_run_noalloc(
        qo.ctypes.data_as(P32), kv.ctypes.data_as(P32), b.batch, b.num_heads, 192, 128, int(b.causal),
        b.sm_scale, b.window_left, b.logits_soft_cap, _vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), _vp(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_planned_run_on_three_calls():
    import chunked_prefill_attention_ragged_gb300 as mla
    lib = mla.library()
    cases = [
        # (batch, caller status word, LSE wanted)
        (wl.random_ragged(71, [700, 129, 1, 300], None, 8), True, True),                        # first call
        (wl.random_ragged(72, [40, 1000], [300, 1000], 4, logits_soft_cap=30.0), True, True),  # other shapes
        (wl.random_ragged(73, [260, 3], None, 2, causal=False), False, False),                  # no status, no LSE
    ]
    for i, (b, with_status, with_lse) in enumerate(cases):
        q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
        plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                    window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)
        o_ref, lse_ref = plan.run(q, k, v)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan")) if with_lse else None
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
        assert _noalloc(lib, b, q, k, v, o, lse, status) == 0
        torch.cuda.synchronize()
        assert plan.status() == 0
        if status is not None:
            assert int(status.item()) == 0
        # Same kernel, same work list: bit for bit.
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)), f"call {i}: O differs"
        if lse is not None:
            assert torch.equal(lse, lse_ref), f"call {i}: LSE differs"
        if i == 0:
            o_or, lse_or = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=b.causal,
                                            sm_scale=b.sm_scale)
            check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_or, lse_or, "noalloc vs oracle")


def test_noalloc_binding_matches_planned_run():
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(74, [300, 17], None, 4)
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, 4, causal=True, sm_scale=b.sm_scale)
    o_ref, lse_ref = plan.run(q, k, v)
    o = torch.empty_like(o_ref)
    lse = torch.empty_like(lse_ref)
    mla._binding.mla_prefill_run_noalloc(b.qo_indptr, b.kv_indptr, 4, q, k, v, o, lse, sm_scale=b.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16)) and torch.equal(lse, lse_ref)


def test_noalloc_rejects_work_beyond_its_array():
    import chunked_prefill_attention_ragged_gb300 as mla
    lib = mla.library()
    qo = np.array([0, 256], dtype=np.int32)          # 2 query tiles x 40000 heads = 80000 units > 65536
    rc = lib.mla_prefill_run_noalloc(qo.ctypes.data_as(P32), qo.ctypes.data_as(P32), 1, 40000, 192, 128, 1, 0.1,
                                     -1, 0.0, None, None, None, None, None, None, None)
    assert rc == -3
