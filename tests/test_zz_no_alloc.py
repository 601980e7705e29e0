"""The allocation-free prefill entry point (GPU).

mla_prefill_run_noalloc is for callers that cannot allocate device memory (a serving
engine whose memory pool already owns the GPU, a host that forbids allocation after
start-up).  It keeps its work list in a fixed array inside the library instead of a
plan-owned workspace.  These tests call it through the C ABI and compare it with the
allocating entry points (mla_prefill_plan + mla_prefill_run) on two calls in a row, so
the second call also shows that the shared array is correctly rewritten.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from gpu_util import check_attention, f64_of_bf16, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

P32 = ctypes.POINTER(ctypes.c_int32)


def _noalloc(lib, b, q, k, v, o, lse, status):
    qo = np.ascontiguousarray(b.qo_indptr, dtype=np.int32)
    kv = np.ascontiguousarray(b.kv_indptr, dtype=np.int32)
    return lib.mla_prefill_run_noalloc(
        qo.ctypes.data_as(P32), kv.ctypes.data_as(P32), b.batch, b.num_heads, 192, 128, int(b.causal),
        b.sm_scale, b.window_left, b.logits_soft_cap, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
        ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_planned_run_on_two_calls():
    import chunked_prefill_attention_ragged_gb300 as mla
    lib = mla.library()
    batches = [
        wl.random_ragged(71, [700, 129, 1, 300], None, 8),                        # first call
        wl.random_ragged(72, [40, 1000], [300, 1000], 4, logits_soft_cap=30.0),  # second call, other shapes
    ]
    for b in batches:
        q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
        plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                    window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)
        o_ref, lse_ref = plan.run(q, k, v)
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, b, q, k, v, o, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), f64_of_bf16(o_ref),
                        lse_ref.double().cpu().numpy(), "noalloc vs planned run")


def test_noalloc_rejects_work_beyond_its_array():
    import chunked_prefill_attention_ragged_gb300 as mla
    lib = mla.library()
    qo = np.array([0, 256], dtype=np.int32)          # 2 query tiles x 40000 heads = 80000 units > 65536
    rc = lib.mla_prefill_run_noalloc(qo.ctypes.data_as(P32), qo.ctypes.data_as(P32), 1, 40000, 192, 128, 1, 0.1,
                                     -1, 0.0, None, None, None, None, None, None, None)
    assert rc == -3
