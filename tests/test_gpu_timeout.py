"""The time-out path of the prefill kernel's bounded pipeline waits (GPU).

Every mbarrier wait of the kernel gives up after a time limit instead of spinning for
ever: the CTA raises an abort flag that the other roles see, records
MLA_DEVSTAT_TIMEOUT in the plan's status word, waits (within a bound) for its own
in-flight copies and tensor-core products, frees its tensor memory and returns.  The
test mode MLA_TEST_FORCE_TIMEOUT_NS (read at plan time) makes the S issuer wait on a
barrier that nothing arrives on, with a short limit, so this path runs on purpose: no
fault, trap or endless loop is involved, and the context must stay usable.
"""
import os

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import ragged_attention
from gpu_util import check_attention, f64_of_bf16, to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ENV = "MLA_TEST_FORCE_TIMEOUT_NS"


def _plan(b, force_ns=None):
    import chunked_prefill_attention_ragged_gb300 as mla
    old = os.environ.pop(ENV, None)
    try:
        if force_ns is not None:
            os.environ[ENV] = str(force_ns)
        return mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale)
    finally:
        os.environ.pop(ENV, None)
        if old is not None:
            os.environ[ENV] = old


@pytest.mark.parametrize("merge", [False, True])
def test_forced_timeout_reports_status_and_context_survives(merge):
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.random_ragged(81, [700, 130, 45], None, 4)
    q, k, v = to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v)
    rows = b.q.shape[0]
    o = torch.zeros(rows, 4, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(rows, 4, dtype=torch.float32, device="cuda")
    bad = _plan(b, force_ns=20_000_000)               # 20 ms
    if merge:
        bad.run_merge(q, k, v, o, lse)
    else:
        bad.run(q, k, v, o, lse)
    torch.cuda.synchronize()                          # the kernel returned by itself
    with pytest.raises(mla.MlaError) as err:
        bad.status()
    assert err.value.code == -5
    assert bad.status() == 0                          # read-and-clear
    # Same process, same context: a normal plan runs and matches the oracle.
    good = _plan(b)
    o2, lse2 = good.run(q, k, v)
    torch.cuda.synchronize()
    assert good.status() == 0
    o_ref, lse_ref = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=True, sm_scale=b.sm_scale)
    check_attention(f64_of_bf16(o2), lse2.double().cpu().numpy(), o_ref, lse_ref, "after a forced time-out")


def test_out_of_range_limit_leaves_test_mode_off():
    b = wl.random_ragged(82, [130], None, 2)
    plan = _plan(b, force_ns=10 ** 12)                # above the 2 s ceiling: ignored
    o, lse = plan.run(to_dev_bf16(b.q), to_dev_bf16(b.k), to_dev_bf16(b.v))
    torch.cuda.synchronize()
    assert plan.status() == 0
    o_ref, lse_ref = ragged_attention(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, causal=True, sm_scale=b.sm_scale)
    check_attention(f64_of_bf16(o), lse.double().cpu().numpy(), o_ref, lse_ref, "limit out of range")
    assert np.isfinite(lse.cpu().numpy()).all()
