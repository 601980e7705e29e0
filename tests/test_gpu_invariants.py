"""Exact invariants of the ragged prefill kernel, GPU against GPU.

* Ragged isolation: a request's rows come out bit for bit the same whether it runs alone
  or inside a batch.  Its units (128-row query tiles from its first row, key tiles from its
  first key) are the same either way; rows and keys of a neighbouring request that share a
  tile are computed but masked or never stored, so they add exact zeros.
* A window at least as long as every request's key range is no window: every row's
  allowed keys, and so every unit and product, are the same.
"""
import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from gpu_util import to_dev_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def run(q_bits, k_bits, v_bits, qo, kv, heads, causal, sm_scale, window_left=-1, cap=0.0):
    import chunked_prefill_attention_ragged_gb300 as mla
    plan = mla.mla_prefill_plan(qo, kv, heads, causal=causal, sm_scale=sm_scale, window_left=window_left,
                                logits_soft_cap=cap)
    o, lse = plan.run(to_dev_bf16(q_bits), to_dev_bf16(k_bits), to_dev_bf16(v_bits))
    torch.cuda.synchronize()
    assert plan.status() == 0
    return o.view(torch.int16).cpu().numpy(), lse.cpu().numpy()


ISOLATION = [
    # name, q_lens, kv_lens, heads, causal, window, cap
    ("causal_ragged", [300, 1, 129, 77, 256], None, 4, True, -1, 0.0),
    ("prefix_longer_kv", [130, 7, 200], [700, 300, 200], 2, True, -1, 0.0),
    ("noncausal", [33, 300, 1], [1000, 129, 5], 2, False, -1, 0.0),
    ("window_and_cap", [400, 90, 260], None, 2, True, 150, 30.0),
]


@pytest.mark.parametrize("name,q_lens,kv_lens,heads,causal,window,cap", ISOLATION, ids=[c[0] for c in ISOLATION])
def test_request_alone_equals_request_in_batch(name, q_lens, kv_lens, heads, causal, window, cap):
    b = wl.random_ragged(700 + [c[0] for c in ISOLATION].index(name), q_lens, kv_lens, heads, causal=causal,
                         window_left=window, logits_soft_cap=cap)
    o_all, l_all = run(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, heads, causal, b.sm_scale, window, cap)
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        k0, k1 = int(b.kv_indptr[r]), int(b.kv_indptr[r + 1])
        if q1 == q0:
            continue
        qo = np.array([0, q1 - q0], dtype=np.int32)
        kv = np.array([0, k1 - k0], dtype=np.int32)
        o_r, l_r = run(b.q[q0:q1], b.k[k0:k1], b.v[k0:k1], qo, kv, heads, causal, b.sm_scale, window, cap)
        np.testing.assert_array_equal(o_r, o_all[q0:q1], err_msg=f"{name}: request {r} O")
        np.testing.assert_array_equal(l_r.view(np.uint32), l_all[q0:q1].view(np.uint32),
                                      err_msg=f"{name}: request {r} LSE")


@pytest.mark.parametrize("causal", [True, False])
def test_window_covering_every_key_equals_no_window(causal):
    b = wl.random_ragged(720, [300, 129, 1], [700, 129, 40], 2, causal=causal)
    o_ref, l_ref = run(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, 2, causal, b.sm_scale, -1)
    longest = int(np.max(np.diff(b.kv_indptr)))
    for window in (longest - 1, longest, 10 * longest):
        o_w, l_w = run(b.q, b.k, b.v, b.qo_indptr, b.kv_indptr, 2, causal, b.sm_scale, window)
        np.testing.assert_array_equal(o_w, o_ref, err_msg=f"window {window} O")
        np.testing.assert_array_equal(l_w.view(np.uint32), l_ref.view(np.uint32), err_msg=f"window {window} LSE")
