"""Merge of two partial attention states by their LSE (test infrastructure only).

Why it exists: vLLM ``vllm.v1.attention.backends.mla.prefill.flashinfer``,
``run_prefill_context_chunk`` always asks for ``return_lse=True``: each
prefix chunk gives a partial (O, LSE) that has to be combined with the others
and with the new-token attention.  The combination is the exact identity
for softmax over the union of two disjoint key sets A and B:

    LSE = ln(exp(LSE_a) + exp(LSE_b))
    O   = (exp(LSE_a) O_a + exp(LSE_b) O_b) / exp(LSE)

evaluated with the larger LSE factored out.  A side whose LSE is -inf (no
key) contributes nothing; both -inf gives O = 0, LSE = -inf.
"""
import numpy as np

from .bf16 import bf16_bits_to_f64


def merge_state(o_a, lse_a, o_b, lse_b):
    """o_*: [rows, H, Dv] (bf16 bits or floats); lse_*: [rows, H].

    Returns (o [rows, H, Dv], lse [rows, H]) in float64.
    """
    oa = bf16_bits_to_f64(o_a) if o_a.dtype == np.uint16 else np.asarray(o_a, np.float64)
    ob = bf16_bits_to_f64(o_b) if o_b.dtype == np.uint16 else np.asarray(o_b, np.float64)
    la = np.asarray(lse_a, np.float64)
    lb = np.asarray(lse_b, np.float64)
    m = np.maximum(la, lb)
    live = np.isfinite(m)
    ms = np.where(live, m, 0.0)
    wa = np.where(live, np.exp(la - ms), 0.0)
    wb = np.where(live, np.exp(lb - ms), 0.0)
    tot = np.where(live, wa + wb, 1.0)
    o = (wa[..., None] * oa + wb[..., None] * ob) / tot[..., None]
    lse = np.where(live, ms + np.log(tot), -np.inf)
    return o, lse
