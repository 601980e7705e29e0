"""What chunked prefill with a cached prefix must equal (test infrastructure only).

vLLM ``vllm.v1.attention.backends.mla.prefill.flashinfer``,
``finalize_attention_metadata``: the new tokens attend causally to themselves
(``prefill_main``, ``kv_indptr = qo_indptr``) and non-causally to each chunk
of the decompressed prefix (``prefill_chunks[i]``, ``causal=False``), every
part returning its LSE so the parts can be merged.  sglang issue #3849: the
prefix is stored compressed (512 latent + 64 rope) and decompressed into
192/128-dim MHA keys and values.

The plain definition of the end result is one unchunked attention per
request over the keys [prefix ; new tokens], where every prefix key is
visible to every new query and new keys are causal -- i.e. bottom-right
causal attention with Lkv = P + Lq.  That is what this function computes;
it never chunks and never merges.

Reading: K/V coming out of the up-projection are bf16 tensors at the
attention call (the call's dtype), so ``kv_as_bf16`` (default on) rounds the
float64 decompressed K/V to bf16 before the attention.  Windows are not
supported on the chunked path (a window would need absolute positions the
chunk calls do not carry); the oracle asserts ``window_left < 0``.
"""
import numpy as np

from .attention import attend_request
from .bf16 import bf16_bits_to_f64, round_f64_to_bf16
from .gather import gather_latent
from .up_proj import up_project


def chunked_prefill_attention(new_q, new_k, new_v, qo_indptr, cache, block_table, prefix_lens,
                              w_kvb, *, sm_scale: float, logits_soft_cap: float = 0.0,
                              window_left: int = -1, rows=None, heads=None,
                              kv_as_bf16: bool = True):
    """Returns (o [n_rows, n_heads, 128], lse [n_rows, n_heads]) in float64.

    new_q/new_k/new_v: ragged [sum Lq, H, *] bf16 bits of the new tokens;
    cache/block_table/prefix_lens describe each request's cached prefix;
    ``rows``: optional per-request row indices; ``heads``: optional subset.
    """
    assert window_left < 0, "chunked prefix attention is defined without a window"
    qo = np.asarray(qo_indptr, dtype=np.int64)
    num_heads = new_q.shape[1]
    heads = list(range(num_heads)) if heads is None else list(heads)
    outs, lses = [], []
    for r in range(len(qo) - 1):
        p = int(prefix_lens[r])
        one_req_table = block_table[r:r + 1]
        latent = gather_latent(cache, one_req_table, np.array([0, p]), np.array([0]))
        q_r = new_q[qo[r]:qo[r + 1]]
        lq = q_r.shape[0]
        sel = np.arange(lq) if rows is None else np.asarray(rows[r], dtype=np.int64)
        o_r = np.zeros((len(sel), len(heads), new_v.shape[2]))
        l_r = np.full((len(sel), len(heads)), -np.inf)
        for hi, h in enumerate(heads):
            w_h = w_kvb[:, h * 256:(h + 1) * 256]
            k_p, v_p = up_project(latent, w_h, 1)
            if kv_as_bf16:
                k_p, v_p = round_f64_to_bf16(k_p), round_f64_to_bf16(v_p)
            k_all = np.concatenate([k_p, bf16_bits_to_f64(new_k[qo[r]:qo[r + 1], h:h + 1])], axis=0)
            v_all = np.concatenate([v_p, bf16_bits_to_f64(new_v[qo[r]:qo[r + 1], h:h + 1])], axis=0)
            o, l = attend_request(bf16_bits_to_f64(q_r[:, h:h + 1]), k_all, v_all, causal=True,
                                  sm_scale=sm_scale, logits_soft_cap=logits_soft_cap, rows=sel)
            o_r[:, hi] = o[:, 0]
            l_r[:, hi] = l[:, 0]
        outs.append(o_r)
        lses.append(l_r)
    return np.concatenate(outs, axis=0), np.concatenate(lses, axis=0)
