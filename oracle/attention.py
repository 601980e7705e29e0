"""Ragged multi-head attention with LSE, in float64 (test infrastructure only).

Source of the definition:
  * vLLM ``vllm.v1.attention.backends.mla.prefill.flashinfer``,
    ``FlashInferPrefillBackend.finalize_attention_metadata``: one ragged
    problem per request given by ``qo_indptr``/``kv_indptr``, as many KV heads
    as query heads, query/key head dim 128 NoPE + 64 RoPE, value head dim 128,
    an explicit ``sm_scale``, ``window_left``, ``logits_soft_cap``; the
    new-token problem is causal with ``kv_indptr = qo_indptr``; prefix chunks
    are non-causal.
  * same page, ``FlashInferPrefillImpl.run_prefill_new_tokens`` and
    ``run_prefill_context_chunk``: ``run(..., return_lse=True)`` returns O and
    an LSE laid out (q_len, num_heads).
  * Apache TVM PR #17674: the softmax scale is always passed explicitly.

Readings where the pages are silent (each listed in the design notes):
  * LSE is the natural log of sum_j exp(s_ij), s_ij being the scaled and
    soft-capped logit.
  * Causal alignment is bottom-right: query row i of a request with Lq
    queries and Lkv keys sits at key position i + (Lkv - Lq).
  * ``window_left = w >= 0`` keeps keys j with i_abs - w <= j (plus the causal
    bound when causal); ``w < 0`` means no window.
  * Soft cap: s = cap * tanh(sm_scale * q.k / cap) when cap > 0 (scale first).
  * A row with no allowed key has O = 0 and LSE = -inf.
"""
from __future__ import annotations

import numpy as np

from .bf16 import bf16_bits_to_f64


def _as_f64(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f64(x) if x.dtype == np.uint16 else np.asarray(x, dtype=np.float64)


def allowed_mask(lq: int, lkv: int, causal: bool, window_left: int,
                 rows: np.ndarray | None = None) -> np.ndarray:
    """Boolean [n_rows, lkv]: may query row i see key j?"""
    i = np.arange(lq) if rows is None else np.asarray(rows)
    i_abs = i[:, None] + (lkv - lq)
    j = np.arange(lkv)[None, :]
    mask = np.ones((len(i), lkv), dtype=bool)
    if causal:
        mask &= j <= i_abs
    if window_left >= 0:
        mask &= j >= i_abs - window_left
    return mask


def attend_request(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, causal: bool,
                   sm_scale: float, window_left: int = -1, logits_soft_cap: float = 0.0,
                   rows: np.ndarray | None = None, heads=None):
    """Attention of one request.

    q: [Lq, H, Dqk], k: [Lkv, H, Dqk], v: [Lkv, H, Dv] (bf16 bits or floats).
    Returns (o [n_rows, n_heads, Dv], lse [n_rows, n_heads]) in float64.
    """
    lq, lkv = q.shape[0], k.shape[0]
    heads = range(q.shape[1]) if heads is None else list(heads)
    row_idx = np.arange(lq) if rows is None else np.asarray(rows, dtype=np.int64)
    n, dv = len(row_idx), v.shape[2]
    o = np.zeros((n, len(heads), dv))
    lse = np.full((n, len(heads)), -np.inf)
    if n == 0 or lkv == 0:
        return o, lse
    mask = allowed_mask(lq, lkv, causal, window_left, row_idx)
    has_key = mask.any(axis=1)
    for hi, h in enumerate(heads):
        qh = _as_f64(q[row_idx, h, :])
        kh = _as_f64(k[:, h, :])
        vh = _as_f64(v[:, h, :])
        x = sm_scale * (qh @ kh.T)                       # [n, Lkv] logits
        if logits_soft_cap > 0:
            s = logits_soft_cap * np.tanh(x / logits_soft_cap)
        else:
            s = x
        s = np.where(mask, s, -np.inf)
        m = np.where(has_key, s.max(axis=1), 0.0)         # row max (0 for empty rows)
        e = np.exp(s - m[:, None])                        # exp(-inf) = 0 on masked keys
        tot = e.sum(axis=1)
        row_lse = np.where(has_key, m + np.log(np.where(has_key, tot, 1.0)), -np.inf)
        p = np.where(has_key[:, None], e / np.where(has_key, tot, 1.0)[:, None], 0.0)
        o[:, hi, :] = p @ vh
        lse[:, hi] = row_lse
    return o, lse


def ragged_attention(q, k, v, qo_indptr, kv_indptr, *, causal: bool, sm_scale: float,
                     window_left: int = -1, logits_soft_cap: float = 0.0,
                     rows=None, heads=None):
    """Attention over every request of a ragged batch.

    q: [sum Lq, H, Dqk], k: [sum Lkv, H, Dqk], v: [sum Lkv, H, Dv].
    ``rows``: optional list (one entry per request) of row indices inside the
    request; the result then stacks those rows request after request.
    Returns (o, lse) with o [n_rows, n_heads, Dv] and lse [n_rows, n_heads].
    """
    qo = np.asarray(qo_indptr, dtype=np.int64)
    kv = np.asarray(kv_indptr, dtype=np.int64)
    outs, lses = [], []
    for r in range(len(qo) - 1):
        sel = None if rows is None else rows[r]
        o, l = attend_request(q[qo[r]:qo[r + 1]], k[kv[r]:kv[r + 1]], v[kv[r]:kv[r + 1]],
                              causal=causal, sm_scale=sm_scale, window_left=window_left,
                              logits_soft_cap=logits_soft_cap, rows=sel, heads=heads)
        outs.append(o)
        lses.append(l)
    nh = q.shape[1] if heads is None else len(list(heads))
    if not outs:
        return np.zeros((0, nh, v.shape[2])), np.zeros((0, nh))
    return np.concatenate(outs, axis=0), np.concatenate(lses, axis=0)
