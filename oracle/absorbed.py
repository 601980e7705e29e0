"""Absorbed-weight MLA attention (MQA over the compressed latent) in float64 -- test
infrastructure only.

Sources: sglang issue #3849 ("[DeepseekR1] How ragged prefill manage kv_cache?"): prefill
with a cached prefix calls ``forward_absorb``, attention over the compressed cache rows
(512 latent + 64 rope) instead of decompressed MHA keys; Apache TVM PR #17674: with MLA
weight absorption the softmax scale can no longer be inferred from the head dim, so
``sm_scale`` is passed explicitly.

What absorption computes (the plain definition, written out).  With the up-projection's
per-head blocks W_UK(h) = W_kv_b[:, 256 h : 256 h + 128] and W_UV(h) = W_kv_b[:, 256 h + 128 :
256 h + 256] (the column layout the up-projection oracle uses), the MHA logit of head h is
q_nope(h) . (c_j W_UK(h)) + q_rope(h) . r_j = (W_UK(h) q_nope(h)) . c_j + q_rope(h) . r_j.
So with the absorbed query q_abs(h) = [W_UK(h) q_nope(h) (512) || q_rope(h) (64)] every head
attends to the one shared 576-wide cache row [c_j || r_j] (multi-query attention, one KV
head, Dqk = 576), with V = c_j (Dv = 512), and the MHA output of head h is O_lat(h) W_UV(h).
The softmax scale is the MHA one (192^-0.5 here), passed explicitly.
"""
import numpy as np

from .attention import allowed_mask
from .bf16 import bf16_bits_to_f64

LORA, ROPE, NOPE = 512, 64, 128


def _f64(x):
    return bf16_bits_to_f64(x) if x.dtype == np.uint16 else np.asarray(x, dtype=np.float64)


def absorb_query(q: np.ndarray, w_kvb: np.ndarray) -> np.ndarray:
    """q [T, H, 192] (128 NoPE + 64 RoPE), w_kvb [512, H*256] -> q_abs [T, H, 576] (float64)."""
    q, w = _f64(q), _f64(w_kvb)
    t, h = q.shape[0], q.shape[1]
    out = np.empty((t, h, LORA + ROPE))
    for hh in range(h):
        w_uk = w[:, hh * 256:hh * 256 + NOPE]                 # [512, 128]
        out[:, hh, :LORA] = q[:, hh, :NOPE] @ w_uk.T           # W_UK(h) q_nope(h)
        out[:, hh, LORA:] = q[:, hh, NOPE:]
    return out


def absorbed_attention(q_abs: np.ndarray, kv: np.ndarray, *, causal: bool, sm_scale: float,
                       logits_soft_cap: float = 0.0, rows=None):
    """One request: q_abs [Lq, H, 576], kv [Lkv, 576] (the compressed cache rows).

    Returns (o_lat [n, H, 512], lse [n, H]): per head, softmax over s = sm_scale * q_abs . kv
    (soft-capped and masked as in ``attend_request``, bottom-right causal) and
    o_lat = sum_j p_j kv_j[:512].  A row with no allowed key has o_lat = 0, LSE = -inf."""
    q, kv = _f64(q_abs), _f64(kv)
    lq, lkv = q.shape[0], kv.shape[0]
    row_idx = np.arange(lq) if rows is None else np.asarray(rows, dtype=np.int64)
    n, h = len(row_idx), q.shape[1]
    o = np.zeros((n, h, LORA))
    lse = np.full((n, h), -np.inf)
    if n == 0 or lkv == 0:
        return o, lse
    mask = allowed_mask(lq, lkv, causal, -1, row_idx)
    has = mask.any(axis=1)
    for hh in range(h):
        x = sm_scale * (q[row_idx, hh, :] @ kv.T)
        s = logits_soft_cap * np.tanh(x / logits_soft_cap) if logits_soft_cap > 0 else x
        s = np.where(mask, s, -np.inf)
        m = np.where(has, s.max(axis=1), 0.0)
        e = np.exp(s - m[:, None])
        tot = e.sum(axis=1)
        lse[:, hh] = np.where(has, m + np.log(np.where(has, tot, 1.0)), -np.inf)
        p = np.where(has[:, None], e / np.where(has, tot, 1.0)[:, None], 0.0)
        o[:, hh, :] = p @ kv[:, :LORA]
    return o, lse


def absorbed_output_to_mha(o_lat: np.ndarray, w_kvb: np.ndarray) -> np.ndarray:
    """o_lat [n, H, 512] -> the MHA output [n, H, 128]: o_lat(h) @ W_UV(h)."""
    w = _f64(w_kvb)
    n, h = o_lat.shape[0], o_lat.shape[1]
    out = np.empty((n, h, 128))
    for hh in range(h):
        out[:, hh, :] = o_lat[:, hh, :] @ w[:, hh * 256 + NOPE:(hh + 1) * 256]
    return out
