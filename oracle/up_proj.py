"""Latent up-projection (decompression) in float64 (test infrastructure only).

sglang issue #3849 ("[DeepseekR1] How ragged prefill manage kv_cache?"):
the cache holds 512 latent ("compressed_kv") + 64 rope dims per token, while
prefill attention runs as MHA with 192-dim Q/K (128 NoPE + 64 RoPE) and
128-dim V.  The decompression multiplies the latent by the kv_b weight to
get each head's K_nope and V, and every head's K takes the one shared rope
part (vLLM ``finalize_attention_metadata``: the latent cache has a single
KV head).

Readings (pages silent): weight columns are grouped per head as
[h*256, h*256+128) -> K_nope of head h, [h*256+128, h*256+256) -> V of head h;
K = [K_nope || rope] in that order; RoPE is taken as already applied.
"""
import numpy as np

from .bf16 import bf16_bits_to_f64

NOPE, ROPE, DV, LORA = 128, 64, 128, 512


def up_project(latent: np.ndarray, w_kvb: np.ndarray, num_heads: int):
    """latent: [T, 576] bf16 bits; w_kvb: [512, H*256] bf16 bits.

    Returns (k [T, H, 192], v [T, H, 128]) in float64, exact products summed
    in float64.
    """
    lat = bf16_bits_to_f64(latent)
    w = bf16_bits_to_f64(w_kvb)
    t = lat.shape[0]
    kv = (lat[:, :LORA] @ w).reshape(t, num_heads, NOPE + DV)
    rope = lat[:, LORA:LORA + ROPE]
    k = np.empty((t, num_heads, NOPE + ROPE))
    k[:, :, :NOPE] = kv[:, :, :NOPE]
    k[:, :, NOPE:] = rope[:, None, :]
    v = kv[:, :, NOPE:].copy()
    return k, v
