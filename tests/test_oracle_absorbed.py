"""Pins for the absorbed-weight attention oracle (CPU only): the absorption identity
against the MHA oracle over decompressed K/V (a separately pinned path), a math.fsum
brute force on tiny inputs, and the first-causal-row invariant."""
import math

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import (absorb_query, absorbed_attention, absorbed_output_to_mha, attend_request, bf16_bits_to_f64,
                    up_project)


def _case(seed, lq, lkv, heads):
    rng = np.random.default_rng(seed)
    q = wl.to_bf16_bits(rng.standard_normal((lq, heads, 192)).astype(np.float32))
    lat = wl.to_bf16_bits(rng.standard_normal((lkv, 576)).astype(np.float32))
    w = wl.to_bf16_bits((rng.standard_normal((512, heads * 256)) * 512 ** -0.5).astype(np.float32))
    return q, lat, w


@pytest.mark.parametrize("lq,lkv,causal,cap", [(7, 7, True, 0.0), (5, 19, True, 0.0), (6, 11, False, 0.0),
                                               (9, 9, True, 4.0), (4, 3, True, 0.0)])
def test_absorption_identity_against_mha(lq, lkv, causal, cap):
    """MQA over the compressed rows with the absorbed query gives the MHA oracle's LSE over
    the decompressed K/V, and its output times W_UV gives the MHA output (exact in fp64)."""
    heads = 3
    q, lat, w = _case(lq * 100 + lkv, lq, lkv, heads)
    scale = 192 ** -0.5
    k, v = up_project(lat, w, heads)                              # fp64, not rounded
    o_mha, l_mha = attend_request(q, k, v, causal=causal, sm_scale=scale, logits_soft_cap=cap)
    o_lat, l_abs = absorbed_attention(absorb_query(q, w), lat, causal=causal, sm_scale=scale, logits_soft_cap=cap)
    fin = np.isfinite(l_mha)
    np.testing.assert_array_equal(np.isneginf(l_abs), np.isneginf(l_mha))
    np.testing.assert_allclose(l_abs[fin], l_mha[fin], rtol=0, atol=1e-11)
    np.testing.assert_allclose(absorbed_output_to_mha(o_lat, w), o_mha, rtol=0, atol=1e-11)


def test_brute_force_tiny():
    q, lat, w = _case(3, 4, 6, 2)
    qa = absorb_query(q, w)
    kv = bf16_bits_to_f64(lat)
    scale = 0.11
    o, l = absorbed_attention(qa, lat, causal=True, sm_scale=scale)
    for i in range(4):
        for h in range(2):
            keys = [j for j in range(6) if j <= i + 2]                    # bottom-right: Lkv - Lq = 2
            s = [scale * math.fsum(qa[i, h, d] * kv[j, d] for d in range(576)) for j in keys]
            m = max(s)
            tot = math.fsum(math.exp(x - m) for x in s)
            assert abs(l[i, h] - (m + math.log(tot))) < 1e-12
            for d in (0, 17, 511):
                ref = math.fsum(math.exp(x - m) / tot * kv[j, d] for x, j in zip(s, keys))
                assert abs(o[i, h, d] - ref) < 1e-12


def test_first_causal_row_is_first_latent_row():
    q, lat, w = _case(4, 5, 5, 2)
    o, l = absorbed_attention(absorb_query(q, w), lat, causal=True, sm_scale=0.07)
    np.testing.assert_array_equal(o[0, 0], bf16_bits_to_f64(lat[0, :512]))
    np.testing.assert_array_equal(o[0, 1], bf16_bits_to_f64(lat[0, :512]))
