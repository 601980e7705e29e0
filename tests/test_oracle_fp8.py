"""Pins for the fp8 latent-cache oracle (CPU only): hand-decoded codes from the format
definitions, every e4m3 code against torch's float8 type, bf16 rounding over the whole
range against torch's float32 -> bfloat16 conversion, and the entry layout by one-hot
entries."""
import json
import os

import numpy as np
import pytest

from chunked_prefill_attention_ragged_gb300 import workloads as wl
from oracle import (bf16_bits_to_f64, dequant_fp8_entries, e4m3_to_f64, f64_to_bf16_bits, gather_latent,
                    gather_latent_fp8, ue8m0_to_f64)

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "fp8_e4m3_hand_codes.json")))
torch = pytest.importorskip("torch")


def _val(v):
    return np.nan if v == "nan" else float(v)


def test_e4m3_hand_codes():
    codes = np.array([int(c, 16) for c, _ in GOLD["codes"]], dtype=np.uint8)
    want = np.array([_val(v) for _, v in GOLD["codes"]])
    got = e4m3_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(want[ok]))   # -0.0 keeps its sign


def test_e4m3_every_code_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_ue8m0_hand_codes_and_torch():
    codes = np.array([int(c, 16) for c, _ in GOLD["ue8m0"]["codes"]], dtype=np.uint8)
    want = np.array([_val(v) for _, v in GOLD["ue8m0"]["codes"]])
    got = ue8m0_to_f64(codes)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    np.testing.assert_array_equal(got[~np.isnan(want)], want[~np.isnan(want)])
    allc = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(allc).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    g = ue8m0_to_f64(allc)
    np.testing.assert_array_equal(np.isnan(g), np.isnan(ref))
    np.testing.assert_array_equal(g[~np.isnan(ref)], ref[~np.isnan(ref)])


def test_bf16_encoder_whole_range():
    # float32 inputs are exact in float64, so one float64 -> bf16 rounding must equal
    # torch's float32 -> bfloat16 (round to nearest even, subnormals, overflow).
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 1 << 32, size=200000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    tiny = (rng.integers(0, 1 << 20, size=20000).astype(np.float32) * np.float32(2.0 ** -149))   # subnormals
    edge = np.array([2.0 ** -133, 1.5 * 2.0 ** -133, 0.5 * 2.0 ** -133, 2.5 * 2.0 ** -133, -0.0, 3.3e38, 3.39e38,
                     np.finfo(np.float32).max, -np.inf, np.inf, 0.0], dtype=np.float32)
    allx = np.concatenate([x, tiny, -tiny, edge])
    ref = torch.from_numpy(allx).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(f64_to_bf16_bits(allx.astype(np.float64)), ref)
    assert f64_to_bf16_bits(np.array([np.nan]))[0] == 0x7FC0


def test_entry_layout_one_hot():
    # Latent bytes all 1.0 (0x38), scale g = 2^(g - 3): value i must be 2^(i // 64 - 3);
    # the rope bytes are copied as 64 little-endian bf16 values.
    e = np.zeros((2, 648), dtype=np.uint8)
    e[:, :512] = 0x38
    e[:, 640:648] = np.arange(8, dtype=np.uint8) + 124
    rope = wl.to_bf16_bits(np.arange(64, dtype=np.float32) - 31.5)
    e[0, 512:640] = rope.view(np.uint8)
    e[1, 3] = 0xC0            # -2.0 in group 0 of entry 1
    out = dequant_fp8_entries(e)
    vals = bf16_bits_to_f64(out[:, :512])
    np.testing.assert_array_equal(vals[0], 2.0 ** (np.arange(512) // 64 - 3))
    np.testing.assert_array_equal(out[0, 512:], rope)
    assert vals[1, 3] == -2.0 * 2.0 ** -3 and vals[1, 4] == 2.0 ** -3


def test_dequant_exact_products_and_gather():
    # Mid-range scales: every product is a bf16 value, so dequant is exact.
    rng = np.random.default_rng(8)
    cache = wl.random_fp8_cache(rng, 6, 4)
    e = cache.reshape(-1, 648)
    lat = bf16_bits_to_f64(dequant_fp8_entries(e)[:, :512])
    exact = e4m3_to_f64(e[:, :512]) * np.repeat(ue8m0_to_f64(e[:, 640:]), 64, axis=1)
    np.testing.assert_array_equal(lat, exact)
    table = rng.permutation(6)[:4].reshape(2, 2).astype(np.int32)
    cu = np.array([0, 5, 8], dtype=np.int32)
    st = np.array([2, 1], dtype=np.int32)
    got = gather_latent_fp8(cache, table, cu, st)
    np.testing.assert_array_equal(got, dequant_fp8_entries(gather_latent(cache, table, cu, st)))
    slot = table[1, 0] * 4 + 3          # row 5 + 2: request 1, position 1 + 2 = 3 -> block index 0, offset 3
    np.testing.assert_array_equal(got[5 + 2], dequant_fp8_entries(e[slot:slot + 1])[0])
