"""bfloat16 <-> float64 for the oracle (test infrastructure only).

bfloat16 is the upper half of an IEEE float32, so decoding is exact.  The
encoder rounds a float64 straight to bfloat16 (7 stored mantissa bits,
round to nearest, ties to even) without passing through float32, so there
is no double rounding.  Used only where a reading says an intermediate is
carried as bf16 (the ABI's K/V and O tensors).
"""
import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """uint16 bfloat16 patterns -> float64 (exact)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    Returns float64 values that are exactly representable in bfloat16.
    Valid for finite inputs inside the normal bfloat16 range, which is all
    the oracle ever feeds it.
    """
    x = np.ascontiguousarray(x, dtype=np.float64)
    u = x.view(np.uint64)
    drop = np.uint64(52 - 7)                       # float64 mantissa bits below bf16's 7
    keep_lsb = (u >> drop) & np.uint64(1)
    half = (np.uint64(1) << (drop - np.uint64(1))) - np.uint64(1)
    r = (u + half + keep_lsb) >> drop << drop
    return r.view(np.float64)
