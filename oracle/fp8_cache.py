"""FP8 latent cache entries and their dequantization (test infrastructure only).

Source: vLLM ``vllm/models/deepseek_v4/sparse_mla.py``, the ``fp8_ds_mla`` cache
dtype: one cache entry per token holds the NoPE part as fp8, then the RoPE part
(128 bytes, i.e. 64 bf16 values), then 8 bytes of fp8 scales (584 bytes for
DeepSeek-V4's 448 NoPE + 64 RoPE).  sglang issue #3849 gives DeepSeek-R1's
compressed row: 512 latent + 64 rope.

Readings (the page prints only the byte budget; each is listed in the design
notes):
  * the R1-shaped entry is 648 bytes: bytes [0, 512) hold the 512 latent values
    as float8 e4m3 (the "fn" variant: no infinities, 0x7F/0xFF are NaN), bytes
    [512, 640) the 64 rope values as bf16 (little-endian), bytes [640, 648)
    eight scale bytes, scale g covering latent values [64 g, 64 g + 64);
  * a scale byte is an unsigned power-of-two exponent (UE8M0): scale = 2^(b - 127),
    b = 255 is NaN;
  * the dequantized latent value is e4m3(x) * scale rounded to bf16 (round to
    nearest even; the product of a 4-bit significand and a power of two is
    exact in fp64, so this is one rounding, which only matters below bf16's
    normal range or above its largest value);
  * the rope part is copied unchanged.
"""
import numpy as np

from .gather import gather_latent

ENTRY_BYTES = 648
LATENT = 512
ROPE = 64
GROUP = 64


def e4m3_to_f64(b: np.ndarray) -> np.ndarray:
    """float8 e4m3 (fn) byte -> float64, from the format's definition: sign bit, 4-bit
    exponent with bias 7, 3-bit mantissa; exponent 0 is subnormal (2^-6 * m/8);
    exponent 15 with mantissa 7 is NaN (there is no infinity)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    out = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, out)


def ue8m0_to_f64(b: np.ndarray) -> np.ndarray:
    """Unsigned power-of-two scale byte -> 2^(b - 127); 255 is NaN."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    return np.where(b == 255, np.nan, np.ldexp(1.0, b - 127))


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, round to nearest even, over bf16's whole range:
    subnormals (multiples of 2^-133 below 2^-126), overflow to infinity, signed zero,
    NaN -> the quiet NaN 0x7FC0."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    nan = np.isnan(x)
    ax = np.abs(np.where(nan, 0.0, x))
    sign = np.signbit(x) & ~nan
    # normal range: keep 8 significant bits (round to nearest even on the float64 bits)
    u = np.where(ax >= 2.0 ** -126, ax, 1.0).view(np.uint64)
    drop = np.uint64(52 - 7)
    r = (u + ((np.uint64(1) << (drop - np.uint64(1))) - np.uint64(1)) + ((u >> drop) & np.uint64(1))) >> drop << drop
    normal = r.view(np.float64)
    # below the normal range: multiples of 2^-133 (np.round rounds half to even)
    sub = np.round(ax * 2.0 ** 133) * 2.0 ** -133
    mag = np.where(ax >= 2.0 ** -126, normal, sub)
    big = mag > np.float64(np.finfo(np.float32).max)       # past bf16's largest value once rounded
    mag32 = np.where(big, np.inf, mag).astype(np.float32)   # exact: bf16 values are float32 values
    bits = (mag32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    out[:] = np.where(sign, bits | np.uint16(0x8000), bits)
    out[nan] = np.uint16(0x7FC0)
    return out


def dequant_fp8_entries(entries: np.ndarray) -> np.ndarray:
    """uint8 [T, 648] cache entries -> bf16 bits [T, 576] (512 dequantized latent + 64 rope)."""
    entries = np.ascontiguousarray(entries, dtype=np.uint8)
    t = entries.shape[0]
    vals = e4m3_to_f64(entries[:, :LATENT])
    scales = ue8m0_to_f64(entries[:, LATENT + 2 * ROPE:ENTRY_BYTES])          # [T, 8]
    lat = vals * np.repeat(scales, GROUP, axis=1)
    out = np.empty((t, LATENT + ROPE), dtype=np.uint16)
    out[:, :LATENT] = f64_to_bf16_bits(lat)
    out[:, LATENT:] = entries[:, LATENT:LATENT + 2 * ROPE].copy().view("<u2")
    return out


def gather_latent_fp8(cache: np.ndarray, block_table: np.ndarray, cu_seq_lens: np.ndarray,
                      chunk_starts: np.ndarray) -> np.ndarray:
    """One prefix chunk out of an fp8 paged cache [num_blocks, block_size, 648] (uint8),
    dequantized: the slot rule of ``gather_latent`` followed by ``dequant_fp8_entries``."""
    return dequant_fp8_entries(gather_latent(cache, block_table, cu_seq_lens, chunk_starts))
