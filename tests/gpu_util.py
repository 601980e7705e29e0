"""Shared helpers for the GPU parity tests (bf16 bit transport and tolerance checks)."""
import numpy as np

from oracle import bf16_bits_to_f64

# Tolerances for bf16 inputs with fp32 accumulation (stated with the workloads):
O_MAX_ABS = 1.5e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 2e-3


def to_dev_bf16(bits: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_dev(arr: np.ndarray, device="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def bits_of(t) -> np.ndarray:
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of_bf16(t) -> np.ndarray:
    return bf16_bits_to_f64(bits_of(t))


def check_attention(o_gpu: np.ndarray, lse_gpu: np.ndarray, o_ref: np.ndarray, lse_ref: np.ndarray, what=""):
    """o_* float64 [rows, H, 128]; lse_* float64 [rows, H]."""
    assert o_gpu.shape == o_ref.shape, (o_gpu.shape, o_ref.shape)
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    err = np.abs(o_gpu - o_ref)
    assert err.max(initial=0) <= O_MAX_ABS, f"{what}: O max err {err.max():.3e}"
    assert (err.mean() if err.size else 0) <= O_MEAN_ABS, f"{what}: O mean err {err.mean():.3e}"
    if lse_gpu is not None:
        ninf_ref = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(lse_gpu), ninf_ref), f"{what}: -inf LSE pattern differs"
        fin = ~ninf_ref
        lerr = np.abs(lse_gpu[fin] - lse_ref[fin])
        assert lerr.max(initial=0) <= LSE_MAX_ABS, f"{what}: LSE max err {lerr.max():.3e}"
        return float(err.max(initial=0)), float(err.mean() if err.size else 0), float(lerr.max(initial=0))
    return float(err.max(initial=0)), float(err.mean() if err.size else 0), 0.0


def sample_rows(q_lens, n_random=128, every_tile=1, seed=0):
    """Per request: first 2, last 2, tile boundaries (every `every_tile`-th) +-1, random rows."""
    rng = np.random.default_rng(seed)
    out = []
    for L in q_lens:
        L = int(L)
        s = {0, 1, L - 2, L - 1}
        for b in range(128 * every_tile, L, 128 * every_tile):
            s.update((b - 1, b, b + 1))
        s.update(rng.integers(0, L, size=min(n_random, L)).tolist())
        out.append(np.array(sorted(x for x in s if 0 <= x < L), dtype=np.int64))
    return out
