"""Shared helpers for the GPU parity tests (bf16 bit transport and tolerance checks)."""
import numpy as np

from oracle import bf16_bits_to_f64

# Tolerances for bf16 inputs with fp32 accumulation (stated with the workloads):
O_MAX_ABS = 1.5e-2
O_MEAN_ABS = 2e-3
LSE_MAX_ABS = 2e-3
# O is a bf16 tensor, so even the exact result, rounded to the nearest bf16, can be half a
# bf16 ulp away from the fp64 oracle: 2^-6 = 0.0156 for |O| in [4, 8), already above
# O_MAX_ABS.  The max bound therefore applies to the error beyond that representation
# step: |O_gpu - O_ref| <= O_MAX_ABS + ulp_bf16(O_ref) / 2.


def half_ulp_bf16(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |x| (8 significant bits), 2^(e - 8) for |x| in [2^e, 2^(e+1))."""
    return 2.0 ** (np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126))) - 8)


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
    beyond = err - half_ulp_bf16(o_ref)
    assert beyond.max(initial=0) <= O_MAX_ABS, (
        f"{what}: O error {beyond.max():.3e} beyond half a bf16 ulp (max raw error {err.max():.3e})")
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


# ---------------------------------------------------------------------------- guard bands
GUARD_BYTES = 4096
_GUARD_BYTE = 0xA5


class Guarded:
    """A device tensor with GUARD_BYTES of sentinel bytes before and after it.

    A kernel that writes past either end of its output (a wrong row stride, a ragged tail
    written in full, a stray store of a masked row) changes the sentinel; ``check()``
    asserts that it did not.  compute-sanitizer stands in for nothing here: this is the
    check that runs with every parity test."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        import torch
        n = 1
        for s in shape:
            n *= int(s)
        esize = torch.empty((), dtype=dtype).element_size()
        nbytes = n * esize
        self.raw = torch.full((2 * GUARD_BYTES + nbytes + 16,), _GUARD_BYTE, dtype=torch.uint8, device=device)
        self.tensor = self.raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(*shape)
        if fill is not None:
            self.tensor.fill_(fill)
        self.nbytes = nbytes

    def check(self, what=""):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.nbytes:]
        assert bool((head == _GUARD_BYTE).all()), f"{what}: bytes before the output were written"
        assert bool((tail == _GUARD_BYTE).all()), f"{what}: bytes after the output were written"


# ---------------------------------------------------------------------------- parallel oracle
def _attend_piece(args):
    from oracle import attend_request
    q, k, v, kw = args
    return attend_request(q, k, v, **kw)


def _chunked_piece(args):
    from oracle import chunked_prefill_attention
    a, kw = args
    return chunked_prefill_attention(*a, **kw)


def _pool(n_jobs):
    import multiprocessing as mp
    import os
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    workers = max(1, min(n_jobs, os.cpu_count() or 1, 16))
    # spawn, never fork: the parent already holds a CUDA context.
    return mp.get_context("spawn").Pool(workers)


def oracle_parallel(b, rows=None):
    """The oracle over every (request, head) of a ragged batch, in a spawned process pool.

    rows: optional per-request row indices (as for ``oracle.ragged_attention``).  Returns
    (o [n_rows, H, 128], lse [n_rows, H]) stacked request after request."""
    qo, kv = b.qo_indptr, b.kv_indptr
    jobs, where = [], []
    for r in range(b.batch):
        sel = None if rows is None else rows[r]
        kw = dict(causal=b.causal, sm_scale=b.sm_scale, window_left=b.window_left,
                  logits_soft_cap=b.logits_soft_cap, rows=sel)
        for h in range(b.num_heads):
            jobs.append((b.q[qo[r]:qo[r + 1], h:h + 1], b.k[kv[r]:kv[r + 1], h:h + 1], b.v[kv[r]:kv[r + 1], h:h + 1],
                         kw))
            where.append((r, h))
    with _pool(len(jobs)) as pool:
        res = pool.map(_attend_piece, jobs, chunksize=1)
    return _stack(b, rows, where, res)


def chunked_oracle_parallel(cb, rows=None, heads_per_job=8):
    """``oracle.chunked_prefill_attention`` over every (request, head group), in a spawned pool.

    Each job gets its request's prefix rows (taken out of the cache by ``oracle.gather_latent``
    here) as a cache of one-row blocks, so the whole cache is not shipped to every worker."""
    from oracle import gather_latent
    b = cb.new
    qo = b.qo_indptr
    H = b.num_heads
    jobs, where = [], []
    for r in range(b.batch):
        p = int(cb.prefix_lens[r])
        lat = gather_latent(cb.cache, cb.block_table[r:r + 1], np.array([0, p]), np.array([0]))
        cache_r = lat.reshape(p, 1, lat.shape[1]) if p else np.zeros((1, 1, lat.shape[1]), dtype=lat.dtype)
        table_r = np.arange(max(p, 1), dtype=np.int32)[None, :]
        sel = None if rows is None else [rows[r]]
        lq = int(qo[r + 1] - qo[r])
        for h0 in range(0, H, heads_per_job):
            hs = slice(h0, min(H, h0 + heads_per_job))
            a = (b.q[qo[r]:qo[r + 1], hs], b.k[qo[r]:qo[r + 1], hs], b.v[qo[r]:qo[r + 1], hs],
                 np.array([0, lq], dtype=np.int32), cache_r, table_r, np.array([p]),
                 cb.w_kvb[:, h0 * 256:hs.stop * 256])
            jobs.append((a, dict(sm_scale=b.sm_scale, logits_soft_cap=b.logits_soft_cap, rows=sel)))
            where.append((r, hs))
    with _pool(len(jobs)) as pool:
        res = pool.map(_chunked_piece, jobs, chunksize=1)
    return _stack(b, rows, where, res)


def _stack(b, rows, where, res):
    H = b.num_heads
    n_r = [int(b.q_lens[r]) if rows is None else len(rows[r]) for r in range(b.batch)]
    off = np.concatenate([[0], np.cumsum(n_r)]).astype(np.int64)
    o = np.zeros((int(off[-1]), H, 128))
    lse = np.full((int(off[-1]), H), -np.inf)
    for (r, h), (o_p, l_p) in zip(where, res):
        if isinstance(h, slice):
            o[off[r]:off[r + 1], h] = o_p
            lse[off[r]:off[r + 1], h] = l_p
        else:
            o[off[r]:off[r + 1], h] = o_p[:, 0]
            lse[off[r]:off[r + 1], h] = l_p[:, 0]
    return o, lse
