"""ctypes binding over libmla_prefill.so (argument marshalling only).

Every function mirrors one C entry point of ``include/mla_prefill.h`` under
the same name.  Tensors are torch tensors: device memory and the current
CUDA stream come from torch, all arithmetic happens in the library's
kernels.  There is no fallback: if the shared library cannot be built or
loaded, the first call raises.
"""
from __future__ import annotations

import ctypes
import threading

import numpy as np

from . import _build

_lib = None
_lock = threading.Lock()

MLA_OK = 0
_c_int, _c_i64, _c_f, _c_vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)

_SIGNATURES = {
    "mla_error_string": (ctypes.c_char_p, [_c_int]),
    "mla_abi_version": (_c_int, []),
    "mla_prefill_plan": (_c_int, [ctypes.POINTER(_c_vp), _i32p, _i32p, _c_int, _c_int, _c_int, _c_int, _c_int,
                                  _c_f, _c_int, _c_f, _c_vp]),
    "mla_prefill_run": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_prefill_run_merge": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_prefill_run_shared_rope": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp, _c_vp, _c_int,
                                             _c_vp]),
    "mla_prefill_status": (_c_int, [_c_vp]),
    "mla_plan_destroy": (_c_int, [_c_vp]),
    "mla_plan_query": (_c_int, [_c_vp, _c_int, _i64p]),
    "mla_plan_units_host": (_c_int, [_i32p, _i32p, _c_int, _c_int, _c_int, _c_int, _c_int, _i32p, _c_i64, _i32p,
                                     _i64p]),
    "mla_gather_latent": (_c_int, [_c_vp, _c_i64, _c_int, _c_int, _c_vp, _c_int, _c_vp, _c_vp, _c_int, _c_i64,
                                   _c_vp, _c_vp, _c_vp]),
    "mla_gather_latent_fp8": (_c_int, [_c_vp, _c_i64, _c_int, _c_int, _c_vp, _c_int, _c_vp, _c_vp, _c_int, _c_i64,
                                       _c_vp, _c_vp, _c_vp]),
    "mla_cache_write": (_c_int, [_c_vp, _c_i64, _c_int, _c_int, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp]),
    "mla_up_proj": (_c_int, [_c_vp, _c_vp, _c_i64, _c_int, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_up_proj_paged": (_c_int, [_c_vp, _c_i64, _c_int, _c_int, _c_vp, _c_int, _c_vp, _c_vp, _c_int, _c_i64,
                                   _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_up_proj_paged_split": (_c_int, [_c_vp, _c_i64, _c_int, _c_int, _c_vp, _c_int, _c_vp, _c_vp, _c_int,
                                         _c_i64, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_merge_state": (_c_int, [_c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_i64, _c_int, _c_int, _c_vp]),
    "mla_prefill_run_noalloc": (_c_int, [_i32p, _i32p, _c_int, _c_int, _c_int, _c_int, _c_int, _c_f, _c_int, _c_f,
                                         _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp]),
    "mla_absorbed_plan": (_c_int, [ctypes.POINTER(_c_vp), _i32p, _i32p, _c_int, _c_int, _c_int, _c_int, _c_f, _c_f,
                                   _c_vp]),
    "mla_absorbed_run": (_c_int, [_c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_int, _c_vp, _c_vp, _c_vp]),
}
EXPORTED = tuple(_SIGNATURES)


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})")


def library(build_if_stale: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the shared library."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_stale else _build.LIB_PATH
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def library_path() -> str:
    return _build.LIB_PATH


def error_string(code: int) -> str:
    return library().mla_error_string(code).decode()


def _check(code: int, what: str):
    if code != MLA_OK:
        raise MlaError(code, what)


def _host_i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_i32p)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t, dtype, name):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------------------- plan
class PrefillPlan:
    """Owns an ``mla_plan_t``; created by :func:`mla_prefill_plan`."""

    def __init__(self, handle: ctypes.c_void_p, num_heads: int, total_q: int, total_kv: int):
        self._h = handle
        self.num_heads = num_heads
        self.total_q = total_q
        self.total_kv = total_kv

    @property
    def handle(self):
        return self._h

    def query(self, which: int) -> int:
        v = ctypes.c_int64(0)
        _check(library().mla_plan_query(self._h, which, ctypes.byref(v)), "mla_plan_query")
        return int(v.value)

    num_units = property(lambda self: self.query(0))
    num_ctas = property(lambda self: self.query(1))
    allowed_pairs = property(lambda self: self.query(4))
    kv_tiles = property(lambda self: self.query(5))
    cta_pairs = property(lambda self: bool(self.query(6)))

    def run(self, q, k, v, o=None, lse=None, return_lse=True, stream=None):
        return mla_prefill_run(self, q, k, v, o, lse, return_lse, stream)

    def run_merge(self, q, k, v, o, lse, stream=None):
        return mla_prefill_run_merge(self, q, k, v, o, lse, stream)

    def status(self) -> int:
        return mla_prefill_status(self)

    def destroy(self):
        if self._h:
            h, self._h = self._h, None
            _check(library().mla_plan_destroy(h), "mla_plan_destroy")

    def __del__(self):
        try:
            if self._h and _lib is not None:
                _lib.mla_plan_destroy(self._h)
                self._h = None
        except Exception:
            pass


def mla_prefill_plan(qo_indptr, kv_indptr, num_heads: int, head_dim_qk: int = 192, head_dim_vo: int = 128,
                     causal: bool = True, sm_scale: float | None = None, window_left: int = -1,
                     logits_soft_cap: float = 0.0, stream=None) -> PrefillPlan:
    """Plan a ragged prefill (host indptrs).  ``sm_scale`` is required, as on the pages."""
    if sm_scale is None:
        raise ValueError("sm_scale must be given explicitly")
    qo, kv = _host_i32(qo_indptr), _host_i32(kv_indptr)
    if qo.ndim != 1 or kv.shape != qo.shape or qo.size < 1:
        raise ValueError("qo_indptr and kv_indptr must be 1-D of equal length batch+1")
    h = ctypes.c_void_p()
    _check(library().mla_prefill_plan(ctypes.byref(h), _ptr(qo), _ptr(kv), qo.size - 1, num_heads, head_dim_qk,
                                      head_dim_vo, int(bool(causal)), float(sm_scale), int(window_left),
                                      float(logits_soft_cap), _stream(stream)), "mla_prefill_plan")
    return PrefillPlan(h, num_heads, int(qo[-1]), int(kv[-1]))


class AbsorbedPlan(PrefillPlan):
    """An ``mla_plan_t`` made by :func:`mla_absorbed_plan` (absorbed-weight MQA prefill over
    the paged latent cache); status, query and destroy as for :class:`PrefillPlan`."""

    def __init__(self, handle, num_heads: int, total_q: int, batch: int, block_size: int, max_kv_blocks: int):
        super().__init__(handle, num_heads, total_q, 0)
        self.batch = batch
        self.block_size = block_size
        self.max_kv_blocks = max_kv_blocks

    def run(self, q_abs, cache, block_table, o=None, lse=None, return_lse=True, stream=None):
        return mla_absorbed_run(self, q_abs, cache, block_table, o, lse, return_lse, stream)

    def run_merge(self, *args, **kwargs):
        raise TypeError("an absorbed plan runs with mla_absorbed_run")


def mla_absorbed_plan(qo_indptr, kv_lens, num_heads: int, block_size: int, causal: bool = True,
                      sm_scale: float | None = None, logits_soft_cap: float = 0.0, stream=None) -> AbsorbedPlan:
    """Plan an absorbed-weight prefill: request r has qo_indptr[r+1]-qo_indptr[r] new query
    rows, the last ones of its kv_lens[r] cache positions.  ``sm_scale`` is required."""
    if sm_scale is None:
        raise ValueError("sm_scale must be given explicitly")
    qo, kl = _host_i32(qo_indptr), _host_i32(kv_lens)
    if qo.ndim != 1 or qo.size < 1 or kl.shape != (qo.size - 1,):
        raise ValueError("qo_indptr must be 1-D [batch+1] and kv_lens [batch]")
    h = ctypes.c_void_p()
    _check(library().mla_absorbed_plan(ctypes.byref(h), _ptr(qo), _ptr(kl), qo.size - 1, num_heads, int(block_size),
                                       int(bool(causal)), float(sm_scale), float(logits_soft_cap), _stream(stream)),
           "mla_absorbed_plan")
    max_blocks = int(max(((int(x) + block_size - 1) // block_size for x in kl), default=0))
    return AbsorbedPlan(h, num_heads, int(qo[-1]), qo.size - 1, int(block_size), max_blocks)


def mla_absorbed_run(plan: AbsorbedPlan, q_abs, cache, block_table, o=None, lse=None, return_lse=True, stream=None):
    """Run an absorbed plan: q_abs [T, H, 576], cache [NB, BS, 576], block_table [B, M] int32
    (device) -> (o_lat [T, H, 512], lse [T, H] or None)."""
    import torch
    H, T = plan.num_heads, plan.total_q
    if tuple(q_abs.shape) != (T, H, 576):
        raise ValueError(f"q_abs must be [{T}, {H}, 576], got {tuple(q_abs.shape)}")
    if cache.dim() != 3 or cache.shape[1] != plan.block_size or cache.shape[2] != 576:
        raise ValueError(f"cache must be [num_blocks, {plan.block_size}, 576], got {tuple(cache.shape)}")
    if block_table.dim() != 2 or block_table.shape[0] != plan.batch or block_table.shape[1] < plan.max_kv_blocks:
        raise ValueError(f"block_table must be [{plan.batch}, >= {plan.max_kv_blocks}], got {tuple(block_table.shape)}")
    if o is None:
        o = torch.empty((T, H, 512), dtype=torch.bfloat16, device=q_abs.device)
    if return_lse and lse is None:
        lse = torch.empty((T, H), dtype=torch.float32, device=q_abs.device)
    if tuple(o.shape) != (T, H, 512) or (lse is not None and tuple(lse.shape) != (T, H)):
        raise ValueError("o/lse shapes do not match the plan")
    bf = torch.bfloat16
    _check(library().mla_absorbed_run(plan.handle, _dev(q_abs, bf, "q_abs"), _dev(cache, bf, "cache"),
                                      int(cache.shape[0]), _dev(block_table, torch.int32, "block_table"),
                                      int(block_table.shape[1]), _dev(o, bf, "o"),
                                      _dev(lse, torch.float32, "lse"), _stream(stream)),
           "mla_absorbed_run")
    return o, lse


def mla_prefill_run(plan: PrefillPlan, q, k, v, o=None, lse=None, return_lse=True, stream=None):
    """Run a plan; returns (o, lse) (lse None when not requested)."""
    import torch
    H = plan.num_heads
    if tuple(q.shape) != (plan.total_q, H, 192):
        raise ValueError(f"q must be [{plan.total_q}, {H}, 192], got {tuple(q.shape)}")
    if tuple(k.shape) != (plan.total_kv, H, 192) or tuple(v.shape) != (plan.total_kv, H, 128):
        raise ValueError("k/v shapes do not match the plan")
    if o is None:
        o = torch.empty((plan.total_q, H, 128), dtype=torch.bfloat16, device=q.device)
    if return_lse and lse is None:
        lse = torch.empty((plan.total_q, H), dtype=torch.float32, device=q.device)
    if tuple(o.shape) != (plan.total_q, H, 128) or (lse is not None and tuple(lse.shape) != (plan.total_q, H)):
        raise ValueError("o/lse shapes do not match the plan")
    bf = torch.bfloat16
    _check(library().mla_prefill_run(plan.handle, _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"),
                                     _dev(o, bf, "o"), _dev(lse, torch.float32, "lse"), _stream(stream)),
           "mla_prefill_run")
    return o, lse


def mla_prefill_run_merge(plan: PrefillPlan, q, k, v, o, lse, stream=None):
    """Run a plan and merge the result into the partial state (o, lse) in place; returns (o, lse)."""
    import torch
    H = plan.num_heads
    if tuple(q.shape) != (plan.total_q, H, 192):
        raise ValueError(f"q must be [{plan.total_q}, {H}, 192], got {tuple(q.shape)}")
    if tuple(k.shape) != (plan.total_kv, H, 192) or tuple(v.shape) != (plan.total_kv, H, 128):
        raise ValueError("k/v shapes do not match the plan")
    if o is None or lse is None:
        raise ValueError("mla_prefill_run_merge needs the partial state o and lse")
    if tuple(o.shape) != (plan.total_q, H, 128) or tuple(lse.shape) != (plan.total_q, H):
        raise ValueError("o/lse shapes do not match the plan")
    bf = torch.bfloat16
    _check(library().mla_prefill_run_merge(plan.handle, _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"),
                                           _dev(o, bf, "o"), _dev(lse, torch.float32, "lse"), _stream(stream)),
           "mla_prefill_run_merge")
    return o, lse


def mla_prefill_run_shared_rope(plan: PrefillPlan, q, k_nope, k_rope, v, o=None, lse=None, merge: bool = False,
                                stream=None):
    """Run a plan with K = [k_nope (per head) || k_rope (one row per key, shared by all heads)].

    k_nope [T_kv, H, 128]; k_rope: a 2-D [T_kv, 64] view whose rows may be strided (e.g.
    latent[:, 512:] of a gathered [T_kv, 576] latent).  merge=True merges into (o, lse)."""
    import torch
    H = plan.num_heads
    if tuple(q.shape) != (plan.total_q, H, 192):
        raise ValueError(f"q must be [{plan.total_q}, {H}, 192], got {tuple(q.shape)}")
    if tuple(k_nope.shape) != (plan.total_kv, H, 128) or tuple(v.shape) != (plan.total_kv, H, 128):
        raise ValueError("k_nope/v shapes do not match the plan")
    if k_rope.dim() != 2 or tuple(k_rope.shape) != (plan.total_kv, 64) or k_rope.stride(1) != 1:
        raise ValueError("k_rope must be a [T_kv, 64] view with unit column stride")
    if merge and (o is None or lse is None):
        raise ValueError("merge needs the partial state o and lse")
    if k_rope.dtype != torch.bfloat16 or not k_rope.is_cuda:
        raise TypeError("k_rope must be a bf16 CUDA tensor")
    if o is None:
        o = torch.empty((plan.total_q, H, 128), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((plan.total_q, H), dtype=torch.float32, device=q.device)
    if tuple(o.shape) != (plan.total_q, H, 128) or tuple(lse.shape) != (plan.total_q, H):
        raise ValueError("o/lse shapes do not match the plan")
    bf = torch.bfloat16
    _check(library().mla_prefill_run_shared_rope(plan.handle, _dev(q, bf, "q"), _dev(k_nope, bf, "k_nope"),
                                                 ctypes.c_void_p(k_rope.data_ptr()), int(k_rope.stride(0)),
                                                 _dev(v, bf, "v"), _dev(o, bf, "o"), _dev(lse, torch.float32, "lse"),
                                                 int(bool(merge)), _stream(stream)), "mla_prefill_run_shared_rope")
    return o, lse


def mla_prefill_status(plan: PrefillPlan) -> int:
    """Read-and-clear the plan's device status word; raises on a device-side error."""
    code = library().mla_prefill_status(plan.handle)
    _check(code, "mla_prefill_status")
    return code


def mla_plan_destroy(plan: PrefillPlan):
    plan.destroy()


def mla_plan_units_host(qo_indptr, kv_indptr, num_heads: int, causal: bool, window_left: int, num_ctas: int):
    """Host planner only: returns (units [n, 8] int32, cta_offsets [num_ctas+1] int32)."""
    qo, kv = _host_i32(qo_indptr), _host_i32(kv_indptr)
    n = ctypes.c_int64(0)
    offs = np.zeros(num_ctas + 1, dtype=np.int32)
    lib = library()
    args = (_ptr(qo), _ptr(kv), qo.size - 1, num_heads, int(bool(causal)), int(window_left), num_ctas)
    code = lib.mla_plan_units_host(*args, None, 0, _ptr(offs), ctypes.byref(n))
    if code not in (MLA_OK, -2):
        _check(code, "mla_plan_units_host")
    units = np.zeros((max(1, n.value), 8), dtype=np.int32)
    _check(lib.mla_plan_units_host(*args, _ptr(units), n.value, _ptr(offs), ctypes.byref(n)),
           "mla_plan_units_host")
    return units[:n.value], offs


# ---------------------------------------------------------------------------- gather / up-proj / merge
def mla_gather_latent(cache, block_table, cu_seq_lens, chunk_starts, total_tokens: int, out=None, status=None,
                      stream=None):
    """Copy one prefix chunk out of the paged latent cache (device tensors)."""
    import torch
    nb, bs, e = cache.shape
    if out is None:
        out = torch.empty((total_tokens, e), dtype=cache.dtype, device=cache.device)
    batch = block_table.shape[0]
    i32 = torch.int32
    _check(library().mla_gather_latent(_dev(cache, torch.bfloat16, "cache"), nb, bs, e,
                                       _dev(block_table, i32, "block_table"), block_table.shape[1],
                                       _dev(cu_seq_lens, i32, "cu_seq_lens"), _dev(chunk_starts, i32, "chunk_starts"),
                                       batch, int(total_tokens), _dev(out, torch.bfloat16, "out"),
                                       _dev(status, i32, "status"), _stream(stream)), "mla_gather_latent")
    return out


def mla_gather_latent_fp8(cache, block_table, cu_seq_lens, chunk_starts, total_tokens: int, out=None, status=None,
                          stream=None):
    """One prefix chunk out of an fp8 paged cache (uint8 [NB, BS, 648]), dequantized to
    bf16 [total_tokens, 576]."""
    import torch
    nb, bs, e = cache.shape
    t = int(total_tokens)
    if out is None:
        out = torch.empty((t, 576), dtype=torch.bfloat16, device=cache.device)
    if tuple(out.shape) != (t, 576):
        raise ValueError(f"out must be [{t}, 576]")
    batch = block_table.shape[0]
    if tuple(cu_seq_lens.shape) != (batch + 1,) or tuple(chunk_starts.shape) != (batch,):
        raise ValueError("cu_seq_lens must be [B+1] and chunk_starts [B] for a block table of B rows")
    i32 = torch.int32
    _check(library().mla_gather_latent_fp8(_dev(cache, torch.uint8, "cache"), nb, bs, e,
                                           _dev(block_table, i32, "block_table"), block_table.shape[1],
                                           _dev(cu_seq_lens, i32, "cu_seq_lens"),
                                           _dev(chunk_starts, i32, "chunk_starts"), batch, t,
                                           _dev(out, torch.bfloat16, "out"), _dev(status, i32, "status"),
                                           _stream(stream)), "mla_gather_latent_fp8")
    return out


def mla_cache_write(cache, latent, slot_mapping, status=None, stream=None):
    """Store latent [T, E] rows into the paged cache [NB, BS, E] at slot_mapping [T] (int64,
    device; negative = padding token).  Returns the cache (written in place)."""
    import torch
    nb, bs, e = cache.shape
    t = latent.shape[0]
    if latent.shape[1] != e or slot_mapping.shape[0] != t:
        raise ValueError("latent must be [T, entry_dim] and slot_mapping [T]")
    _check(library().mla_cache_write(_dev(cache, torch.bfloat16, "cache"), nb, bs, e,
                                     _dev(latent, torch.bfloat16, "latent"),
                                     _dev(slot_mapping, torch.int64, "slot_mapping"), int(t),
                                     _dev(status, torch.int32, "status"), _stream(stream)), "mla_cache_write")
    return cache


def mla_up_proj(latent, w_kvb, num_heads: int, k_out=None, v_out=None, status=None, stream=None):
    """latent [T, 576] x w_kvb [512, H*256] -> K [T, H, 192], V [T, H, 128]."""
    import torch
    t = latent.shape[0]
    if tuple(latent.shape[1:]) != (576,) or tuple(w_kvb.shape) != (512, num_heads * 256):
        raise ValueError("latent must be [T, 576] and w_kvb [512, H*256]")
    if k_out is None:
        k_out = torch.empty((t, num_heads, 192), dtype=torch.bfloat16, device=latent.device)
    if v_out is None:
        v_out = torch.empty((t, num_heads, 128), dtype=torch.bfloat16, device=latent.device)
    bf = torch.bfloat16
    _check(library().mla_up_proj(_dev(latent, bf, "latent"), _dev(w_kvb, bf, "w_kvb"), t, num_heads,
                                 _dev(k_out, bf, "k_out"), _dev(v_out, bf, "v_out"),
                                 _dev(status, torch.int32, "status"), _stream(stream)), "mla_up_proj")
    return k_out, v_out


def mla_up_proj_paged(cache, block_table, cu_seq_lens, chunk_starts, total_tokens: int, w_kvb, num_heads: int,
                      k_out=None, v_out=None, status=None, stream=None):
    """One prefix chunk decompressed straight from the paged cache [NB, BS, 576]:
    K [T, H, 192], V [T, H, 128] (T = total_tokens), as gather + up-projection would give."""
    import torch
    nb, bs, e = cache.shape
    t = int(total_tokens)
    if e != 576 or tuple(w_kvb.shape) != (512, num_heads * 256):
        raise ValueError("cache must be [NB, BS, 576] and w_kvb [512, H*256]")
    batch = block_table.shape[0]
    if tuple(cu_seq_lens.shape) != (batch + 1,) or tuple(chunk_starts.shape) != (batch,):
        raise ValueError("cu_seq_lens must be [B+1] and chunk_starts [B] for a block table of B rows")
    if k_out is None:
        k_out = torch.empty((t, num_heads, 192), dtype=torch.bfloat16, device=cache.device)
    if v_out is None:
        v_out = torch.empty((t, num_heads, 128), dtype=torch.bfloat16, device=cache.device)
    if tuple(k_out.shape) != (t, num_heads, 192) or tuple(v_out.shape) != (t, num_heads, 128):
        raise ValueError("k_out/v_out shapes do not match total_tokens and num_heads")
    bf, i32 = torch.bfloat16, torch.int32
    _check(library().mla_up_proj_paged(_dev(cache, bf, "cache"), nb, bs, e, _dev(block_table, i32, "block_table"),
                                       block_table.shape[1], _dev(cu_seq_lens, i32, "cu_seq_lens"),
                                       _dev(chunk_starts, i32, "chunk_starts"), batch, t, _dev(w_kvb, bf, "w_kvb"),
                                       num_heads, _dev(k_out, bf, "k_out"), _dev(v_out, bf, "v_out"),
                                       _dev(status, i32, "status"), _stream(stream)), "mla_up_proj_paged")
    return k_out, v_out


def mla_up_proj_paged_split(cache, block_table, cu_seq_lens, chunk_starts, total_tokens: int, w_kvb, num_heads: int,
                            k_nope_out=None, v_out=None, rope_out=None, status=None, stream=None):
    """mla_up_proj_paged with K split into K_nope [T, H, 128] and one rope row per token [T, 64]."""
    import torch
    nb, bs, e = cache.shape
    t = int(total_tokens)
    if e != 576 or tuple(w_kvb.shape) != (512, num_heads * 256):
        raise ValueError("cache must be [NB, BS, 576] and w_kvb [512, H*256]")
    batch = block_table.shape[0]
    if tuple(cu_seq_lens.shape) != (batch + 1,) or tuple(chunk_starts.shape) != (batch,):
        raise ValueError("cu_seq_lens must be [B+1] and chunk_starts [B] for a block table of B rows")
    bf, i32 = torch.bfloat16, torch.int32
    if k_nope_out is None:
        k_nope_out = torch.empty((t, num_heads, 128), dtype=bf, device=cache.device)
    if v_out is None:
        v_out = torch.empty((t, num_heads, 128), dtype=bf, device=cache.device)
    if rope_out is None:
        rope_out = torch.empty((t, 64), dtype=bf, device=cache.device)
    if (tuple(k_nope_out.shape) != (t, num_heads, 128) or tuple(v_out.shape) != (t, num_heads, 128)
            or tuple(rope_out.shape) != (t, 64)):
        raise ValueError("k_nope_out/v_out/rope_out shapes do not match total_tokens and num_heads")
    _check(library().mla_up_proj_paged_split(_dev(cache, bf, "cache"), nb, bs, e, _dev(block_table, i32, "block_table"),
                                             block_table.shape[1], _dev(cu_seq_lens, i32, "cu_seq_lens"),
                                             _dev(chunk_starts, i32, "chunk_starts"), batch, t,
                                             _dev(w_kvb, bf, "w_kvb"), num_heads, _dev(k_nope_out, bf, "k_nope_out"),
                                             _dev(v_out, bf, "v_out"), _dev(rope_out, bf, "rope_out"),
                                             _dev(status, i32, "status"), _stream(stream)), "mla_up_proj_paged_split")
    return k_nope_out, v_out, rope_out


def mla_merge_state(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """Merge two partial states by LSE; o_out/lse_out may be o_a/lse_a (in place)."""
    import torch
    rows, h, d = o_a.shape
    if tuple(o_b.shape) != (rows, h, d):
        raise ValueError(f"o_b must be {(rows, h, d)} like o_a, got {tuple(o_b.shape)}")
    if tuple(lse_a.shape) != (rows, h) or tuple(lse_b.shape) != (rows, h):
        raise ValueError(f"lse_a and lse_b must be {(rows, h)}")
    if o_out is not None and tuple(o_out.shape) != (rows, h, d):
        raise ValueError(f"o_out must be {(rows, h, d)}")
    if lse_out is not None and tuple(lse_out.shape) != (rows, h):
        raise ValueError(f"lse_out must be {(rows, h)}")
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    bf, f32 = torch.bfloat16, torch.float32
    _check(library().mla_merge_state(_dev(o_a, bf, "o_a"), _dev(lse_a, f32, "lse_a"), _dev(o_b, bf, "o_b"),
                                     _dev(lse_b, f32, "lse_b"), _dev(o_out, bf, "o_out"),
                                     _dev(lse_out, f32, "lse_out"), rows, h, d, _stream(stream)),
           "mla_merge_state")
    return o_out, lse_out


def mla_prefill_run_noalloc(qo_indptr, kv_indptr, num_heads: int, q, k, v, o, lse=None, *, causal: bool = True,
                            sm_scale: float, window_left: int = -1, logits_soft_cap: float = 0.0, status=None,
                            stream=None):
    """Plan + run without any device allocation by the library (outputs are caller-provided).

    For callers that cannot allocate device memory; the work list goes into a fixed
    array inside the library, so overlapping calls must be serialised by the caller."""
    import torch
    qo, kv = _host_i32(qo_indptr), _host_i32(kv_indptr)
    if qo.ndim != 1 or kv.shape != qo.shape or qo.size < 1:
        raise ValueError("qo_indptr and kv_indptr must be 1-D of equal length batch+1")
    total_q, total_kv = int(qo[-1]), int(kv[-1])
    H = int(num_heads)
    for t, shape, name in ((q, (total_q, H, 192), "q"), (k, (total_kv, H, 192), "k"), (v, (total_kv, H, 128), "v"),
                           (o, (total_q, H, 128), "o")):
        if t is None or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}, got {None if t is None else tuple(t.shape)}")
    if lse is not None and tuple(lse.shape) != (total_q, H):
        raise ValueError(f"lse must be [{total_q}, {H}], got {tuple(lse.shape)}")
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold at least one int32 word")
    bf = torch.bfloat16
    _check(library().mla_prefill_run_noalloc(
        _ptr(qo), _ptr(kv), qo.size - 1, num_heads, 192, 128, int(bool(causal)), float(sm_scale), int(window_left),
        float(logits_soft_cap), _dev(q, bf, "q"), _dev(k, bf, "k"), _dev(v, bf, "v"), _dev(o, bf, "o"),
        _dev(lse, torch.float32, "lse"), _dev(status, torch.int32, "status"), _stream(stream)),
        "mla_prefill_run_noalloc")
    return o, lse
