"""Chunked prefill with a cached, compressed prefix, as a sequence of C-ABI calls.

vLLM "vllm.v1.attention.backends.mla.prefill.flashinfer",
FlashInferPrefillBackend.finalize_attention_metadata: one causal plan over the
new tokens (kv_indptr = qo_indptr) and one non-causal plan per prefix chunk
(kv_indptr = chunked_context.cu_seq_lens[i]), all sharing sm_scale,
window_left and logits_soft_cap; run_prefill_context_chunk returns each
chunk's LSE so the partial outputs can be merged.  sglang issue #3849: the
prefix lives in the paged cache as 512 latent + 64 rope per token and is
decompressed before attention.

Per run: new-token attention -> for every chunk: the chunk's K/V decompressed
straight out of the paged cache (mla_up_proj_paged_split: gather and
up-projection in one kernel, no gathered latent buffer, K as per-head K_nope
plus one rope row per token, since every head's K carries the same rope) ->
non-causal attention merged into the running (O, LSE) by the attention
kernel's epilogue (mla_prefill_run_shared_rope with merge).
Variants, the same result up to rounding: with paged_up_proj=False one gather
of every chunk's latent rows (one launch, large enough to run near HBM
bandwidth) feeds mla_up_proj; with fuse_merge=False the attention writes its
own O/LSE and mla_merge_state merges them.  With cache_fp8=True the cache holds
648-byte fp8 entries (vLLM sparse_mla.py's fp8_ds_mla layout, see
mla_gather_latent_fp8): one dequantizing gather of every chunk feeds
mla_up_proj.  Chunking bounds the decompressed
K/V (per chunk tokens x heads x 640 bytes).  Every step is a kernel of
libmla_prefill.so; this class only owns buffers and orders the calls on one
stream.
"""
from __future__ import annotations

import numpy as np

from ._binding import (mla_gather_latent, mla_gather_latent_fp8, mla_merge_state, mla_prefill_plan,
                       mla_prefill_run_shared_rope, mla_up_proj, mla_up_proj_paged, mla_up_proj_paged_split)


class ChunkedPrefill:
    """Plans once (host metadata + device work lists), runs per layer.

    qo_indptr: host [B+1]; cu_seq_lens: host [C, B+1] (chunk kv_indptrs);
    chunk_starts: host [C, B] (first prefix position of each chunk per request).
    """

    def __init__(self, qo_indptr, cu_seq_lens, chunk_starts, num_heads: int, *, sm_scale: float,
                 logits_soft_cap: float = 0.0, device="cuda", stream=None, fuse_merge: bool = True,
                 paged_up_proj: bool = True, cache_fp8: bool = False):
        import torch
        self.num_heads = num_heads
        qo = np.asarray(qo_indptr, dtype=np.int32)
        cu = np.atleast_2d(np.asarray(cu_seq_lens, dtype=np.int32))
        st = np.atleast_2d(np.asarray(chunk_starts, dtype=np.int32))
        self.qo = qo
        self.cu = cu
        self.total_q = int(qo[-1])
        self.main = mla_prefill_plan(qo, qo, num_heads, causal=True, sm_scale=sm_scale,
                                     logits_soft_cap=logits_soft_cap, stream=stream)
        self.chunks = [mla_prefill_plan(qo, cu[c], num_heads, causal=False, sm_scale=sm_scale,
                                        logits_soft_cap=logits_soft_cap, stream=stream)
                       for c in range(cu.shape[0])]
        self.chunk_tokens = [int(cu[c, -1]) for c in range(cu.shape[0])]
        self.cu_dev = torch.from_numpy(cu.copy()).to(device)
        self.starts_dev = torch.from_numpy(st.copy()).to(device)
        # All chunks in one gather: (chunk, request) pairs become the rows' "requests",
        # chunk c's rows are latent[row0[c] : row0[c] + chunk_tokens[c]], and the block
        # table is repeated once per chunk.
        n_chunks, batch = cu.shape[0], cu.shape[1] - 1
        self.num_chunks, self.batch = n_chunks, batch
        self.row0 = [0]
        for t in self.chunk_tokens:
            self.row0.append(self.row0[-1] + t)
        lens_all = np.diff(cu, axis=1).reshape(-1)
        cu_all = np.zeros(n_chunks * batch + 1, dtype=np.int32)
        np.cumsum(lens_all, out=cu_all[1:])
        self.cu_all_dev = torch.from_numpy(cu_all).to(device)
        self.starts_all_dev = torch.from_numpy(st.reshape(-1).astype(np.int32).copy()).to(device)
        self.total_prefix = int(cu_all[-1])
        self.table_all = None
        self._table_key = None
        t_max = max(self.chunk_tokens, default=0)
        h = num_heads
        bf = torch.bfloat16
        self.cache_fp8 = bool(cache_fp8)
        self.paged_up_proj = bool(paged_up_proj) and not self.cache_fp8
        self.latent = None if self.paged_up_proj else torch.empty((max(self.total_prefix, 1), 576), dtype=bf,
                                                                   device=device)
        # K of a chunk: [T, H, 192], or with the shared rope K_nope [T, H, 128] + rope [T, 64]
        self.shared_rope = self.paged_up_proj
        self.k_c = torch.empty((max(t_max, 1), h, 128 if self.shared_rope else 192), dtype=bf, device=device)
        self.rope_c = torch.empty((max(t_max, 1), 64), dtype=bf, device=device) if self.shared_rope else None
        self.v_c = torch.empty((max(t_max, 1), h, 128), dtype=bf, device=device)
        self.fuse_merge = bool(fuse_merge)
        if self.fuse_merge:
            self.o_c = self.lse_c = None
        else:
            self.o_c = torch.empty((max(self.total_q, 1), h, 128), dtype=bf, device=device)
            self.lse_c = torch.empty((max(self.total_q, 1), h), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def chunk_table(self, block_table):
        """The block table repeated once per chunk (rows of the one gather launch).

        Rebuilt only when the caller's table changed (another tensor, or written in
        place since the last call), so layers that share a batch's table pay once."""
        import torch
        key = (block_table.data_ptr(), block_table._version, tuple(block_table.shape), block_table.device)
        if self.table_all is not None and key == self._table_key:
            return self.table_all
        shape = (self.num_chunks * self.batch, block_table.shape[1])
        self.table_all = torch.empty(shape, dtype=torch.int32, device=block_table.device)
        self.table_all.view(self.num_chunks, self.batch, -1).copy_(block_table.unsqueeze(0).expand(
            self.num_chunks, -1, -1))
        self._table_key = key
        return self.table_all

    def gather_all(self, cache, block_table, stream=None):
        """Every chunk's latent rows, one launch: self.latent[row0[c]:row0[c+1]] is chunk c."""
        import torch
        if self.latent is None:
            self.latent = torch.empty((max(self.total_prefix, 1), 576), dtype=torch.bfloat16, device=cache.device)
        if self.total_prefix:
            gather = mla_gather_latent_fp8 if self.cache_fp8 else mla_gather_latent
            gather(cache, self.chunk_table(block_table), self.cu_all_dev, self.starts_all_dev, self.total_prefix,
                   self.latent[:self.total_prefix], self.status, stream)
        return self.latent

    def run(self, q, k, v, cache, block_table, w_kvb, o=None, lse=None, stream=None):
        """q/k/v: new tokens; cache [NB, BS, 576] bf16 (or [NB, BS, 648] uint8 with cache_fp8);
        block_table [B, M] int32 (device)."""
        o, lse = self.main.run(q, k, v, o, lse, True, stream)
        if not self.paged_up_proj:
            self.gather_all(cache, block_table, stream)
        for c, plan in enumerate(self.chunks):
            t = self.chunk_tokens[c]
            if t == 0:
                continue
            kc, vc = self.k_c[:t], self.v_c[:t]
            self.decompress(c, cache, block_table, w_kvb, kc, vc, stream)
            self.chunk_attention(c, q, o, lse, stream)
        return o, lse

    def chunk_attention(self, c, q, o, lse, stream=None):
        """Chunk c's non-causal attention over its decompressed K/V, merged into (o, lse)."""
        t, plan = self.chunk_tokens[c], self.chunks[c]
        kc, vc = self.k_c[:t], self.v_c[:t]
        if self.fuse_merge:
            if self.shared_rope:
                mla_prefill_run_shared_rope(plan, q, kc, self.rope_c[:t], vc, o, lse, True, stream)
            else:
                plan.run_merge(q, kc, vc, o, lse, stream)
        else:
            oc, lc = self.o_c[:self.total_q], self.lse_c[:self.total_q]
            if self.shared_rope:
                mla_prefill_run_shared_rope(plan, q, kc, self.rope_c[:t], vc, oc, lc, False, stream)
            else:
                plan.run(q, kc, vc, oc, lc, True, stream)
            mla_merge_state(o, lse, oc, lc, o, lse, stream)

    def decompress(self, c, cache, block_table, w_kvb, kc, vc, stream=None):
        """Chunk c's K and V [T, H, 128] into kc, vc (K [T, H, 192], or K_nope [T, H, 128] with
        the rope rows in self.rope_c when the rope is shared)."""
        t = self.chunk_tokens[c]
        if self.shared_rope:
            mla_up_proj_paged_split(cache, block_table, self.cu_dev[c], self.starts_dev[c], t, w_kvb, self.num_heads,
                                    kc, vc, self.rope_c[:t], self.status, stream)
        elif self.paged_up_proj:
            mla_up_proj_paged(cache, block_table, self.cu_dev[c], self.starts_dev[c], t, w_kvb, self.num_heads, kc, vc,
                              self.status, stream)
        else:
            lat = self.latent[self.row0[c]:self.row0[c] + t]
            mla_up_proj(lat, w_kvb, self.num_heads, kc, vc, self.status, stream)

    def check_status(self):
        """Raise if any kernel of the pipeline reported a device-side problem."""
        from ._binding import MlaError
        word = int(self.status.item())
        if word:
            self.status.zero_()
            raise MlaError(-5 if word & 1 else -6, "chunked prefill pipeline")
        self.main.status()
        for p in self.chunks:
            p.status()
