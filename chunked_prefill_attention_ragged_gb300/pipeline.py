"""Chunked prefill with a cached, compressed prefix, as a sequence of C-ABI calls.

vLLM "vllm.v1.attention.backends.mla.prefill.flashinfer",
FlashInferPrefillBackend.finalize_attention_metadata: one causal plan over the
new tokens (kv_indptr = qo_indptr) and one non-causal plan per prefix chunk
(kv_indptr = chunked_context.cu_seq_lens[i]), all sharing sm_scale,
window_left and logits_soft_cap; run_prefill_context_chunk returns each
chunk's LSE so the partial outputs can be merged.  sglang issue #3849: the
prefix lives in the paged cache as 512 latent + 64 rope per token and is
decompressed before attention.

Per run: new-token attention -> for every chunk: gather -> up-projection ->
non-causal attention -> in-place LSE merge into the running (O, LSE).  Every
step is a kernel of libmla_prefill.so; this class only owns buffers and
orders the calls on one stream.
"""
from __future__ import annotations

import numpy as np

from ._binding import (mla_gather_latent, mla_merge_state, mla_prefill_plan, mla_up_proj)


class ChunkedPrefill:
    """Plans once (host metadata + device work lists), runs per layer.

    qo_indptr: host [B+1]; cu_seq_lens: host [C, B+1] (chunk kv_indptrs);
    chunk_starts: host [C, B] (first prefix position of each chunk per request).
    """

    def __init__(self, qo_indptr, cu_seq_lens, chunk_starts, num_heads: int, *, sm_scale: float,
                 logits_soft_cap: float = 0.0, device="cuda", stream=None):
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
        t_max = max(self.chunk_tokens, default=0)
        h = num_heads
        bf = torch.bfloat16
        self.latent = torch.empty((max(t_max, 1), 576), dtype=bf, device=device)
        self.k_c = torch.empty((max(t_max, 1), h, 192), dtype=bf, device=device)
        self.v_c = torch.empty((max(t_max, 1), h, 128), dtype=bf, device=device)
        self.o_c = torch.empty((max(self.total_q, 1), h, 128), dtype=bf, device=device)
        self.lse_c = torch.empty((max(self.total_q, 1), h), dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def run(self, q, k, v, cache, block_table, w_kvb, o=None, lse=None, stream=None):
        """q/k/v: new tokens; cache [NB, BS, 576]; block_table [B, M] int32 (device)."""
        o, lse = self.main.run(q, k, v, o, lse, True, stream)
        for c, plan in enumerate(self.chunks):
            t = self.chunk_tokens[c]
            if t == 0:
                continue
            lat = self.latent[:t]
            mla_gather_latent(cache, block_table, self.cu_dev[c], self.starts_dev[c], t, lat, self.status, stream)
            kc, vc = self.k_c[:t], self.v_c[:t]
            mla_up_proj(lat, w_kvb, self.num_heads, kc, vc, self.status, stream)
            oc, lc = self.o_c[:self.total_q], self.lse_c[:self.total_q]
            plan.run(q, kc, vc, oc, lc, True, stream)
            mla_merge_state(o, lse, oc, lc, o, lse, stream)
        return o, lse

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
