"""Paged latent gather, written as plain loops (test infrastructure only).

Addressing rule: vLLM ``vllm/models/deepseek_v4/sparse_mla.py``,
``_build_c128a_topk_metadata_kernel``, decode branch: a token at position p
of request r lives in physical block ``block_table[r, p // block_size]`` at
offset ``p % block_size``, i.e. flat slot ``block * block_size + offset``.

What is gathered: sglang issue #3849 ("[DeepseekR1] How ragged prefill
manage kv_cache?"): the cache keeps one compressed row per token (512 latent
then 64 rope); chunked prefill pulls a prefix chunk out of it before
decompressing.

Chunk convention (vLLM ``finalize_attention_metadata``: chunk i's kv_indptr
is ``chunked_context.cu_seq_lens[i]``): output row ``cu_seq_lens[r] + t``
holds prefix position ``chunk_starts[r] + t`` of request r, for
t < cu_seq_lens[r+1] - cu_seq_lens[r].
"""
import numpy as np


def slot_of(block_table: np.ndarray, r: int, pos: int, block_size: int) -> int:
    """Flat cache slot of prefix position ``pos`` of request ``r``."""
    block = int(block_table[r, pos // block_size])
    return block * block_size + pos % block_size


def gather_latent(cache: np.ndarray, block_table: np.ndarray, cu_seq_lens: np.ndarray,
                  chunk_starts: np.ndarray) -> np.ndarray:
    """Copy one prefix chunk out of the paged cache.

    cache: [num_blocks, block_size, E]; block_table: [B, max_blocks];
    cu_seq_lens: [B+1]; chunk_starts: [B].  Returns [cu_seq_lens[B], E] with
    the cache's dtype (a bit copy).
    """
    num_blocks, block_size, e = cache.shape
    flat = cache.reshape(num_blocks * block_size, e)
    cu = [int(c) for c in cu_seq_lens]
    out = np.zeros((cu[-1], e), dtype=cache.dtype)
    for r in range(len(cu) - 1):
        for t in range(cu[r + 1] - cu[r]):
            out[cu[r] + t] = flat[slot_of(block_table, r, int(chunk_starts[r]) + t, block_size)]
    return out
