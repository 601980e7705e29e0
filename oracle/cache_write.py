"""Paged latent cache write by slot mapping, written as a plain loop (test infrastructure only).

What is written: sglang issue #3849 ("[DeepseekR1] How ragged prefill manage
kv_cache?"): ragged prefill saves the new tokens' compressed rows (512 latent
then 64 rope) into the paged cache before attention runs.

Where: vLLM ``vllm/models/deepseek_v4/sparse_mla.py``: each token carries a flat
cache slot in ``slot_mapping`` (``block * block_size + offset``, the same flat
index the gather reads through ``slot_of``); in the decode branch of
``_build_c128a_topk_metadata_kernel`` a token is valid when its slot is >= 0,
so a negative slot marks a padding token, which writes nothing.

Reading taken where the pages are silent: if two tokens name the same slot, the
later token's row is what the oracle leaves there (a sequential loop); the GPU
path may leave either, so tests compare such slots against both candidates.
"""
import numpy as np


def cache_write(cache: np.ndarray, latent: np.ndarray, slot_mapping: np.ndarray) -> np.ndarray:
    """Return a copy of ``cache`` [num_blocks, block_size, E] with row ``t`` of
    ``latent`` [T, E] stored at flat slot ``slot_mapping[t]`` for every token whose
    slot is >= 0.  Slots past the cache are an error here (the kernel skips and flags
    them)."""
    num_blocks, block_size, e = cache.shape
    assert latent.shape == (len(slot_mapping), e)
    out = cache.copy()
    flat = out.reshape(num_blocks * block_size, e)
    for t, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        assert slot < num_blocks * block_size, "slot past the cache"
        flat[slot] = latent[t]
    return out
