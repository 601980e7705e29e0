"""fp64 CPU oracle for MLA ragged prefill -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct restatement of what the CUDA path
computes, written from the pages' definitions:

  * ragged (varlen) multi-head attention with an explicit softmax scale,
    optional causal mask (bottom-right aligned), sliding window and logits
    soft cap, returning O and the per-row natural-log LSE
    (vLLM ``vllm.v1.attention.backends.mla.prefill.flashinfer``:
    ``finalize_attention_metadata`` plans ``prefill_main`` causal and
    ``prefill_chunks[i]`` non-causal; ``run_prefill_new_tokens`` /
    ``run_prefill_context_chunk`` return (O, LSE));
  * the paged latent gather (slot = block_table[req, pos // block_size] *
    block_size + pos % block_size, from the decode branch of
    ``_build_c128a_topk_metadata_kernel`` in vLLM's
    ``vllm/models/deepseek_v4/sparse_mla.py``);
  * the paged cache write of new tokens' compressed rows by slot mapping
    (negative slot = padding token, sglang issue #3849 / vLLM sparse_mla.py);
  * the latent up-projection into per-head K = [K_nope || k_rope] and V
    (sglang issue #3849: 512 latent + 64 rope cached, attention runs as MHA
    with 192-dim Q/K and 128-dim V);
  * the LSE merge of two partial attention states;
  * the fp8 latent cache entry (fp8 latent with power-of-two scales per 64
    values, bf16 rope; vLLM ``sparse_mla.py``'s ``fp8_ds_mla`` layout) and its
    dequantizing gather;
  * the unchunked attention that chunked prefill must reproduce;
  * absorbed-weight attention (multi-query over the 576-wide compressed rows,
    sglang issue #3849's forward_absorb; explicit sm_scale per TVM PR #17674).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
and never imports it; its inputs come from the seeded generators in
``chunked_prefill_attention_ragged_gb300.workloads`` (as bf16 bit patterns)
or from hand-written fixtures.

Every function here is pinned by ``-m "not gpu"`` tests against brute force,
closed forms and invariants.  Parity pins: attention (brute force, closed
forms, invariants), gather (hand fixture + brute force), cache write (hand
fixture, round trip through the gather, padding slots), up-projection
(hand fixture + triple loop), merge (closed forms + split/merge identity),
chunked pipeline (split/merge identity), absorbed attention (the
absorption identity against the MHA oracle over decompressed K/V, brute force),
fp8 entries (hand-decoded codes, every
e4m3 code against the library's float8 type, exact products).  No function is "parity unpinned".
"""
from .bf16 import bf16_bits_to_f64, round_f64_to_bf16
from .attention import allowed_mask, attend_request, ragged_attention
from .gather import gather_latent, slot_of
from .cache_write import cache_write
from .up_proj import up_project
from .merge import merge_state
from .chunked import chunked_prefill_attention
from .absorbed import absorb_query, absorbed_attention, absorbed_output_to_mha
from .fp8_cache import (dequant_fp8_entries, e4m3_to_f64, f64_to_bf16_bits, gather_latent_fp8,
                        ue8m0_to_f64)

__all__ = [
    "bf16_bits_to_f64", "round_f64_to_bf16", "allowed_mask", "attend_request",
    "ragged_attention", "gather_latent", "slot_of", "cache_write", "up_project", "merge_state",
    "chunked_prefill_attention", "dequant_fp8_entries", "e4m3_to_f64", "f64_to_bf16_bits",
    "gather_latent_fp8", "ue8m0_to_f64", "absorb_query", "absorbed_attention", "absorbed_output_to_mha",
]
