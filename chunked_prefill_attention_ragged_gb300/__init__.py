"""GB300-native (sm_103a) MLA ragged prefill attention.

The compute lives in ``libmla_prefill.so`` (C ABI in ``include/mla_prefill.h``):
hand-written tcgen05/TMA kernels for ragged causal and non-causal attention with
LSE, the paged latent gather and cache write, the latent up-projection and the
LSE merge, and the absorbed-weight (MQA over the latent) prefill.  This package is a thin ctypes binding with the same entry-point
names, plus the seeded workload generators.  Importing it loads nothing; the first call builds
(if needed) and loads the library, and raises if that fails.
"""
from ._binding import (EXPORTED, AbsorbedPlan, MlaError, PrefillPlan, error_string, library, library_path,
                       mla_absorbed_plan, mla_absorbed_run,
                       mla_cache_write, mla_gather_latent, mla_gather_latent_fp8, mla_merge_state, mla_plan_destroy, mla_plan_units_host,
                       mla_prefill_plan, mla_prefill_run, mla_prefill_run_merge, mla_prefill_run_noalloc,
                       mla_prefill_run_shared_rope, mla_prefill_status, mla_up_proj, mla_up_proj_paged,
                       mla_up_proj_paged_split)

__all__ = [
    "EXPORTED", "AbsorbedPlan", "MlaError", "PrefillPlan", "error_string", "library", "library_path",
    "mla_absorbed_plan", "mla_absorbed_run",
    "mla_cache_write", "mla_gather_latent", "mla_gather_latent_fp8", "mla_merge_state", "mla_plan_destroy", "mla_plan_units_host",
    "mla_prefill_plan", "mla_prefill_run", "mla_prefill_run_merge", "mla_prefill_run_noalloc", "mla_prefill_status",
    "mla_up_proj",
    "mla_up_proj_paged", "mla_up_proj_paged_split", "mla_prefill_run_shared_rope",
]
