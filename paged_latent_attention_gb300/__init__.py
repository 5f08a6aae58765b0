"""paged_latent_attention_gb300: gated MLA decode over a flat paged KV pool on GB300.

The compute path is the CUDA library libplmla.so (C ABI in include/plmla.h);
this package only marshals torch tensors into it.
"""
from .api import (  # noqa: F401
    DEFAULT_SCALE,
    allocate_workspace,
    device_status,
    get_page_checks,
    get_split_mode,
    get_team_clusters,
    mla_dcp_shard,
    mla_decode,
    mla_decode_fp8,
    mla_decode_layers,
    mla_kv_append,
    mla_kv_append_fp8,
    mla_merge_partials,
    mla_plan_splits,
    mla_quantize_queries_fp8,
    mla_split_budget,
    mla_split_combine,
    mla_workspace_size,
    mla_workspace_size_fp8,
    set_page_checks,
    set_split_mode,
    set_team_clusters,
)
