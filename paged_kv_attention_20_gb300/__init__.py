"""GB300-native paged attention over a block-table KV cache.

Python face of libpagedattn.so (C ABI declared in include/paged_attn.h).  The
functions carry the C names and only marshal arguments; all work runs in the
library's sm_103a kernels:

    paged_attn_plan           build + upload a schedule (per-query seq/pos/slot, work lists)
    paged_kv_store            append new K/V rows at the plan's slots (bit-exact copy)
    paged_attn_forward        paged MHA/GQA attention (decode + chunked causal prefill)
    paged_attn_forward_split  split-KV form with an fp32 LSE-merge workspace
    paged_mla_forward         MLA over a shared latent head + rotated position cache
    paged_attn_split_heuristic, paged_attn_decode_sms_beside_prefill, workspace_bytes,
    make_workspace, device_status
"""
from ._binding import (EXPORTED, MAX_SPLITS, PagedAttentionError, Plan, device_status, lib_path, load,
                       make_workspace, paged_attn_decode_sms_beside_prefill, paged_attn_forward,
                       paged_attn_forward_split, paged_attn_plan, paged_attn_plan_advance,
                       paged_attn_split_heuristic, paged_kv_store, paged_mla_forward, paged_mla_split_heuristic,
                       time_next_kernel, workspace_bytes)
from .buildlib import build

__all__ = ["EXPORTED", "MAX_SPLITS", "PagedAttentionError", "Plan", "build", "device_status", "lib_path",
           "load", "make_workspace", "paged_attn_decode_sms_beside_prefill", "paged_attn_forward",
           "paged_attn_forward_split", "paged_attn_plan",
           "paged_attn_plan_advance",
           "paged_attn_split_heuristic", "paged_kv_store", "paged_mla_forward", "paged_mla_split_heuristic",
           "time_next_kernel", "workspace_bytes"]
