"""Operands that are not this GPU's device memory are refused before launch.

The kernels' TMA tensor maps and loads address only the current GPU's own
memory (ruDNN 0.1.7, src/paged_attention/mod.rs, `check_tensor`: every operand
on Q's device).  Through the C ABI, a pinned host buffer passed as a cache,
as q, as the output or as the workspace -- on a plan with prefill tiles (the
tensor-core prefill kernel), a decode plan and an MLA plan -- must return
PA_ERR_ARG, leave the output untouched and launch nothing (the device status
word stays clear).
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_attention_20_gb300 as pka
from helpers import plan_for
from workloads import build_case, decode_queries

pytestmark = pytest.mark.gpu

PA_ERR_ARG = 1


def _mixed_case():
    lens = [400, 90]
    queries = [(0, 200 + i) for i in range(150)] + [(1, 89)]
    return build_case("ptr_mixed", 41, lens, queries, 16, 4, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))


def test_pinned_host_operands_are_refused(cuda_device):
    lib = pka.load()
    for case in (_mixed_case(), build_case("ptr_decode", 42, [70, 300], decode_queries([70, 300]), 32, 8, 128, 128,
                                           16, torch.bfloat16, 1 / math.sqrt(128))):
        dc = case.to("cuda")
        plan = plan_for(case)
        out = torch.full((case.num_queries, case.hq, case.dv), float("nan"), dtype=case.dtype, device="cuda")
        host_k = case.k_cache.pin_memory()
        host_q = case.q.pin_memory()
        host_out = torch.empty_like(out, device="cpu").pin_memory()
        stream = torch.cuda.current_stream().cuda_stream
        torch.cuda.synchronize()
        for q, k, o, what in ((dc.q, host_k, out, "k_cache"), (host_q, dc.k_cache, out, "q"),
                              (dc.q, dc.k_cache, host_out, "out")):
            rc = lib.paged_attn_forward(plan.handle, q.data_ptr(), k.data_ptr(), dc.v_cache.data_ptr(),
                                        o.data_ptr(), case.hq, case.hkv, case.d, case.dv, case.scale, 1, 0, 2, stream)
            assert rc == PA_ERR_ARG, (case.name, what, rc)
            assert "device memory" in lib.pa_last_error().decode()
        # the split form: a pinned host workspace
        ws = torch.empty(pka.workspace_bytes(case.num_queries, case.hq, case.dv, 3), dtype=torch.uint8).pin_memory()
        rc = lib.paged_attn_forward_split(plan.handle, dc.q.data_ptr(), dc.k_cache.data_ptr(), dc.v_cache.data_ptr(),
                                          out.data_ptr(), case.hq, case.hkv, case.d, case.dv, case.scale, 1, 0, 2,
                                          ws.data_ptr(), ws.numel(), 3, stream)
        assert rc == PA_ERR_ARG
        # the append into a pinned host cache
        rc = lib.paged_kv_store(plan.handle, dc.new_k.data_ptr(), dc.new_v.data_ptr(), host_k.data_ptr(),
                                dc.v_cache.data_ptr(), case.hkv, case.d, case.dv, 2, stream)
        assert rc == PA_ERR_ARG
        torch.cuda.synchronize()
        assert torch.isnan(out.float()).all(), "a refused call wrote the output"
        assert pka.device_status() == 0


def test_pinned_host_mla_cache_is_refused(cuda_device):
    lib = pka.load()
    lens = [70, 300]
    case = build_case("ptr_mla", 43, lens, decode_queries(lens), 128, 1, 512, 64, 64, torch.bfloat16,
                      1 / math.sqrt(192), mla_p=64)
    dc = case.to("cuda")
    plan = plan_for(case)
    out = torch.full((case.num_queries, case.hq, case.d), float("nan"), dtype=case.dtype, device="cuda")
    host_lat = case.k_cache.pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.paged_mla_forward(plan.handle, dc.q.data_ptr(), dc.qp.data_ptr(), host_lat.data_ptr(),
                               dc.v_cache.data_ptr(), out.data_ptr(), case.hq, case.d, case.p, case.scale, 1, 0, 2,
                               None, 0, 1, stream)
    assert rc == PA_ERR_ARG
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
    # and the same call on device memory runs
    rc = lib.paged_mla_forward(plan.handle, dc.q.data_ptr(), dc.qp.data_ptr(), dc.k_cache.data_ptr(),
                               dc.v_cache.data_ptr(), out.data_ptr(), case.hq, case.d, case.p, case.scale, 1, 0, 2,
                               None, 0, 1, stream)
    assert rc == 0, lib.pa_last_error().decode()
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and pka.device_status() == 0
