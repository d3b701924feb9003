"""The allocation-free split forward against the workspace split forward.

paged_attn_forward_split_static serves callers that cannot give the library a
workspace (a host runtime that owns every device allocation, or a decode loop
that must not hit cudaMalloc's device-wide synchronisation): its split
partials live in a static device array inside the library.  This file checks,
through the C ABI, that two calls in a row -- different plans and shapes, so
the second call runs over the first one's leftovers -- give the same result as
paged_attn_forward_split with a caller workspace, within the bf16 tolerance of
the parity tests, and that an oversize request is refused.  It is collected
last and also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_attention_20_gb300 as pka
from helpers import HALF_ABS, plan_for
from workloads import build_case, decode_queries, gqa_decode_bf16

pytestmark = pytest.mark.gpu

PA_ERR_WORKSPACE = 6
SCRATCH_BYTES = 16 << 20


def _static_fn():
    lib = pka.load()
    fn = lib.paged_attn_forward_split_static
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, i32, i32, ctypes.c_int, i32, vp]
    fn.restype = ctypes.c_int
    return lib, fn


def _run_both(case, splits):
    lib, fn = _static_fn()
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    ref = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits)
    out = torch.full_like(ref, float("nan"))
    stream = torch.cuda.current_stream().cuda_stream
    rc = fn(plan.handle, dc.q.data_ptr(), dc.k_cache.data_ptr(), dc.v_cache.data_ptr(), out.data_ptr(),
            case.hq, case.hkv, case.d, case.dv, case.scale, 1, 0, 2, splits, stream)
    assert rc == 0, lib.pa_last_error().decode()
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), ref.float().cpu().numpy()


def test_static_scratch_matches_workspace_split(cuda_device):
    # first call: the GQA decode layer (64 queries, 32 heads, contexts up to 8K), 4 splits
    got, ref = _run_both(gqa_decode_bf16(), 4)
    assert np.isfinite(got).all()
    assert float(np.max(np.abs(got - ref))) <= HALF_ABS
    # second call in a row: another plan and shape over the same (now stale) scratch
    seq_lens = [1, 33, 700, 2500, 90]
    case = build_case("static2", 23, seq_lens, decode_queries(seq_lens), 16, 2, 128, 128, 16,
                      torch.bfloat16, 1 / math.sqrt(128))
    got, ref = _run_both(case, 7)
    assert np.isfinite(got).all()
    assert float(np.max(np.abs(got - ref))) <= HALF_ABS


def test_static_scratch_refuses_oversize(cuda_device):
    lib, fn = _static_fn()
    plan = pka.paged_attn_plan([64], [[0, 1, 2, 3]], [0], [63], 16, 4, device="cuda")
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check fails first
    # 1 query x 1024 heads x 1024 dims x 64 splits x 4 B = 256 MiB > 16 MiB
    assert pka.workspace_bytes(1, 1024, 1024, 64) > SCRATCH_BYTES
    rc = fn(plan.handle, fake, fake, fake, fake, 1024, 1024, 1024, 1024, 0.1, 1, 0, 2, 64, None)
    assert rc == PA_ERR_WORKSPACE
    assert "PA_STATIC_SCRATCH_BYTES" in lib.pa_last_error().decode()
