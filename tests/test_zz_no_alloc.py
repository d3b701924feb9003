"""The allocation-free split forward against the fp64 oracle.

paged_attn_forward_split_static serves callers that cannot give the library a
workspace (a host runtime that owns every device allocation, or a decode loop
that must not hit cudaMalloc's device-wide synchronisation): its split
partials live in a static device array inside the library, which keeps
whatever the previous call left there.  This file calls it through the C ABI
three times in a row -- the GQA decode layer, then another decode plan and
shape over the first call's leftovers, then a mixed plan whose prefill tiles
write their split partials (rows with no key in a split included) into the
same array -- and checks each output against the oracle within the bf16
tolerance of the parity tests, and against the workspace form of the call.  An
oversize request is refused, and an invalid call gets the status the
workspace form gives even when its size would not fit.  It is collected last
and also passes on its own in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, oracle_after_store, plan_for
from workloads import build_case, decode_queries, gqa_decode_bf16

pytestmark = pytest.mark.gpu

PA_ERR_DTYPE = 3
PA_ERR_WORKSPACE = 6
SCRATCH_BYTES = 16 << 20


def _static_fn():
    lib = pka.load()
    fn = lib.paged_attn_forward_split_static
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, i32, i32, ctypes.c_int, i32, vp]
    fn.restype = ctypes.c_int
    return lib, fn


def _check_static(case, splits, rows=None, window=0):
    lib, fn = _static_fn()
    assert pka.workspace_bytes(case.num_queries, case.hq, case.dv, splits) <= SCRATCH_BYTES
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    out = torch.full((case.num_queries, case.hq, case.dv), float("nan"), dtype=case.dtype, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = fn(plan.handle, dc.q.data_ptr(), dc.k_cache.data_ptr(), dc.v_cache.data_ptr(), out.data_ptr(),
            case.hq, case.hkv, case.d, case.dv, case.scale, 1, window, 2, splits, stream)
    assert rc == 0, lib.pa_last_error().decode()
    ws_out = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits, window=window)
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    got = out.double().cpu().numpy()
    ref, _, _, _ = oracle_after_store(case, rows=rows, window=window)
    flat = got.reshape(-1, case.dv)
    if rows is not None:
        flat = flat[np.asarray(rows)]
    assert_close(flat, ref.reshape(flat.shape), case.dtype, f"{case.name} static split {splits}")
    # the workspace form runs the same kernels on the same partition: the same bits
    assert torch.equal(out.cpu().view(torch.int16), ws_out.cpu().view(torch.int16))


def test_static_scratch_matches_oracle_three_calls(cuda_device):
    # 1: the GQA decode layer (64 queries, 32 heads, contexts up to 8K), 4 splits, sampled rows
    case = gqa_decode_bf16()
    rng = np.random.default_rng(11)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=256, replace=False))
    _check_static(case, 4, rows=rows)
    # 2: another decode plan and shape over the first call's leftovers, 7 splits
    seq_lens = [1, 33, 700, 2500, 90]
    case = build_case("static2", 23, seq_lens, decode_queries(seq_lens), 16, 2, 128, 128, 16,
                      torch.bfloat16, 1 / math.sqrt(128))
    _check_static(case, 7)
    # 3: prefill tiles and decode items with 5 splits: the chunk starts at
    # position 0, so its first rows see fewer keys than 5 page-rounded splits
    # cover and their last splits are empty (lse = -inf written over the
    # stale array); then the same plan under a sliding window
    lens = [300, 1200, 50]
    queries = [(0, i) for i in range(160)] + [(1, 1199), (2, 49)]
    case = build_case("static3", 31, lens, queries, 16, 4, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    _check_static(case, 5)
    _check_static(case, 3, window=200)


def test_static_scratch_refuses_oversize(cuda_device):
    lib, fn = _static_fn()
    plan = pka.paged_attn_plan([64], [[0, 1, 2, 3]], [0], [63], 16, 4, device="cuda")
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check fails first
    # 1 query x 1024 heads x 1024 dims x 64 splits x 4 B = 256 MiB > 16 MiB
    assert pka.workspace_bytes(1, 1024, 1024, 64) > SCRATCH_BYTES
    rc = fn(plan.handle, fake, fake, fake, fake, 1024, 1024, 1024, 1024, 0.1, 1, 0, 2, 64, None)
    assert rc == PA_ERR_WORKSPACE
    assert "PA_STATIC_SCRATCH_BYTES" in lib.pa_last_error().decode()
    # an invalid dtype is reported as such, although the size would not fit either
    rc = fn(plan.handle, fake, fake, fake, fake, 1024, 1024, 1024, 1024, 0.1, 1, 0, 7, 64, None)
    assert rc == PA_ERR_DTYPE
