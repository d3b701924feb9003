"""Dependent calls issued back to back, with no synchronisation between them.

Every kernel of the library may start before the kernel ahead of it in the
stream has finished (programmatic dependent launch) and waits for it before
touching memory; these tests issue chains whose every step depends on the one
before and read the results only at the end: a decode loop (the schedule
advanced on the device, the new rows appended, attention over them) for a
CUDA-core and a tensor-core group size, and a mixed prefill + decode plan whose
appended rows change from call to call.  Each step is compared with the fp64
oracle (ruDNN 0.1.7, src/paged_attention/mod.rs: `append_with_report`, then
`DevicePlan::attention`).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import assert_close
from workloads import build_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("hq,hkv,splits", [(16, 4, 3), (64, 8, 5)])
def test_decode_loop_without_syncs(cuda_device, hq, hkv, splits):
    ctx0 = [40, 300, 129, 1000]
    steps = 5
    final = [c + steps for c in ctx0]
    queries = [(s, c - 1) for s, c in enumerate(ctx0)]
    case = build_case("b2b", 101, final, queries, hq, hkv, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    gen = torch.Generator().manual_seed(5)
    step_k = [torch.randn(len(ctx0), hkv, 128, generator=gen).bfloat16() for _ in range(steps)]
    step_v = [torch.randn(len(ctx0), hkv, 128, generator=gen).bfloat16() for _ in range(steps)]
    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos, case.page_size,
                               case.num_pages, device=dev)
    ks = [k.to(dev) for k in step_k]
    vs = [v.to(dev) for v in step_v]
    ws = pka.make_workspace(plan, hq, 128, splits)
    outs = []
    torch.cuda.synchronize()
    for i in range(steps):          # nothing waits for the GPU inside this loop
        pka.paged_attn_plan_advance(plan)
        pka.paged_kv_store(plan, ks[i], vs[i], dc.k_cache, dc.v_cache)
        outs.append(pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits,
                                                 workspace=ws))
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    kc, vc = case.k_cache.clone(), case.v_cache.clone()
    for i in range(steps):
        pos = np.array([c - 1 + i + 1 for c in ctx0], dtype=np.int32)
        kc, vc = oracle.kv_store(step_k[i], step_v[i], kc, vc, case.block_table, case.query_seq, pos)
        ref, _ = oracle.attention(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq, pos, case.scale)
        assert_close(outs[i].cpu().double().numpy(), ref, torch.bfloat16, f"step {i} G={hq // hkv}")


def test_mixed_plan_restored_between_calls(cuda_device):
    """A prefill chunk + decode queries; each call appends different rows, then attends."""
    seq_lens = [400, 700, 90]
    queries = [(0, 100 + i) for i in range(300)] + [(1, 699), (2, 89)]
    case = build_case("b2b_mixed", 102, seq_lens, queries, 16, 4, 128, 128, 16, torch.bfloat16,
                      1 / math.sqrt(128))
    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos, case.page_size,
                               case.num_pages, device=dev)
    assert plan.n_tiles > 0 and plan.n_decode > 0
    gen = torch.Generator().manual_seed(6)
    news = [(torch.randn(case.num_queries, 4, 128, generator=gen).bfloat16(),
             torch.randn(case.num_queries, 4, 128, generator=gen).bfloat16()) for _ in range(3)]
    outs = []
    torch.cuda.synchronize()
    for k, v in news:
        pka.paged_kv_store(plan, k.to(dev), v.to(dev), dc.k_cache, dc.v_cache)
        outs.append(pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale))
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    for i, (k, v) in enumerate(news):
        kc, vc = oracle.kv_store(k, v, case.k_cache, case.v_cache, case.block_table, case.query_seq, case.query_pos)
        ref, _ = oracle.attention(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                                  case.scale)
        assert_close(outs[i].cpu().double().numpy(), ref, torch.bfloat16, f"call {i}")
