"""A captured decode step replayed with a device-resident schedule.

libmir-cuda 0.1.0, src/backend/attention/graph/mod.rs captures one decode
attention layer (store, then attention) into a CUDA graph; boostr 0.1.0,
src/inference/decode_graph.rs keeps the per-step scalars (write position
seq_len, attention length seq_len + 1) in device memory so one graph replays
the loop without re-capture.  Here the graph holds pa_plan_advance +
paged_kv_store + paged_attn_forward; each replay moves every query one
position on, appends that step's rows and attends, and every step is checked
against the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, oracle_after_store
from workloads import build_case, decode_queries

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("split", [False, True])
def test_captured_decode_step_replays(cuda_device, split):
    ctx0 = [30, 77, 128, 200]          # keys present before the first replayed step
    steps = 6
    final = [c + steps for c in ctx0]  # pages are reserved up to here
    queries = [(s, c - 1) for s, c in enumerate(ctx0)]
    case = build_case("graph", 41, final, queries, 16, 4, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    gen = torch.Generator().manual_seed(9)
    step_k = [torch.randn(4, 4, 128, generator=gen).bfloat16() for _ in range(steps)]
    step_v = [torch.randn(4, 4, 128, generator=gen).bfloat16() for _ in range(steps)]

    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                               case.page_size, case.num_pages, device=dev)
    new_k = torch.empty(4, 4, 128, dtype=torch.bfloat16, device=dev)
    new_v = torch.empty_like(new_k)
    out = torch.empty(4, 16, 128, dtype=torch.bfloat16, device=dev)
    ws = pka.make_workspace(plan, 16, 128, 3) if split else None

    def attend():
        if split:
            pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, 3, workspace=ws, out=out)
        else:
            pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, out=out)

    attend()                           # one plain call first (kernel attributes are set outside capture)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pka.paged_attn_plan_advance(plan)
        pka.paged_kv_store(plan, new_k, new_v, dc.k_cache, dc.v_cache)
        attend()

    kc_ref, vc_ref = case.k_cache.clone(), case.v_cache.clone()
    for step in range(steps):
        new_k.copy_(step_k[step])
        new_v.copy_(step_v[step])
        graph.replay()
        torch.cuda.synchronize()
        assert pka.device_status() == 0
        pos = np.array([c - 1 + step + 1 for c in ctx0], dtype=np.int32)
        kc_ref, vc_ref = oracle.kv_store(step_k[step], step_v[step], kc_ref, vc_ref, case.block_table,
                                         case.query_seq, pos)
        ref, _ = oracle.attention(case.q, kc_ref, vc_ref, case.seq_lens, case.block_table, case.query_seq,
                                  pos, case.scale)
        assert_close(out.cpu().double().numpy(), ref, torch.bfloat16, f"replay step {step}")


def test_advance_past_reserved_pages_is_flagged(cuda_device):
    # one sequence filling its only page; the next position has no page
    plan = pka.paged_attn_plan([16], [[0]], [0], [15], 16, 1, device="cuda")
    pka.paged_attn_plan_advance(plan)
    torch.cuda.synchronize()
    assert pka.device_status(clear=True) == 4          # PA_DEVICE_RANGE
    # a table entry of -1 for the next page is refused the same way
    plan = pka.paged_attn_plan([16], [[0, -1]], [0], [15], 16, 1, device="cuda")
    pka.paged_attn_plan_advance(plan)
    torch.cuda.synchronize()
    assert pka.device_status(clear=True) == 4


def test_staged_plans_replayed_from_one_graph(cuda_device):
    """Plan.stage + a pinned copy inside the graph: each replay runs the schedule staged last.

    Two plans with the same counts but different page assignments (and caches)
    are staged in turn into the same pinned and device buffers; every replay is
    checked against the oracle for the plan staged before it.
    """
    seq_lens = [70, 333, 5, 1000]
    queries = decode_queries(seq_lens) + [(3, 500)]
    cases = [build_case("staged", seed, seq_lens, queries, 16, 4, 128, 128, 16, torch.bfloat16,
                        1 / math.sqrt(128)) for seed in (71, 72)]
    plans = [pka.paged_attn_plan(c.seq_lens, c.block_table, c.query_seq, c.query_pos, c.page_size, c.num_pages,
                                 upload=False) for c in cases]
    assert plans[0].device_bytes() == plans[1].device_bytes()
    n = plans[0].device_bytes()
    dev = torch.device("cuda")
    words = torch.empty(n, dtype=torch.uint8, device=dev)
    words_host = torch.empty(n, dtype=torch.uint8).pin_memory()
    dc = cases[0].to(dev)
    out = torch.empty(cases[0].num_queries, 16, 128, dtype=torch.bfloat16, device=dev)
    plans[0].stage(words_host, words)
    ws = pka.make_workspace(plans[0], 16, 128, 3)
    state = {"plan": plans[0]}

    def body():
        words.copy_(words_host, non_blocking=True)
        pka.paged_kv_store(state["plan"], dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
        pka.paged_attn_forward_split(state["plan"], dc.q, dc.k_cache, dc.v_cache, cases[0].scale, 3,
                                     workspace=ws, out=out)

    body()                             # one plain run first (kernel attributes are set outside capture)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        body()
    for i in (1, 0, 1):
        c = cases[i]
        plans[i].stage(words_host, words)          # host-side only; the replay copies it
        for name in ("q", "k_cache", "v_cache", "new_k", "new_v"):
            getattr(dc, name).copy_(getattr(c, name))
        graph.replay()
        torch.cuda.synchronize()
        assert pka.device_status() == 0
        ref, _, _, _ = oracle_after_store(c)
        assert_close(out.cpu().double().numpy(), ref, torch.bfloat16, f"staged plan {i}")
