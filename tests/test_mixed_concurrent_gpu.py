"""The mixed prefill + decode call with its decode items beside its prefill tiles.

ruDNN 0.1.7, src/paged_attention/mod.rs, module doc and `DevicePlan::attention`:
one call serves a batch that mixes chunked-prefill queries and decode queries.
At the mixed workload's size the library runs the decode kernel on a second
stream of the calling thread, on a share of the SMs, while the prefill kernel
runs on the others, and joins it back into the caller's stream.  A call made
while the caller's stream is being captured, on a thread that has no second
stream yet, runs the two kernels one after the other instead.  Every form must
give the same output, bit for bit, and that output must match the oracle.
"""
import math
import threading

import numpy as np
import pytest
import torch

import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, oracle_after_store
from workloads import build_case, mixed_prefill_decode_bf16

pytestmark = pytest.mark.gpu


def _in_thread(fn):
    box = {}

    def run():
        try:
            box["value"] = fn()
        except BaseException as e:  # reported in the calling thread
            box["error"] = e

    t = threading.Thread(target=run)
    t.start()
    t.join()
    if "error" in box:
        raise box["error"]
    return box["value"]


def test_mixed_call_same_bits_in_every_form(cuda_device):
    case = mixed_prefill_decode_bf16()
    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                               case.page_size, case.num_pages, device=dev)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    assert plan.n_tiles > 0 and plan.n_decode > 0

    def call(out):
        pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, out=out)

    def fresh():
        return torch.full((case.num_queries, case.hq, case.dv), float("nan"), dtype=case.dtype, device=dev)

    eager_main = fresh()
    call(eager_main)                   # kernel attributes are set outside capture
    torch.cuda.synchronize()

    def second_thread():
        outs = {}
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            # captured before this thread made any call: no second stream yet, so serial
            outs["captured_serial"] = fresh()
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1):
                call(outs["captured_serial"])
            g1.replay()
            # an eager call creates the thread's second stream and runs the kernels side by side
            outs["eager"] = fresh()
            call(outs["eager"])
            # captured again: the fork and join into the second stream are part of the graph
            outs["captured_side"] = fresh()
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2):
                call(outs["captured_side"])
            for _ in range(3):
                g2.replay()
        s.synchronize()
        assert pka.device_status() == 0
        return outs

    outs = _in_thread(second_thread)
    for name, out in outs.items():
        assert torch.equal(out, eager_main), name
    assert not torch.isnan(eager_main.float()).any()

    # the output against the oracle: decode rows and rows of every prefill chunk
    rng = np.random.default_rng(17)
    npq = case.meta["n_prefill"] * case.meta["chunk"]
    qs = np.concatenate([rng.choice(npq, 12, replace=False),
                         npq + rng.choice(case.num_queries - npq, 12, replace=False)])
    rows = np.sort(np.concatenate([q * case.hq + rng.choice(case.hq, 2, replace=False) for q in qs]))
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = eager_main.double().cpu().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, "mixed call beside")


def test_mixed_call_split_workspace_same_bits(cuda_device):
    # with splits > 1 both kernels write partials and one merge after the join covers every query
    case = mixed_prefill_decode_bf16()
    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                               case.page_size, case.num_pages, device=dev)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    ws = pka.make_workspace(plan, case.hq, case.dv, 2)
    outs = []
    for _ in range(3):
        out = torch.full((case.num_queries, case.hq, case.dv), float("nan"), dtype=case.dtype, device=dev)
        pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, 2, workspace=ws, out=out)
        outs.append(out)
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    rng = np.random.default_rng(23)
    rows = np.sort(rng.choice(case.num_queries * case.hq, 48, replace=False))
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = outs[0].double().cpu().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, "mixed split call beside")


def test_mixed_call_tensor_core_decode_beside(cuda_device):
    # groups of 8 query heads per KV head: the decode items run on the persistent
    # tensor-core decode kernel, its grid capped to the SMs the prefill leaves
    gen = np.random.default_rng(31)
    offs = [int(x) for x in gen.integers(1024, 3072, size=4)]
    dctx = [int(x) for x in gen.integers(2048, 6144, size=64)]
    chunk = 512
    seq_lens = [o + chunk for o in offs] + dctx
    queries = [(s, o + i) for s, o in enumerate(offs) for i in range(chunk)]
    queries += [(len(offs) + s, n - 1) for s, n in enumerate(dctx)]
    case = build_case("mixed_g8", 37, seq_lens, queries, 64, 8, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                               case.page_size, case.num_pages, device=dev)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)

    def fresh():
        return torch.full((case.num_queries, case.hq, case.dv), float("nan"), dtype=case.dtype, device=dev)

    def call(out):
        pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, out=out)

    warm = fresh()
    call(warm)                         # kernel attributes are set outside capture
    torch.cuda.synchronize()

    def serial_then_beside():
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            serial = fresh()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):  # no second stream on this thread yet: one after the other
                call(serial)
            g.replay()
            beside = fresh()
            call(beside)
        s.synchronize()
        return serial, beside

    serial, beside = _in_thread(serial_then_beside)
    assert pka.device_status() == 0
    assert torch.equal(serial, beside)
    assert torch.equal(warm, beside)
    rng = np.random.default_rng(5)
    npq = len(offs) * chunk
    qs = np.concatenate([rng.choice(npq, 8, replace=False), npq + rng.choice(len(dctx), 8, replace=False)])
    rows = np.sort(np.concatenate([q * case.hq + rng.choice(case.hq, 2, replace=False) for q in qs]))
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = beside.double().cpu().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, "mixed call, tensor-core decode beside")


@pytest.mark.parametrize("dtype,causal,window", [(torch.float16, True, 0), (torch.bfloat16, False, 0),
                                                 (torch.bfloat16, True, 2048)])
def test_mixed_call_beside_fp16_and_non_causal(cuda_device, dtype, causal, window):
    # the mixed workload's layout in fp16, non-causal (every query sees its whole sequence),
    # and under a sliding window
    base = mixed_prefill_decode_bf16()
    offs, chunk = base.meta["prefill_offsets"], base.meta["chunk"]
    npf = len(offs)
    dctx = [int(n) for n in base.seq_lens[npf:]]
    seq_lens = [o + chunk for o in offs] + dctx
    queries = [(s, o + i) for s, o in enumerate(offs) for i in range(chunk)]
    queries += [(npf + s, n - 1) for s, n in enumerate(dctx)]
    case = build_case("mixed_variant", 43, seq_lens, queries, 32, 8, 128, 128, 16, dtype, 1 / math.sqrt(128),
                      causal=causal)
    dev = torch.device("cuda")
    dc = case.to(dev)
    plan = pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                               case.page_size, case.num_pages, device=dev)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    assert pka.paged_attn_decode_sms_beside_prefill(plan, 32, 8, 128, 128, causal=causal, window=window,
                                                    dtype=dtype) > 0

    def fresh():
        return torch.full((case.num_queries, case.hq, case.dv), float("nan"), dtype=case.dtype, device=dev)

    def call(out):
        pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, causal=causal, window=window,
                               out=out)

    beside = fresh()
    call(beside)                       # kernel attributes are set outside capture

    def serial_form():
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            out = fresh()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):  # no second stream on this thread yet: one after the other
                call(out)
            g.replay()
        s.synchronize()
        return out

    serial = _in_thread(serial_form)
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    assert torch.equal(serial, beside)
    rng = np.random.default_rng(11)
    npq = npf * chunk
    qs = np.concatenate([rng.choice(npq, 8, replace=False), npq + rng.choice(len(dctx), 8, replace=False)])
    rows = np.sort(np.concatenate([q * case.hq + rng.choice(case.hq, 2, replace=False) for q in qs]))
    ref, _, _, _ = oracle_after_store(case, rows=rows, causal=causal, window=window)
    got = beside.double().cpu().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, f"mixed call beside ({dtype}, causal={causal}, window={window})")
