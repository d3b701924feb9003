"""Full-size tensor-core parity on whole row blocks, not random samples.

ruDNN 0.1.7, src/paged_attention/mod.rs (`DevicePlan::attention` over packed
decode and chunked prefill at absolute positions; `DevicePlan::mla`): at the
mixed and MLA workloads' full sizes, in the launch configuration the
benchmark times (the library's split heuristic), every output row of the
blocks most likely to expose a tiling or scheduling fault is compared with
the fp64 oracle:
  * mixed prefill + decode: every (query, head) row of the longest prefill
    chunk (its diagonal tiles and its deepest key tiles, 512 queries x 32
    heads) and of every decode item;
  * MLA decode: all 128 heads of the 8 queries with the longest histories
    (the units that bound the persistent walk), plus 8 of the shortest.
The bf16 tolerance is the parity bar's 2e-2 absolute.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, oracle_after_store, plan_for
from workloads import mixed_prefill_decode_bf16, mla_decode_bf16

pytestmark = pytest.mark.gpu


def _run(case, splits):
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    if case.is_mla:
        ws = pka.make_workspace(plan, case.hq, case.dv, splits) if splits > 1 else None
        out = pka.paged_mla_forward(plan, dc.q, dc.qp, dc.k_cache, dc.v_cache, case.scale, workspace=ws,
                                    splits=splits)
    else:
        out = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits)
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    return out.cpu().double().numpy().reshape(-1, case.dv)


def test_mixed_longest_chunk_and_all_decode_rows(cuda_device):
    case = mixed_prefill_decode_bf16()
    plan = plan_for(case)
    splits = pka.paged_attn_split_heuristic(plan, case.hq, case.hkv)
    chunk, offs = case.meta["chunk"], case.meta["prefill_offsets"]
    longest = int(np.argmax(offs))
    first = longest * chunk                      # chunks are packed first, in sequence order
    npq = case.meta["n_prefill"] * chunk
    queries = list(range(first, first + chunk)) + list(range(npq, case.num_queries))
    rows = (np.asarray(queries)[:, None] * case.hq + np.arange(case.hq)[None, :]).reshape(-1)
    got = _run(case, splits)[rows]
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    assert_close(got, ref, case.dtype, f"mixed: chunk at offset {offs[longest]} + decode rows, splits {splits}")


def test_mla_longest_and_shortest_histories_all_heads(cuda_device):
    case = mla_decode_bf16()
    plan = plan_for(case)
    splits = pka.paged_mla_split_heuristic(plan, case.hq)
    order = np.argsort(case.query_pos)
    queries = np.concatenate([order[-8:], order[:8]])
    rows = (queries[:, None] * case.hq + np.arange(case.hq)[None, :]).reshape(-1)
    got = _run(case, splits)[rows]
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    assert_close(got, ref, case.dtype, f"mla: 16 queries x 128 heads, splits {splits}")


@pytest.mark.parametrize("splits", [2, 3])
def test_mla_split_partials_full_size(cuda_device, splits):
    """The MLA workload with its histories split: the fp32 partials (written through the
    epilogue's lane-group transpose) and the merge, on the longest histories' heads."""
    case = mla_decode_bf16()
    order = np.argsort(case.query_pos)
    queries = np.concatenate([order[-4:], order[:2]])
    rows = (queries[:, None] * case.hq + np.arange(case.hq)[None, :]).reshape(-1)
    got = _run(case, splits)[rows]
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    assert_close(got, ref, case.dtype, f"mla: 6 queries x 128 heads, splits {splits}")


def test_mixed_split_partials_longest_chunk(cuda_device):
    """The mixed workload at 3 splits: the prefill kernel's fp32 partials for every row of
    the longest chunk, merged with the decode items' partials."""
    case = mixed_prefill_decode_bf16()
    chunk, offs = case.meta["chunk"], case.meta["prefill_offsets"]
    longest = int(np.argmax(offs))
    first = longest * chunk
    rows = (np.arange(first, first + chunk)[:, None] * case.hq + np.arange(case.hq)[None, :]).reshape(-1)
    got = _run(case, 3)[rows]
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    assert_close(got, ref, case.dtype, "mixed: longest chunk, splits 3")
