"""Tensor-core decode for GQA groups of 8 or more heads per KV head, against the fp64 oracle.

ruDNN 0.1.7, src/paged_attention/mod.rs (`DevicePlan::attention`,
`attention_into_split`): the same paged decode as every other path; here the
query group of one KV head sits in the first rows of a 128-row tensor-core
tile.  Groups 8..128 (powers of two and 12, 24, 40, 96), page sizes 8..256,
ragged histories (1 key, one short of and one past a 128-key tile), splits
whose first tile starts mid-tile, sliding windows, non-causal queries and fp16
are compared element by element, and the per-split partials and LSE with the
oracle's partition.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, gpu_store_and_attend, oracle_after_store, plan_for
from workloads import build_case, decode_queries

pytestmark = pytest.mark.gpu

LENS = [1, 15, 127, 128, 129, 700, 2100]


def _compare(case, splits=None, causal=None, window=0, what=""):
    out, _, _, _ = gpu_store_and_attend(case, splits=splits, causal=causal, window=window)
    ref, _, _, _ = oracle_after_store(case, causal=causal, window=window)
    return assert_close(out.double().numpy(), ref, case.dtype, f"{what} splits={splits} window={window}")


@pytest.mark.parametrize("hq,hkv", [(8, 1), (64, 8), (32, 2), (64, 1), (128, 1), (24, 2), (48, 2), (40, 1), (96, 1)])
def test_groups(cuda_device, hq, hkv):
    case = build_case("tc_groups", 81, LENS, decode_queries(LENS), hq, hkv, 128, 128, 16, torch.bfloat16,
                      1 / math.sqrt(128))
    _compare(case, what=f"G={hq // hkv}")
    _compare(case, splits=5, what=f"G={hq // hkv}")


@pytest.mark.parametrize("ps", [8, 32, 64, 128, 256])
def test_page_sizes(cuda_device, ps):
    case = build_case("tc_ps", 82, LENS, decode_queries(LENS), 32, 4, 128, 128, ps, torch.bfloat16,
                      1 / math.sqrt(128))
    _compare(case, what=f"ps={ps}")
    _compare(case, splits=3, what=f"ps={ps}")


def test_fp16_non_causal_window(cuda_device):
    seq_lens = [40, 300, 1500]
    queries = [(0, 10), (0, 39), (1, 0), (1, 150), (1, 299), (2, 777), (2, 1499)]
    case = build_case("tc_misc", 83, seq_lens, queries, 16, 2, 128, 128, 16, torch.float16, 0.07)
    _compare(case, what="fp16")
    _compare(case, causal=False, what="fp16 non-causal")
    _compare(case, causal=False, splits=4, what="fp16 non-causal")
    for w in (1, 100, 129, 1000):
        _compare(case, window=w, what="fp16")
        _compare(case, window=w, splits=3, what="fp16")


def test_split_partials_follow_the_partition(cuda_device):
    seq_lens = [90, 700, 1500, 4097]
    case = build_case("tc_parts", 84, seq_lens, decode_queries(seq_lens), 64, 8, 128, 128, 16, torch.bfloat16,
                      0.1)
    splits, window = 6, 1333
    for w in (0, window):
        dc = case.to("cuda")
        plan = plan_for(case)
        pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
        ws = pka.make_workspace(plan, case.hq, case.dv, splits)
        pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits, workspace=ws,
                                     window=w)
        torch.cuda.synchronize()
        assert pka.device_status() == 0
        nrows = case.num_queries * case.hq
        o_bytes = (splits * nrows * case.dv * 4 + 255) // 256 * 256
        wsb = ws.view(torch.uint8).cpu()
        o_part = wsb[:splits * nrows * case.dv * 4].view(torch.float32).view(splits, nrows, case.dv).double().numpy()
        lse_part = wsb[o_bytes:o_bytes + splits * nrows * 4].view(torch.float32).view(splits, nrows).double().numpy()
        kc, vc = oracle.kv_store(case.new_k, case.new_v, case.k_cache, case.v_cache, case.block_table,
                                 case.query_seq, case.query_pos)
        ro, rl = oracle.attention_split(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq,
                                        case.query_pos, case.scale, splits, window=w)
        finite = np.isfinite(rl)
        assert np.array_equal(finite, np.isfinite(lse_part)), "empty splits must carry lse = -inf"
        np.testing.assert_allclose(lse_part[finite], rl[finite], rtol=0, atol=2e-3)
        for s in range(splits):
            sel = finite[s]
            assert_close(o_part[s][sel], ro[s][sel], torch.bfloat16, f"partial {s} window={w}")
            assert np.all(o_part[s][~sel] == 0.0)


def test_repeatable(cuda_device):
    """Twenty runs give the same bits (one warp's softmax, lazy rescale of O)."""
    seq_lens = [3000, 129, 4500]
    case = build_case("tc_rep", 85, seq_lens, decode_queries(seq_lens), 64, 8, 128, 128, 16, torch.bfloat16,
                      1 / math.sqrt(128))
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    first = None
    for _ in range(20):
        out = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, 7, window=777)
        torch.cuda.synchronize()
        assert pka.device_status() == 0
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))
