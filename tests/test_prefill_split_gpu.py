"""Split-KV for prefill tiles against the fp64 oracle.

ruDNN 0.1.7, src/paged_attention/mod.rs, doc of `attention_into_split`: the
visible history is split over several planes whose FP32 statistics are merged.
Every row of a prefill tile has its own visible range (causal at its absolute
position, a sliding window's lower end), and each range is cut by the same
partition as a decode query's.  The tests compare the per-split fp32 partials
and natural-log LSE of prefill rows with the oracle's partition, and the merged
output for chunks at the start, in the middle and deep into a long sequence.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, gpu_store_and_attend, oracle_after_store, plan_for
from workloads import build_case

pytestmark = pytest.mark.gpu


def _partials(case, splits, window=0):
    dc = case.to("cuda")
    plan = plan_for(case)
    assert plan.n_tiles > 0
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    ws = pka.make_workspace(plan, case.hq, case.dv, splits)
    out = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits, workspace=ws,
                                       window=window)
    torch.cuda.synchronize()
    assert pka.device_status() == 0
    nrows = case.num_queries * case.hq
    o_bytes = (splits * nrows * case.dv * 4 + 255) // 256 * 256
    wsb = ws.view(torch.uint8).cpu()
    o_part = wsb[:splits * nrows * case.dv * 4].view(torch.float32).view(splits, nrows, case.dv).double().numpy()
    lse_part = wsb[o_bytes:o_bytes + splits * nrows * 4].view(torch.float32).view(splits, nrows).double().numpy()
    return out.cpu(), o_part, lse_part


@pytest.mark.parametrize("window", [0, 150])
def test_prefill_split_partials_follow_the_partition(cuda_device, window):
    """Per-split partials and LSE of prefill rows equal the oracle's, row by row."""
    seq_lens = [700, 300]
    queries = [(0, 300 + i) for i in range(260)] + [(1, i) for i in range(140)]
    case = build_case("pf_split", 61, seq_lens, queries, 8, 2, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    splits = 3
    out, o_part, lse_part = _partials(case, splits, window)
    kc, vc = oracle.kv_store(case.new_k, case.new_v, case.k_cache, case.v_cache, case.block_table,
                             case.query_seq, case.query_pos)
    ro, rl = oracle.attention_split(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq,
                                    case.query_pos, case.scale, splits, window=window)
    finite = np.isfinite(rl)
    assert np.array_equal(finite, np.isfinite(lse_part)), "empty splits must carry lse = -inf"
    np.testing.assert_allclose(lse_part[finite], rl[finite], rtol=0, atol=2e-3)
    for s in range(splits):
        sel = finite[s]
        assert_close(o_part[s][sel], ro[s][sel], torch.bfloat16, f"prefill partial {s}")
        assert np.all(o_part[s][~sel] == 0.0)
    ref, _ = oracle.attention(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                              case.scale, window=window)
    assert_close(out.double().numpy(), ref, torch.bfloat16, "merged prefill split")


@pytest.mark.parametrize("ps,dtype", [(16, torch.bfloat16), (64, torch.float16)])
def test_prefill_split_merged(cuda_device, ps, dtype):
    """Mixed chunks + decode items through the split path, several split counts."""
    seq_lens = [300, 900, 129, 40]
    queries = [(0, i) for i in range(300)]
    queries += [(1, 500 + i) for i in range(260)]
    queries += [(2, 128)]
    queries += [(3, 20 + i) for i in range(20)]
    case = build_case("pf_split_m", 62, seq_lens, queries, 16, 4, 128, 128, ps, dtype, 1 / math.sqrt(128))
    ref, _, _, _ = oracle_after_store(case)
    for splits in (2, 5, 16):
        out, _, _, _ = gpu_store_and_attend(case, splits=splits)
        assert_close(out.double().numpy(), ref, dtype, f"prefill split {splits} ps={ps}")
    out, _, _, _ = gpu_store_and_attend(case, splits=4, window=97)
    refw, _, _, _ = oracle_after_store(case, window=97)
    assert_close(out.double().numpy(), refw, dtype, "prefill split with window")


def test_long_context_prefill_chunk_split(cuda_device):
    """A 128-query chunk at position ~24K: 32 heads give 32 CTAs unsplit; 12 splits spread it."""
    ctx = 24_000
    queries = [(0, ctx - 128 + i) for i in range(128)]
    case = build_case("pf_long", 63, [ctx], queries, 32, 8, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=64, replace=False))
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    out, _, _, _ = gpu_store_and_attend(case, splits=12)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, torch.bfloat16, "long-context prefill chunk, 12 splits")
