"""Sliding-window attention through the C ABI against the fp64 oracle.

A layer's attention carries a `window` next to its head geometry
(libmir-cuda 0.1.0, src/backend/attention/graph/mod.rs, `Geometry`; the split
configuration is chosen from the token count and that window).  The pages name
the field only; the reading here, shared with the oracle, is that a query at
absolute position p sees keys p - window + 1 .. (its causal or non-causal upper
end), and window = 0 is no window.  Windows that start mid-page and mid-tile,
W = 1, windows longer than the history, splits, prefill chunks (where every
row of a tile has its own lower end) and MLA are all compared with the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, gpu_store_and_attend, oracle_after_store, plan_for
from workloads import build_case, decode_queries, long_context_decode_bf16

pytestmark = pytest.mark.gpu


def _compare(case, window, splits=None, causal=None, rows=None, what=""):
    out, _, _, _ = gpu_store_and_attend(case, splits=splits, causal=causal, window=window)
    ref, _, _, _ = oracle_after_store(case, causal=causal, window=window, rows=rows)
    got = out.double().numpy()
    if rows is not None:
        got = got.reshape(-1, got.shape[-1])[np.asarray(rows)]
    return assert_close(got, ref, case.dtype, f"{what or case.name} window={window} splits={splits}")


@pytest.mark.parametrize("ps", [8, 16, 64])
def test_decode_window_bf16(cuda_device, ps):
    seq_lens = [1, 15, 16, 17, 100, 777, 2049]
    case = build_case("win_dec", 51, seq_lens, decode_queries(seq_lens), 32, 8, 128, 128, ps,
                      torch.bfloat16, 1 / math.sqrt(128))
    for w in (1, 5, 16, 37, 300, 5000):
        _compare(case, w)
        _compare(case, w, splits=3)
    _compare(case, 700, splits=16)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float16])
def test_decode_window_other_dtypes(cuda_device, dtype):
    seq_lens = [3, 60, 333]
    case = build_case("win_dt", 52, seq_lens, decode_queries(seq_lens) + [(2, 100)], 8, 2, 64, 64, 16,
                      dtype, 0.125)
    for w in (1, 10, 64):
        _compare(case, w)
        _compare(case, w, splits=4)


def test_decode_window_non_causal(cuda_device):
    seq_lens = [40, 300]
    queries = [(0, 10), (0, 39), (1, 0), (1, 150), (1, 299)]
    case = build_case("win_nc", 53, seq_lens, queries, 16, 4, 128, 128, 16, torch.bfloat16, 0.09)
    for w in (1, 33, 200):
        _compare(case, w, causal=False)
        _compare(case, w, causal=False, splits=5)


def test_window_split_partials_follow_the_partition(cuda_device):
    """Per-split fp32 partials and LSE under a window match the oracle's windowed partition."""
    seq_lens = [90, 700, 1500]
    case = build_case("win_ws", 54, seq_lens, decode_queries(seq_lens), 8, 2, 128, 128, 16, torch.bfloat16, 0.1)
    splits, window = 5, 333
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    ws = pka.make_workspace(plan, case.hq, case.dv, splits)
    pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits, workspace=ws,
                                 window=window)
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
                                    case.query_pos, case.scale, splits, window=window)
    finite = np.isfinite(rl)
    assert np.array_equal(finite, np.isfinite(lse_part)), "empty splits must carry lse = -inf"
    np.testing.assert_allclose(lse_part[finite], rl[finite], rtol=0, atol=2e-3)
    for s in range(splits):
        sel = finite[s]
        assert_close(o_part[s][sel], ro[s][sel], torch.bfloat16, f"windowed partial {s}")


@pytest.mark.parametrize("ps,dtype", [(16, torch.bfloat16), (64, torch.bfloat16), (32, torch.float16)])
def test_prefill_window(cuda_device, ps, dtype):
    """Prefill tiles: each query row has its own window start inside the tile."""
    seq_lens = [300, 900, 40]
    queries = [(0, i) for i in range(300)]                   # from position 0: windows start at 0 early on
    queries += [(1, 500 + i) for i in range(260)]            # mid-sequence chunk, partial last tile
    queries += [(2, 20 + i) for i in range(20)]
    case = build_case("win_pf", 55, seq_lens, queries, 16, 4, 128, 128, ps, dtype, 1 / math.sqrt(128))
    for w in (1, 50, 129, 256, 1000):
        _compare(case, w, what=f"prefill ps={ps}")
    _compare(case, 77, causal=False, what=f"prefill non-causal ps={ps}")
    _compare(case, 200, splits=3, what=f"prefill + split decode ps={ps}")


@pytest.mark.parametrize("ps", [16, 64, 128])
def test_mla_window(cuda_device, ps):
    seq_lens = [1, 64, 65, 500, 3000]
    queries = decode_queries(seq_lens) + [(4, 1234)]
    case = build_case("win_mla", 56, seq_lens, queries, 128, 1, 512, 64, ps, torch.bfloat16,
                      1 / math.sqrt(192), mla_p=64)
    for w in (1, 63, 100, 2048):
        _compare(case, w, what=f"mla ps={ps}")
    _compare(case, 1000, splits=3, what=f"mla split ps={ps}")


def test_long_context_window_sampled(cuda_device):
    """The 128K long-context decode with a 4096-key window at the heuristic split, sampled rows."""
    case = long_context_decode_bf16()
    window = 4096
    plan = plan_for(case)
    splits = pka.paged_attn_split_heuristic(plan, case.hq, case.hkv, window=window)
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=24, replace=False))
    _compare(case, window, splits=splits, rows=rows, what="long context")
    _compare(case, window, rows=rows, what="long context unsplit")


@pytest.mark.parametrize("ps", [64, 128])
def test_mla_window_repeatable(cuda_device, ps):
    """Thirty runs of a windowed MLA layer give the same bits every time.

    A short first window tile sets a low reference maximum, so later tiles
    rescale O often; the softmax warps then drift apart, which once let a
    warp already on the next tile complete the current tile's P barrier
    (seen as NaN in one warp's rows on one CTA of the pair).
    """
    seq_lens = [1, 64, 65, 500, 3000]
    queries = decode_queries(seq_lens) + [(4, 1234)]
    case = build_case("win_mla_rep", 56, seq_lens, queries, 128, 1, 512, 64, ps, torch.bfloat16,
                      1 / math.sqrt(192), mla_p=64)
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    first = None
    for _ in range(30):
        out = pka.paged_mla_forward(plan, dc.q, dc.qp, dc.k_cache, dc.v_cache, case.scale, window=2048)
        torch.cuda.synchronize()
        assert pka.device_status() == 0
        assert torch.isfinite(out.float()).all()
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))


def test_prefill_window_repeatable(cuda_device):
    """The same for prefill tiles, whose softmax warps can be two tiles apart."""
    seq_lens = [900, 2000]
    queries = [(0, 400 + i) for i in range(500)] + [(1, 1500 + i) for i in range(500)]
    case = build_case("win_pf_rep", 57, seq_lens, queries, 32, 8, 128, 128, 16, torch.bfloat16,
                      1 / math.sqrt(128))
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    first = None
    for _ in range(30):
        out = pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, window=37)
        torch.cuda.synchronize()
        assert pka.device_status() == 0
        assert torch.isfinite(out.float()).all()
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out.view(torch.int16), first.view(torch.int16))


def test_mla_fp16_split_window(cuda_device):
    """MLA in fp16 through the split path, with and without a window."""
    seq_lens = [70, 500, 1300]
    case = build_case("win_mla16", 58, seq_lens, decode_queries(seq_lens) + [(2, 640)], 128, 1, 512, 64, 64,
                      torch.float16, 1 / math.sqrt(192), mla_p=64)
    for w in (0, 300):
        _compare(case, w, splits=3, what="mla fp16")


def test_prefill_window_split_tile_range(cuda_device):
    # With a window the page-rounded split chunk can shrink as a tile's rows
    # move their base to the next page, so split s > 1 of a later row may start
    # before that of an earlier row: the tile's key range has to cover every row,
    # not only the first and the last.  Windows and split counts chosen so some
    # tiles of this layout have such rows, causal and not.
    seq_lens = [300, 900]
    queries = [(0, i) for i in range(300)] + [(1, 500 + i) for i in range(200)]
    case = build_case("win_pf_nc", 59, seq_lens, queries, 16, 4, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    for w in (0, 77, 400):
        _compare(case, w, causal=False, splits=3, what="prefill non-causal split")
    _compare(case, 82, splits=3, what="prefill causal split")
    _compare(case, 50, splits=4, what="prefill causal split")
