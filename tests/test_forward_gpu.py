"""Paged attention through the C ABI against the fp64 oracle.

Follows ruDNN 0.1.7, src/paged_attention/mod.rs (`DevicePlan::attention`,
`attention_into_split`, `DevicePlan::mla`): every case appends its new rows
with paged_kv_store first, then attends, and the oracle does the same on the
host.  Caches carry NaN in every unreferenced page and tail slot, so any read
outside the visible keys shows up as a non-finite output.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, bits_equal, gpu_store_and_attend, oracle_after_store, plan_for
from workloads import (build_case, decode_queries, gqa_decode_bf16, long_context_decode_bf16,
                       mixed_prefill_decode_bf16, mla_decode_bf16, tiny_fp32_mha_decode)

pytestmark = pytest.mark.gpu


def _compare(case, splits=None, rows=None, causal=None, what=""):
    out, _, _, _ = gpu_store_and_attend(case, splits=splits, causal=causal)
    ref, _, _, _ = oracle_after_store(case, rows=rows, causal=causal)
    got = out.double().numpy()
    if rows is not None:
        got = got.reshape(-1, got.shape[-1])[np.asarray(rows)]
    return assert_close(got, ref, case.dtype, what or case.name)


# ------------------------------------------------------------ named shapes --

def test_tiny_fp32_mha_decode(cuda_device):
    _compare(tiny_fp32_mha_decode())


def test_tiny_fp32_split(cuda_device):
    for s in (1, 2, 3, 16, 64):
        _compare(tiny_fp32_mha_decode(), splits=s, what=f"tiny split {s}")


def test_gqa_decode_bf16_full(cuda_device):
    """The Llama-3-8B-like decode layer at full size, every (query, head) row."""
    _compare(gqa_decode_bf16())


def test_gqa_decode_bf16_heuristic_split(cuda_device):
    case = gqa_decode_bf16()
    plan = plan_for(case)
    s = pka.paged_attn_split_heuristic(plan, case.hq, case.hkv)
    assert 1 <= s <= 64
    _compare(case, splits=s, what=f"gqa heuristic split {s}")


@pytest.mark.parametrize("splits", [1, 2, 4, 8, 16, 32, 64])
def test_long_context_split_sampled(cuda_device, splits):
    """Contexts 32K..128K, sampled rows against the oracle, for every split count."""
    case = _long_case()
    rng = np.random.default_rng(3)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=24, replace=False))
    ref = _long_ref(case, tuple(rows))
    out, _, _, _ = gpu_store_and_attend(case, splits=splits)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, f"long split {splits}")


_LONG = {}


def _long_case():
    if "case" not in _LONG:
        _LONG["case"] = long_context_decode_bf16()
    return _LONG["case"]


def _long_ref(case, rows):
    if rows not in _LONG:
        _LONG[rows] = oracle_after_store(case, rows=np.array(rows))[0]
    return _LONG[rows]


def test_mixed_prefill_decode_small(cuda_device):
    case = mixed_prefill_decode_bf16(n_prefill=3, chunk=300, off_hi=700, n_decode=12, dec_lo=20, dec_hi=900)
    _compare(case)


def test_mla_decode_small(cuda_device):
    case = mla_decode_bf16(num_seqs=6, heads=16, ctx_lo=1, ctx_hi=700)
    _compare(case)


def test_mla_decode_small_split(cuda_device):
    case = mla_decode_bf16(num_seqs=5, heads=8, ctx_lo=60, ctx_hi=500)
    _compare(case, splits=4, what="mla split 4")


# -------------------------------------------------------------- edge cases --

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (64, 4), (12, 3)])
def test_gqa_group_sizes(cuda_device, dtype, hq, hkv):
    seq_lens = [1, 15, 16, 17, 90]
    case = build_case("groups", 11, seq_lens, decode_queries(seq_lens), hq, hkv, 128, 128, 16, dtype,
                      1 / math.sqrt(128))
    _compare(case, what=f"G={hq // hkv} {dtype}")


@pytest.mark.parametrize("d", [64, 128, 256, 40, 96])
@pytest.mark.parametrize("ps", [16, 64, 1, 3])
def test_head_dims_and_page_sizes(cuda_device, d, ps):
    seq_lens = [1, ps, ps + 1, 5 * ps - 1 if ps > 1 else 7, 130]
    case = build_case("dims", 12, seq_lens, decode_queries(seq_lens), 8, 2, d, d, ps, torch.bfloat16,
                      1 / math.sqrt(d), pool_pages=None)
    _compare(case, what=f"d={d} ps={ps}")


def test_value_dim_differs(cuda_device):
    seq_lens = [3, 40, 77]
    case = build_case("dv", 13, seq_lens, decode_queries(seq_lens), 4, 2, 64, 32, 16, torch.bfloat16, 0.125)
    _compare(case)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_non_causal_and_mid_positions(cuda_device, dtype):
    seq_lens = [50, 120, 33]
    queries = [(0, 3), (1, 60), (2, 32), (1, 0), (0, 49)]
    case = build_case("noncausal", 14, seq_lens, queries, 8, 2, 128, 128, 16, dtype, 0.09)
    _compare(case, causal=False, what="non-causal")
    _compare(case, causal=True, what="causal mid positions")
    _compare(case, causal=False, splits=5, what="non-causal split")


def test_splits_exceed_pages(cuda_device):
    seq_lens = [1, 2, 17, 33]
    case = build_case("many_splits", 15, seq_lens, decode_queries(seq_lens), 8, 2, 128, 128, 16,
                      torch.bfloat16, 0.1)
    for s in (7, 64):
        _compare(case, splits=s, what=f"splits {s} > pages")


def test_split_partials_and_lse_match_oracle(cuda_device):
    """The workspace's per-split fp32 outputs and log-sum-exp match the oracle's partition."""
    seq_lens = [1, 100, 700, 1500]
    case = build_case("ws", 16, seq_lens, decode_queries(seq_lens), 8, 2, 128, 128, 16, torch.bfloat16, 0.1)
    splits = 5
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    ws = pka.make_workspace(plan, case.hq, case.dv, splits)
    pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits, workspace=ws)
    torch.cuda.synchronize()
    nrows = case.num_queries * case.hq
    o_bytes = (splits * nrows * case.dv * 4 + 255) // 256 * 256
    wsb = ws.view(torch.uint8).cpu()
    o_part = wsb[:splits * nrows * case.dv * 4].view(torch.float32).view(splits, nrows, case.dv).double().numpy()
    lse_part = wsb[o_bytes:o_bytes + splits * nrows * 4].view(torch.float32).view(splits, nrows).double().numpy()
    kc, vc = oracle.kv_store(case.new_k, case.new_v, case.k_cache, case.v_cache, case.block_table,
                             case.query_seq, case.query_pos)
    ro, rl = oracle.attention_split(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq,
                                    case.query_pos, case.scale, splits)
    finite = np.isfinite(rl)
    assert np.array_equal(finite, np.isfinite(lse_part)), "empty splits must carry lse = -inf"
    assert np.all(lse_part[~finite] == -np.inf)
    np.testing.assert_allclose(lse_part[finite], rl[finite], rtol=0, atol=2e-3)
    for s in range(splits):
        sel = finite[s]
        assert_close(o_part[s][sel], ro[s][sel], torch.bfloat16, f"partial {s}")


def test_single_visible_key_is_exact(cuda_device):
    """A causal query at position 0 sees only its own key: out equals its value row bit for bit."""
    seq_lens = [1, 30, 64]
    queries = [(0, 0), (1, 0), (2, 0)]
    for dtype in (torch.bfloat16, torch.float32):
        case = build_case("single", 17, seq_lens, queries, 8, 2, 128, 128, 16, dtype, 0.1)
        out, _, _, _ = gpu_store_and_attend(case)
        expect = case.new_v.repeat_interleave(4, dim=1)
        assert bits_equal(out, expect)


def test_page_permutation_bit_invariance(cuda_device):
    """Same logical data under two physical page permutations: identical output bits."""
    base = build_case("perm", 18, [37, 200, 513], decode_queries([37, 200, 513]), 16, 4, 128, 128, 16,
                      torch.bfloat16, 0.1, poison=False)
    out_a, _, _, _ = gpu_store_and_attend(base)
    # Rebuild the caches under another permutation of the same logical rows.
    perm = torch.randperm(base.num_pages, generator=torch.Generator().manual_seed(5)).numpy()
    inv_table = perm[base.block_table]
    kc = torch.empty_like(base.k_cache)
    vc = torch.empty_like(base.v_cache)
    kc[perm] = base.k_cache
    vc[perm] = base.v_cache
    moved = base.to("cpu")
    moved.block_table = inv_table.astype(np.int32)
    moved.k_cache, moved.v_cache = kc, vc
    out_b, _, _, _ = gpu_store_and_attend(moved)
    assert bits_equal(out_a, out_b)


def test_zero_queries_launches_nothing(cuda_device):
    plan = pka.paged_attn_plan([5], [[0]], [], [], 16, 1, device="cuda")
    q = torch.empty(0, 4, 64, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(1, 16, 4, 64, device="cuda", dtype=torch.bfloat16)
    out = pka.paged_attn_forward(plan, q, kc, kc.clone(), 0.1)
    assert out.shape == (0, 4, 64)


def test_finite_with_poisoned_neighbours(cuda_device):
    """Pages and tail slots full of NaN next to every sequence never leak into outputs."""
    seq_lens = [5, 16, 31, 47]
    case = build_case("poison", 19, seq_lens, decode_queries(seq_lens), 8, 8, 128, 128, 16,
                      torch.bfloat16, 0.1, pool_pages=64)
    out, _, _, _ = gpu_store_and_attend(case)
    assert torch.isfinite(out.float()).all()


def test_repeat_calls_reuse_workspace_across_plans(cuda_device):
    """One workspace serves two plans of compatible shape on the same stream."""
    a = build_case("ws1", 20, [100, 300], decode_queries([100, 300]), 8, 2, 128, 128, 16, torch.bfloat16, 0.1)
    b = build_case("ws2", 21, [40, 999], decode_queries([40, 999]), 8, 2, 128, 128, 16, torch.bfloat16, 0.1)
    plan_a = plan_for(a)
    ws = pka.make_workspace(plan_a, 8, 128, 8)
    for case in (a, b):
        dc = case.to("cuda")
        plan = plan_for(case)
        pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
        out = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, 8, workspace=ws)
        ref, _, _, _ = oracle_after_store(case)
        assert_close(out.cpu().double().numpy(), ref, case.dtype, case.name)


# ------------------------------------------------ tensor-core paths (sm_103a) --

def _sampled(case, nrows, seed, splits=None):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=nrows, replace=False))
    out, _, _, _ = gpu_store_and_attend(case, splits=splits)
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    return assert_close(got, ref, case.dtype, case.name)


def test_mixed_prefill_decode_full_sampled(cuda_device):
    """8 prefill chunks of 512 queries at offsets up to 4096 plus 120 decode queries."""
    _sampled(mixed_prefill_decode_bf16(), 96, 4)


def test_mla_decode_full_sampled(cuda_device):
    """128 queries x 128 heads, latent 512 + position 64, contexts up to 16K, page size 64."""
    _sampled(mla_decode_bf16(), 64, 5)


@pytest.mark.parametrize("heads,ps,dtype", [(256, 64, torch.bfloat16), (128, 16, torch.bfloat16),
                                            (100, 64, torch.float16), (128, 128, torch.bfloat16)])
def test_mla_shapes(cuda_device, heads, ps, dtype):
    case = mla_decode_bf16(num_seqs=4, heads=heads, ctx_lo=1, ctx_hi=600)
    if ps != 64 or dtype != torch.bfloat16:
        ctx = list(case.seq_lens)
        case = build_case("mla_shapes", 31, ctx, decode_queries(ctx), heads, 1, 512, 64, ps, dtype,
                          1 / math.sqrt(192), mla_p=64)
    _compare(case, what=f"mla H={heads} ps={ps} {dtype}")


def test_mla_non_causal_and_splits(cuda_device):
    seq_lens = [70, 300, 129]
    queries = [(0, 5), (1, 299), (2, 64)]
    case = build_case("mla_nc", 32, seq_lens, queries, 128, 1, 512, 64, 64, torch.bfloat16,
                      1 / math.sqrt(192), mla_p=64)
    _compare(case, causal=False, what="mla non-causal")
    for s in (2, 3, 8):
        _compare(case, splits=s, what=f"mla split {s}")


@pytest.mark.parametrize("ps,dtype", [(16, torch.bfloat16), (64, torch.bfloat16), (16, torch.float16),
                                      (32, torch.bfloat16)])
def test_prefill_chunks(cuda_device, ps, dtype):
    """Chunks at offset 0 and mid-sequence, run lengths that leave partial 128-query tiles."""
    seq_lens = [300, 700, 129, 40]
    queries = [(0, i) for i in range(300)]                       # whole sequence from position 0
    queries += [(1, 400 + i) for i in range(200)]                # mid-sequence chunk, partial tile
    queries += [(2, 128 + 0)]                                    # decode query
    queries += [(3, 20 + i) for i in range(20)]                  # short run (still a tile: >= 16)
    case = build_case("prefill", 33, seq_lens, queries, 16, 4, 128, 128, ps, dtype, 1 / math.sqrt(128))
    _compare(case, what=f"prefill ps={ps} {dtype}")
    _compare(case, causal=False, what=f"prefill non-causal ps={ps}")
    _compare(case, splits=4, what=f"prefill + split decode ps={ps}")
