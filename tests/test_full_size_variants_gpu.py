"""The named workloads at full size in other dtypes and page sizes.

ruDNN 0.1.7, src/paged_attention/mod.rs: the attention calls take F16 as well
as BF16 and F32 tensors (`check_tensor`), with the output in the inputs' dtype.
The benchmark's workloads are bf16; these cases lay out the same schedules
and shapes in fp16, so the fp16 forms of the CUDA-core decode, the
tensor-core decode (groups of 8) and the MLA kernel run at the sizes and
occupancies the benchmark measures, against the fp64 oracle.  The page size
is any power of two (`HostPlan`); the mixed and MLA schedules are also laid
out in other page sizes than the benchmark's, which changes how many TMA
boxes the prefill and MLA kernels issue per key tile.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_attention_20_gb300 as pka
from helpers import assert_close, gpu_store_and_attend, oracle_after_store, plan_for
from workloads import build_case, decode_queries, gqa_decode_bf16, long_context_decode_bf16, mla_decode_bf16

pytestmark = pytest.mark.gpu


def _as_fp16(case, seed):
    ctx = [int(n) for n in case.seq_lens]
    return build_case(case.name + "_fp16", seed, ctx, decode_queries(ctx), case.hq, case.hkv, case.d,
                      case.p if case.is_mla else case.dv, case.page_size, torch.float16, case.scale,
                      mla_p=case.p)


def test_gqa_decode_fp16_full_every_row(cuda_device):
    """The GQA decode layer's schedule in fp16 at the heuristic split, every (query, head) row."""
    case = _as_fp16(gqa_decode_bf16(), 21)
    s = pka.paged_attn_split_heuristic(plan_for(case), case.hq, case.hkv)
    out, _, _, _ = gpu_store_and_attend(case, splits=s)
    ref, _, _, _ = oracle_after_store(case)
    assert_close(out.double().numpy(), ref, case.dtype, f"gqa fp16, split {s}")


def test_long_context_fp16_sampled(cuda_device):
    """32K..128K histories, 64 query heads per 8 KV heads (the tensor-core decode) in fp16."""
    case = _as_fp16(long_context_decode_bf16(), 22)
    s = pka.paged_attn_split_heuristic(plan_for(case), case.hq, case.hkv)
    rng = np.random.default_rng(22)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=32, replace=False))
    out, _, _, _ = gpu_store_and_attend(case, splits=s)
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, f"long-context fp16, split {s}")


def test_mla_decode_fp16_sampled(cuda_device):
    """The MLA workload's schedule (128 queries x 128 heads, R=512, P=64) in fp16."""
    case = _as_fp16(mla_decode_bf16(), 23)
    assert case.is_mla and case.dtype == torch.float16
    rng = np.random.default_rng(23)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=48, replace=False))
    out, _, _, _ = gpu_store_and_attend(case)
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, "mla fp16")


@pytest.mark.parametrize("ps", [32, 128])
def test_mixed_layout_other_page_sizes(cuda_device, ps):
    """The mixed workload's schedule with larger pages (fewer, bigger TMA boxes per key tile)."""
    from workloads import mixed_prefill_decode_bf16
    base = mixed_prefill_decode_bf16()
    offs, chunk = base.meta["prefill_offsets"], base.meta["chunk"]
    npf = len(offs)
    dctx = [int(n) for n in base.seq_lens[npf:]]
    seq_lens = [o + chunk for o in offs] + dctx
    queries = [(s, o + i) for s, o in enumerate(offs) for i in range(chunk)]
    queries += [(npf + s, n - 1) for s, n in enumerate(dctx)]
    case = build_case(f"mixed_ps{ps}", 24, seq_lens, queries, 32, 8, 128, 128, ps, torch.bfloat16,
                      1 / math.sqrt(128))
    rng = np.random.default_rng(ps)
    npq = npf * chunk
    qs = np.concatenate([rng.choice(npq, 16, replace=False), npq + rng.choice(len(dctx), 8, replace=False)])
    rows = np.sort(np.concatenate([q * case.hq + rng.choice(case.hq, 2, replace=False) for q in qs]))
    out, _, _, _ = gpu_store_and_attend(case)
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, f"mixed, page size {ps}")


def test_mla_layout_small_pages(cuda_device):
    """The MLA workload's schedule stored in 16-row pages (four TMA boxes per 64-key tile)."""
    base = mla_decode_bf16()
    ctx = [int(n) for n in base.seq_lens]
    case = build_case("mla_ps16", 25, ctx, decode_queries(ctx), base.hq, 1, 512, 64, 16, torch.bfloat16,
                      base.scale, mla_p=64)
    rng = np.random.default_rng(25)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=48, replace=False))
    out, _, _, _ = gpu_store_and_attend(case)
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    got = out.double().numpy().reshape(-1, case.dv)[rows]
    assert_close(got, ref, case.dtype, "mla, page size 16")
