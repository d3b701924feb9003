"""The named decode workloads at full size in fp16.

ruDNN 0.1.7, src/paged_attention/mod.rs: the attention calls take F16 as well
as BF16 and F32 tensors (`check_tensor`), with the output in the inputs' dtype.
The benchmark's workloads are bf16; these cases lay out the same schedules,
shapes and page sizes in fp16, so the fp16 forms of the CUDA-core decode, the
tensor-core decode (groups of 8) and the MLA kernel run at the sizes and
occupancies the benchmark measures, against the fp64 oracle.
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
