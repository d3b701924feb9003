"""Shapes at the edges of what the C ABI accepts, against the fp64 oracle.

ruDNN 0.1.7, src/paged_attention/mod.rs (`DevicePlan::attention` head-dim and
position-dim checks, `DevicePlan::mla`): head dims run from 1 to 1024, the MLA
position dim from 1 to 256, and any page size is allowed.  The smallest and
largest head and position dims (odd ones included, which no 16-byte row
copy covers) go through the generic kernel; pages larger than a key tile go
through the TMA decode, the tensor-core MLA, and prefill chunks whose pages
exceed the prefill tile.  Every case appends its new rows first and is
compared with and without a split.
"""
import math

import numpy as np
import pytest
import torch

from helpers import assert_close, gpu_store_and_attend, oracle_after_store
from workloads import build_case, decode_queries

pytestmark = pytest.mark.gpu


def _compare(case, splits=None, what=""):
    out, _, _, _ = gpu_store_and_attend(case, splits=splits)
    ref, _, _, _ = oracle_after_store(case)
    assert np.isfinite(out.double().numpy()).all()
    return assert_close(out.double().numpy(), ref, case.dtype, f"{what or case.name} splits={splits}")


@pytest.mark.parametrize("d,dv,dtype", [(1, 1, torch.float32), (1, 1, torch.bfloat16), (1024, 1024, torch.bfloat16),
                                        (1024, 1024, torch.float32), (1024, 3, torch.float16),
                                        (7, 1024, torch.bfloat16)])
def test_head_dim_extremes(cuda_device, d, dv, dtype):
    seq_lens = [1, 17, 300]
    case = build_case("dim_ext", 71, seq_lens, decode_queries(seq_lens), 4, 2, d, dv, 16, dtype, 1 / math.sqrt(d))
    for splits in (None, 3):
        _compare(case, splits, what=f"d={d} dv={dv} {dtype}")


@pytest.mark.parametrize("r,p,ps,dtype", [(1024, 256, 64, torch.bfloat16), (8, 1, 16, torch.float32),
                                          (512, 256, 16, torch.float16)])
def test_mla_dim_extremes(cuda_device, r, p, ps, dtype):
    seq_lens = [1, 64, 700]
    case = build_case("mla_ext", 72, seq_lens, decode_queries(seq_lens), 16, 1, r, p, ps, dtype,
                      1 / math.sqrt(r + p), mla_p=p)
    for splits in (None, 2):
        _compare(case, splits, what=f"mla R={r} P={p} ps={ps} {dtype}")


@pytest.mark.parametrize("ps", [256, 512])
def test_large_pages_decode(cuda_device, ps):
    # GQA groups of 4 (TMA decode): histories ending mid-page, on a page edge, and one key
    seq_lens = [1, ps - 1, ps, ps + 1, 3 * ps + 77]
    case = build_case("big_pages", 73, seq_lens, decode_queries(seq_lens), 32, 8, 128, 128, ps, torch.bfloat16,
                      1 / math.sqrt(128))
    for splits in (None, 4):
        _compare(case, splits, what=f"decode ps={ps}")


def test_large_pages_mla(cuda_device):
    seq_lens = [1, 255, 256, 1000]
    case = build_case("big_pages_mla", 74, seq_lens, decode_queries(seq_lens), 128, 1, 512, 64, 256, torch.bfloat16,
                      1 / math.sqrt(192), mla_p=64)
    for splits in (None, 3):
        _compare(case, splits, what="mla ps=256")


@pytest.mark.parametrize("ps", [256, 512])
def test_large_pages_prefill(cuda_device, ps):
    # a chunk of 200 queries starting mid-page next to two decode queries
    seq_lens = [ps + 300, 900]
    queries = [(0, ps + 100 + i) for i in range(200)] + [(1, 899)]
    case = build_case("big_pages_pf", 75, seq_lens, queries, 16, 4, 128, 128, ps, torch.bfloat16,
                      1 / math.sqrt(128))
    for splits in (None, 3):
        _compare(case, splits, what=f"prefill ps={ps}")


@pytest.mark.parametrize("dv,dtype,splits", [(64, torch.bfloat16, 3), (3, torch.bfloat16, 3), (5, torch.float32, 2),
                                             (64, torch.float16, 16)])
def test_merge_paths(cuda_device, dv, dtype, splits):
    # 64 queries x 16 heads = 1024 rows: below 16 splits the merge takes one warp
    # per row (value dims under one warp's column chunk leave lanes idle), at 16
    # or more one block per row; the small cases above cover the block path too
    rng = np.random.default_rng(76)
    seq_lens = [int(x) for x in rng.integers(1, 300, size=64)]
    case = build_case("merge_paths", 76, seq_lens, decode_queries(seq_lens), 16, 4, 32, dv, 16, dtype,
                      1 / math.sqrt(32))
    _compare(case, splits, what=f"merge dv={dv} {dtype}")
