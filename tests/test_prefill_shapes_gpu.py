"""Chunked prefill for head layouts outside the 4-head groups of the other tests.

ruDNN 0.1.7, src/paged_attention/mod.rs (`DevicePlan::attention`, module doc:
packed decode and chunked prefill at absolute positions).  The tensor-core
prefill pairs the query heads of a KV head in two-CTA clusters when the group
size is even and runs single CTAs otherwise; both walk their share of the work
units persistently.  MHA (group 1), odd groups (3), groups of 8 (whose decode
items in the same call go to the tensor-core decode) and a case with more
units than CTAs resident at once are compared with the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

from helpers import assert_close, gpu_store_and_attend, oracle_after_store
from workloads import build_case

pytestmark = pytest.mark.gpu


def _mixed(seq_lens, chunks, decodes):
    """Prefill chunks (seq, first position, length) then one decode query per listed sequence."""
    queries = []
    for s, p0, n in chunks:
        queries += [(s, p0 + i) for i in range(n)]
    queries += [(s, seq_lens[s] - 1) for s in decodes]
    return queries


@pytest.mark.parametrize("hq,hkv", [(4, 4), (6, 2), (8, 1), (32, 4)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_head_layouts(cuda_device, hq, hkv, dtype):
    seq_lens = [300, 700, 129, 60]
    queries = _mixed(seq_lens, [(0, 0, 300), (1, 450, 250), (2, 1, 128)], [3])
    case = build_case("pf_heads", 91, seq_lens, queries, hq, hkv, 128, 128, 16, dtype, 1 / math.sqrt(128))
    ref, _, _, _ = oracle_after_store(case)
    for splits in (None, 3):
        out, _, _, _ = gpu_store_and_attend(case, splits=splits)
        assert_close(out.double().numpy(), ref, dtype, f"hq={hq} hkv={hkv} splits={splits}")


def test_more_units_than_resident_ctas(cuda_device):
    """Group 3 (single CTAs): 16 query tiles x 24 heads = 384 units over at most 152 CTAs."""
    offs = [0, 700, 1500, 2600]
    seq_lens = [o + 512 for o in offs]
    queries = _mixed(seq_lens, [(s, o, 512) for s, o in enumerate(offs)], [])
    case = build_case("pf_units", 92, seq_lens, queries, 24, 8, 128, 128, 16, torch.bfloat16, 1 / math.sqrt(128))
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(case.num_queries * case.hq, size=96, replace=False))
    ref, _, _, _ = oracle_after_store(case, rows=rows)
    for splits in (None, 2):
        out, _, _, _ = gpu_store_and_attend(case, splits=splits)
        got = out.double().numpy().reshape(-1, case.dv)[rows]
        assert_close(got, ref, torch.bfloat16, f"384 units splits={splits}")
