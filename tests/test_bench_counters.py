"""The benchmark's algorithmic counters against a brute-force count (host only).

Every reported GB/s and TFLOP/s divides one of two counts by a time: the K/V
bytes a query's visible keys occupy (each KV head read once for its whole
query group; latent plus position row for MLA) and the multiply-add flops of
the causal-visible (query, key, head) triples (4*D per triple for MHA/GQA with
D = Dv; 2*(R+P) + 2*R for MLA).  Here both are recounted key by key from the
case's own positions and lengths, including a split at a query index as the
mixed workload's prefill part uses.
"""
import math

import numpy as np
import pytest
import torch

import bench
from workloads import build_case, decode_queries


def _brute(case, first=0, count=None):
    last = case.num_queries if count is None else first + count
    keys = 0
    for i in range(first, last):
        s, p = int(case.query_seq[i]), int(case.query_pos[i])
        end = p + 1 if case.causal else int(case.seq_lens[s])
        keys += sum(1 for j in range(int(case.seq_lens[s])) if j < end)
    elt = torch.empty((), dtype=case.dtype).element_size()
    if case.is_mla:
        return keys * (case.d + case.p) * elt, keys * case.hq * (2 * (case.d + case.p) + 2 * case.d)
    return keys * case.hkv * (case.d + case.dv) * elt, keys * case.hq * (2 * case.d + 2 * case.dv)


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_counts(causal):
    seq_lens = [1, 17, 64, 200]
    queries = decode_queries(seq_lens) + [(3, 100 + i) for i in range(20)]
    case = build_case("count", 3, seq_lens, queries, 8, 2, 64, 64, 16, torch.bfloat16, 0.125, causal=causal)
    b, f = _brute(case)
    assert bench.kv_bytes(case) == b and bench.attn_flops(case) == f
    # the prefill part alone (queries 4.. on) and its byte count from a query index on
    b2, f2 = _brute(case, 4, 20)
    assert bench.attn_flops(case, 4, 20) == f2 and bench.kv_bytes(case, 4) == b2


def test_mla_counts():
    seq_lens = [5, 300]
    case = build_case("count_mla", 4, seq_lens, decode_queries(seq_lens), 16, 1, 512, 64, 64, torch.bfloat16,
                      1 / math.sqrt(192), mla_p=64)
    b, f = _brute(case)
    assert bench.kv_bytes(case) == b == 305 * 576 * 2
    assert bench.attn_flops(case) == f == 305 * 16 * (2 * 576 + 2 * 512)


def test_long_context_closed_form():
    # four decode queries at the ends of histories of 32, 64, 96 and 128 keys
    # (the long-context layout at 1/1024 scale): sum of contexts x Hkv x (D + Dv) x 2 bytes
    ctx = [32, 64, 96, 128]
    case = build_case("count_long", 5, ctx, decode_queries(ctx), 64, 8, 128, 128, 16, torch.bfloat16, 0.088)
    assert bench.kv_bytes(case) == sum(ctx) * 8 * 256 * 2
    assert bench.attn_flops(case) == sum(ctx) * 64 * 4 * 128
    assert np.array_equal(bench.visible_counts(case), np.array(ctx))
