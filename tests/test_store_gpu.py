"""Cache append (paged_kv_store) against the oracle's host scatter: bit-exact.

ruDNN 0.1.7, src/paged_attention/mod.rs, `append_with_report`: new rows
[queries, heads, d|dv] land at the plan's positions; a zero-size append does
nothing.
"""
import pytest
import torch

import oracle
import paged_kv_attention_20_gb300 as pka
from helpers import bits_equal, plan_for
from workloads import build_case, decode_queries, gqa_decode_bf16, mixed_prefill_decode_bf16

pytestmark = pytest.mark.gpu


def _store_matches(case):
    dc = case.to("cuda")
    plan = plan_for(case)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    torch.cuda.synchronize()
    ek, ev = oracle.kv_store(case.new_k, case.new_v, case.k_cache, case.v_cache, case.block_table,
                             case.query_seq, case.query_pos)
    assert bits_equal(dc.k_cache.cpu(), ek)
    assert bits_equal(dc.v_cache.cpu(), ev)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("d,dv,heads,ps", [(128, 128, 8, 16), (64, 64, 4, 16), (40, 24, 3, 5), (7, 5, 1, 3),
                                           (512, 64, 1, 64)])
def test_store_bit_exact(cuda_device, dtype, d, dv, heads, ps):
    seq_lens = [1, ps - 1 if ps > 1 else 1, ps, ps + 1, 3 * ps + 2]
    queries = decode_queries(seq_lens) + [(4, 0), (4, ps)]
    case = build_case("store", 7, seq_lens, queries, heads, heads, d, dv, ps, dtype, 0.1, pool_pages=40)
    _store_matches(case)


def test_store_gqa_decode_full_size(cuda_device):
    _store_matches(gqa_decode_bf16())


def test_store_prefill_chunks(cuda_device):
    _store_matches(mixed_prefill_decode_bf16(n_prefill=3, chunk=300, off_hi=700, n_decode=9,
                                             dec_lo=20, dec_hi=900))


def test_store_unaligned_rows(cuda_device):
    """Rows that are not 16-byte multiples or start unaligned take the element path."""
    case = build_case("store", 8, [9, 33], decode_queries([9, 33]), 2, 2, 6, 10, 4, torch.bfloat16, 0.1)
    dc = case.to("cuda")
    plan = plan_for(case)
    big_k = torch.zeros(case.new_k.numel() + 1, dtype=case.dtype, device="cuda")
    nk = big_k[1:].view(case.new_k.shape)      # 2-byte offset -> not 16-byte aligned
    nk.copy_(dc.new_k)
    pka.paged_kv_store(plan, nk, dc.new_v, dc.k_cache, dc.v_cache)
    torch.cuda.synchronize()
    ek, ev = oracle.kv_store(case.new_k, case.new_v, case.k_cache, case.v_cache, case.block_table,
                             case.query_seq, case.query_pos)
    assert bits_equal(dc.k_cache.cpu(), ek) and bits_equal(dc.v_cache.cpu(), ev)


def test_store_empty_plan_is_noop(cuda_device):
    plan = pka.paged_attn_plan([3], [[0]], [], [], 4, 1, device="cuda")
    kc = torch.full((1, 4, 1, 8), 3.0, device="cuda")
    pka.paged_kv_store(plan, torch.empty(0, 1, 8, device="cuda"), torch.empty(0, 1, 8, device="cuda"), kc,
                       kc.clone())
    torch.cuda.synchronize()
    assert torch.all(kc == 3.0)
