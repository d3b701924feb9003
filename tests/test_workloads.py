"""The seeded synthetic inputs follow their stated recipe (host only).

Both the oracle and the CUDA path read these cases, so their structure is
pinned here: shapes and dtypes of the five workloads, context ranges,
decode queries at ctx - 1, prefill chunks at o .. o + chunk - 1 with
seq_len = o + chunk (packed before the decode queries), distinct physical pages
drawn from a shuffled pool, NaN in every unreferenced page and every tail slot
past a sequence's end (so a read outside the visible keys cannot go unnoticed),
finite values everywhere else, and bit-for-bit repeatable draws per seed.
"""
import math

import numpy as np
import torch

import workloads


def _check_layout(c):
    ps = c.page_size
    n_pages = [(int(n) + ps - 1) // ps for n in c.seq_lens]
    used = np.concatenate([c.block_table[s, :n] for s, n in enumerate(n_pages)]) if n_pages else np.zeros(0)
    assert len(set(used.tolist())) == len(used), "every used page belongs to one sequence"
    assert used.min() >= 0 and used.max() < c.num_pages
    dead = sorted(set(range(c.num_pages)) - set(used.tolist()))
    for cache in (c.k_cache, c.v_cache):
        assert cache.shape[:2] == (c.num_pages, ps)
        if dead:
            assert torch.isnan(cache[dead].float()).all()
        for s, n in enumerate(n_pages):
            rows = cache[torch.as_tensor(c.block_table[s, :n], dtype=torch.long)].reshape(n * ps, *cache.shape[2:])
            live = int(c.seq_lens[s])
            assert torch.isfinite(rows[:live].float()).all()
            assert torch.isnan(rows[live:].float()).all()
    for t in (c.q, c.new_k, c.new_v) + ((c.qp,) if c.qp is not None else ()):
        assert t.dtype == c.dtype and torch.isfinite(t.float()).all()
    assert c.q.shape == (c.num_queries, c.hq, c.d)
    assert c.new_k.shape == (c.num_queries, c.hkv, c.d) and c.new_v.shape[:2] == (c.num_queries, c.hkv)
    assert np.all(c.query_pos < c.seq_lens[c.query_seq]) and np.all(c.query_pos >= 0)


def test_tiny_fp32_mha_decode():
    c = workloads.tiny_fp32_mha_decode()
    assert c.dtype == torch.float32 and (c.hq, c.hkv, c.d, c.dv, c.page_size) == (4, 4, 64, 64, 16)
    assert c.num_pages == 64 and c.seq_lens.tolist() == [1, 17, 64, 200] and c.scale == 1 / 8
    assert c.query_pos.tolist() == [0, 16, 63, 199] and c.query_seq.tolist() == [0, 1, 2, 3]
    _check_layout(c)
    assert int(np.isnan(c.k_cache.numpy().reshape(64, -1)).all(axis=1).sum()) >= 64 - 20


def test_gqa_and_long_context_shapes():
    c = workloads.gqa_decode_bf16(num_seqs=6, ctx_lo=20, ctx_hi=90)
    assert c.dtype == torch.bfloat16 and (c.hq, c.hkv, c.d, c.dv, c.page_size) == (32, 8, 128, 128, 16)
    assert all(20 <= n <= 90 for n in c.seq_lens) and c.query_pos.tolist() == [n - 1 for n in c.seq_lens]
    assert math.isclose(c.scale, 1 / math.sqrt(128))
    _check_layout(c)
    lc = workloads.long_context_decode_bf16(ctx=(40, 80))
    assert (lc.hq, lc.hkv, lc.d) == (64, 8, 128) and lc.seq_lens.tolist() == [40, 80]
    _check_layout(lc)


def test_mixed_prefill_decode_structure():
    c = workloads.mixed_prefill_decode_bf16(n_prefill=3, chunk=20, off_hi=50, n_decode=4, dec_lo=10, dec_hi=30)
    offs, chunk = c.meta["prefill_offsets"], c.meta["chunk"]
    assert len(offs) == 3 and all(0 <= o <= 50 for o in offs)
    for s, o in enumerate(offs):
        assert c.seq_lens[s] == o + chunk
        sel = c.query_seq == s
        assert c.query_pos[sel].tolist() == list(range(o, o + chunk))
    assert c.query_seq[:3 * chunk].tolist() == sorted(c.query_seq[:3 * chunk].tolist())   # prefill first
    dec = c.seq_lens[3:]
    assert all(10 <= n <= 30 for n in dec) and c.query_pos[3 * chunk:].tolist() == [n - 1 for n in dec]
    _check_layout(c)


def test_mla_structure():
    c = workloads.mla_decode_bf16(num_seqs=3, heads=4, ctx_lo=1, ctx_hi=200)
    assert c.is_mla and (c.hq, c.hkv, c.d, c.dv, c.p, c.page_size) == (4, 1, 512, 512, 64, 64)
    assert c.qp.shape == (3, 4, 64) and c.v_cache.shape[-1] == 64        # position cache rides in v_cache
    assert math.isclose(c.scale, 1 / math.sqrt(192))
    _check_layout(c)


def test_draws_repeat_per_seed():
    a = workloads.gqa_decode_bf16(num_seqs=3, ctx_lo=5, ctx_hi=40)
    b = workloads.gqa_decode_bf16(num_seqs=3, ctx_lo=5, ctx_hi=40)
    c = workloads.gqa_decode_bf16(seed=9, num_seqs=3, ctx_lo=5, ctx_hi=40)
    for name in ("q", "k_cache", "v_cache", "new_k", "new_v"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    assert np.array_equal(a.block_table, b.block_table) and np.array_equal(a.seq_lens, b.seq_lens)
    assert not torch.equal(a.q, c.q)
