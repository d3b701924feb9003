"""Pins of the fp64 oracle against things other than itself (CPU only).

Each pin checks the oracle against an independent statement of what paged
attention computes (ruDNN 0.1.7, src/paged_attention/mod.rs, doc comments of
`DevicePlan::attention`, `DevicePlan::mla`, `attention_into_split`; the
append in `append_with_report`; boostr 0.1.0, src/inference/decode_graph.rs,
`DeviceScalars::update` for the write-then-attend convention):

  * library attention (torch SDPA, float64, explicit absolute-position mask)
    on contiguous per-sequence data that the test itself scatters into pages;
  * MLA as ordinary attention with K = [latent | kp], V = latent, one KV head;
  * invariance of the bits under a new physical page permutation;
  * split + merge equal to the unsplit result for 1..64 splits;
  * one visible key -> the value row exactly; equal scores -> mean of V;
  * log-sum-exp against scipy.special.logsumexp;
  * a naive pure-Python loop on tiny inputs;
  * the sliding window (a layer's `window`, libmir-cuda 0.1.0,
    src/backend/attention/graph/mod.rs, `Geometry`; read as: a query at
    position p sees keys p - W + 1 and later) against SDPA with a band mask,
    its two limits (W = 1: the own key's value row; W > p: no window), split
    invariance and brute force;
  * closed-form worked examples in tests/golden/closed_forms.json;
  * the append as a page-level round trip.

`test_planted_mistakes_are_caught` recompiles the oracle with one deliberate
mistake at a time and checks that some pin fails for each.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

import oracle
from workloads import build_case, decode_queries

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


# ----------------------------------------------------------------- helpers --

def paged_from_contiguous(per_seq, table, page_size, pages, fill=float("nan")):
    """Scatter contiguous per-sequence rows [n, H, E] into a fresh paged cache,
    one whole page at a time (logical page g of sequence s -> table[s, g])."""
    h, e = per_seq[0].shape[1:]
    cache = torch.full((pages, page_size, h, e), fill, dtype=per_seq[0].dtype)
    for s, rows in enumerate(per_seq):
        n = rows.shape[0]
        for g in range((n + page_size - 1) // page_size):
            chunk = rows[g * page_size:(g + 1) * page_size]
            cache[int(table[s, g]), :chunk.shape[0]] = chunk
    return cache


def random_layout(seed, seq_lens, page_size, extra_pages=3):
    gen = torch.Generator().manual_seed(seed)
    n_pages = [(n + page_size - 1) // page_size for n in seq_lens]
    pool = sum(n_pages) + extra_pages
    perm = torch.randperm(pool, generator=gen).numpy()
    table = np.full((len(seq_lens), max(n_pages)), -1, dtype=np.int32)
    off = 0
    for s, n in enumerate(n_pages):
        table[s, :n] = perm[off:off + n]
        off += n
    return table, pool


def sdpa_reference(q, k_seq, v_seq, query_seq, query_pos, scale, causal, hkv, window=0):
    """float64 SDPA per query on contiguous data; GQA by repeat_interleave;
    window > 0 adds a band mask (keys j >= pos - window + 1)."""
    nq, hq, _ = q.shape
    outs = []
    for i in range(nq):
        s, pos = int(query_seq[i]), int(query_pos[i])
        k = k_seq[s].double().repeat_interleave(hq // hkv, dim=1)     # [n, Hq, D]
        v = v_seq[s].double().repeat_interleave(hq // hkv, dim=1)
        n = k.shape[0]
        mask = torch.ones(1, n, dtype=torch.bool)
        if causal:
            mask = (torch.arange(n) <= pos).view(1, n)
        if window > 0:
            mask = mask & (torch.arange(n) >= pos - window + 1).view(1, n)
        o = F.scaled_dot_product_attention(
            q[i].double().unsqueeze(1),            # [Hq, 1, D]
            k.transpose(0, 1), v.transpose(0, 1),  # [Hq, n, D]
            attn_mask=mask, scale=scale)
        outs.append(o.squeeze(1))
    return torch.stack(outs).numpy()


def contiguous_problem(seed, seq_lens, queries, hq, hkv, d, dv, page_size, dtype, causal, p=0):
    gen = torch.Generator().manual_seed(seed)
    k_seq = [torch.randn(n, hkv, d, generator=gen).to(dtype) for n in seq_lens]
    v_seq = [torch.randn(n, hkv, dv, generator=gen).to(dtype) for n in seq_lens]
    kp_seq = [torch.randn(n, 1, p, generator=gen).to(dtype) for n in seq_lens] if p else None
    q = torch.randn(len(queries), hq, d, generator=gen).to(dtype)
    qp = torch.randn(len(queries), hq, p, generator=gen).to(dtype) if p else None
    table, pool = random_layout(seed + 1, seq_lens, page_size)
    qseq = np.array([a for a, _ in queries], dtype=np.int32)
    qpos = np.array([b for _, b in queries], dtype=np.int32)
    return dict(k_seq=k_seq, v_seq=v_seq, kp_seq=kp_seq, q=q, qp=qp, table=table, pool=pool,
                qseq=qseq, qpos=qpos, seq_lens=np.array(seq_lens, dtype=np.int32))


# -------------------------------------------------------------------- pins --

def pin_sdpa_mha_gqa(plant=0):
    for (hq, hkv, causal, dtype, ps) in [(4, 4, True, torch.float32, 4), (8, 2, True, torch.bfloat16, 8),
                                         (6, 3, False, torch.float16, 4), (4, 1, True, torch.float32, 16)]:
        seq_lens = [1, 5, 17, 33]
        queries = decode_queries(seq_lens) + [(3, 10), (2, 0), (1, 2), (3, 31)]
        pr = contiguous_problem(11 + hq, seq_lens, queries, hq, hkv, 16, 12, ps, dtype, causal)
        kc = paged_from_contiguous(pr["k_seq"], pr["table"], ps, pr["pool"])
        vc = paged_from_contiguous(pr["v_seq"], pr["table"], ps, pr["pool"])
        out, _ = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                                  0.37, causal=causal, plant=plant)
        ref = sdpa_reference(pr["q"], pr["k_seq"], pr["v_seq"], pr["qseq"], pr["qpos"], 0.37, causal, hkv)
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def pin_sdpa_mla(plant=0):
    seq_lens = [3, 40, 65]
    queries = decode_queries(seq_lens) + [(2, 7)]
    pr = contiguous_problem(5, seq_lens, queries, 8, 1, 24, 24, 16, torch.bfloat16, True, p=6)
    lat = paged_from_contiguous(pr["k_seq"], pr["table"], 16, pr["pool"])
    kpc = paged_from_contiguous(pr["kp_seq"], pr["table"], 16, pr["pool"])
    out, _ = oracle.attention(pr["q"], lat, lat, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                              0.21, causal=True, qp=pr["qp"], kp_cache=kpc, plant=plant)
    kcat = [torch.cat([k, kp], dim=-1) for k, kp in zip(pr["k_seq"], pr["kp_seq"])]
    qcat = torch.cat([pr["q"], pr["qp"]], dim=-1)
    ref = sdpa_reference(qcat, kcat, pr["k_seq"], pr["qseq"], pr["qpos"], 0.21, True, 1)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def pin_permutation_invariance(plant=0):
    seq_lens = [9, 30, 47]
    queries = decode_queries(seq_lens) + [(1, 3), (2, 20)]
    pr = contiguous_problem(21, seq_lens, queries, 4, 2, 8, 8, 4, torch.bfloat16, True)
    results = []
    for layout_seed in (100, 200, 300):
        table, pool = random_layout(layout_seed, seq_lens, 4, extra_pages=5)
        kc = paged_from_contiguous(pr["k_seq"], table, 4, pool)
        vc = paged_from_contiguous(pr["v_seq"], table, 4, pool)
        out, lse = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], table, pr["qseq"], pr["qpos"],
                                    0.5, causal=True, plant=plant)
        results.append((out, lse))
    for out, lse in results[1:]:
        assert np.array_equal(out, results[0][0]) and np.array_equal(lse, results[0][1])


def pin_split_invariance(plant=0):
    seq_lens = [1, 16, 17, 100, 257]
    case = build_case("split", 31, seq_lens, decode_queries(seq_lens) + [(4, 130)], 4, 2, 16, 16, 16,
                      torch.float32, 0.25)
    args = (case.q, case.k_cache, case.v_cache, case.seq_lens, case.block_table, case.query_seq,
            case.query_pos, case.scale)
    out, lse = oracle.attention(*args, plant=plant)
    for s in (1, 2, 3, 7, 16, 64):
        op, lp = oracle.attention_split(*args, splits=s, plant=plant)
        mo, ml = oracle.merge(op, lp)
        np.testing.assert_allclose(mo.reshape(out.shape), out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(ml.reshape(lse.shape), lse, rtol=1e-12, atol=1e-12)


def pin_single_key(plant=0):
    # Every query sits at position 0 (causal): it sees exactly its own key.
    seq_lens = [1, 5, 20]
    queries = [(0, 0), (1, 0), (2, 0)]
    pr = contiguous_problem(41, seq_lens, queries, 4, 2, 8, 8, 4, torch.float32, True)
    kc = paged_from_contiguous(pr["k_seq"], pr["table"], 4, pr["pool"])
    vc = paged_from_contiguous(pr["v_seq"], pr["table"], 4, pr["pool"])
    out, lse = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                                0.3, causal=True, plant=plant)
    for i, (s, _) in enumerate(queries):
        v0 = pr["v_seq"][s][0].double().repeat_interleave(2, dim=0).numpy()
        assert np.array_equal(out[i], v0)
        k0 = pr["k_seq"][s][0].double().repeat_interleave(2, dim=0)
        sc = 0.3 * (pr["q"][i].double() * k0).sum(-1).numpy()
        np.testing.assert_allclose(lse[i], sc, rtol=1e-13, atol=1e-13)


def pin_equal_scores(plant=0):
    seq_lens = [7, 40]
    queries = decode_queries(seq_lens) + [(1, 12)]
    pr = contiguous_problem(51, seq_lens, queries, 2, 1, 8, 8, 8, torch.float32, True)
    pr["q"].zero_()
    kc = paged_from_contiguous(pr["k_seq"], pr["table"], 8, pr["pool"])
    vc = paged_from_contiguous(pr["v_seq"], pr["table"], 8, pr["pool"])
    out, lse = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                                1.0, causal=True, plant=plant)
    for i, (s, pos) in enumerate(queries):
        mean = pr["v_seq"][s][:pos + 1, 0].double().mean(0).numpy()
        for h in range(2):
            np.testing.assert_allclose(out[i, h], mean, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse[i, h], math.log(pos + 1), rtol=1e-13)


def pin_logsumexp(plant=0):
    seq_lens = [23, 64]
    queries = decode_queries(seq_lens) + [(1, 5)]
    pr = contiguous_problem(61, seq_lens, queries, 4, 2, 16, 16, 16, torch.bfloat16, True)
    kc = paged_from_contiguous(pr["k_seq"], pr["table"], 16, pr["pool"])
    vc = paged_from_contiguous(pr["v_seq"], pr["table"], 16, pr["pool"])
    _, lse = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                              0.125, causal=True, plant=plant)
    for i, (s, pos) in enumerate(queries):
        k = pr["k_seq"][s][:pos + 1].double()                         # [n, Hkv, D]
        for h in range(4):
            sc = 0.125 * (k[:, h // 2, :] @ pr["q"][i, h].double()).numpy()
            np.testing.assert_allclose(lse[i, h], logsumexp(sc), rtol=1e-13, atol=1e-13)


def naive_python(q, k_seq, v_seq, qseq, qpos, scale, causal, window=0):
    nq, hq, d = len(q), len(q[0]), len(q[0][0])
    out = []
    for i in range(nq):
        rows = []
        for h in range(hq):
            kk, vv = k_seq[qseq[i]], v_seq[qseq[i]]
            hkv = len(kk[0])
            g = hq // hkv
            n = qpos[i] + 1 if causal else len(kk)
            first = max(0, qpos[i] - window + 1) if window > 0 else 0
            keys = list(range(first, n))
            sc = [scale * sum(q[i][h][e] * kk[j][h // g][e] for e in range(d)) for j in keys]
            m = max(sc)
            w = [math.exp(x - m) for x in sc]
            tot = sum(w)
            rows.append([sum(w[t] * vv[j][h // g][e] for t, j in enumerate(keys)) / tot
                         for e in range(len(vv[0][0]))])
        out.append(rows)
    return np.array(out)


def pin_brute_force(plant=0):
    seq_lens = [3, 8, 6]
    queries = [(0, 2), (1, 7), (1, 4), (2, 5), (2, 0)]
    for causal in (True, False):
        pr = contiguous_problem(71, seq_lens, queries, 4, 2, 4, 3, 2, torch.float32, causal)
        kc = paged_from_contiguous(pr["k_seq"], pr["table"], 2, pr["pool"])
        vc = paged_from_contiguous(pr["v_seq"], pr["table"], 2, pr["pool"])
        out, _ = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                                  0.7, causal=causal, plant=plant)
        ref = naive_python(pr["q"].double().tolist(), [k.double().tolist() for k in pr["k_seq"]],
                           [v.double().tolist() for v in pr["v_seq"]], pr["qseq"].tolist(),
                           pr["qpos"].tolist(), 0.7, causal)
        np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-14)


def pin_window(plant=0):
    """Sliding window: SDPA with a band mask, the limits W = 1 and W > p,
    split invariance under the window, and brute force."""
    seq_lens = [1, 9, 33, 70]
    queries = decode_queries(seq_lens) + [(3, 40), (2, 5), (3, 0), (1, 3)]
    for (hq, hkv, causal, dtype, ps) in [(4, 2, True, torch.float32, 8), (6, 3, False, torch.bfloat16, 4)]:
        pr = contiguous_problem(91 + hq, seq_lens, queries, hq, hkv, 16, 12, ps, dtype, causal)
        kc = paged_from_contiguous(pr["k_seq"], pr["table"], ps, pr["pool"])
        vc = paged_from_contiguous(pr["v_seq"], pr["table"], ps, pr["pool"])
        args = (pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"], 0.41)
        for w in (1, 2, 5, 17, 64):
            out, lse = oracle.attention(*args, causal=causal, window=w, plant=plant)
            ref = sdpa_reference(pr["q"], pr["k_seq"], pr["v_seq"], pr["qseq"], pr["qpos"], 0.41, causal, hkv,
                                 window=w)
            np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
            for sp in (2, 3, 8):
                op, lp = oracle.attention_split(*args, splits=sp, causal=causal, window=w, plant=plant)
                mo, ml = oracle.merge(op, lp)
                np.testing.assert_allclose(mo.reshape(out.shape), out, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(ml.reshape(lse.shape), lse, rtol=1e-12, atol=1e-12)
        if causal:
            # W = 1: each query sees only its own key
            out, _ = oracle.attention(*args, causal=True, window=1, plant=plant)
            for i, (sq, pos) in enumerate(queries):
                v = pr["v_seq"][sq][pos].double().repeat_interleave(hq // hkv, dim=0).numpy()
                assert np.array_equal(out[i], v)
        # a window longer than every position is no window, bit for bit
        o0, l0 = oracle.attention(*args, causal=causal, plant=plant)
        o1, l1 = oracle.attention(*args, causal=causal, window=1000, plant=plant)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    # brute force on a tiny case
    seq_lens = [3, 8, 6]
    queries = [(0, 2), (1, 7), (1, 4), (2, 5), (2, 0)]
    pr = contiguous_problem(97, seq_lens, queries, 4, 2, 4, 3, 2, torch.float32, True)
    kc = paged_from_contiguous(pr["k_seq"], pr["table"], 2, pr["pool"])
    vc = paged_from_contiguous(pr["v_seq"], pr["table"], 2, pr["pool"])
    for w in (2, 3):
        out, _ = oracle.attention(pr["q"], kc, vc, pr["seq_lens"], pr["table"], pr["qseq"], pr["qpos"],
                                  0.7, causal=True, window=w, plant=plant)
        ref = naive_python(pr["q"].double().tolist(), [k.double().tolist() for k in pr["k_seq"]],
                           [v.double().tolist() for v in pr["v_seq"]], pr["qseq"].tolist(),
                           pr["qpos"].tolist(), 0.7, True, window=w)
        np.testing.assert_allclose(out, ref, rtol=1e-14, atol=1e-14)


def _nan_tensor(x):
    a = np.array(x, dtype=object)
    a = np.where(a == None, np.nan, a).astype(np.float64)  # noqa: E711
    return torch.from_numpy(a).float()


def pin_golden(plant=0):
    doc = json.load(open(GOLDEN))
    for c in doc["cases"]:
        q = _nan_tensor(c["q"])
        table = np.array(c["block_table"], dtype=np.int32)
        kw = {}
        if "latent" in c:
            kc = vc = _nan_tensor(c["latent"])
            kw = dict(qp=_nan_tensor(c["qp"]), kp_cache=_nan_tensor(c["kp_cache"]))
        else:
            kc, vc = _nan_tensor(c["k_cache"]), _nan_tensor(c["v_cache"])
        for mode in ("causal", "noncausal"):
            if mode not in c:
                continue
            out, lse = oracle.attention(q, kc, vc, c["seq_lens"], table, c["query_seq"], c["query_pos"],
                                        c["scale"], causal=(mode == "causal"), plant=plant, **kw)
            np.testing.assert_allclose(out, np.array(c[mode]["out"]), rtol=1e-14, atol=1e-15)
            np.testing.assert_allclose(lse, np.array(c[mode]["lse"]), rtol=1e-14, atol=1e-15)


def pin_store_round_trip(plant=0):
    seq_lens = [5, 18, 33]
    queries = [(0, 4), (1, 16), (1, 17), (2, 0), (2, 32)]
    pr = contiguous_problem(81, seq_lens, queries, 2, 2, 8, 4, 4, torch.bfloat16, True)
    kc = paged_from_contiguous(pr["k_seq"], pr["table"], 4, pr["pool"], fill=-7.0)
    vc = paged_from_contiguous(pr["v_seq"], pr["table"], 4, pr["pool"], fill=-7.0)
    gen = torch.Generator().manual_seed(3)
    new_k = torch.randn(len(queries), 2, 8, generator=gen).bfloat16()
    new_v = torch.randn(len(queries), 2, 4, generator=gen).bfloat16()
    k2, v2 = oracle.kv_store(new_k, new_v, kc, vc, pr["table"], pr["qseq"], pr["qpos"])
    # Expected: contiguous sequences with the queried positions overwritten, re-paged whole.
    ek = [k.clone() for k in pr["k_seq"]]
    ev = [v.clone() for v in pr["v_seq"]]
    for i, (s, pos) in enumerate(queries):
        ek[s][pos] = new_k[i]
        ev[s][pos] = new_v[i]
    assert torch.equal(k2.view(torch.int16), paged_from_contiguous(ek, pr["table"], 4, pr["pool"], -7.0).view(torch.int16))
    assert torch.equal(v2.view(torch.int16), paged_from_contiguous(ev, pr["table"], 4, pr["pool"], -7.0).view(torch.int16))


PINS = [pin_sdpa_mha_gqa, pin_sdpa_mla, pin_permutation_invariance, pin_split_invariance,
        pin_single_key, pin_equal_scores, pin_logsumexp, pin_brute_force, pin_golden,
        pin_store_round_trip, pin_window]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin()


def test_split_range_partition():
    """Splits tile [0, n) in page-multiple chunks, in order, with no gap or overlap."""
    for n in (1, 15, 16, 17, 100, 4096, 131072):
        for s_count in (1, 2, 3, 8, 64):
            prev = 0
            for s in range(s_count):
                a, b = oracle.split_range(n, s_count, s, 16)
                assert a == prev and b >= a
                assert (b - a) % 16 == 0 or b == n
                prev = b
            assert prev == n
    # under a window the visible keys start at lo; later split starts fall on page boundaries
    for lo, n in ((5, 40), (37, 100), (64, 65), (1000, 131072)):
        for s_count in (1, 2, 5, 64):
            prev = lo
            for s in range(s_count):
                a, b = oracle.split_range(n, s_count, s, 16, lo=lo)
                assert a == prev and b >= a
                assert a == lo or a % 16 == 0 or a == n
                prev = b
            assert prev == n


def test_workload_shapes():
    c = build_case("t", 1, [1, 17], decode_queries([1, 17]), 4, 2, 8, 8, 16, torch.bfloat16, 0.3,
                   pool_pages=5)
    assert c.k_cache.shape == (5, 16, 2, 8)
    assert c.block_table.shape == (2, 2)
    # unreferenced pages and tail slots are NaN
    used = set(c.block_table[c.block_table >= 0].tolist())
    for pgi in range(5):
        if pgi not in used:
            assert torch.isnan(c.k_cache[pgi].float()).all()
    assert torch.isnan(c.k_cache[int(c.block_table[0, 0]), 1:].float()).all()
    assert not torch.isnan(c.k_cache[int(c.block_table[0, 0]), 0].float()).any()


@pytest.mark.parametrize("plant", [1, 2, 3, 4, 5, 6])
def test_planted_mistakes_are_caught(plant):
    """Each deliberately broken oracle build must fail at least one pin."""
    failures = 0
    for pin in PINS:
        try:
            pin(plant=plant)
        except AssertionError:
            failures += 1
    assert failures >= 1, f"planted mistake {plant} slipped through every pin"


def test_rows_and_thread_counts_give_the_same_bits():
    """The sampled parity tests ask the oracle for chosen (query, head) rows on
    many threads: those must be exactly the rows of the full single-threaded
    result, for plain, windowed and split attention and for MLA."""
    import workloads
    rng = np.random.default_rng(11)
    c = workloads.gqa_decode_bf16(num_seqs=5, ctx_lo=30, ctx_hi=400)
    args = (c.q, c.k_cache, c.v_cache, c.seq_lens, c.block_table, c.query_seq, c.query_pos, c.scale)
    nrows = c.num_queries * c.hq
    rows = np.sort(rng.choice(nrows, 37, replace=False))
    for window in (0, 50):
        full, lse = oracle.attention(*args, window=window, nthreads=1)
        many, lse_many = oracle.attention(*args, window=window, nthreads=8)
        assert np.array_equal(full, many) and np.array_equal(lse, lse_many)
        sub, lse_sub = oracle.attention(*args, window=window, rows=rows, nthreads=3)
        assert np.array_equal(sub, full.reshape(nrows, -1)[rows]) and np.array_equal(lse_sub, lse.reshape(-1)[rows])
        part, lpart = oracle.attention_split(*args, splits=5, window=window, nthreads=1)
        psub, lpsub = oracle.attention_split(*args, splits=5, window=window, rows=rows, nthreads=4)
        assert np.array_equal(psub, part[:, rows]) and np.array_equal(lpsub, lpart[:, rows])
    m = workloads.mla_decode_bf16(num_seqs=3, heads=8, ctx_lo=10, ctx_hi=300)
    margs = (m.q, m.k_cache, m.k_cache, m.seq_lens, m.block_table, m.query_seq, m.query_pos, m.scale)
    mfull, _ = oracle.attention(*margs, qp=m.qp, kp_cache=m.v_cache, nthreads=1)
    mrows = np.array([0, 5, 9, 23])
    msub, _ = oracle.attention(*margs, qp=m.qp, kp_cache=m.v_cache, rows=mrows, nthreads=6)
    assert np.array_equal(msub, mfull.reshape(m.num_queries * m.hq, -1)[mrows])
