"""Seeded synthetic inputs for the paged-attention workloads.

Shared by the tests and the benchmark.  This module only draws random numbers
and lays them out: it holds none of the attention arithmetic (no scores, no
softmax, no gather, no cache writes).  Every case is reproducible from its seed.

A case holds:
  * the schedule: seq_lens [S], block_table [S, W] (unused entries -1),
    query_seq [Q], query_pos [Q], page_size, num_pages;
  * packed Q [Q, Hq, D] (and position Q [Q, H, P] for MLA);
  * paged caches [pages, page_size, Hkv, D|Dv] filled with N(0, 1) draws in the
    case's dtype, with every page that no sequence references and every slot
    past a sequence's length set to NaN, so a stray read shows in the output;
  * new rows [Q, Hkv, D|Dv] that a cache append writes at the queries' slots.

For MLA the "k" cache is the latent cache [pages, ps, 1, R] and the "v" cache
the rotated position cache [pages, ps, 1, P] (the append writes both); the
attention reads the latent as key and value.

The named workloads follow the page shapes of the paged-attention problem
statement: tiny fp32 MHA decode, Llama-3-8B-like GQA decode, long-context
split decode, mixed chunked prefill + decode, and MLA decode.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass
class PagedCase:
    name: str
    dtype: torch.dtype
    seq_lens: np.ndarray
    block_table: np.ndarray
    query_seq: np.ndarray
    query_pos: np.ndarray
    page_size: int
    num_pages: int
    hq: int
    hkv: int
    d: int
    dv: int
    scale: float
    causal: bool
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    new_k: torch.Tensor
    new_v: torch.Tensor
    qp: torch.Tensor | None = None      # MLA position Q [Q, H, P]
    p: int = 0                          # MLA position dim (0 = not MLA)
    meta: dict = field(default_factory=dict)

    @property
    def num_queries(self) -> int:
        return int(self.query_seq.shape[0])

    @property
    def is_mla(self) -> bool:
        return self.qp is not None

    def to(self, device) -> "PagedCase":
        """Copy of the case with every tensor on ``device``."""
        kw = dict(self.__dict__)
        for name in ("q", "k_cache", "v_cache", "new_k", "new_v", "qp"):
            if kw[name] is not None:
                kw[name] = kw[name].to(device)
        kw["meta"] = dict(self.meta)
        return PagedCase(**kw)


def _randn(gen: torch.Generator, shape, dtype, chunk=1 << 24) -> torch.Tensor:
    """N(0,1) draws made in fp32, rounded once to ``dtype`` (chunked to bound memory)."""
    out = torch.empty(shape, dtype=dtype)
    flat = out.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, dtype=torch.float32).to(dtype)
    return out


def build_case(name, seed, seq_lens, queries, hq, hkv, d, dv, page_size, dtype, scale,
               causal=True, pool_pages=None, mla_p=0, poison=True) -> PagedCase:
    """Lay out a paged problem.

    seq_lens: context length of each sequence (keys present after the append).
    queries:  list of (seq, absolute position) in packing order.
    pool_pages: physical pool size (default: exactly the pages used).
    mla_p: > 0 makes an MLA case (hkv must be 1, dv is the position dim P).
    """
    gen = torch.Generator().manual_seed(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    n_pages = [(int(n) + page_size - 1) // page_size for n in seq_lens]
    used = int(sum(n_pages))
    pool = used if pool_pages is None else int(pool_pages)
    if pool < used:
        raise ValueError("pool smaller than the pages in use")
    width = max(1, max(n_pages) if n_pages else 1)
    perm = torch.randperm(pool, generator=gen).numpy().astype(np.int64)
    table = np.full((len(seq_lens), width), -1, dtype=np.int64)
    off = 0
    for s, n in enumerate(n_pages):
        table[s, :n] = perm[off:off + n]
        off += n

    nq = len(queries)
    qseq = np.array([int(a) for a, _ in queries], dtype=np.int32)
    qpos = np.array([int(b) for _, b in queries], dtype=np.int32)
    if mla_p:
        if hkv != 1:
            raise ValueError("MLA cases have one latent head")
        q = _randn(gen, (nq, hq, d), dtype)
        qp = _randn(gen, (nq, hq, mla_p), dtype)
    else:
        q = _randn(gen, (nq, hq, d), dtype)
        qp = None
    k_cache = _randn(gen, (pool, page_size, hkv, d), dtype)
    v_cache = _randn(gen, (pool, page_size, hkv, dv), dtype)
    new_k = _randn(gen, (nq, hkv, d), dtype)
    new_v = _randn(gen, (nq, hkv, dv), dtype)

    if poison:
        referenced = np.zeros(pool, dtype=bool)
        for s, n in enumerate(n_pages):
            referenced[table[s, :n]] = True
            tail = int(seq_lens[s]) - (n - 1) * page_size   # live rows in the last page
            if n and tail < page_size:
                last = int(table[s, n - 1])
                k_cache[last, tail:] = float("nan")
                v_cache[last, tail:] = float("nan")
        dead = torch.from_numpy(np.nonzero(~referenced)[0])
        if dead.numel():
            k_cache[dead] = float("nan")
            v_cache[dead] = float("nan")

    return PagedCase(name=name, dtype=dtype, seq_lens=seq_lens.astype(np.int32),
                     block_table=table.astype(np.int32), query_seq=qseq, query_pos=qpos,
                     page_size=page_size, num_pages=pool, hq=hq, hkv=hkv, d=d,
                     dv=(d if mla_p else dv), scale=float(scale), causal=causal, q=q,
                     k_cache=k_cache, v_cache=v_cache, new_k=new_k, new_v=new_v, qp=qp,
                     p=int(mla_p), meta={"seed": seed})


def _uniform_ints(gen: torch.Generator, n, lo, hi) -> list[int]:
    """n integers uniform in [lo, hi] inclusive."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def decode_queries(seq_lens):
    """One decode query per sequence at position ctx - 1 (its own key is the newest)."""
    return [(s, int(n) - 1) for s, n in enumerate(seq_lens)]


# ---------------------------------------------------------------------------
# Named workloads.  Their keyword arguments shrink batch sizes and context
# ranges for parity cases the oracle finishes in seconds, keeping the structure.
# ---------------------------------------------------------------------------

def tiny_fp32_mha_decode(seed=1) -> PagedCase:
    """4 sequences, contexts {1,17,64,200}, Hq=Hkv=4, D=Dv=64, ps=16, 64-page pool, fp32."""
    ctx = [1, 17, 64, 200]
    c = build_case("tiny_fp32_mha_decode", seed, ctx, decode_queries(ctx), 4, 4, 64, 64, 16,
                   torch.float32, 1.0 / 8.0, pool_pages=64)
    return c


def gqa_decode_bf16(seed=2, num_seqs=64, ctx_lo=512, ctx_hi=8192) -> PagedCase:
    """Llama-3-8B-like decode layer: Hq=32, Hkv=8, D=Dv=128, ps=16, bf16, contexts U[lo,hi]."""
    gen = torch.Generator().manual_seed(seed * 7919 + 1)
    ctx = _uniform_ints(gen, num_seqs, ctx_lo, ctx_hi)
    return build_case("gqa_decode_bf16", seed, ctx, decode_queries(ctx), 32, 8, 128, 128, 16,
                      torch.bfloat16, 1.0 / math.sqrt(128))


def long_context_decode_bf16(seed=3, ctx=(32768, 65536, 98304, 131072)) -> PagedCase:
    """Long-context split-KV decode: Hq=64, Hkv=8, D=Dv=128, ps=16, bf16."""
    return build_case("long_context_split_decode_bf16", seed, list(ctx), decode_queries(ctx), 64, 8,
                      128, 128, 16, torch.bfloat16, 1.0 / math.sqrt(128))


def mixed_prefill_decode_bf16(seed=4, n_prefill=8, chunk=512, off_hi=4096, n_decode=120,
                              dec_lo=1024, dec_hi=4096) -> PagedCase:
    """Chunked prefill (n_prefill chunks of `chunk` queries at offsets U[0, off_hi]) + decode.

    Prefill sequence i holds o_i cached keys and appends a chunk at positions
    o_i .. o_i + chunk - 1 (seq_len = o_i + chunk); decode sequences have
    contexts U[dec_lo, dec_hi] with their query at ctx - 1.  Queries are packed
    in sequence order, prefill chunks first.  Hq=32, Hkv=8, D=Dv=128, ps=16.
    """
    gen = torch.Generator().manual_seed(seed * 7919 + 1)
    offs = _uniform_ints(gen, n_prefill, 0, off_hi)
    dctx = _uniform_ints(gen, n_decode, dec_lo, dec_hi)
    seq_lens = [o + chunk for o in offs] + dctx
    queries = []
    for s, o in enumerate(offs):
        queries += [(s, o + i) for i in range(chunk)]
    queries += [(n_prefill + s, n - 1) for s, n in enumerate(dctx)]
    c = build_case("mixed_prefill_decode_bf16", seed, seq_lens, queries, 32, 8, 128, 128, 16,
                   torch.bfloat16, 1.0 / math.sqrt(128))
    c.meta.update(prefill_offsets=offs, chunk=chunk, n_prefill=n_prefill, n_decode=n_decode)
    return c


def mla_decode_bf16(seed=5, num_seqs=128, heads=128, ctx_lo=1024, ctx_hi=16384) -> PagedCase:
    """MLA decode: H heads, latent R=512, position P=64, ps=64, scale 1/sqrt(128+64)."""
    gen = torch.Generator().manual_seed(seed * 7919 + 1)
    ctx = _uniform_ints(gen, num_seqs, ctx_lo, ctx_hi)
    return build_case("mla_decode_bf16", seed, ctx, decode_queries(ctx), heads, 1, 512, 64, 64,
                      torch.bfloat16, 1.0 / math.sqrt(192), mla_p=64)


WORKLOADS = {
    "tiny_fp32_mha_decode": tiny_fp32_mha_decode,
    "gqa_decode_bf16": gqa_decode_bf16,
    "long_context_split_decode_bf16": long_context_decode_bf16,
    "mixed_prefill_decode_bf16": mixed_prefill_decode_bf16,
    "mla_decode_bf16": mla_decode_bf16,
}

