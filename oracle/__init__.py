"""fp64 CPU oracle for paged attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library package never does, and the
two share no code: this module compiles ``paged_attn_oracle.c`` with the host C
compiler (plain loops, binary64, OpenMP over (query, head) rows) and calls it
through ctypes.

The functions follow ruDNN 0.1.7, src/paged_attention/mod.rs (the doc comments
of ``DevicePlan::attention``, ``DevicePlan::mla``, ``attention_into_split`` and
the body of ``append_with_report``) and boostr 0.1.0,
src/inference/decode_graph.rs (``DeviceScalars::update``: write at seq_len,
attend over seq_len + 1 keys).  The C file lists every passage and every
reading taken where the pages are silent.

Pins: every function here is checked in tests/test_oracle.py against things
other than itself (library attention on contiguous data, permutation and split
invariance, closed forms, brute force, golden fixtures).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "paged_attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS: dict[int, ctypes.CDLL] = {}

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p


def lib_path(plant: int = 0) -> str:
    return os.path.join(_BUILD, f"libpaoracle_p{plant}.so")


def build(plant: int = 0, force: bool = False) -> str:
    """Compile the oracle (optionally with a planted mistake) and return the .so path."""
    out = lib_path(plant)
    with _LOCK:
        if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
            os.makedirs(_BUILD, exist_ok=True)
            tmp = f"{out}.{os.getpid()}.tmp"
            cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                   "-shared", "-fPIC", f"-DPLANT={plant}", _SRC, "-o", tmp, "-lm"]
            subprocess.check_call(cmd)
            os.replace(tmp, out)
    return out


def _lib(plant: int = 0) -> ctypes.CDLL:
    if plant not in _LIBS:
        lib = ctypes.CDLL(build(plant))
        prob = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _i64, _i64, _i64, _i64,
                _vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64, ctypes.c_double, ctypes.c_int, _i64]
        lib.pa_oracle_attention.argtypes = prob + [_vp, _i64, _vp, _vp, ctypes.c_int]
        lib.pa_oracle_attention.restype = ctypes.c_int
        lib.pa_oracle_attention_split.argtypes = prob + [_vp, _i64, _i64, _vp, _vp, ctypes.c_int]
        lib.pa_oracle_attention_split.restype = ctypes.c_int
        lib.pa_oracle_merge.argtypes = [_vp, _vp, _i64, _i64, _i64, _vp, _vp]
        lib.pa_oracle_merge.restype = None
        lib.pa_oracle_split_range.argtypes = [_i64, _i64, _i64, _i64, _i64,
                                              ctypes.POINTER(_i64), ctypes.POINTER(_i64)]
        lib.pa_oracle_kv_store.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                           _vp, _i64, _vp, _vp, _i64]
        lib.pa_oracle_kv_store.restype = None
        lib.pa_oracle_plant.restype = ctypes.c_int
        lib.pa_oracle_threads.restype = ctypes.c_int
        _LIBS[plant] = lib
    return _LIBS[plant]


def threads() -> int:
    """Number of OpenMP threads the oracle uses by default."""
    return int(_lib().pa_oracle_threads())


def _cpu(t):
    """Contiguous CPU tensor (no copy when already so)."""
    if t is None:
        return None
    return t.detach().to("cpu").contiguous()


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _problem(q, k_cache, v_cache, seq_lens, block_table, query_seq, query_pos, scale, causal,
             qp=None, kp_cache=None, window=0):
    """Marshal tensors to the C problem arguments. Returns (args, keepalive, hq, dv)."""
    q, k_cache, v_cache, qp, kp_cache = (_cpu(t) for t in (q, k_cache, v_cache, qp, kp_cache))
    if q.dtype not in _DTYPE_CODE:
        raise TypeError(f"oracle: unsupported dtype {q.dtype}")
    for t in (k_cache, v_cache, qp, kp_cache):
        if t is not None and t.dtype != q.dtype:
            raise TypeError("oracle: all operands must share Q's dtype")
    seq_lens, query_seq, query_pos = _i32(seq_lens), _i32(query_seq), _i32(query_pos)
    block_table = _i32(block_table)
    if block_table.ndim != 2:
        block_table = block_table.reshape(len(seq_lens), -1)
    nq, hq, d = q.shape
    pages, ps, hkv, _ = k_cache.shape
    dv = v_cache.shape[3]
    p = qp.shape[2] if qp is not None else 0
    if qp is not None:
        if hkv != 1:
            raise ValueError("oracle: MLA latent cache must have one head")
        dv = d  # the latent is the value
    args = [_ptr(q), _ptr(qp), _ptr(k_cache), _ptr(v_cache), _ptr(kp_cache), _DTYPE_CODE[q.dtype],
            nq, hq, hkv, d, dv, p, _ptr(seq_lens), len(seq_lens), _ptr(block_table),
            block_table.shape[1], _ptr(query_seq), _ptr(query_pos), ps, pages, float(scale),
            1 if causal else 0, int(window)]
    keep = (q, k_cache, v_cache, qp, kp_cache, seq_lens, block_table, query_seq, query_pos)
    return args, keep, nq, hq, dv


def _rows_arg(rows, nq, hq):
    if rows is None:
        return None, nq * hq
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    if r.size and (r.min() < 0 or r.max() >= nq * hq):
        raise ValueError("oracle: row index out of range")
    return r, r.size


def attention(q, k_cache, v_cache, seq_lens, block_table, query_seq, query_pos, scale,
              causal=True, qp=None, kp_cache=None, rows=None, nthreads=0, plant=0, window=0):
    """fp64 paged attention.

    Returns (out, lse): out is float64 [Q, Hq, Dv] when rows is None, else
    [len(rows), Dv] for the flat (q * Hq + h) indices in ``rows``.  For MLA pass
    the latent cache as both k_cache and v_cache plus qp / kp_cache.  window > 0
    limits a query at position p to keys p - window + 1 and later.
    """
    args, keep, nq, hq, dv = _problem(q, k_cache, v_cache, seq_lens, block_table, query_seq,
                                      query_pos, scale, causal, qp, kp_cache, window)
    r, nrows = _rows_arg(rows, nq, hq)
    out = np.zeros((nrows, dv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = _lib(plant).pa_oracle_attention(*args, _ptr(r), nrows, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle: scratch allocation failed")
    del keep
    if rows is None:
        return out.reshape(nq, hq, dv), lse.reshape(nq, hq)
    return out, lse


def attention_split(q, k_cache, v_cache, seq_lens, block_table, query_seq, query_pos, scale,
                    splits, causal=True, qp=None, kp_cache=None, rows=None, nthreads=0, plant=0,
                    window=0):
    """Per-split partials: (out_part [S, rows, Dv], lse_part [S, rows]) in fp64."""
    args, keep, nq, hq, dv = _problem(q, k_cache, v_cache, seq_lens, block_table, query_seq,
                                      query_pos, scale, causal, qp, kp_cache, window)
    r, nrows = _rows_arg(rows, nq, hq)
    out = np.zeros((splits, nrows, dv), dtype=np.float64)
    lse = np.zeros((splits, nrows), dtype=np.float64)
    rc = _lib(plant).pa_oracle_attention_split(*args, _ptr(r), nrows, int(splits), _ptr(out),
                                               _ptr(lse), int(nthreads))
    if rc != 0:
        raise MemoryError("oracle: scratch allocation failed")
    del keep
    return out, lse


def merge(out_part, lse_part):
    """Merge split partials ([S, rows, Dv], [S, rows]) -> (out [rows, Dv], lse [rows])."""
    out_part = np.ascontiguousarray(out_part, dtype=np.float64)
    lse_part = np.ascontiguousarray(lse_part, dtype=np.float64)
    s, nrows, dv = out_part.shape
    out = np.zeros((nrows, dv), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    _lib().pa_oracle_merge(_ptr(out_part), _ptr(lse_part), s, nrows, dv, _ptr(out), _ptr(lse))
    return out, lse


def split_range(n, splits, s, page_size, lo=0):
    """[j0, j1) of split s of the visible keys [lo, n), as the oracle partitions them."""
    a, b = _i64(), _i64()
    _lib().pa_oracle_split_range(int(lo), int(n), int(splits), int(s), int(page_size),
                                 ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def kv_store(new_k, new_v, k_cache, v_cache, block_table, query_seq, query_pos):
    """Host scatter of new rows into copies of the caches; returns (k_cache', v_cache')."""
    new_k, new_v = _cpu(new_k), _cpu(new_v)
    kc, vc = _cpu(k_cache).clone(), _cpu(v_cache).clone()
    block_table = _i32(block_table)
    query_seq, query_pos = _i32(query_seq), _i32(query_pos)
    nq, heads, d = new_k.shape
    dv = new_v.shape[2]
    ps = kc.shape[1]
    _lib().pa_oracle_kv_store(_ptr(new_k), _ptr(new_v), _ptr(kc), _ptr(vc), new_k.element_size(),
                              nq, heads, d, dv, _ptr(block_table), block_table.shape[-1],
                              _ptr(query_seq), _ptr(query_pos), ps)
    return kc, vc
