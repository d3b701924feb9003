"""The kernels' split partition against the oracle's, on the host.

ruDNN 0.1.7, src/paged_attention/mod.rs (`attention_into_split`: the visible
history is split, each split's FP32 statistics merged) and libmir-cuda 0.1.0,
src/backend/attention/graph/mod.rs (`Geometry::window`).  The kernels take
every query's visible range and split ranges from two inline host/device
helpers; here those helpers are compiled for the host and compared, over
random positions, lengths, windows, split counts and page sizes, with the
oracle's own partition, and the ranges are checked to tile the visible keys:
in order, without gap or overlap, every split but the first starting on a
page boundary.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    so = str(tmp_path_factory.mktemp("probe") / "split_probe.so")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "paged_kv_attention_20_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "native", "split_probe.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    i, p = ctypes.c_int, ctypes.POINTER(ctypes.c_longlong)
    lib.probe_split_bounds.argtypes = [i, i, i, i, i, i, i, p, p, p, p]
    lib.probe_split_bounds.restype = None
    return lib


def _kernel_split(lib, pos, seq_len, causal, window, splits, s, ps):
    v = [ctypes.c_longlong() for _ in range(4)]
    lib.probe_split_bounds(pos, seq_len, causal, window, splits, s, ps, *[ctypes.byref(x) for x in v])
    return tuple(x.value for x in v)


def test_kernel_partition_matches_the_oracle(probe):
    rng = np.random.default_rng(8)
    checked = 0
    for _ in range(4000):
        ps = int(rng.choice([1, 3, 8, 16, 64, 256]))
        seq_len = int(rng.integers(1, 20000))
        pos = int(rng.integers(0, seq_len))
        causal = int(rng.integers(0, 2))
        window = int(rng.choice([0, 0, 1, int(rng.integers(1, 3000)), 100000]))
        splits = int(rng.choice([1, 2, 3, 5, 8, 19, 64]))
        # the documented visible range: [pos - W + 1 (W > 0), causal end pos + 1 or seq_len)
        lo = max(0, pos - window + 1) if window > 0 else 0
        hi = pos + 1 if causal else seq_len
        prev = lo
        for s in range(splits):
            klo, khi, j0, j1 = _kernel_split(probe, pos, seq_len, causal, window, splits, s, ps)
            assert (klo, khi) == (lo, hi)
            assert (j0, j1) == oracle.split_range(hi, splits, s, ps, lo), (pos, seq_len, causal, window, splits, s, ps)
            if j1 > j0:
                assert j0 == prev, "splits must tile the range in order"
                assert s == 0 or j0 % ps == 0 or j0 == lo
                prev = j1
            checked += 1
        assert prev == hi, "the splits together cover every visible key"
    assert checked > 20000
