"""A bounded device-side wait that runs out reports through the status word.

ruDNN 0.1.7, src/paged_attention/mod.rs, `PagedAttentionError`: every failure
is a status, nothing traps.  Every wait of the library's kernels is
pa::tc::mbar_wait with a cycle limit; when it gives up, the kernel records a
PA_DEVICE_TIMEOUT_* code in the library's device status word and returns.
Here a test-only kernel (tests/native/wait_probe.cu, linked against the
library) waits on an mbarrier that no thread arrives on, with a limit of a
few thousand cycles: the kernel must return, the status word must read
PA_DEVICE_TIMEOUT_MMA, and pa_device_status with clear must reset it.  The
same probe with its arrival made must wait successfully and leave the word
clear.  Nothing else is in flight while it runs (no cluster, TMA or MMA).
"""
import ctypes
import os
import shutil
import subprocess

import pytest

import paged_kv_attention_20_gb300 as pka

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PA_DEVICE_TIMEOUT_MMA = 2


@pytest.fixture(scope="module")
def probe(built_lib, tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    pkg = os.path.join(ROOT, "paged_kv_attention_20_gb300")
    so = str(tmp_path_factory.mktemp("waitprobe") / "wait_probe.so")
    subprocess.run([nvcc, "-O2", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                    "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", os.path.join(pkg, "csrc"),
                    os.path.join(ROOT, "tests", "native", "wait_probe.cu"), "-o", so, "-L", pkg, "-lpagedattn",
                    "-Xlinker", "-rpath," + pkg], check=True)
    lib = ctypes.CDLL(so)
    lib.probe_wait.argtypes = [ctypes.c_longlong, ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
    lib.probe_wait.restype = ctypes.c_int
    return lib


def _run(probe, limit, arrive):
    out = (ctypes.c_int32 * 2)()
    assert probe.probe_wait(limit, arrive, out) == 0
    return out[0], out[1]


def test_wait_that_runs_out_sets_and_clears_the_status(cuda_device, probe):
    assert pka.device_status(clear=True) == 0          # start clear
    result, cycles = _run(probe, 4000, arrive=0)
    assert result == 2, "the wait on a barrier nobody arrives on must give up"
    assert cycles >= 4000
    assert pka.device_status(clear=False) == PA_DEVICE_TIMEOUT_MMA
    assert pka.device_status(clear=True) == PA_DEVICE_TIMEOUT_MMA   # read, then cleared
    assert pka.device_status(clear=False) == 0


def test_wait_that_completes_leaves_the_status_clear(cuda_device, probe):
    result, _ = _run(probe, 4000, arrive=1)
    assert result == 1
    assert pka.device_status(clear=True) == 0
