"""Shared test plumbing: run a workload through the C ABI and through the oracle.

Tolerances (the paged-attention parity bar):
  * fp32 operands: max |gpu - oracle| <= 1e-5 * RMS(oracle output);
  * bf16 / fp16 operands: max |gpu - oracle| <= 2e-2 absolute (fp32 accumulation),
    the oracle reading the same rounded inputs;
  * the cache append: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_attention_20_gb300 as pka

FP32_REL_RMS = 1e-5
HALF_ABS = 2e-2


def tolerance(dtype, ref: np.ndarray) -> float:
    if dtype == torch.float32:
        rms = float(np.sqrt(np.mean(ref.astype(np.float64) ** 2))) if ref.size else 1.0
        return FP32_REL_RMS * rms
    return HALF_ABS


def assert_close(gpu: np.ndarray, ref: np.ndarray, dtype, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, f"{what}: shape {gpu.shape} vs {ref.shape}"
    assert np.isfinite(gpu).all(), f"{what}: non-finite GPU output"
    err = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    tol = tolerance(dtype, ref)
    assert err <= tol, f"{what}: max abs err {err:.3e} > tol {tol:.3e}"
    return err


def plan_for(case, device="cuda"):
    return pka.paged_attn_plan(case.seq_lens, case.block_table, case.query_seq, case.query_pos,
                               case.page_size, case.num_pages, device=device)


def gpu_store_and_attend(case, splits=None, workspace=None, causal=None, device="cuda", window=0):
    """Append the case's new rows, then attend.  Returns (out_cpu, k_cache_cpu, v_cache_cpu, plan)."""
    dc = case.to(device)
    plan = plan_for(case, device)
    pka.paged_kv_store(plan, dc.new_k, dc.new_v, dc.k_cache, dc.v_cache)
    causal = case.causal if causal is None else causal
    if case.is_mla:
        out = pka.paged_mla_forward(plan, dc.q, dc.qp, dc.k_cache, dc.v_cache, case.scale, causal=causal,
                                    workspace=workspace, splits=splits or 1, window=window)
    elif splits is None:
        out = pka.paged_attn_forward(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, causal=causal,
                                     window=window)
    else:
        out = pka.paged_attn_forward_split(plan, dc.q, dc.k_cache, dc.v_cache, case.scale, splits,
                                           workspace=workspace, causal=causal, window=window)
    torch.cuda.synchronize()
    assert pka.device_status() == 0, "a device-side wait timed out"
    return out.cpu(), dc.k_cache.cpu(), dc.v_cache.cpu(), plan


def oracle_after_store(case, rows=None, causal=None, nthreads=0, window=0):
    """Oracle: host append of the new rows, then fp64 attention (optionally on sampled rows)."""
    kc, vc = oracle.kv_store(case.new_k, case.new_v, case.k_cache, case.v_cache, case.block_table,
                             case.query_seq, case.query_pos)
    causal = case.causal if causal is None else causal
    if case.is_mla:
        out, lse = oracle.attention(case.q, kc, kc, case.seq_lens, case.block_table, case.query_seq,
                                    case.query_pos, case.scale, causal=causal, qp=case.qp, kp_cache=vc,
                                    rows=rows, nthreads=nthreads, window=window)
    else:
        out, lse = oracle.attention(case.q, kc, vc, case.seq_lens, case.block_table, case.query_seq,
                                    case.query_pos, case.scale, causal=causal, rows=rows, nthreads=nthreads,
                                    window=window)
    return out, lse, kc, vc


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a.view(torch.int16), b.view(torch.int16))
