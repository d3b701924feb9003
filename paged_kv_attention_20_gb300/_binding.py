"""ctypes binding of libpagedattn.so: argument marshalling only.

Every computation happens in the library's CUDA kernels.  This module checks
what only the Python side can see (tensor device, dtype, contiguity, rank,
storage overlap of the output with the inputs -- ruDNN 0.1.7,
src/paged_attention/mod.rs, `attention_into`: "the PyTorch adapter enforces
storage-overlap checks"), passes raw pointers and the current CUDA stream, and
turns non-OK statuses into exceptions.  If the library is missing it raises;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import buildlib as _build

_LIB = None

PA_OK = 0
STATUS_NAMES = {0: "PA_OK", 1: "PA_ERR_ARG", 2: "PA_ERR_SHAPE", 3: "PA_ERR_DTYPE", 4: "PA_ERR_RANGE",
                5: "PA_ERR_WRITE_CONFLICT", 6: "PA_ERR_WORKSPACE", 7: "PA_ERR_SPLITS", 8: "PA_ERR_LIMIT",
                9: "PA_ERR_CUDA", 10: "PA_ERR_STATE"}
_DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
MAX_SPLITS = 64

EXPORTED = ["pa_last_error", "pa_status_string", "pa_abi_version", "paged_attn_plan",
            "pa_plan_device_bytes", "pa_plan_upload", "pa_plan_stage", "pa_plan_destroy", "pa_plan_describe",
            "pa_workspace_bytes", "paged_attn_split_heuristic", "paged_mla_split_heuristic",
            "paged_attn_decode_sms_beside_prefill", "paged_kv_store", "paged_attn_forward",
            "paged_attn_forward_split", "paged_mla_forward", "pa_plan_advance", "pa_time_next_kernel",
            "pa_device_status"]


class PagedAttentionError(RuntimeError):
    """A library call returned a status other than PA_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libpagedattn.so (built by build.build()); raise if it is missing."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with paged_kv_attention_20_gb300.build() "
                           "(nvcc, sm_103a); there is no fallback path")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.pa_last_error.restype = ctypes.c_char_p
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_abi_version.restype = i32
    lib.paged_attn_plan.argtypes = [vp, i32, vp, i32, vp, vp, i32, i32, i32, ctypes.POINTER(vp)]
    lib.paged_attn_plan.restype = ctypes.c_int
    lib.pa_plan_device_bytes.argtypes = [vp]
    lib.pa_plan_device_bytes.restype = sz
    lib.pa_plan_upload.argtypes = [vp, vp, sz, vp]
    lib.pa_plan_upload.restype = ctypes.c_int
    lib.pa_plan_stage.argtypes = [vp, vp, sz, vp, sz]
    lib.pa_plan_stage.restype = ctypes.c_int
    lib.pa_plan_destroy.argtypes = [vp]
    lib.pa_plan_destroy.restype = None
    lib.pa_plan_describe.argtypes = [vp, ctypes.POINTER(i64)]
    lib.pa_plan_describe.restype = ctypes.c_int
    lib.pa_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.pa_workspace_bytes.restype = sz
    lib.paged_attn_split_heuristic.argtypes = [vp, i32, i32, i32, i32]
    lib.paged_attn_split_heuristic.restype = i32
    lib.paged_mla_split_heuristic.argtypes = [vp, i32, i32, i32]
    lib.paged_mla_split_heuristic.restype = i32
    lib.paged_attn_decode_sms_beside_prefill.argtypes = [vp, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.paged_attn_decode_sms_beside_prefill.restype = i32
    lib.paged_kv_store.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int, vp]
    lib.paged_kv_store.restype = ctypes.c_int
    lib.paged_attn_forward.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, i32, i32,
                                       ctypes.c_int, vp]
    lib.paged_attn_forward.restype = ctypes.c_int
    lib.paged_attn_forward_split.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, ctypes.c_float, i32,
                                             i32, ctypes.c_int, vp, sz, i32, vp]
    lib.paged_attn_forward_split.restype = ctypes.c_int
    lib.paged_mla_forward.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_float, i32, i32,
                                      ctypes.c_int, vp, sz, i32, vp]
    lib.paged_mla_forward.restype = ctypes.c_int
    lib.pa_plan_advance.argtypes = [vp, vp]
    lib.pa_plan_advance.restype = ctypes.c_int
    lib.pa_time_next_kernel.argtypes = [vp, vp]
    lib.pa_time_next_kernel.restype = ctypes.c_int
    lib.pa_device_status.argtypes = [ctypes.POINTER(i32), i32]
    lib.pa_device_status.restype = ctypes.c_int
    _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, load().pa_last_error().decode())


def _i32_array(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


class Plan:
    """A validated schedule (`paged_attn_plan`) and, once uploaded, its device copy."""

    def __init__(self, handle: int, counts: np.ndarray):
        self._handle = ctypes.c_void_p(handle)
        self.queries, self.sequences, self.width, self.page_size, self.pages = (int(x) for x in counts[:5])
        self.n_decode, self.n_tiles, self.n_tile_queries = (int(x) for x in counts[5:8])
        self.words = None
        self.device = None

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._handle

    def device_bytes(self) -> int:
        return int(load().pa_plan_device_bytes(self._handle))

    def upload(self, device=None) -> "Plan":
        """Allocate the metadata buffer on `device` and enqueue its upload on the current stream."""
        device = torch.device(device if device is not None else "cuda")
        n = self.device_bytes()
        self.words = torch.empty(max(16, n), dtype=torch.uint8, device=device)
        self.device = self.words.device
        _check(load().pa_plan_upload(self._handle, self.words.data_ptr(), self.words.numel(),
                                     _stream(self.device)))
        return self

    def upload_into(self, words: torch.Tensor) -> "Plan":
        """Upload into a caller-provided device byte buffer (reused across steps)."""
        self.words = words
        self.device = words.device
        _check(load().pa_plan_upload(self._handle, words.data_ptr(), words.numel(), _stream(words.device)))
        return self

    def stage(self, host_words: torch.Tensor, device_words: torch.Tensor) -> "Plan":
        """Write the device image into `host_words` (CPU uint8, e.g. pinned) and bind `device_words`.

        Nothing is copied to the device: the caller copies host_words into
        device_words on its stream (capturable in a CUDA graph) before the
        next call that uses this plan.
        """
        for t, name, on_cuda in ((host_words, "host_words", False), (device_words, "device_words", True)):
            if t.dtype != torch.uint8 or not t.is_contiguous() or t.is_cuda != on_cuda:
                raise ValueError(f"{name} must be a contiguous uint8 {'CUDA' if on_cuda else 'CPU'} tensor")
        _check(load().pa_plan_stage(self._handle, host_words.data_ptr(), host_words.numel(),
                                    device_words.data_ptr(), device_words.numel()))
        self.words = device_words
        self.device = device_words.device
        return self

    def __del__(self):
        h = getattr(self, "_handle", None)
        if h is not None and h.value and _LIB is not None:
            _LIB.pa_plan_destroy(h)
            self._handle = ctypes.c_void_p(0)


def paged_attn_plan(seq_lens, block_table, query_seq, query_pos, page_size: int, num_pages: int,
                    device=None, upload: bool = True) -> Plan:
    """Build (and by default upload) a schedule; see paged_attn_plan in paged_attn.h."""
    lib = load()
    seq_lens = _i32_array(seq_lens)
    bt = _i32_array(block_table)
    if bt.ndim == 1:
        bt = bt.reshape(len(seq_lens), -1) if len(seq_lens) else bt.reshape(0, 0)
    width = int(bt.shape[1]) if bt.ndim == 2 else 0
    qs, qp = _i32_array(query_seq), _i32_array(query_pos)
    if qs.shape != qp.shape:
        raise ValueError("query_seq and query_pos must have the same length")
    handle = ctypes.c_void_p()
    _check(lib.paged_attn_plan(seq_lens.ctypes.data, len(seq_lens), bt.ctypes.data, width, qs.ctypes.data,
                               qp.ctypes.data, len(qs), int(page_size), int(num_pages), ctypes.byref(handle)))
    counts = (ctypes.c_int64 * 8)()
    _check(lib.pa_plan_describe(handle, counts))
    plan = Plan(handle.value, np.array(counts[:], dtype=np.int64))
    if upload:
        plan.upload(device)
    return plan


def _tensor(t: torch.Tensor, name: str, dtype, device, rank: int) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dim() != rank:
        raise ValueError(f"{name} must have rank {rank}")


def _storage_span(t: torch.Tensor):
    start = t.data_ptr()
    return start, start + t.numel() * t.element_size()


def _check_disjoint(out: torch.Tensor, *inputs) -> None:
    o0, o1 = _storage_span(out)
    for t in inputs:
        if t is None or t.numel() == 0:
            continue
        a0, a1 = _storage_span(t)
        if a0 < o1 and o0 < a1:
            raise ValueError("output overlaps an input tensor")


def _plan_ready(plan: Plan, device) -> None:
    if plan.words is None:
        raise ValueError("plan has not been uploaded")
    if plan.device != device:
        raise ValueError(f"plan metadata is on {plan.device}, tensors on {device}")


def workspace_bytes(queries: int, heads: int, value_dim: int, splits: int) -> int:
    return int(load().pa_workspace_bytes(int(queries), int(heads), int(value_dim), int(splits)))


def make_workspace(plan: Plan, heads: int, value_dim: int, splits: int, device=None) -> torch.Tensor:
    """Caller-owned fp32 workspace sized for `splits` partials."""
    n = workspace_bytes(plan.queries, heads, value_dim, splits)
    return torch.empty((n + 3) // 4, dtype=torch.float32, device=device or plan.device)


def paged_attn_split_heuristic(plan: Plan, num_heads: int, num_kv_heads: int, num_sms: int | None = None,
                               window: int = 0) -> int:
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(plan.device or 0).multi_processor_count
    return int(load().paged_attn_split_heuristic(plan.handle, int(num_heads), int(num_kv_heads), int(window),
                                                 int(num_sms)))


def paged_mla_split_heuristic(plan: Plan, num_heads: int, num_sms: int | None = None, window: int = 0) -> int:
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(plan.device or 0).multi_processor_count
    return int(load().paged_mla_split_heuristic(plan.handle, int(num_heads), int(window), int(num_sms)))


def paged_attn_decode_sms_beside_prefill(plan: Plan, num_heads: int, num_kv_heads: int, head_dim: int,
                                         value_dim: int, causal: bool = True, window: int = 0,
                                         dtype=torch.bfloat16, num_sms: int | None = None) -> int:
    """SMs an attention call on this plan leaves to its decode items beside the prefill tiles (0: serial)."""
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(plan.device or 0).multi_processor_count
    return int(load().paged_attn_decode_sms_beside_prefill(plan.handle, int(num_heads), int(num_kv_heads),
                                                           int(head_dim), int(value_dim), 1 if causal else 0,
                                                           int(window), _DTYPES[dtype], int(num_sms)))


def paged_kv_store(plan: Plan, new_k, new_v, k_cache, v_cache) -> None:
    """Append new_k [Q, H, d] / new_v [Q, H, dv] into the caches at the plan's slots."""
    dev = k_cache.device
    dt = k_cache.dtype
    for name, t, r in (("new_k", new_k, 3), ("new_v", new_v, 3), ("k_cache", k_cache, 4), ("v_cache", v_cache, 4)):
        _tensor(t, name, dt, dev, r)
    _plan_ready(plan, dev)
    heads, d, dv = k_cache.shape[2], k_cache.shape[3], v_cache.shape[3]
    if tuple(k_cache.shape[:3]) != tuple(v_cache.shape[:3]) or k_cache.shape[0] != plan.pages \
            or k_cache.shape[1] != plan.page_size:
        raise ValueError("cache shapes do not match the plan")
    if tuple(new_k.shape) != (plan.queries, heads, d) or tuple(new_v.shape) != (plan.queries, heads, dv):
        raise ValueError("new rows must be [queries, heads, d|dv]")
    _check(load().paged_kv_store(plan.handle, new_k.data_ptr(), new_v.data_ptr(), k_cache.data_ptr(),
                                 v_cache.data_ptr(), heads, d, dv, _DTYPES[dt], _stream(dev)))


def _attn_common(plan, q, k_cache, v_cache, out):
    dev, dt = q.device, q.dtype
    if dt not in _DTYPES:
        raise TypeError("dtype must be float32, float16 or bfloat16")
    _tensor(q, "q", dt, dev, 3)
    _tensor(k_cache, "k_cache", dt, dev, 4)
    _tensor(v_cache, "v_cache", dt, dev, 4)
    _plan_ready(plan, dev)
    if k_cache.shape[0] != plan.pages or k_cache.shape[1] != plan.page_size \
            or tuple(k_cache.shape[:3]) != tuple(v_cache.shape[:3]):
        raise ValueError("cache shapes do not match the plan")
    if q.shape[0] != plan.queries or q.shape[2] != k_cache.shape[3]:
        raise ValueError("q must be [queries, num_heads, head_dim] matching the plan and cache")
    shape = (q.shape[0], q.shape[1], v_cache.shape[3])
    if out is None:
        out = torch.empty(shape, dtype=dt, device=dev)
    else:
        _tensor(out, "out", dt, dev, 3)
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    _check_disjoint(out, q, k_cache, v_cache)
    return out


def paged_attn_forward(plan: Plan, q, k_cache, v_cache, scale: float, causal: bool = True, out=None,
                       window: int = 0):
    """Paged MHA/GQA attention; returns out [queries, num_heads, value_dim].
    window > 0: a query at position p sees keys p - window + 1 and later."""
    out = _attn_common(plan, q, k_cache, v_cache, out)
    _check(load().paged_attn_forward(plan.handle, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                     out.data_ptr(), q.shape[1], k_cache.shape[2], q.shape[2],
                                     v_cache.shape[3], float(scale), 1 if causal else 0, int(window),
                                     _DTYPES[q.dtype], _stream(q.device)))
    return out


def paged_attn_forward_split(plan: Plan, q, k_cache, v_cache, scale: float, splits: int, workspace=None,
                             causal: bool = True, out=None, window: int = 0):
    """Split-KV paged attention with an fp32 workspace (allocated here when not given)."""
    out = _attn_common(plan, q, k_cache, v_cache, out)
    if workspace is None:
        workspace = make_workspace(plan, q.shape[1], v_cache.shape[3], splits, q.device)
    _check_disjoint(out, workspace)
    _check(load().paged_attn_forward_split(plan.handle, q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           out.data_ptr(), q.shape[1], k_cache.shape[2], q.shape[2],
                                           v_cache.shape[3], float(scale), 1 if causal else 0, int(window),
                                           _DTYPES[q.dtype], workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(), int(splits),
                                           _stream(q.device)))
    return out


def paged_mla_forward(plan: Plan, q, qp, latent_cache, pos_cache, scale: float, causal: bool = True,
                      workspace=None, splits: int = 1, out=None, window: int = 0):
    """MLA attention over a shared latent head plus a rotated position cache."""
    dev, dt = q.device, q.dtype
    if dt not in _DTYPES:
        raise TypeError("dtype must be float32, float16 or bfloat16")
    _tensor(q, "q", dt, dev, 3)
    _tensor(qp, "qp", dt, dev, 3)
    _tensor(latent_cache, "latent_cache", dt, dev, 4)
    _tensor(pos_cache, "pos_cache", dt, dev, 4)
    _plan_ready(plan, dev)
    if latent_cache.shape[2] != 1 or pos_cache.shape[2] != 1:
        raise ValueError("MLA latent cache must have one shared head")
    if latent_cache.shape[0] != plan.pages or latent_cache.shape[1] != plan.page_size \
            or tuple(pos_cache.shape[:2]) != tuple(latent_cache.shape[:2]):
        raise ValueError("cache shapes do not match the plan")
    if q.shape[0] != plan.queries or q.shape[2] != latent_cache.shape[3] or tuple(qp.shape[:2]) != tuple(q.shape[:2]) \
            or qp.shape[2] != pos_cache.shape[3]:
        raise ValueError("incompatible MLA query / cache dimensions")
    shape = tuple(q.shape)
    if out is None:
        out = torch.empty(shape, dtype=dt, device=dev)
    else:
        _tensor(out, "out", dt, dev, 3)
        if tuple(out.shape) != shape:
            raise ValueError(f"out must have shape {shape}")
    if splits > 1 and workspace is None:
        workspace = make_workspace(plan, q.shape[1], q.shape[2], splits, dev)
    _check_disjoint(out, q, qp, latent_cache, pos_cache, workspace)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().paged_mla_forward(plan.handle, q.data_ptr(), qp.data_ptr(), latent_cache.data_ptr(),
                                    pos_cache.data_ptr(), out.data_ptr(), q.shape[1], q.shape[2], qp.shape[2],
                                    float(scale), 1 if causal else 0, int(window), _DTYPES[dt], ws_ptr, ws_bytes,
                                    int(splits), _stream(dev)))
    return out


def paged_attn_plan_advance(plan: Plan) -> None:
    """Move every query of a decode plan one position forward, on the device (graph-capturable)."""
    if plan.words is None:
        raise ValueError("plan has not been uploaded")
    _check(load().pa_plan_advance(plan.handle, _stream(plan.device)))


def time_next_kernel(start: torch.cuda.Event, stop: torch.cuda.Event) -> None:
    """Have the next attention call record `start`/`stop` around its main kernel."""
    for ev in (start, stop):
        if not ev.cuda_event:   # torch creates the CUDA event lazily
            ev.record()
    _check(load().pa_time_next_kernel(start.cuda_event, stop.cuda_event))


def device_status(clear: bool = True) -> int:
    """Synchronise and read (and clear) the device timeout word; 0 means no wait ran out."""
    code = ctypes.c_int32(0)
    _check(load().pa_device_status(ctypes.byref(code), 1 if clear else 0))
    return int(code.value)
