"""Host-only checks of the C ABI (no GPU calls).

* libpagedattn.so loads and exports every function include/paged_attn.h declares;
* schedule validation (ruDNN 0.1.7, src/paged_attention/mod.rs, `HostPlan` use,
  `validate_writes`, `bounded`) rejects bad input with the documented status;
* argument checks of the attention entry points (`execute_attention_into`)
  fire before anything touches the device;
* the work lists, workspace sizing and split heuristic behave as documented.
"""
import ctypes
import os
import re

import numpy as np
import torch
import pytest

import paged_kv_attention_20_gb300 as pka
from paged_kv_attention_20_gb300._binding import PagedAttentionError

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "paged_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if not n.startswith("defined")))


def test_header_functions_are_exported(built_lib):
    names = declared_functions()
    assert "paged_attn_forward" in names and "paged_kv_store" in names and len(names) >= 15
    for n in names:
        assert hasattr(built_lib, n), f"{n} declared in paged_attn.h but not exported"
    assert set(pka.EXPORTED) <= set(names)
    assert built_lib.pa_abi_version() == 3


def _status_of(fn, *a, **k):
    with pytest.raises(PagedAttentionError) as ei:
        fn(*a, **k)
    return ei.value.status


def plan(*a, **k):
    return pka.paged_attn_plan(*a, upload=False, **k)


def test_plan_validation_statuses(built_lib):
    ok = plan([5, 20], [[0, 1], [2, 3]], [0, 1], [4, 19], 16, 4)
    assert ok.queries == 2 and ok.n_decode == 2 and ok.n_tiles == 0
    # page id outside the pool
    assert _status_of(plan, [5, 20], [[0, 1], [2, 9]], [0, 1], [4, 19], 16, 4) == 4
    # position beyond the sequence
    assert _status_of(plan, [5, 20], [[0, 1], [2, 3]], [0, 1], [5, 19], 16, 4) == 4
    # negative position
    assert _status_of(plan, [5, 20], [[0, 1], [2, 3]], [0, 1], [-1, 19], 16, 4) == 4
    # sequence longer than its table row
    assert _status_of(plan, [5, 40], [[0, 1], [2, 3]], [0, 1], [4, 19], 16, 4) == 4
    # query names a missing sequence
    assert _status_of(plan, [5, 20], [[0, 1], [2, 3]], [0, 2], [4, 19], 16, 4) == 4
    # two queries of one plan write the same slot (also across sequences sharing a page)
    assert _status_of(plan, [5, 20], [[0, 1], [2, 3]], [1, 1], [19, 19], 16, 4) == 5
    assert _status_of(plan, [5, 5], [[0, 1], [0, 3]], [0, 1], [4, 4], 16, 4) == 5
    # page_size must be positive
    assert _status_of(plan, [5], [[0]], [0], [4], 0, 4) == 1
    # slot indexing beyond 32 bits
    assert _status_of(plan, [5], [[0]], [0], [4], 1 << 16, 1 << 16) == 4


def test_shared_pages_for_reads_are_allowed(built_lib):
    # two sequences share physical page 0 as a common prefix; they write different pages
    p = plan([20, 20], [[0, 1], [0, 2]], [0, 1], [19, 19], 16, 3)
    assert p.n_decode == 2


def test_unused_table_entries_are_ignored(built_lib):
    p = plan([5], [[2, -1, 77]], [0], [4], 16, 3)
    assert p.queries == 1


def test_work_lists_split_runs_into_tiles(built_lib):
    # sequence 0: a 300-query prefill run; sequence 1: a 10-query run (decode items);
    # sequence 2: one decode query
    q_seq = [0] * 300 + [1] * 10 + [2]
    q_pos = list(range(100, 400)) + list(range(50, 60)) + [7]
    p = plan([400, 60, 8], [[i for i in range(25)], [30 + i for i in range(25)], [60] + [0] * 24],
             q_seq, q_pos, 16, 61)
    assert p.n_tiles == 3 and p.n_tile_queries == 300      # 128 + 128 + 44
    assert p.n_decode == 11


def test_empty_plan(built_lib):
    p = plan([], np.zeros((0, 0), dtype=np.int32), [], [], 16, 0)
    assert p.queries == 0 and p.device_bytes() % 16 == 0


def test_workspace_bytes(built_lib):
    n = pka.workspace_bytes(4, 64, 128, 64)
    assert n == ((64 * 4 * 64 * 128 * 4 + 255) // 256 * 256) + ((64 * 4 * 64 * 4 + 255) // 256 * 256)
    assert pka.workspace_bytes(4, 0, 128, 2) == 0
    assert pka.workspace_bytes(4, 64, 128, 0) == 0


def test_split_heuristic(built_lib):
    lens = [32768, 65536, 98304, 131072]
    table = np.arange(sum(n // 16 for n in lens), dtype=np.int32)
    rows, off = [], 0
    for n in lens:
        rows.append(np.pad(table[off:off + n // 16], (0, 8192 - n // 16)))
        off += n // 16
    p = plan(lens, np.stack(rows), [0, 1, 2, 3], [n - 1 for n in lens], 16, int(table.size))
    s = pka.paged_attn_split_heuristic(p, 64, 8, num_sms=152)
    assert 8 <= s <= 64
    small = plan([20], [[0, 1]], [0], [19], 16, 2)
    assert pka.paged_attn_split_heuristic(small, 8, 8, num_sms=152) == 1   # one page: no split
    # a sliding window bounds the history the heuristic splits
    assert pka.paged_attn_split_heuristic(p, 64, 8, num_sms=152, window=64) == 1
    assert pka.paged_attn_split_heuristic(p, 64, 8, num_sms=152, window=4096) <= 4096 // 64


def test_split_heuristic_fills_rounds_for_large_groups(built_lib):
    """Groups of 8+ (persistent tensor-core decode): about four rounds of units, last round nearly full."""
    lens = [32768, 65536, 98304, 131072]
    table = np.arange(sum(n // 16 for n in lens), dtype=np.int32)
    rows, off = [], 0
    for n in lens:
        rows.append(np.pad(table[off:off + n // 16], (0, 8192 - n // 16)))
        off += n // 16
    p = plan(lens, np.stack(rows), [0, 1, 2, 3], [n - 1 for n in lens], 16, int(table.size))
    for sms in (152, 148, 100, 132):
        s = pka.paged_attn_split_heuristic(p, 64, 8, num_sms=sms)
        units = 4 * 8 * s
        rounds = -(-units // sms)
        assert 3 <= rounds <= 6, (sms, s)
        assert units / (rounds * sms) >= 0.9, (sms, s)     # the last round is (nearly) full
    assert pka.paged_attn_split_heuristic(p, 64, 8, num_sms=152) == 19    # 608 units = 4 x 152


def test_plan_stage_writes_the_device_image(built_lib):
    """pa_plan_stage: the image goes to a host buffer, the device buffer is only bound."""
    import torch
    lens, table = [5, 40], [[3, -1, -1], [2, 4, 1]]
    p = plan(lens, np.array(table), [0, 1, 1], [4, 38, 39], 16, 5)
    n = p.device_bytes()
    host = torch.zeros(n + 64, dtype=torch.uint8)
    fake = 0x10000                                     # bound, never dereferenced on the host
    lib = _lib()
    assert lib.pa_plan_stage(p.handle, host.data_ptr(), n + 64, ctypes.c_void_p(fake), n) == 0
    words = host[:n].view(torch.int32).numpy()
    assert np.all(host[n:].numpy() == 0)               # nothing past the image is written
    flat = np.array(table, dtype=np.int32).ravel()
    hits = [i for i in range(words.size - flat.size + 1) if np.array_equal(words[i:i + flat.size], flat)]
    assert hits and hits[0] % 4 == 0                   # the block table sits in a 16-byte aligned section
    again = torch.zeros(n, dtype=torch.uint8)
    assert lib.pa_plan_stage(p.handle, again.data_ptr(), n, ctypes.c_void_p(fake), n) == 0
    assert torch.equal(again, host[:n])
    assert lib.pa_plan_stage(p.handle, host.data_ptr(), n - 1, ctypes.c_void_p(fake), n) == 1   # short host
    assert lib.pa_plan_stage(p.handle, host.data_ptr(), n, ctypes.c_void_p(fake), n - 16) == 1  # short device
    assert lib.pa_plan_stage(p.handle, host.data_ptr(), n, ctypes.c_void_p(fake + 4), n) == 1   # misaligned
    assert lib.pa_plan_stage(p.handle, None, n, ctypes.c_void_p(fake), n) == 1


def _mla_plan(lens):
    """One decode query per history, pages laid out back to back (ps = 64)."""
    pages = [(n + 63) // 64 for n in lens]
    width = max(pages)
    table, off = np.zeros((len(lens), width), dtype=np.int32), 0
    for i, n in enumerate(pages):
        table[i, :n] = np.arange(off, off + n)
        off += n
    return plan(lens, table, list(range(len(lens))), [n - 1 for n in lens], 64, off)


def test_mla_split_heuristic(built_lib):
    """The MLA kernel is tensor-bound: split only to fill SM pairs or to cut a dominant history."""
    rng = np.random.default_rng(0)
    many = _mla_plan([int(x) for x in rng.integers(1024, 16385, size=128)])
    assert pka.paged_mla_split_heuristic(many, 128, num_sms=152) == 1        # 128 pairs already cover 76 slots
    few = _mla_plan([8192] * 4)
    s = pka.paged_mla_split_heuristic(few, 128, num_sms=152)
    assert 19 <= s <= 8192 // 256                                            # 4 x s items fill 76 pair slots
    skew = _mla_plan([131072] + [1024] * 100)                                # one history holds most keys
    assert pka.paged_mla_split_heuristic(skew, 128, num_sms=152) > 1
    assert pka.paged_mla_split_heuristic(few, 128, num_sms=152, window=1024) == 4   # >= 256 keys per split
    assert pka.paged_mla_split_heuristic(_mla_plan([100]), 128, num_sms=152) == 1
    assert 1 <= pka.paged_mla_split_heuristic(_mla_plan([1 << 20]), 128, num_sms=4096) <= 64


def _lib():
    return pka.load()


def test_attention_argument_checks_before_launch(built_lib):
    """Bad heads, dims, scale, splits or workspace are refused with no device work."""
    lib = _lib()
    p = plan([5], [[0]], [0], [4], 16, 1)
    h = p.handle
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails validation first
    f = lib.paged_attn_forward
    assert f(h, fake, fake, fake, fake, 6, 4, 64, 64, 0.1, 1, 0, 2, None) == 2          # Hq % Hkv
    assert f(h, fake, fake, fake, fake, 0, 1, 64, 64, 0.1, 1, 0, 2, None) == 2          # Hq == 0
    assert f(h, fake, fake, fake, fake, 4, 4, 1025, 64, 0.1, 1, 0, 2, None) == 8        # d > 1024
    assert f(h, fake, fake, fake, fake, 4, 4, 64, 0, 0.1, 1, 0, 2, None) == 2           # dv == 0
    assert f(h, fake, fake, fake, fake, 4, 4, 64, 64, float("nan"), 1, 0, 2, None) == 2  # scale NaN
    assert f(h, fake, fake, fake, fake, 4, 4, 64, 64, -1.0, 1, 0, 2, None) == 2         # scale <= 0
    assert f(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 7, None) == 3          # dtype
    assert f(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, -1, 2, None) == 1         # window < 0
    assert f(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 2, None) == 10         # not uploaded
    fs = lib.paged_attn_forward_split
    assert fs(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 2, fake, 1 << 20, 65, None) == 7
    assert fs(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 2, fake, 1 << 20, 0, None) == 7
    assert fs(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 2, fake, 16, 4, None) == 6   # too small
    assert fs(h, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 2, None, 1 << 20, 4, None) == 6
    m = lib.paged_mla_forward
    assert m(h, fake, fake, fake, fake, fake, 4, 64, 0, 0.1, 1, 0, 2, None, 0, 1, None) == 8     # P == 0
    assert m(h, fake, fake, fake, fake, fake, 4, 64, 257, 0.1, 1, 0, 2, None, 0, 1, None) == 8   # P > 256
    assert m(h, fake, fake, fake, fake, fake, 4, 64, 64, 0.1, 1, 0, 2, None, 0, 2, None) == 7    # split w/o ws
    assert m(h, fake, fake, fake, fake, fake, 4, 64, 64, 0.1, 1, -3, 2, None, 0, 1, None) == 1   # window < 0
    st = lib.paged_kv_store
    assert st(h, fake, fake, fake, fake, 0, 64, 64, 2, None) == 2
    assert st(h, fake, fake, fake, fake, 1, 64, 64, 9, None) == 3
    assert st(h, fake, fake, fake, fake, 1, 64, 64, 2, None) == 10                     # not uploaded
    assert st(None, fake, fake, fake, fake, 1, 64, 64, 2, None) == 1
    assert lib.pa_last_error().decode().startswith("paged_kv_store")


def test_zero_queries_is_ok_without_launch(built_lib):
    lib = _lib()
    p = plan([5], [[0]], [], [], 16, 1)
    fake = ctypes.c_void_p(0x1000)
    assert lib.paged_attn_forward(p.handle, fake, fake, fake, fake, 4, 4, 64, 64, 0.1, 1, 0, 2, None) == 0
    assert lib.paged_kv_store(p.handle, fake, fake, fake, fake, 1, 64, 64, 2, None) == 0


def test_plan_advance_refusals(built_lib):
    lib = _lib()
    # a plan with a prefill run (>= 16 consecutive positions) cannot advance
    p = plan([40], [[0, 1, 2]], [0] * 20, list(range(20)), 16, 3)
    assert p.n_tiles == 1
    assert lib.pa_plan_advance(p.handle, None) == 10
    # a decode plan must be uploaded first
    d = plan([5], [[0]], [0], [4], 16, 1)
    assert lib.pa_plan_advance(d.handle, None) == 10
    assert lib.pa_plan_advance(None, None) == 1


def test_status_names_and_per_thread_messages(built_lib):
    """pa_status_string names every status the header declares; a failed call's
    message stays with the thread that made it."""
    import threading
    lib = _lib()
    text = open(HEADER).read()
    enum = re.search(r"typedef enum \{(.*?)\} pa_status;", text, flags=re.S).group(1)
    codes = {name: int(v) for name, v in re.findall(r"(PA_[A-Z_]+)\s*=\s*(\d+)", enum)}
    assert codes["PA_OK"] == 0 and len(codes) == 11
    for name, v in codes.items():
        assert lib.pa_status_string(v).decode() == name
    assert lib.pa_status_string(99).decode() == "PA_UNKNOWN"
    with pytest.raises(PagedAttentionError) as ei:
        plan([5], [[0]], [0], [9], 16, 1)                      # position past the sequence
    assert ei.value.status == codes["PA_ERR_RANGE"]
    assert "position" in lib.pa_last_error().decode()
    seen = {}
    t = threading.Thread(target=lambda: seen.setdefault("msg", lib.pa_last_error().decode()))
    t.start()
    t.join()
    assert seen["msg"] == ""                                     # nothing failed on that thread


def _mixed_plan(offs, chunk, dctx, ps=16):
    """Prefill chunks (chunk queries at offsets offs) then one decode query per history in dctx."""
    lens = [o + chunk for o in offs] + list(dctx)
    pages = [(n + ps - 1) // ps for n in lens]
    width = max(pages)
    table, off = np.full((len(lens), width), -1, dtype=np.int32), 0
    for i, n in enumerate(pages):
        table[i, :n] = np.arange(off, off + n)
        off += n
    qs, qp = [], []
    for s, o in enumerate(offs):
        qs += [s] * chunk
        qp += list(range(o, o + chunk))
    for i, n in enumerate(dctx):
        qs.append(len(offs) + i)
        qp.append(n - 1)
    return plan(lens, table, qs, qp, ps, off)


def test_decode_sms_beside_prefill(built_lib):
    """Mixed calls share the SMs only when both halves are large; the share stays a minority."""
    rng = np.random.default_rng(4)
    offs = [int(x) for x in rng.integers(0, 4097, size=8)]
    dctx = [int(x) for x in rng.integers(1024, 4097, size=120)]
    big = _mixed_plan(offs, 512, dctx)
    n = pka.paged_attn_decode_sms_beside_prefill(big, 32, 8, 128, 128, num_sms=152)
    assert 8 <= n <= 60, n                                   # the mixed workload's size: a share for the decode
    assert pka.paged_attn_decode_sms_beside_prefill(big, 32, 8, 128, 128, dtype=torch.float16, num_sms=152) == n
    # prefill tiles that the tensor-core prefill kernel does not take (fp32, other head sizes) stay serial
    assert pka.paged_attn_decode_sms_beside_prefill(big, 32, 8, 128, 128, dtype=torch.float32, num_sms=152) == 0
    assert pka.paged_attn_decode_sms_beside_prefill(big, 32, 8, 64, 64, num_sms=152) == 0
    # no decode items, or no prefill tiles, or halves too small: one after the other
    assert pka.paged_attn_decode_sms_beside_prefill(_mixed_plan(offs, 512, []), 32, 8, 128, 128, num_sms=152) == 0
    assert pka.paged_attn_decode_sms_beside_prefill(_mixed_plan([], 512, dctx), 32, 8, 128, 128, num_sms=152) == 0
    small = _mixed_plan([100], 64, [300, 500])
    assert pka.paged_attn_decode_sms_beside_prefill(small, 32, 8, 128, 128, num_sms=152) == 0
    # a window shrinks both halves; a tiny window leaves nothing worth splitting
    assert pka.paged_attn_decode_sms_beside_prefill(big, 32, 8, 128, 128, window=64, num_sms=152) == 0
    # invalid arguments
    assert pka.paged_attn_decode_sms_beside_prefill(big, 0, 8, 128, 128, num_sms=152) == 0
    assert pka.paged_attn_decode_sms_beside_prefill(big, 32, 8, 128, 128, num_sms=0) == 0
    lib = pka.load()
    assert lib.paged_attn_decode_sms_beside_prefill(None, 32, 8, 128, 128, 1, 0, 2, 152) == 0
    assert lib.paged_attn_decode_sms_beside_prefill(big.handle, 32, 8, 128, 128, 1, 0, 7, 152) == 0   # bad dtype
