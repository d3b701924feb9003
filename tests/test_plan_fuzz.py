"""Randomised schedules against the documented plan rules (host only, no GPU).

ruDNN 0.1.7, src/paged_attention/mod.rs: the schedule a caller hands over
(`HostPlan`: per-query sequence and absolute position, per-sequence length and
block-table row) is checked before anything is uploaded (`validate_writes`,
`bounded`).  Here a few thousand small random schedules, most of them valid and
the rest broken in one or more ways, go through paged_attn_plan; the status is
compared with the rules as paged_attn.h states them, and every accepted plan's
word image (staged to host memory) with what those rules and the documented
work lists give: per query (seq, pos, slot = table[seq][pos / ps] * ps +
pos % ps), runs of at least 16 consecutive positions of one sequence cut into
prefill tiles of at most 128 queries (heaviest last position first), every
other query a decode item (largest position first, ties in packing order),
and every query once more in that order.
"""
import ctypes

import numpy as np

import paged_kv_attention_20_gb300 as pka
from paged_kv_attention_20_gb300._binding import PagedAttentionError

PA_OK, PA_ERR_RANGE, PA_ERR_WRITE_CONFLICT = 0, 4, 5
MIN_RUN, TILE_M = 16, 128


def expected_status(seq_lens, table, qseq, qpos, ps, pages):
    width = table.shape[1]
    for s, n in enumerate(seq_lens):
        if n < 0 or n > width * ps:
            return PA_ERR_RANGE
        for g in range(-(-n // ps)):
            if not 0 <= table[s, g] < pages:
                return PA_ERR_RANGE
    slots = []
    for s, p in zip(qseq, qpos):
        if not 0 <= s < len(seq_lens) or not 0 <= p < seq_lens[s]:
            return PA_ERR_RANGE
        slots.append(int(table[s, p // ps]) * ps + p % ps)
    if len(set(slots)) != len(slots):
        return PA_ERR_WRITE_CONFLICT
    return PA_OK


def expected_work(qseq, qpos):
    tiles, decode, i, n = [], [], 0, len(qseq)
    while i < n:
        j = i + 1
        while j < n and qseq[j] == qseq[i] and qpos[j] == qpos[j - 1] + 1:
            j += 1
        if j - i >= MIN_RUN:
            tiles += [(qseq[i], b, min(TILE_M, j - b), qpos[b]) for b in range(i, j, TILE_M)]
        else:
            decode += list(range(i, j))
        i = j
    decode.sort(key=lambda q: -qpos[q])                                 # stable: ties keep packing order
    tiles.sort(key=lambda t: -(t[3] + t[2] - 1))
    return decode, tiles


def random_schedule(rng):
    ps = int(rng.choice([1, 2, 3, 4, 16]))
    ns = int(rng.integers(0, 5))
    width = int(rng.integers(0, 13 if ps == 16 else 7)) if ns else 0
    pages = int(rng.integers(0, 3 * max(ns * width, 1) + 1))
    seq_lens = [int(rng.integers(0, width * ps + 1)) for _ in range(ns)]
    # pages drawn without repeats where the pool allows, so most schedules are valid
    need = ns * width
    pool = rng.permutation(pages) if pages >= need else rng.integers(0, max(pages, 1), size=need)
    table = np.asarray(pool[:need], dtype=np.int64).reshape(ns, width) if need else np.zeros((ns, width), np.int64)
    for s in range(ns):                                                 # unused entries: anything
        table[s, -(-seq_lens[s] // ps):] = rng.integers(-1, pages + 5, size=width - (-(-seq_lens[s] // ps)))
    qseq, qpos = [], []
    for s in rng.permutation(ns):
        n = seq_lens[s]
        if n == 0 or rng.random() < 0.3:
            continue
        if rng.random() < 0.5:                                          # a run ending at the last key
            k = int(rng.integers(1, n + 1))
            qseq += [int(s)] * k
            qpos += list(range(n - k, n))
        else:                                                           # scattered positions
            for p in sorted(rng.choice(n, size=int(rng.integers(1, min(n, 6) + 1)), replace=False)):
                qseq.append(int(s))
                qpos.append(int(p))
    # break it in a few ways, now and then
    r = rng.random()
    if r < 0.06 and ns:
        seq_lens[int(rng.integers(ns))] = width * ps + 1                # longer than its table row
    elif r < 0.12 and ns and width:
        table[int(rng.integers(ns)), 0] = rng.choice([-1, pages])       # outside the pool (if used)
    elif r < 0.18 and qseq:
        qpos[int(rng.integers(len(qpos)))] += int(rng.choice([-10**6, 10**6]))
    elif r < 0.24 and qseq:
        qseq[int(rng.integers(len(qseq)))] = int(rng.choice([-1, ns]))
    elif r < 0.32 and qseq:
        i = int(rng.integers(len(qseq)))                                # a second write of a slot
        qseq.append(qseq[i])
        qpos.append(qpos[i])
    elif r < 0.36 and ns:
        seq_lens[int(rng.integers(ns))] = -1
    return seq_lens, table.astype(np.int32), qseq, qpos, ps, pages


def staged_words(plan):
    n = plan.device_bytes()
    buf = (ctypes.c_int32 * (n // 4))()
    fake = 0x10000                                                      # bound only, never dereferenced
    assert pka.load().pa_plan_stage(plan.handle, ctypes.addressof(buf), n, ctypes.c_void_p(fake), n) == 0
    return np.frombuffer(buf, dtype=np.int32).copy()


def test_random_schedules_follow_the_rules(built_lib):
    rng = np.random.default_rng(20261203)
    seen = {PA_OK: 0, PA_ERR_RANGE: 0, PA_ERR_WRITE_CONFLICT: 0}
    tiles_seen = 0
    for _ in range(3000):
        seq_lens, table, qseq, qpos, ps, pages = random_schedule(rng)
        want = expected_status(seq_lens, table, qseq, qpos, ps, pages)
        seen[want] += 1
        try:
            plan = pka.paged_attn_plan(seq_lens, table, qseq, qpos, ps, pages, upload=False)
            got = PA_OK
        except PagedAttentionError as e:
            got = e.status
        assert got == want, (seq_lens, table.tolist(), qseq, qpos, ps, pages)
        if got != PA_OK:
            continue
        w = staged_words(plan)
        nq, ns, width = len(qseq), len(seq_lens), table.shape[1]
        assert list(w[1:8]) == [nq, ns, width, ps, pages, plan.n_decode, plan.n_tiles]
        o_q, o_len, o_tab, o_dec, o_til = (int(x) for x in w[8:13])
        assert all(x % 4 == 0 for x in (o_q, o_len, o_tab, o_dec, o_til))
        meta = w[o_q:o_q + 4 * nq].reshape(nq, 4)
        for i in range(nq):
            slot = int(table[qseq[i], qpos[i] // ps]) * ps + qpos[i] % ps
            assert list(meta[i]) == [qseq[i], qpos[i], slot, 0]
        assert list(w[o_len:o_len + ns]) == seq_lens
        assert np.array_equal(w[o_tab:o_tab + ns * width], table.ravel())
        decode, tiles = expected_work(qseq, qpos)
        assert list(w[o_dec:o_dec + len(decode)]) == decode
        got_tiles = [tuple(int(x) for x in w[o_til + 4 * t:o_til + 4 * t + 4]) for t in range(plan.n_tiles)]
        assert got_tiles == tiles
        assert plan.n_tile_queries == sum(t[2] for t in tiles)
        # the last section: every query, largest position first (ties in packing order)
        o_ord = o_til + 4 * plan.n_tiles
        assert list(w[o_ord:o_ord + nq]) == sorted(range(nq), key=lambda q: -qpos[q])
        assert int(w[13]) == -(-(o_ord + nq) // 4) * 4 and int(w[0]) == 0x50414731
        tiles_seen += len(tiles)
    # the draw reaches every outcome and builds prefill tiles, so the checks above bite
    assert min(seen.values()) > 100 and tiles_seen > 100, (seen, tiles_seen)
