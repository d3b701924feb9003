"""The benchmark's multi-rank path on the host: a job over several GPUs times
the decode workloads only.  Its main function runs here with every GPU step
replaced by a recorder, under WORLD_SIZE=2, and must never ask for the mixed
prefill or the MLA workload (the kernels that run as thread-block clusters),
while a one-rank run keeps them."""
import sys
import types

import pytest

import bench


@pytest.mark.parametrize("world", [2, 4, 8])
def test_secondary_for_run_drops_prefill_and_mla(world):
    for requested in ("long,mixed,mla", "mixed", "mla", "gqa,mla,long", ""):
        which = bench.secondary_for_run(requested, world)
        assert "mixed" not in which and "mla" not in which
        assert set(which) <= set(bench.DECODE_ONLY)
    assert bench.secondary_for_run("long,mixed,mla", 1) == ["long", "mixed", "mla"]


def _run_main(monkeypatch, world, rank):
    calls = {"secondary": [], "cases": []}

    class FakeStep:
        def __init__(self, case, device, splits=None):
            calls["cases"].append(case.name)
            self.splits = 1

        def kernels_per_step(self):
            return 2

    fake_pka = types.SimpleNamespace(build=lambda: None)
    monkeypatch.setitem(sys.modules, "paged_kv_attention_20_gb300", fake_pka)
    monkeypatch.setenv("WORLD_SIZE", str(world))
    monkeypatch.setenv("RANK", str(rank))
    monkeypatch.setenv("LOCAL_RANK", str(rank))
    monkeypatch.setattr(bench.torch.cuda, "set_device", lambda d: None)
    import torch.distributed as dist
    monkeypatch.setattr(dist, "init_process_group", lambda *a, **k: None)
    monkeypatch.setattr(bench, "DecodeStep", FakeStep)
    monkeypatch.setattr(bench, "time_step", lambda *a, **k: (10.0, [0.01], [0.2], [0.19], {"samples": 5}))
    monkeypatch.setattr(bench, "whole_job_rate", lambda u, s, ms, w, d: (w * u * s / (ms / 1e3), ms))
    monkeypatch.setattr(bench, "barrier", lambda w: None)
    monkeypatch.setattr(bench, "e2e_leg", lambda *a, **k: {"value": 1.0})
    monkeypatch.setattr(bench, "cpu_baseline", lambda *a, **k: {"value": 1.0})
    monkeypatch.setattr(bench, "profile_traffic", lambda *a, **k: None)
    monkeypatch.setattr(bench, "secondary", lambda device, w, s, peaks, which, **k: calls["secondary"].append(list(which)) or {})
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", str(world), "--steps", "2", "--warmup", "3",
                                      "--no-cpu-baseline"])
    bench.main()
    return calls


def test_multi_rank_main_never_requests_prefill_or_mla(monkeypatch, capsys):
    calls = _run_main(monkeypatch, 2, 0)
    assert calls["secondary"], "rank 0 should still time the decode workloads"
    for which in calls["secondary"]:
        assert "mixed" not in which and "mla" not in which
    assert all("mla" not in c and "mixed" not in c for c in calls["cases"])


def test_single_rank_main_keeps_every_workload(monkeypatch, capsys):
    calls = _run_main(monkeypatch, 1, 0)
    assert calls["secondary"] == [["long", "mixed", "mla"]]
