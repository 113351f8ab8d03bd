"""bench.py host logic on CPU: rank reduction over gloo, throughput, JSON lines."""

import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = bench.rank_env()
    dist = bench.init_dist(w, "gloo")
    bench.barrier(dist)
    # rank r pretends its timed region took (r + 1) seconds
    slowest = bench.max_over_ranks(dist, float(r + 1))
    value = bench.aggregate_value(updates_per_step=10**9, steps=4, world=w, max_seconds=slowest)
    out.put((r, w, local, slowest, value))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == [0, 1]
    for rank, world, local, slowest, value in results:
        assert world == 2 and local == rank
        assert slowest == 2.0
        # both ranks' updates over the slowest rank's time
        assert value == pytest.approx(2 * 4 * 10**9 / 2.0 / 1e9)


def test_single_rank_has_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_clock_summary_window():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.samples = [(10.0, 1900.0, 2070.0, []), (11.0, 2070.0, 2070.0, ["sw_power_cap"]),
                 (12.0, 2000.0, 2070.0, []), (20.0, 500.0, 2070.0, [])]
    out = s.summary(10.5, 12.5)
    assert out["sm_mhz"] == 2035.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 2
    assert s.summary(30.0, 31.0)["window"].startswith("whole run")


def test_clock_sampler_waits_for_its_first_sample():
    import threading
    import time
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc, s.samples = object(), []
    threading.Timer(0.1, lambda: s.samples.append((0.0, 2070.0, 2070.0, []))).start()
    t = time.time()
    s.wait_first(timeout=5.0)
    assert s.samples and time.time() - t < 2.0
    s.samples = []
    t = time.time()
    s.wait_first(timeout=0.2)                  # none arrive: bounded
    assert not s.samples and 0.15 < time.time() - t < 2.0


def test_reference_arm_json(capsys):
    rc = bench.main(["--impl", "reference", "--config", "tiny_stripmap", "--steps", "2",
                     "--warmup", "3", "--ref-step-seconds", "0.05"])
    assert rc == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "Gupd/s"
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_cpu_baseline_reports_one_thread_and_extrapolation():
    from synth import scenes
    sc = scenes.make_scene(scenes.CONFIGS[0])
    cb = bench.cpu_baseline(sc, 0.2)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["one_thread"]["value"] > 0 and cb["one_thread"]["unit"] == "Gupd/s"
    ex = cb["extrapolated_full_image_s"]
    updates = sc.params["na"] * sc.params["nx"] * sc.params["ny"]
    assert abs(ex["one_thread"] * cb["one_thread"]["value"] * 1e9 - updates) <= 1e-6 * updates
    assert cb["cpu_model"] and cb["page_figure"]["one_thread_cpu_s"] == 56.0


def test_traffic_is_reported_only_for_the_captured_kernel(monkeypatch):
    """The ncu traffic figure belongs to one revision of the kernel sources:
    the same sources report it, any other revision reports null."""
    now = bench.kernel_sources_sha256()
    monkeypatch.setattr(bench, "MAIN_KERNEL_TRAFFIC_SHA256", now)
    assert bench.main_kernel_traffic() == bench.MAIN_KERNEL_TRAFFIC
    monkeypatch.setattr(bench, "MAIN_KERNEL_TRAFFIC_SHA256", "0" * 64)
    assert bench.main_kernel_traffic() is None
    monkeypatch.setattr(bench, "MAIN_KERNEL_TRAFFIC_SOURCES", ("no/such/file.cu",))
    monkeypatch.setattr(bench, "MAIN_KERNEL_TRAFFIC_SHA256", now)
    assert bench.main_kernel_traffic() is None
