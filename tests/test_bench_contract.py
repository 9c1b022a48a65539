"""bench.py on CPU: the reference arm's JSON line, the non-zero-rank exit, and the
multi-process aggregation (max over ranks) with the gloo backend, world size 2."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0",
              "--cpu-seconds", "1"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"]:
        assert key in j, key
    assert j["impl"] == "reference" and j["warmup"] >= 3 and j["value"] > 0
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["cpu_baseline"]["kind"] == "oracle"
    assert j["config"]["workload"] == "tiny"


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"],
             {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [3.0, 5.0][rank]
    m = bench.max_over_ranks(ms)
    q.put((rank, m, bench.job_tokens_per_s(world, 16384, m)))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [5.0, 5.0]
    # whole-job throughput: both replicas' tokens over the slowest replica's step time
    assert got[0][2] == 2 * 16384 / 5e-3


def test_single_process_passthrough():
    assert bench.max_over_ranks(7.5) == 7.5


def test_clock_summary_keeps_the_timed_region_only(tmp_path):
    """Samples taken before the timed region (idle or warming up, full clocks) are left
    out of the clock summary; throttle reasons come from the region's samples."""
    import datetime

    import bench

    c = bench.ClockSampler(0)
    path = tmp_path / "clocks.csv"
    now = datetime.datetime(2026, 1, 2, 3, 4, 5)
    with open(path, "w") as f:
        for i in range(10):
            ts = (now + datetime.timedelta(milliseconds=100 * i)).strftime("%Y/%m/%d %H:%M:%S.%f")
            busy = i >= 3
            f.write(f"{ts[:-3]}, {1400 if busy else 2070}, 2070, 1300.5, Not Active, Not Active, "
                    f"Not Active, {'Active' if busy else 'Not Active'}\n")
    c.file = open(path)
    c.proc = object()  # the sampler process has already ended
    c.t0 = now + datetime.timedelta(milliseconds=250)
    c.t1 = now + datetime.timedelta(milliseconds=950)
    s = c.summary()
    assert s["samples"] == 7 and s["window"] == "timed region"
    assert s["sm_mhz"] == 1400 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]


def test_producer_launch_time_counts_overlap_once():
    """Launches of two batches in flight overlap: each moment of any producer running
    counts once, and gaps between launches count not at all."""
    ns = 1_000_000  # 1 ms in ns
    one = [(0, 2 * ns)]
    assert abs(bench.producer_launch_ms(one) - 2.0) < 1e-12
    # two launches sharing 0.5 ms, then one after a gap: (2.5 + 1) ms busy over 3
    spans = [(0, 2 * ns), (int(1.5 * ns), int(2.5 * ns)), (10 * ns, 11 * ns)]
    assert abs(bench.producer_launch_ms(spans) - 3.5 / 3) < 1e-12
    # order of the records does not matter; a launch inside another adds nothing
    spans2 = [(10 * ns, 11 * ns), (int(0.5 * ns), ns), (0, 2 * ns)]
    assert abs(bench.producer_launch_ms(spans2) - 3.0 / 3) < 1e-12


def test_source_fingerprint_ignores_comments(tmp_path, monkeypatch):
    csrc = tmp_path / "tile_signaled_grouped_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("int a = 1;  // one\n\n/* block\n comment */\nint b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fp = bench.source_fingerprint(("k.cu",))
    (csrc / "k.cu").write_text("// header\nint a = 1;\n\n\nint b = 2;  // two\n")
    assert bench.source_fingerprint(("k.cu",)) == fp
    (csrc / "k.cu").write_text("int a = 1;\nint b = 3;\n")
    assert bench.source_fingerprint(("k.cu",)) != fp


def test_peak_follows_the_clock_regime_of_the_timed_region():
    full = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "window": "timed region"}
    capped = {"sm_mhz": 1758.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
              "window": "timed region"}
    at_max = dict(capped, sm_mhz=2070.0)  # the cap flagged, the clock still at its maximum
    outside = dict(capped, window="whole sampler run (none inside the region)")
    assert bench.pick_bf16_peak(0.035, full, 1945.0, 1707.2) == (1945.0, "burst", False)
    assert bench.pick_bf16_peak(0.4, capped, 1945.0, 1707.2) == (1707.2, "sustained", True)
    assert bench.pick_bf16_peak(0.4, at_max, 1945.0, 1707.2) == (1945.0, "burst", False)
    assert bench.pick_bf16_peak(0.4, outside, 1945.0, 1707.2) == (1945.0, "burst", False)
    assert bench.pick_bf16_peak(3.0, full, 1945.0, 1707.2) == (1707.2, "sustained", False)
    assert bench.pick_bf16_peak(0.035, None, 1945.0, 1707.2) == (1945.0, "burst", False)
