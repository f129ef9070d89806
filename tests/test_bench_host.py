"""Host-side logic of bench.py on CPU: the max-over-ranks reduction with two gloo
ranks, the reference arm's JSON line, and non-zero ranks exiting quietly."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    ms = 10.0 * (rank + 1)  # rank 1 is the slowest
    got = bench._max_over_ranks(ms, world, "cpu")
    bench._barrier(world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 20.0, 1: 20.0}


def _bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, timeout=300)


def test_reference_arm_json_line():
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["value"] > 0


@pytest.mark.parametrize("rank", ["1"])
def test_reference_arm_other_ranks_exit_quietly(rank):
    r = _bench(["--impl", "reference", "--steps", "1", "--warmup", "3"], {"RANK": rank, "WORLD_SIZE": "2"})
    assert r.returncode == 0 and not r.stdout.strip()


def test_clock_sampler_with_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """The sampler waits for its first sample, keeps every line the tool prints
    while the region runs, and reports the median loaded clock and any active
    throttle reason."""
    import time

    sys.path.insert(0, ROOT)
    import bench

    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "i=0\n"
                    "while true; do\n"
                    "  if [ $i -eq 2 ]; then r='Active'; else r='Not Active'; fi\n"
                    "  echo \"2055, 2070, 900.0, Not Active, Not Active, Not Active, $r\"\n"
                    "  i=$((i+1)); sleep 0.02\n"
                    "done\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    with bench.ClockSampler(0) as clk:
        assert clk.lines, "the timed region must not start before the first sample"
        time.sleep(0.3)
    s = clk.summary()
    assert s["samples"] >= 5
    assert s["sm_mhz"] == 2055.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("PATH", str(tmp_path))  # no nvidia-smi anywhere
    with bench.ClockSampler(0) as clk:
        pass
    assert clk.summary()["samples"] == 0


def test_live_pair_counts_match_a_brute_force_count():
    # the exact flop counts of the mask-variant workloads rest on live_pairs()
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench

    for Sq, Sk, causal, window in ((5, 2, True, (-1, -1)), (2, 5, True, (-1, -1)), (7, 7, False, (2, 1)),
                                   (9, 4, False, (0, 0)), (6, 11, True, (3, -1)), (8, 8, False, (-1, -1))):
        wl, wr = window
        if causal:
            wr = 0
        n = 0
        for i in range(Sq):
            for j in range(Sk):
                c = i + Sk - Sq
                n += (wl < 0 or j >= c - wl) and (wr < 0 or j <= c + wr)
        assert bench.live_pairs(Sq, Sk, causal, window) == n, (Sq, Sk, causal, window)
    # the three mask variants' per-head counts
    assert bench.live_pairs(2048, 8192, True, (-1, -1)) == 14681088
    assert bench.live_pairs(16384, 16384, False, (4096, 0)) == 58734592
    assert bench.live_pairs(4096, 4096, True, (-1, -1)) == 8390656
    assert np.isclose(bench.workload_flops(bench.WORKLOADS[0])[1], 4 * 2 * 16 * 128 * 14681088)
