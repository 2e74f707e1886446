"""Host-side logic of bench.py that needs no GPU.

* world_size-2 gloo ranks: barrier, max-over-ranks timing and the whole-job
  rate that rank 0 reports (each rank runs its own independent problems; the
  only collective is on the timing scalar).
* the reference arm (CPU oracle) prints one well-formed JSON line, and ranks
  other than 0 print nothing.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.init_dist(world, "gloo")
    bench.barrier(d)
    ms = 2.0 + rank  # rank 1 is the slower one
    worst = bench.max_over_ranks(ms, d)
    rate = bench.whole_job_rate(1e9, world, worst)
    q.put((rank, worst, rate))
    d.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.0, 3.0]
    # 2 ranks x 1 GFLOP per step in 3 ms -> 666.7 GFLOP/s for the whole job
    assert abs(res[0][2] - 2e9 / 3e-3 / 1e9) < 1e-6


def test_single_rank_helpers():
    assert bench.max_over_ranks(1.5, None) == 1.5
    assert bench.whole_job_rate(3e9, 1, 1.0) == pytest.approx(3000.0)
    p3, ptf32, hbm = bench.roofline_peaks({"bf16_tflops": 2250.0, "hbm_gbs": 7000.0})
    assert ptf32 == pytest.approx(1100.0) and p3 == pytest.approx(1100.0 / 3)
    # 2047 MAC/clk/SM x 2 flop x 152 SMs x 2.07 GHz / 3 MMAs per product
    assert bench.probe_peak_3xtf32(152, 2070.0) == pytest.approx(429.37, abs=0.01)


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       env=env, timeout=900)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["higher_is_better"] is True and d["metric"] == bench.METRIC


def _no_dist_env():
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    return env


def test_launch_ranks_starts_every_rank():
    """bench.launch_ranks (the path --gpus N takes outside torchrun) starts N
    processes that form one process group; rank 0 alone prints."""
    probe = os.path.join(ROOT, "tests", "rank_probe.py")
    r = subprocess.run([sys.executable, "-c",
                        "import sys; sys.path.insert(0, sys.argv[1]); import bench; "
                        "sys.exit(bench.launch_ranks(2, [], script=sys.argv[2]))", ROOT, probe],
                       capture_output=True, text=True, env=_no_dist_env(), timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["ranks"] == [0, 1] and d["ms_per_step"] == 2.0
    assert d["value"] == pytest.approx(2e9 / 2e-3 / 1e9)


def test_gpus_flag_launches_the_ranks_itself():
    """bench.py --gpus 2 without torchrun runs two ranks (the reference arm
    needs no GPU): one JSON line, from rank 0, with n_gpus 2."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"], capture_output=True,
                       text=True, env=_no_dist_env(), timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2


def test_reference_arm_other_ranks_are_silent():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
