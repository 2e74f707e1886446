"""Throughput benchmark of the fp32 addmm + implicit-im2col conv2d hot path.

One step = the two operations of the path on their largest workloads, both in
the default (fp32-accurate, 3xTF32 tensor-core) mode:
  * addmm   out[8192,4096] = self[4096] + mat1[8192,4096] @ mat2[4096,4096]
            (operands ~ N(0,1)/64, self ~ N(0,1))
  * conv2d  B=8, IC=OC=256, 56x56, 3x3, stride 1, pad 1, dilation 1, bias
            (x ~ N(0,1), w ~ N(0,1/48), bias ~ N(0,0.02))
Metric: GFLOP/s counted as 2*M*N*K per operation (conv: M=OC, N=B*OH*OW,
K=IC*KH*KW, padding taps included).  Inputs are synthetic (seeded SplitMix64
draws), resident in HBM before the timed region; L2 is flushed (a 256 MB
write) before every step, outside the step's own CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs the same per-GPU step on its own GPU (weak
scaling, no collective on the data path); rank 0 prints one JSON line.
``--gpus N`` with N > 1 outside torchrun starts the N ranks itself (one
process per GPU through torch.distributed.run on 127.0.0.1).
``--impl reference`` times the CPU oracle (fp64, the plain definition) on a
bounded sample of the same workload instead.
After the timed steps the same step is repeated back to back for
``--sustain-seconds`` (default 3 s) and reported as the sustained rate with the
SM clock sampled during it.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GFLOP/s (2MNK) addmm & im2col-conv2d fp32 at 1 GB300; % of 3xTF32 roofline"
UNIT = "GFLOP/s"
ADDMM_CASE = "large_8192x4096x4096"
CONV_CASE = "body_56_3x3_d1"
WORKLOAD = ("addmm 8192x4096x4096 self[N] + conv2d B8 IC256 OC256 56x56 3x3 s1 p1 d1 (bias), "
            "fp32 in/out, default 3xTF32 mode")
FLUSH_BYTES = 256 << 20
# Nominal dense TF32 / BF16 tensor throughput of the GB300 (1.1 vs 2.25 PFLOP/s).
TF32_PER_BF16 = 1.1 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# tcgen05.mma kind::tf32 multiply-adds per clock per SM, measured on GB300 with
# back-to-back 128x256x8 MMAs (a probe outside the product); times the SM
# count and the SM clock sampled during the run it gives a clock-true peak.
TF32_MAC_PER_CLK_SM = 2047.0


def addmm_flops(M, N, K):
    return 2.0 * M * N * K


def conv_dims(c):
    OH = (c["H"] + 2 * c["pad"] - c["dilation"] * (c["KH"] - 1) - 1) // c["stride"] + 1
    OW = (c["W"] + 2 * c["pad"] - c["dilation"] * (c["KW"] - 1) - 1) // c["stride"] + 1
    return OH, OW, c["OC"], c["B"] * OH * OW, c["IC"] * c["KH"] * c["KW"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured (MEASURED_PEAKS.json)"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback (profiling recipe)"


def roofline_peaks(peaks):
    """3xTF32-adjusted tensor peak in TFLOP/s of metric flops, and HBM GB/s."""
    tf32 = peaks["bf16_tflops"] * TF32_PER_BF16
    return tf32 / 3.0, tf32, peaks["hbm_gbs"]


def probe_peak_3xtf32(sms: int, sm_mhz: float) -> float:
    """3xTF32 peak in TFLOP/s of metric flops from the probed MMA rate at the
    given SM count and clock (three MMAs per product)."""
    return TF32_MAC_PER_CLK_SM * 2.0 * sms * sm_mhz * 1e6 / 3.0 / 1e12


# ------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def _free_port() -> int:
    import socket
    sk = socket.socket()
    sk.bind(("127.0.0.1", 0))
    port = sk.getsockname()[1]
    sk.close()
    return port


def launch_ranks(n: int, argv, script: str | None = None) -> int:
    """Runs `script` (this file by default) as n ranks on one node, one
    process per GPU, through torch.distributed.run with its rendezvous on
    127.0.0.1; returns the exit status.  The ranks inherit stdout, so rank 0's
    JSON line is the output."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port",
           str(_free_port()), script or os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def barrier(dist_mod, device=None):
    if dist_mod is not None:
        if device is not None:
            dist_mod.barrier(device_ids=[device.index])
        else:
            dist_mod.barrier()


def max_over_ranks(value: float, dist_mod, device=None) -> float:
    """Maximum of a per-rank float over all ranks (the timing rule's max)."""
    if dist_mod is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_step_per_rank: float, world_size: int, max_ms_per_step: float):
    """GFLOP/s of all ranks together: every rank runs the same step (weak scaling)."""
    return flops_per_step_per_rank * world_size / (max_ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def device_record(device):
    """Name, SM count, driver and CUDA runtime of the GPU the numbers come from."""
    import torch
    props = torch.cuda.get_device_properties(device)
    rec = {"name": props.name, "sms": props.multi_processor_count,
           "cc": f"{props.major}.{props.minor}", "cuda_runtime": torch.version.cuda}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(device.index or 0)], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        rec["driver"] = out or None
    except (OSError, subprocess.SubprocessError):
        rec["driver"] = None
    return rec


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="imc_clocks_", suffix=".csv")
        self.proc = None
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return None
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) < 10:
                        continue
                    try:
                        ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                        rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
                    except ValueError:
                        continue
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_mod = init_dist(ws, "nccl")

    from addmm_implicit_im2col_gb300 import binding, build, synth
    build.build()
    binding.load()

    ca, s_np, a_np, b_np = synth.make_addmm_case(ADDMM_CASE)
    cc, x_np, w_np, bias_np = synth.make_conv_case(CONV_CASE)
    OH, OW, cM, cN, cK = conv_dims(cc)
    fl_addmm = addmm_flops(ca["M"], ca["N"], ca["K"])
    fl_conv = addmm_flops(cM, cN, cK)
    flops_step = fl_addmm + fl_conv

    S, A, Bm = (torch.from_numpy(t).to(device) for t in (s_np, a_np, b_np))
    X, Wt, Bias = (torch.from_numpy(t).to(device) for t in (x_np, w_np, bias_np))
    out_a = torch.empty((ca["M"], ca["N"]), dtype=torch.float32, device=device)
    out_c = torch.empty((cc["B"], cc["OC"], OH, OW), dtype=torch.float32, device=device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        binding.addmm(S, A, Bm, beta=ca["beta"], alpha=ca["alpha"], out=out_a)
        binding.conv2d(X, Wt, Bias, cc["stride"], cc["pad"], cc["dilation"], out=out_c)

    for _ in range(args.warmup):
        flush.fill_(0.0)
        step()
    kern_a = kern_c = None
    binding.addmm(S, A, Bm, beta=ca["beta"], alpha=ca["alpha"], out=out_a)
    kern_a = binding.last_kernel()
    binding.conv2d(X, Wt, Bias, cc["stride"], cc["pad"], cc["dilation"], out=out_c)
    kern_c = binding.last_kernel()
    torch.cuda.synchronize(device)

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(dist_mod, device)
    torch.cuda.synchronize(device)
    launches0 = binding.launch_count()
    t0 = time.time()
    for i in range(args.steps):
        flush.fill_(float(i))  # evict the previous step's data from L2
        ev[i][0].record(stream)
        binding.addmm(S, A, Bm, beta=ca["beta"], alpha=ca["alpha"], out=out_a)
        ev[i][1].record(stream)
        binding.conv2d(X, Wt, Bias, cc["stride"], cc["pad"], cc["dilation"], out=out_c)
        ev[i][2].record(stream)
    torch.cuda.synchronize(device)
    t1 = time.time()
    barrier(dist_mod, device)
    launches = binding.launch_count() - launches0
    clocks = None
    if sampler:
        time.sleep(0.1)
        sampler.stop()
        clocks = sampler.summary(t0, t1)

    ms_addmm = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    ms_conv = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    ms_step_local = (sum(ms_addmm) + sum(ms_conv)) / args.steps
    ms_step = max_over_ranks(ms_step_local, dist_mod, device)
    value = whole_job_rate(flops_step, ws, ms_step)

    # ---- end to end through the host-buffer entry points: every step hands the
    # library its six inputs in pinned host memory and takes both results back
    # in pinned host memory (gemm_addmm_f32_host + conv2d_gemm_f32_host: the
    # library copies the inputs in, computes and copies the results out, all on
    # the step's stream).  Steps rotate over --e2e-streams streams, so step i+1's
    # inputs go in while step i computes and its results come out; the per-step
    # inputs (229 MB) are larger than L2.  The same steps on one stream are
    # reported beside it.
    h_in = [torch.from_numpy(t).pin_memory() for t in (s_np, a_np, b_np, x_np, w_np, bias_np)]
    h_out = [torch.empty(out_a.shape, dtype=torch.float32).pin_memory(),
             torch.empty(out_c.shape, dtype=torch.float32).pin_memory()]
    h2d = sum(t.numel() * 4 for t in h_in)
    d2h = sum(t.numel() * 4 for t in h_out)
    e2e_steps = max(4, args.steps)  # the same steps as the device-resident figure
    # the addmm and the conv are independent problems: each has its own ring
    e2e_streams = [(torch.cuda.Stream(device), torch.cuda.Stream(device))
                   for _ in range(args.e2e_streams)]

    def host_step(st):
        binding.addmm_host(h_in[0], h_in[1], h_in[2], beta=ca["beta"], alpha=ca["alpha"],
                           out=h_out[0], stream=st[0])
        binding.conv2d_host(h_in[3], h_in[4], h_in[5], cc["stride"], cc["pad"], cc["dilation"],
                            out=h_out[1], stream=st[1])

    def e2e_run(n, rings):
        streams = list(dict.fromkeys(st for pair in rings for st in pair))
        first = streams[0]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        start.record(first)
        for st in streams[1:]:
            st.wait_event(start)
        for i in range(n):
            host_step(rings[i % len(rings)])
        for st in streams[1:]:
            done = torch.cuda.Event()
            done.record(st)
            first.wait_event(done)
        end.record(first)
        end.synchronize()
        return start.elapsed_time(end) / n

    one_stream = [(e2e_streams[0][0], e2e_streams[0][0])]
    e2e_run(2, one_stream)
    e2e_run(len(e2e_streams), e2e_streams)
    barrier(dist_mod, device)
    serial_ms = max_over_ranks(e2e_run(e2e_steps, one_stream), dist_mod, device)
    barrier(dist_mod, device)
    e2e_ms = max_over_ranks(e2e_run(e2e_steps, e2e_streams), dist_mod, device)
    e2e_value = whole_job_rate(flops_step, ws, e2e_ms)
    # the last step's results, as copied to the host, equal the device-resident run's
    e2e_ok = (torch.equal(h_out[0], out_a.cpu()) and torch.equal(h_out[1], out_c.cpu()))
    # The pages' one published figure is the implicit-im2col GEMM's speed-up
    # over their direct conv kernel; time the same ratio here (outside the
    # timed region, after it).
    direct = None
    if rank == 0 and not args.no_direct_baseline:
        d_ms = []
        for _ in range(3):
            flush.fill_(0.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            binding.conv2d(X, Wt, Bias, cc["stride"], cc["pad"], cc["dilation"], mode="direct",
                           out=out_c)
            e1.record(stream)
            e1.synchronize()
            d_ms.append(e0.elapsed_time(e1))
        dm = statistics.median(d_ms)
        direct = {"workload": "the step's conv2d", "direct_ms": round(dm, 4),
                  "gemm_ms": round(sum(ms_conv) / len(ms_conv), 4),
                  "speedup": round(dm / (sum(ms_conv) / len(ms_conv)), 2)}
    # ---- sustained: the same step (with its L2 flush) back to back for
    # --sustain-seconds, long enough for the power limit to set the clock;
    # device time of the steps from per-step events, SM clock sampled meanwhile
    sustained = None
    if args.sustain_seconds > 0:
        n_sus = max(args.steps, int(np.ceil(args.sustain_seconds * 1e3 / max(ms_step, 1e-3))))
        sampler_s = ClockSampler(local) if rank == 0 else None
        time.sleep(0.3 if sampler_s else 0.0)
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_sus)]
        barrier(dist_mod, device)
        torch.cuda.synchronize(device)
        ts0 = time.time()
        for i in range(n_sus):
            flush.fill_(float(i))
            sev[i][0].record(stream)
            step()
            sev[i][1].record(stream)
            if i % 256 == 255:
                sev[i][1].synchronize()  # keeps the queue of launches short
        torch.cuda.synchronize(device)
        ts1 = time.time()
        barrier(dist_mod, device)
        sus_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in sev) / n_sus, dist_mod, device)
        clocks_s = None
        if sampler_s:
            time.sleep(0.1)
            sampler_s.stop()
            clocks_s = sampler_s.summary(ts0, ts1)
        sustained = {"value": round(whole_job_rate(flops_step, ws, sus_ms), 1), "unit": UNIT,
                     "ms_per_step": round(sus_ms, 4), "steps": n_sus,
                     "wall_s": round(ts1 - ts0, 2), "clocks": clocks_s,
                     "how": "the timed step (L2 flush outside each step's events) repeated back "
                            "to back; device time summed over per-step CUDA events"}
    status = binding.check_device_error(None)

    if rank != 0:
        if dist_mod is not None:
            dist_mod.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    p3, ptf32, hbm = roofline_peaks(peaks)
    avg_addmm = sum(ms_addmm) / len(ms_addmm)
    avg_conv = sum(ms_conv) / len(ms_conv)
    ach_a = fl_addmm / (avg_addmm * 1e-3) / 1e12
    ach_c = fl_conv / (avg_conv * 1e-3) / 1e12
    traffic = load_profiled_traffic("k_tc_gemm")
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    p_probe = probe_peak_3xtf32(sms, sm_mhz)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded SplitMix64 uniform / Box-Muller normal draws)",
        "config": {"workload": WORKLOAD, "addmm": [ca["M"], ca["N"], ca["K"]],
                   "conv_gemm": [cM, cN, cK], "mode": "default",
                   "kernels": {"addmm": kern_a, "conv2d": kern_c},
                   "l2": "flushed by a 256 MB write before every step, outside the step events",
                   "parallelism": f"replicas x{ws} (independent problems per GPU)"},
        "roofline": {"bound": "tensor", "achieved": round(ach_a, 2), "peak": round(p3, 2),
                     "unit": "TFLOP/s", "frac": round(ach_a / p3, 4), "traffic": traffic,
                     "kernel": f"addmm {kern_a} (k_tc_gemm)",
                     "peak_source": f"{peak_src}: bf16 {peaks['bf16_tflops']} TFLOP/s x 1.1/2.25 "
                                    f"(nominal TF32/BF16) = {ptf32:.1f} TF32, /3 for 3xTF32",
                     "achieved_basis": "2*M*N*K metric flops / CUDA-event average launch time",
                     "peak_probe": round(p_probe, 2), "frac_probe": round(ach_a / p_probe, 4),
                     "peak_probe_basis": f"{TF32_MAC_PER_CLK_SM:.0f} MAC/clk/SM (tcgen05 kind::tf32 "
                                         f"probe) x 2 x {sms} SMs x {sm_mhz:.0f} MHz (median SM "
                                         f"clock sampled in the timed region) / 3"},
        "parts": {
            "addmm": {"ms": round(avg_addmm, 4), "TFLOP/s": round(ach_a, 2),
                      "frac": round(ach_a / p3, 4)},
            "conv2d": {"ms": round(avg_conv, 4), "TFLOP/s": round(ach_c, 2),
                       "frac": round(ach_c / p3, 4), "frac_probe": round(ach_c / p_probe, 4)},
        },
        "sustained": sustained,
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4), "steps": e2e_steps,
                "path": "every step: gemm_addmm_f32_host + conv2d_gemm_f32_host on pinned "
                        "host buffers (the library copies the 6 inputs in, computes and "
                        "copies both results out on the call's stream; one copy queue per "
                        "direction); the addmm and the conv each rotate over "
                        f"{args.e2e_streams} streams",
                "serial_ms_per_step": round(serial_ms, 4), "results_match_device_run": e2e_ok,
                "serial_value": round(whole_job_rate(flops_step, ws, serial_ms), 1)},
        "gpu_launches": launches,
        "conv_gemm_vs_direct": direct,
        "clocks": clocks,
        "device": device_record(device),
        "watchdog": status,
    }
    if not args.no_cpu_baseline and ws == 1:  # the host cores' baseline is an N=1 figure
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if dist_mod is not None:
        dist_mod.destroy_process_group()
    return line


def load_profiled_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or a source file it lists has changed since the capture."""
    import glob
    import hashlib
    import re
    pat = re.compile(r"^TRAFFIC kernel=(\S+) bytes_per_launch=(\d+) source_sha256_16=(\w+) "
                     r"sources=(\S+)$")
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.match(line.strip())
                if not m or m.group(1) != kernel:
                    continue
                digest = hashlib.sha256()
                try:
                    for src in m.group(4).split(","):
                        with open(os.path.join(ROOT, src), "rb") as g:
                            digest.update(g.read())
                except OSError:
                    return None
                return int(m.group(2)) if digest.hexdigest()[:16] == m.group(3) else None
    return None


# ------------------------------------------------------- CPU baseline arm
def oracle_sample_step(nthreads, addmm_rows, conv_channels):
    """One bounded sample of the step on the oracle: ``addmm_rows`` output rows
    of the addmm and ``conv_channels`` output channels of the first image of the
    conv.  Returns (flops, seconds)."""
    import oracle
    from addmm_implicit_im2col_gb300 import synth
    ca, s, a, b = _cached("addmm", lambda: synth.make_addmm_case(ADDMM_CASE))
    cc, x, w, bias = _cached("conv", lambda: synth.make_conv_case(CONV_CASE))
    OH, OW, _, _, cK = conv_dims(cc)
    rows = synth.checked_rows(ADDMM_CASE, ca["M"], addmm_rows)
    chans = np.arange(conv_channels, dtype=np.int64)
    t = time.perf_counter()
    oracle.addmm(s, a, b, beta=ca["beta"], alpha=ca["alpha"], rows=rows, nthreads=nthreads)
    oracle.conv2d(x[:1], w, bias, cc["stride"], cc["pad"], cc["dilation"], channels=chans,
                  nthreads=nthreads)
    dt = time.perf_counter() - t
    flops = 2.0 * len(rows) * ca["N"] * ca["K"] + 2.0 * conv_channels * OH * OW * cK
    return flops, dt


_CACHE = {}


def _cached(key, fn):
    if key not in _CACHE:
        _CACHE[key] = fn()
    return _CACHE[key]


def cpu_baseline(target_seconds=1.0):
    import oracle
    cores = oracle.default_threads()
    rows, chans = 256, 128
    flops, dt = oracle_sample_step(cores, rows, chans)
    return {"value": round(flops / dt / 1e9, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{rows} seeded rows of the 8192x4096x4096 addmm + {chans} output channels "
                      f"of image 0 of the conv ({flops / 1e9:.2f} GFLOP, {dt:.2f} s wall on "
                      f"{cores} threads, fp64 oracle as committed)"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    cores = oracle.default_threads()
    rows, chans = 16, 16
    for _ in range(args.warmup):
        oracle_sample_step(cores, rows, chans)
    tot_f, tot_t = 0.0, 0.0
    for _ in range(args.steps):
        f, t = oracle_sample_step(cores, rows, chans)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e9
    sample = (f"per step: {rows} seeded rows of the 8192x4096x4096 addmm + {chans} output "
              f"channels of image 0 of the conv ({tot_f / args.steps / 1e9:.3f} GFLOP)")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 uniform / Box-Muller normal draws)",
        "config": {"workload": WORKLOAD, "sample": sample,
                   "impl": "CPU oracle (plain C, fp64) on the host cores"},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["imc", "reference"], default="imc")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-direct-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=1.0)
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams each problem's end-to-end calls rotate over")
    ap.add_argument("--sustain-seconds", type=float, default=3.0,
                    help="repeat the step back to back this long for the sustained rate "
                         "(0: skip)")
    raw = list(sys.argv[1:] if argv is None else argv)
    args = ap.parse_args(raw)
    args.warmup = max(args.warmup, 3)  # the timing rules want at least 3 warm-up steps
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(args.gpus, raw))
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
