"""Benchmark: dgrad useful-MAC TFLOP/s on one GB300, printed as one JSON line.

Default workload: the dgrad shape of page "Non-unit stride input backward different
input and dispatches between BOO and Fusilli" (bf16 NHWC, N=16, Hi=1, Wi=512,
C=K=2048, 1x2 filter, stride (1, 2), pad 0 -> dy 16x1x256x2048), seeded
synthetic inputs N(0,1)*0.02 rounded to bf16.  A "step" is one
conv_bwd_data_run (every kernel of the path) with dy and w resident in HBM;
L2 is flushed (a 512 MiB write) before every step, outside the step's events.
The line also carries `per_workload`: every other workload (the fp32 sweep,
the grouped layer, the stress set, the fp32 tensor-core shapes) timed the same
way, each with its own roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the CPU oracle, timed on host cores)

Under torchrun (N > 1) every rank runs an independent replica of the same
workload on its own GPU (the op needs no exchange); the time is the max over
ranks and the value the work of all ranks divided by it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dgrad useful-MAC TFLOP/s and % of GB300 bf16 dense peak, 1 GPU"
# Pages' number for this workload: IREE "BOO" lowering, 551 us on an AMD GPU
# whose model the page does not name (6.872e10 useful FLOP -> 124.7 TFLOP/s).
PAGE_TFLOPS = 124.7
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
# Per-launch DRAM traffic of each workload's GEMM kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only while the kernel's
# sources are unchanged (hash below) and the plan launches the same tile shape.
TF32_PER_BF16 = 1.1 / 2.25  # NOMINAL dense TF32 / bf16 tensor rates of the part (no measured TF32 peak)
TC2_SOURCES = ("tc_common.cuh", "tc2_sm103.cu", "internal.h")
TC_SOURCES = ("tc_common.cuh", "tc_sm103.cu", "internal.h")
BAND_SOURCES = ("tc_common.cuh", "tc_band_sm103.cu", "band.h", "internal.h")
TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, tc2_dgrad_kernel<512, false>, one launch on the
    # 16x1x512x2048 shape (after an L2 flush): 33.69 MB + 0.86 MB (dx stays in L2 at kernel end)
    "bf16_16x1x512x2048_1x2_s1x2": {"files": TC2_SOURCES, "tile": (256, 512, 2), "kernel": "tc2_dgrad_kernel<512>",
                                    "sha": "4e32a809679716a0", "bytes": 34.556e6},
    # ncu --set full, tc_band_dgrad_kernel on the 64x56x56x256 G=32 layer: 25.81 MB + 41.42 MB (the rest of
    # dx stays in L2 at kernel end)
    "bf16_resnext_64x56x56x256_g32_3x3_s2": {"files": BAND_SOURCES, "tile": (128, 64, 1),
                                             "kernel": "tc_band_dgrad_kernel", "sha": "17f1d15c09232dd0",
                                             "bytes": 67.227e6},
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, tc_dgrad_kernel<256, true> (class pairs) on the
    # 32x57x57x128 5x5 stride-3 layer: 3.83 MB read (dy + w) + 0 written (dx stays in L2 at kernel end)
    "bf16_32x57x57x128_5x5_s3_p2": {"files": TC_SOURCES, "tile": (128, 256, 1), "kernel": "tc_dgrad_kernel<256>",
                                    "sha": "b675ce02e42d2d4f", "bytes": 3.830e6},
}


def traffic_for(case, plan, label):
    """Recorded per-launch DRAM traffic of the workload's kernel, or None when
    the kernel's sources, tile shape or kernel differ from the capture's."""
    tr = TRAFFIC.get(case.name)
    if not tr or tr["sha"] != kernel_sha(tr["files"]) or tuple(plan.tile()) != tr["tile"] or tr["kernel"] != label:
        return None
    return tr["bytes"]


def kernel_sha(files=TC2_SOURCES) -> str:
    """Hash of the sources that define a kernel launch's behaviour."""
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "conv2d_backward_implicit_bwd_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def _find_key(d, key):
    """First value stored under `key` in a JSON document, searched breadth-first
    (the peaks file may hold them at the top level or under a per-device entry)."""
    todo = [d]
    while todo:
        cur = todo.pop(0)
        if isinstance(cur, dict):
            if key in cur and isinstance(cur[key], (int, float)):
                return float(cur[key])
            todo.extend(cur.values())
        elif isinstance(cur, list):
            todo.extend(cur)
    return None


def load_peaks(root=None):
    path = os.path.join(root or ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            out = {"source": "measured"}
            for k in ("bf16_tflops", "bf16_tflops_sustained", "hbm_gbs"):
                v = _find_key(d, k)
                if v is not None and v > 0:
                    out[k] = v
            if "bf16_tflops" in out and "hbm_gbs" in out:
                return out
        except Exception:
            pass
    return {"source": "fallback", **FALLBACK_PEAKS}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank gets max(x) (identity when world == 1).
    The tensor lives on ``device`` (a CUDA device under NCCL, CPU under gloo)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(useful_flop_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput of ``world`` replicas, each doing the same work,
    timed by the slowest rank (weak scaling)."""
    return useful_flop_per_rank * world / (ms * 1e-3) / 1e12


def make_inputs(case, plan):
    from conv2d_backward_implicit_bwd_gb300 import workloads as wl
    dy_s, w_s, dx_s = plan.shapes()
    dy, w = wl.draw(case, dy_s, w_s)
    return dy, w, dx_s


def oracle_sample(case, dy, w, step: int, max_channels: int = 256):
    """One bounded oracle sample: image (step mod N), a block of up to 256
    input channels of every group starting at a step-dependent offset.
    Returns (seconds, fraction of the workload, threads that had work)."""
    import oracle
    from conv2d_backward_implicit_bwd_gb300 import workloads as wl
    g = oracle.geom(case.N, case.C, case.K, case.Hi, case.Wi, case.Y, case.X, case.pad, case.stride, case.dil,
                    case.groups)
    lay = oracle.LAYOUT_NCHW if case.layout == wl.NCHW else oracle.LAYOUT_NHWC
    Cg = case.C // case.groups
    cb = min(max_channels, Cg)
    nblk = max(1, Cg // cb)
    c0 = (step % nblk) * cb
    n0 = step % case.N
    t0 = time.perf_counter()
    oracle.dgrad(g, lay, dy, w, n_range=(n0, n0 + 1), c_range=(c0, c0 + cb), with_absdot=False)
    dt = time.perf_counter() - t0
    items = case.groups * ((cb + 15) // 16)  # the oracle's OpenMP work items (16-channel blocks)
    return dt, cb / Cg / case.N, min(oracle.num_threads(), items)


def run_reference(args, case):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    from conv2d_backward_implicit_bwd_gb300 import workloads as wl
    g = oracle.geom(case.N, case.C, case.K, case.Hi, case.Wi, case.Y, case.X, case.pad, case.stride, case.dil,
                    case.groups)
    lay = oracle.LAYOUT_NCHW if case.layout == wl.NCHW else oracle.LAYOUT_NHWC
    dy_s, w_s, _ = oracle.shapes(g, lay)
    dy, w = wl.draw(case, dy_s, w_s)
    useful = useful_flop_bruteforce(case, g)
    # keep the whole run to a few minutes: shrink the per-step sample for long runs
    mc = max(16, min(256, (256 * 300 // max(1, args.steps + args.warmup)) // 16 * 16))
    for s in range(args.warmup):
        oracle_sample(case, dy, w, s, mc)
    times, fracs = [], []
    threads = 1
    for s in range(args.steps):
        dt, frac, threads = oracle_sample(case, dy, w, args.warmup + s, mc)
        times.append(dt)
        fracs.append(frac)
    total_t = sum(times)
    value = useful * sum(fracs) / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; identical inputs to the GPU arm)",
        "config": {"workload": case.name, "sample_per_step": f"one image x {mc} input channels of every group"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: one image x {mc} input channels of every group (scatter loop, fp64)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def useful_flop_bruteforce(case, g):
    def taps(In, Out, F, s, d, p):
        return sum(1 for o in range(Out) for f in range(F) if 0 <= o * s - p + f * d < In)
    th = taps(case.Hi, g.Ho, case.Y, case.stride[0], case.dil[0], case.pad[0])
    tw = taps(case.Wi, g.Wo, case.X, case.stride[1], case.dil[1], case.pad[1])
    return 2.0 * case.N * case.K * (case.C // case.groups) * th * tw


FP32_FFMA_PER_SM_CLK = 128  # fp32 lanes per SM (one FFMA = 2 FLOP per lane per clock)


def kernel_label(path, plan, case):
    tm, tn, tsms = plan.tile()
    return {"tcgen05": (f"tc2_dgrad_kernel<{tn}>" if tsms >= 2 else f"tc_dgrad_kernel<{tn}>"),
            "grouped": {"band": "tc_band_dgrad_kernel", "tc": "tc_grouped_dgrad_kernel"}.get(
                plan.grouped_kernel(), f"grouped_dgrad_kernel<{case.C // case.groups}>"),
            "simt": "simt_dgrad_kernel", "tf32": "tf32_dgrad_kernel"}[path]


def roofline_of(path, case, useful, algo_bytes, kmean_ms, peaks, sm_max_mhz=None, num_sms=None):
    """Roofline of a workload's dominant kernel.  Tensor-core bf16 kernels are
    placed against the measured dense bf16 peak, the narrow-group kernel
    against the measured HBM copy rate; workloads near the ridge (the 1x1 and
    5x5 stress layers) report both and are graded on the larger fraction."""
    tflops = useful / (kmean_ms * 1e-3) / 1e12
    gbs = algo_bytes / (kmean_ms * 1e-3) / 1e9
    t = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
         "peak_source": peaks["source"] + " (bf16 dense, burst)"}
    h = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
         "peak_source": peaks["source"] + " (HBM copy)"}
    t["frac"] = t["achieved"] / t["peak"]
    h["frac"] = h["achieved"] / h["peak"]
    if path == "tf32":
        # three TF32 products per useful fp32 multiply-add; no TF32 peak is
        # measured on this machine, so the ceiling is the measured bf16 rate times
        # the part's NOMINAL dense TF32/bf16 ratio (1.1/2.25 PFLOP/s), over 3
        t["peak"] = peaks["bf16_tflops"] * TF32_PER_BF16 / 3.0
        t["frac"] = t["achieved"] / t["peak"]
        t["peak_source"] = (peaks["source"] + " bf16 dense (burst) x nominal TF32/bf16 ratio 1.1/2.25 / 3 products "
                            "per MAC; nominal ceiling, not a measured TF32 peak")
        return dict(t, hbm_frac=h["frac"])
    if path == "simt":
        # CUDA-core FFMA: 152 SMs x 128 lanes x 2 FLOP x max SM clock
        mhz = sm_max_mhz or 2070.0
        sms = num_sms or 152
        peak = sms * FP32_FFMA_PER_SM_CLK * 2 * mhz * 1e6 / 1e12
        a = {"bound": "alu", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
             "peak_source": f"{sms} SMs x {FP32_FFMA_PER_SM_CLK} fp32 lanes x 2 FLOP x {mhz:.0f} MHz (FFMA)"}
        return dict(a, hbm_frac=h["frac"])
    tags = case.tags[0] if case.tags else ""
    if path == "grouped" or tags == "grouped":
        return dict(h, tensor_frac=t["frac"])
    if tags == "ridge":
        best = t if t["frac"] >= h["frac"] else h
        return dict(best, tensor_frac=t["frac"], hbm_frac=h["frac"], graded_on="max(tensor, hbm)")
    return dict(t, hbm_frac=h["frac"])


def device_inputs(case, plan):
    import numpy as np
    import torch
    from conv2d_backward_implicit_bwd_gb300 import workloads as wl
    dy, w, dx_s = make_inputs(case, plan)
    tdt = torch.bfloat16 if case.dtype == wl.BF16 else torch.float32
    if case.dtype == wl.BF16:
        dy_h = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16)
        w_h = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16)
    else:
        dy_h, w_h = torch.from_numpy(dy), torch.from_numpy(w)
    return dy, w, dy_h, w_h, dy_h.cuda(), w_h.cuda(), torch.empty(dx_s, dtype=tdt, device="cuda"), dx_s, tdt


def timed_steps(plan, dy_d, w_d, dx_d, flush, stream, steps):
    """Per-step device times (ms): L2 flushed before every step, outside the
    step's events; the flush kernel also keeps the stream busy while the next
    step is enqueued, so no host latency lands inside a step's events."""
    import torch
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(stream)
        plan.run(dy_d, w_d, dx_d, stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def kernel_steps(plan, launches, step_ms, dy_d, w_d, dx_d, flush, stream, steps):
    """Device time of the dominant (sub-GEMM) kernel per step: the step itself
    when it is one launch, else the library's own events around that kernel."""
    if launches == 1:
        return step_ms
    plan.set_timing(True)
    out = []
    for _ in range(steps):
        flush.zero_()
        plan.run(dy_d, w_d, dx_d, stream)
        out.append(plan.last_timing()[1])
    plan.set_timing(False)
    return out


def measure_workload(B, case, steps, warmup, flush, stream, peaks, num_sms, env=None):
    """One per-workload entry: the same timing method as the headline line.
    `env`: planner overrides in force while the plan is created."""
    saved = {k: os.environ.get(k) for k in (env or {})}
    os.environ.update(env or {})
    try:
        plan = B.Plan.from_case(case)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    path, launches = plan.path()
    useful, algo_bytes = plan.work()
    _, _, _, _, dy_d, w_d, dx_d, _, _ = device_inputs(case, plan)
    for _ in range(warmup):
        flush.zero_()
        plan.run(dy_d, w_d, dx_d, stream)
    st, det = plan.status(stream)
    if st != B.OK:
        raise RuntimeError(f"{case.name}: device status {B.status_string(st)} {det:#x}")
    step_ms = timed_steps(plan, dy_d, w_d, dx_d, flush, stream, steps)
    kern_ms = kernel_steps(plan, launches, step_ms, dy_d, w_d, dx_d, flush, stream, steps)
    st, det = plan.status(stream)
    if st != B.OK:
        raise RuntimeError(f"{case.name}: device status {B.status_string(st)} {det:#x}")
    ms = sum(step_ms) / len(step_ms)
    kms = sum(kern_ms) / len(kern_ms)
    roof = roofline_of(path, case, useful, algo_bytes, kms, peaks, num_sms=num_sms)
    roof["kernel"] = kernel_label(path, plan, case)
    roof["kernel_ms"] = kms
    roof["traffic"] = traffic_for(case, plan, roof["kernel"])
    return {"ms_per_step": ms, "tflops": useful / (ms * 1e-3) / 1e12, "gbs": algo_bytes / (ms * 1e-3) / 1e9,
            "dtype": case.dtype, "path": path, "launches_per_step": launches, "tile": list(plan.tile()),
            "a_operand": plan.a_operand(), "k_splits": plan.k_splits(),
            "useful_flop": useful, "algo_bytes": algo_bytes, "steps": steps, "warmup": warmup,
            "roofline": roof}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_16x1x512x2048_1x2_s1x2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true")
    ap.add_argument("--pw-steps", type=int, default=30, help="timed steps of each per-workload entry (>= 20)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    args.pw_steps = max(args.pw_steps, 20)

    from conv2d_backward_implicit_bwd_gb300 import workloads as wl
    case = wl.case(args.workload)
    if args.impl == "reference":
        return run_reference(args, case)

    import numpy as np
    import torch
    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from conv2d_backward_implicit_bwd_gb300 import build as cbuild
    cbuild.build()
    from conv2d_backward_implicit_bwd_gb300 import binding as B

    plan = B.Plan.from_case(case)
    path, launches = plan.path()
    useful, algo_bytes = plan.work()
    dy, w, dy_h, w_h, dy_d, w_d, dx_d, dx_s, tdt = device_inputs(case, plan)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    num_sms = torch.cuda.get_device_properties(local_rank).multi_processor_count

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        flush.zero_()
        plan.run(dy_d, w_d, dx_d, stream)
    st, det = plan.status(stream)
    if st != B.OK:
        raise RuntimeError(f"device status {B.status_string(st)} {det:#x}")

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.2)
    barrier()
    t_wall = time.perf_counter()
    step_ms = timed_steps(plan, dy_d, w_d, dx_d, flush, stream, args.steps)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    st, det = plan.status(stream)
    if st != B.OK:
        raise RuntimeError(f"device status {B.status_string(st)} {det:#x}")
    mean_ms = sum(step_ms) / len(step_ms)
    kern_ms = kernel_steps(plan, launches, step_ms, dy_d, w_d, dx_d, flush, stream, args.steps)
    mean_ms = max_over_ranks(mean_ms, world, "cuda")
    value = job_tflops(useful, world, mean_ms)

    # end-to-end through the host-buffer entry point (pinned host memory)
    dy_p, w_p = dy_h.pin_memory(), w_h.pin_memory()
    dx_p = torch.empty(dx_s, dtype=tdt).pin_memory()
    e2e_ms = []
    for i in range(args.e2e_steps + 2):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan.run_host(dy_p, w_p, dx_p, dy_d, w_d, dx_d, stream)
        b.record(stream)
        b.synchronize()
        if i >= 2:
            e2e_ms.append(a.elapsed_time(b))
    e2e_mean = sum(e2e_ms) / len(e2e_ms)
    e2e_mean = max_over_ranks(e2e_mean, world, "cuda")
    esz = 2 if case.dtype == wl.BF16 else 4

    peaks = load_peaks()
    kmean = sum(kern_ms) / len(kern_ms)
    roof = roofline_of(path, case, useful, algo_bytes, kmean, peaks, sm_max_mhz=clocks.get("sm_max_mhz"),
                       num_sms=num_sms)
    roof["kernel"] = kernel_label(path, plan, case)
    roof["kernel_ms"] = kmean
    roof["traffic"] = traffic_for(case, plan, roof["kernel"])

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / PAGE_TFLOPS if case.name.startswith("bf16_16x1x512x2048") else None,
        "dtype": case.dtype, "data": f"synthetic (seeded {case.dist}, sigma {case.sigma}, {case.dtype} RNE)",
        "config": {"workload": case.name, "N": case.N, "C": case.C, "K": case.K, "Hi": case.Hi, "Wi": case.Wi,
                   "Y": case.Y, "X": case.X, "pad": list(case.pad), "stride": list(case.stride),
                   "dil": list(case.dil), "groups": case.groups, "layout": case.layout,
                   "l2": "flushed before every step (512 MiB write, outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "kernel_path": path, "tile": list(plan.tile()), "k_splits": plan.k_splits(),
                   "useful_flop_per_step": useful, "algo_bytes_per_step": algo_bytes},
        "pct_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "roofline": roof,
        "e2e": {"value": job_tflops(useful, world, e2e_mean), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(dy_h.numel() + w_h.numel()) * esz,
                "d2h_bytes_per_step": int(np.prod(dx_s)) * esz, "ms_per_step": e2e_mean},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if not args.no_per_workload:
        # every other workload, timed the same way (L2 flushed outside each
        # step's events, >= 20 steps), on this rank's GPU
        pw = {}
        for c in wl.CASES:
            if c.name == case.name:
                continue
            pw[c.name] = measure_workload(B, c, args.pw_steps, args.warmup, flush, stream, peaks, num_sms)
        line["per_workload"] = pw
        # the shape-specialised SM-pair kernel (dy as a plain matrix, 2-D tiled
        # loads) against the dynamic im2col kernel on the workloads it applies
        # to -- the static-vs-dynamic comparison of "[igemm_dynamic] v4r1 bwd
        # dynamic kernel" (dynamic within 10% of static there)
        sd = {}
        for c in wl.CASES:
            pl = B.Plan.from_case(c)
            dyn = pw[c.name]["ms_per_step"] if c.name in pw else mean_ms
            os.environ["CONVBWD_DEBUG_A"] = "plain"
            try:
                eligible = B.Plan.from_case(c).a_operand() == "plain" and pl.a_operand() == "im2col"
            finally:
                os.environ.pop("CONVBWD_DEBUG_A", None)
            if not eligible:
                continue
            spec = measure_workload(B, c, args.pw_steps, args.warmup, flush, stream, peaks, num_sms,
                                    env={"CONVBWD_DEBUG_A": "plain"})
            sd[c.name] = {"dynamic_ms": dyn, "specialised_ms": spec["ms_per_step"],
                          "dynamic_over_specialised": dyn / spec["ms_per_step"],
                          "specialised_tflops": spec["tflops"]}
        line["static_vs_dynamic"] = sd
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # bounded oracle sample on the host cores (a reported baseline only)
        dts, fr, thr = [], 0.0, 1
        s = 0
        t_start = time.perf_counter()
        while time.perf_counter() - t_start < 10.0 and s < 256:
            dt, f, thr = oracle_sample(case, dy, w, s)
            dts.append(dt)
            fr += f
            s += 1
        line["cpu_baseline"] = {"value": useful * fr / sum(dts) / 1e12, "unit": "TFLOP/s", "cores": thr,
                                "kind": "oracle",
                                "sample": f"{s} oracle calls, each one image x 256 input channels "
                                          f"({100 * fr / max(s, 1):.2f}% of the workload per call, "
                                          f"{sum(dts):.1f} s in total)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
