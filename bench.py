"""Throughput of the exact-attention hot path on GB300: one step = forward + backward
(D preprocess, dK/dV, dQ) over one batch of seeded synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line on rank 0. `value` is whole-job TFLOPS with inputs resident in HBM
(counted FLOPs: forward 4·B·H·N²·d, backward 10·B·H·N²·d, both halved when causal);
`e2e` is the same metric through the C ABI with host buffers (pinned host -> device
copies of q, k, v, dO and device -> host copies of o, lse, dq, dk, dv inside the timed
region). `--impl reference` times the fp64 CPU oracle on bounded samples instead.
N > 1 (torchrun): every rank runs an independent replica of the workload on its own
GPU (weak scaling, no collective on the data path); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "B4_H32_N4096_d128_bf16_causal"
METRIC = "attention fwd/bwd TFLOPS (causal-adjusted) and % of GB300 dense BF16 peak"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}


def flops(w, part: str) -> float:
    """Counted FLOPs of one pass over the whole workload."""
    base = 4.0 * w.B * w.H * w.N * w.N * w.d
    f = {"fwd": base, "bwd": 2.5 * base, "dkv": 2.0 * base, "dq": 1.5 * base}[part]
    return f / 2 if w.causal else f


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    return dict(FALLBACK_PEAKS)


# ------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------
class NvmlClockSampler:
    """SM clock and clock-event reasons of one GPU polled every ~0.5 ms through NVML (the
    driver's management library, loaded with ctypes; reads only), so that even a timed
    region of a few tens of milliseconds gets a few dozen samples. start()/stop() as for
    ClockSampler; unavailable (None from create) where the library cannot be loaded."""

    # clock-event reason bits of the public NVML API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    @classmethod
    def create(cls, index: int):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            handle = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(handle)) != 0:
                return None
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
            if reasons is None:
                reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except (OSError, AttributeError):
            return None
        return cls(lib, handle, reasons)

    def __init__(self, lib, handle, reasons_fn):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib, self.handle, self.reasons_fn = lib, handle, reasons_fn
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        mx = ctypes.c_uint(0)
        lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))  # NVML_CLOCK_SM = 1
        self.max_mhz = float(mx.value)

    def _run(self):
        ct = self.ct
        clk, rs = ct.c_uint(0), ct.c_ulonglong(0)
        while not self.stop_flag.is_set():
            t = time.time()
            ok = self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(clk)) == 0
            ok = ok and self.reasons_fn(self.handle, ct.byref(rs)) == 0
            if ok:
                self.samples.append((t, float(clk.value), int(rs.value)))
            time.sleep(0.0005)

    def start(self):
        self.thread.start()

    def stop(self, t0: float | None = None, t1: float | None = None) -> dict | None:
        self.stop_flag.set()
        self.thread.join(timeout=5)
        inside = [x for x in self.samples if t0 is None or t0 <= x[0] <= t1]
        if not inside:
            return None
        reasons = sorted({name for _, _, r in inside for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(c for _, c, _ in inside),
                "sm_max_mhz": self.max_mhz, "samples": len(inside), "reasons": reasons,
                "window": "NVML samples taken inside the timed region, every ~0.5 ms"}


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"attn_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0: float | None = None, t1: float | None = None) -> dict | None:
        """Median SM clock of the samples taken between host times t0 and t1 (the timed
        region); throttle reasons seen in that window."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        import datetime
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, clk_max = float(parts[1]), float(parts[2])
                except ValueError:
                    continue
                if t0 is not None and not (t0 <= ts <= t1):
                    continue
                sm.append(clk)
                mx.append(clk_max)
                for name, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons),
                "window": "samples taken inside the timed region, every 50 ms"}


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------
def dist_setup():
    """Rank, world size and local rank from the torchrun environment; for N > 1 joins the
    process group: NCCL, or gloo without CUDA or with BENCH_DIST_BACKEND=gloo (the
    host-side logic is tested that way on the CPU)."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    use_cuda = torch.cuda.is_available() and os.environ.get("BENCH_DIST_BACKEND") != "gloo"
    if world > 1:
        import torch.distributed as dist
        if use_cuda:
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if use_cuda else "gloo")
    elif use_cuda:
        torch.cuda.set_device(0)
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_workload(w, rank: int):
    """Rank r's replica of workload w (weak scaling: every rank runs the whole workload on
    its own GPU, with inputs of its own seed)."""
    from exact_attention_tcgen05_gb300 import inputs as I
    if rank == 0:
        return w
    return I.Workload(w.name, w.B, w.H, w.N, w.d, w.dtype, w.causal, w.seed + 7919 * rank,
                      w.qk_gain, w.spike, w.spike_frac, w.oracle_slices)


def job_tflops(tflop_per_step: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return world * tflop_per_step * steps / (max_ms * 1e-3)


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_baseline(w, budget_s: float = 12.0, max_slices: int = 32) -> dict:
    """The fp64 oracle on (b, h) slices of the workload, in a fresh process (so its BLAS
    thread count is set before numpy loads), until about `budget_s` seconds."""
    cores = os.cpu_count() or 1
    code = f"""
import json, sys, time
sys.path.insert(0, {ROOT!r})
from exact_attention_tcgen05_gb300 import inputs as I
import oracle.attention as OA
w = I.BY_NAME[{w.name!r}]
slices = I.sampled_slices(w, min(w.BH, {max_slices}))
done, t_total = 0, 0.0
for b, h in slices:
    q, k, v, do = (I.to_f64(I.make_slice(w, b, h, t)) for t in ("q", "k", "v", "do"))
    t0 = time.perf_counter()
    OA.attention_forward(q, k, v, w.causal, w.scale)
    OA.attention_backward(q, k, v, do, w.causal, w.scale)
    t_total += time.perf_counter() - t0
    done += 1
    if t_total > {budget_s}:
        break
print(json.dumps({{"slices": done, "seconds": t_total}}))
"""
    env = dict(os.environ, OPENBLAS_NUM_THREADS=str(cores), OMP_NUM_THREADS=str(cores),
               MKL_NUM_THREADS=str(cores))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=600)
    if res.returncode != 0:
        return {"value": None, "error": res.stderr.strip().splitlines()[-1:]}
    r = json.loads(res.stdout.strip().splitlines()[-1])
    per_slice = (flops(w, "fwd") + flops(w, "bwd")) / w.BH
    return {"value": per_slice * r["slices"] / r["seconds"] / 1e12, "unit": "TFLOPS",
            "cores": cores, "kind": "oracle",
            "sample": f"{r['slices']} (b,h) slices of {w.name}, forward + backward in fp64 "
                      f"(numpy; BLAS on {cores} threads, elementwise steps single-threaded), "
                      f"{r['seconds']:.1f} s"}


def launches_per_step(w) -> int:
    """Kernels one forward + backward step launches: forward, D, dK/dV (two passes, dV then
    dK, for head dims above 128), dQ."""
    return 5 if w.d > 128 else 4


def workload_of(args):
    """The workload named by --workload, or the shape given by --custom (smaller cases for
    profiling: "B,H,N,d,dtype,causal|full", inputs drawn by the same generator)."""
    from exact_attention_tcgen05_gb300 import inputs as I
    if not args.custom:
        return I.BY_NAME[args.workload]
    B, H, N, d, dt, mask = args.custom.split(",")
    return I.custom(int(B), int(H), int(N), int(d), dt, mask == "causal", seed=1002)


def config_of(w, world: int) -> dict:
    """The `config` object of the JSON line (both arms print the same one)."""
    f = flops(w, "fwd") + flops(w, "bwd")
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "scale": w.scale, "counted_tflop_per_step": f / 1e12,
            "l2": f"inputs larger than L2: each of q,k,v,dO is "
                  f"{w.B * w.H * w.N * w.d * 2 / 2**20:.0f} MiB > {L2_BYTES / 2**20:.0f} MiB",
            "parallelism": f"replicas x{world}"}


def time_workload(w, steps: int, warmup: int) -> dict:
    """Per-kernel times (ms, averaged) of `steps` forward + backward passes over workload w,
    inputs resident, after `warmup` untimed ones; CUDA events on the launch stream."""
    import torch
    from exact_attention_tcgen05_gb300 import binding
    from exact_attention_tcgen05_gb300 import inputs as I
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    delta = torch.empty_like(lse)
    stream = torch.cuda.current_stream()
    kern = (
        lambda: binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse),
        lambda: binding.attn_bwd_preprocess(o, do, delta),
        lambda: binding.attn_bwd_dkv(q, k, v, lse, delta, do, causal=w.causal, scale=w.scale,
                                     dk=dk, dv=dv),
        lambda: binding.attn_bwd_dq(q, k, v, lse, delta, do, causal=w.causal, scale=w.scale,
                                    dq=dq),
    )
    for _ in range(warmup):
        for fn in kern:
            fn()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(stream)
        for j, fn in enumerate(kern):
            fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    code, where = binding.attn_last_kernel_status()
    if code != binding.ATTN_OK:
        raise RuntimeError(f"{w.name}: a kernel reported status {code} (site {where:#x})")
    out = {n: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps)) / steps
           for j, n in enumerate(("fwd", "delta", "dkv", "dq"))}
    out["step"] = ev[0][0].elapsed_time(ev[-1][4]) / steps
    del q, k, v, do, o, lse, dq, dk, dv, delta
    torch.cuda.empty_cache()
    return out


def measure_workloads(args, peaks: dict, skip: str) -> dict:
    """Forward and backward throughput of the other quoted workloads (the one the line is
    about is skipped) and of the head-dim-256 workload, measured after the main timed
    region, each on its own."""
    from exact_attention_tcgen05_gb300 import inputs as I
    burst = peaks["bf16_tflops"]
    steps = max(10, min(args.steps, 30))
    out = {}
    for w in I.WORKLOADS + I.HEAD_DIM_WORKLOADS:
        if w.name == skip:
            continue
        t = time_workload(w, steps, max(3, args.warmup))
        f_fwd, f_bwd = flops(w, "fwd"), flops(w, "bwd")
        bwd_ms = t["delta"] + t["dkv"] + t["dq"]
        fwd_tf = f_fwd / (t["fwd"] * 1e-3) / 1e12
        bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
        out[w.name] = {
            "steps": steps, "ms_per_step": t["step"],
            "step_tflops": (f_fwd + f_bwd) / (t["step"] * 1e-3) / 1e12,
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "fwd_frac_of_burst": fwd_tf / burst, "bwd_frac_of_burst": bwd_tf / burst,
            "kernels_ms": {n: t[n] for n in ("fwd", "delta", "dkv", "dq")}}
    return out


def run_ours(args) -> None:
    import torch
    from exact_attention_tcgen05_gb300 import binding
    from exact_attention_tcgen05_gb300 import inputs as I

    rank, world, local = dist_setup()
    w = workload_of(args)
    w = replica_workload(w, rank)  # each rank: its own replica (weak scaling)
    binding.load()
    host = {t: I.make_tensor(w, t).pin_memory() for t in ("q", "k", "v", "do")}
    dev = {t: x.cuda(non_blocking=True) for t, x in host.items()}
    q, k, v, do = dev["q"], dev["k"], dev["v"], dev["do"]
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    delta = torch.empty_like(lse)
    stream = torch.cuda.current_stream()

    def step():
        binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse)
        binding.attn_bwd_preprocess(o, do, delta)
        binding.attn_bwd_dkv(q, k, v, lse, delta, do, causal=w.causal, scale=w.scale, dk=dk,
                             dv=dv)
        binding.attn_bwd_dq(q, k, v, lse, delta, do, causal=w.causal, scale=w.scale, dq=dq)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # --- device-timed region: inputs resident, per-kernel events on the launch stream.
    names = ("fwd", "delta", "dkv", "dq")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = NvmlClockSampler.create(local) or ClockSampler(local)
    barrier(world)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_host0 = time.time()
    for i in range(args.steps):
        e = ev[i]
        e[0].record(stream)
        binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, o=o, lse=lse)
        e[1].record(stream)
        binding.attn_bwd_preprocess(o, do, delta)
        e[2].record(stream)
        binding.attn_bwd_dkv(q, k, v, lse, delta, do, causal=w.causal, scale=w.scale, dk=dk,
                             dv=dv)
        e[3].record(stream)
        binding.attn_bwd_dq(q, k, v, lse, delta, do, causal=w.causal, scale=w.scale, dq=dq)
        e[4].record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    time.sleep(0.1)
    clock_info = clocks.stop(t_host0, t_host1)
    barrier(world)
    total_ms = ev[0][0].elapsed_time(ev[-1][4])
    per_kernel = {n: [ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps)]
                  for j, n in enumerate(names)}
    code, where = binding.attn_last_kernel_status()
    if code != binding.ATTN_OK:
        raise RuntimeError(f"a bounded wait ran out inside a kernel (site {where:#x})")
    total_ms = max_over_ranks(total_ms, world)
    ms_step = total_ms / args.steps
    f_fwd, f_bwd = flops(w, "fwd"), flops(w, "bwd")
    value = job_tflops((f_fwd + f_bwd) / 1e12, args.steps, total_ms, world)

    # --- end to end through the C ABI with host buffers: attn_step_host copies the step's
    # inputs in from pinned host memory and its results out, overlapped with the kernels.
    e2e = None
    if not args.no_e2e:
        out_host = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
        h2d = sum(x.numel() * x.element_size() for x in host.values())
        d2h = sum(x.numel() * x.element_size() for x in out_host.values())
        scratch = torch.empty(binding.attn_step_host_scratch_bytes(w.B, w.H, w.N, w.d,
                                                                   E2E_CHUNKS),
                              dtype=torch.uint8, device="cuda")

        def host_step():
            binding.attn_step_host(host["q"], host["k"], host["v"], host["do"], out_host["o"],
                                   out_host["lse"], out_host["dq"], out_host["dk"],
                                   out_host["dv"], scratch, causal=w.causal, scale=w.scale,
                                   chunks=E2E_CHUNKS)

        host_step()  # warm-up of the host path
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e_start.record(stream)
        for _ in range(args.steps):
            host_step()
            # the step's results are on the host when it ends, as a caller reading them
            # needs (back-to-back calls also filled the driver's queue, and about one run in
            # ten of 20 such steps then took 4.4-6.3 ms per step instead of 3.7)
            stream.synchronize()
        e_end.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), world)
        e2e = {"value": job_tflops((f_fwd + f_bwd) / 1e12, args.steps, e2e_ms, world),
               "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "api": f"attn_step_host, {E2E_CHUNKS} chunks of (b, h) slices, copies "
                      f"overlapped with the kernels, stream synchronised after each step"}
        del scratch

    if rank != 0:
        return
    peaks = load_peaks()
    avg = {n: sum(x) / len(x) for n, x in per_kernel.items()}
    share = {n: avg[n] / ms_step for n in names}
    dominant = max(("fwd", "dkv", "dq"), key=lambda n: avg[n])
    dom_flops = flops(w, dominant)
    achieved = dom_flops / (avg[dominant] * 1e-3) / 1e12
    sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    burst = peaks["bf16_tflops"]
    fwd_t = f_fwd / (avg["fwd"] * 1e-3) / 1e12
    bwd_ms = avg["delta"] + avg["dkv"] + avg["dq"]
    bwd_t = f_bwd / (bwd_ms * 1e-3) / 1e12
    delta_bytes = 2 * w.B * w.H * w.N * w.d * 2 + w.B * w.H * w.N * 4
    traffic = load_traffic(dominant, w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) inputs, see exact_attention_tcgen05_gb300/inputs.py)",
        "config": config_of(w, world),
        "fwd_tflops": fwd_t, "bwd_tflops": bwd_t,
        "frac_of_peak": {"fwd": fwd_t / peaks["bf16_tflops"], "bwd": bwd_t / peaks["bf16_tflops"],
                         "peak_tflops": peaks["bf16_tflops"], "peak_source": peaks["source"],
                         "fwd_of_sustained": fwd_t / sustained, "bwd_of_sustained": bwd_t / sustained},
        "kernels": {n: {"ms": avg[n], "share": share[n]} for n in names},
        "delta_kernel": {"achieved_gbs": delta_bytes / (avg["delta"] * 1e-3) / 1e9,
                         "peak_gbs": peaks["hbm_gbs"],
                         "frac": delta_bytes / (avg["delta"] * 1e-3) / 1e9 / peaks["hbm_gbs"]},
        # The kernels are timed inside a region of well under a second, so the burst peak
        # (a GEMM timed alone) is the one to compare with, not the seconds-long sustained one.
        "roofline": {"kernel": dominant, "bound": "tensor", "achieved": achieved,
                     "peak": burst, "unit": "TFLOP/s", "frac": achieved / burst,
                     "peak_kind": f"bf16 burst ({peaks['source']})",
                     "frac_of_sustained": achieved / sustained,
                     "algorithmic_tflop_per_launch": dom_flops / 1e12, "traffic": traffic},
        "e2e": e2e, "clocks": clock_info, "gpu_launches": launches_per_step(w) * args.steps,
        "env": {"gpu": torch.cuda.get_device_name(), "torch": torch.__version__,
                "cuda": torch.version.cuda,
                "sm_count": torch.cuda.get_device_properties(0).multi_processor_count},
    }
    if not args.no_workloads:
        line["workloads"] = measure_workloads(args, peaks, w.name)
    if not args.no_decode:
        line["decode"] = measure_decode(args, peaks)
    if not args.no_varlen:
        line["varlen"] = measure_varlen(args, peaks)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


# Split-KV decoding, measured after the step (outside its timed region): one query row per
# (b, h) against a K/V cache larger than L2, inputs resident, partial + merge per call.
E2E_CHUNKS = 13  # chunks of (b, h) slices in the host-buffer step

DECODE_WORKLOAD = dict(name="decode_B8_H32_Nk32768_d128_bf16", B=8, H=32, Nk=32768, d=128,
                       dtype="bf16", seed=2024)


def measure_decode(args, peaks: dict) -> dict:
    import torch
    from exact_attention_tcgen05_gb300 import binding
    from exact_attention_tcgen05_gb300 import inputs as I

    c = DECODE_WORKLOAD
    B, H, Nk, d = c["B"], c["H"], c["Nk"], c["d"]
    wq = I.custom(B, H, 1, d, c["dtype"], False, seed=c["seed"])
    wk = I.custom(B, H, Nk, d, c["dtype"], False, seed=c["seed"] + 1)
    q, k, v = I.make_tensor_cuda(wq, "q"), I.make_tensor_cuda(wk, "k"), I.make_tensor_cuda(wk, "v")
    splits = binding.attn_decode_splits(B, H, Nk)
    parts = torch.empty((B, H, splits, d + 4), dtype=torch.float32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        binding.attn_decode(q, k, v, num_splits=splits, o=o, lse=lse, partials=parts)
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 100))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        binding.attn_decode_partial(q, k, v, num_splits=splits, partials=parts)
        ev[i][1].record(stream)
        binding.attn_decode_merge(parts, q.dtype, o=o, lse=lse)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    code, where = binding.attn_last_kernel_status()
    if code != binding.ATTN_OK:
        raise RuntimeError(f"a bounded wait ran out inside a decode kernel (site {where:#x})")
    part_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    merge_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / n
    kv_bytes = 2 * B * H * Nk * d * 2
    rec_bytes = B * H * splits * (d + 4) * 4
    total_bytes = kv_bytes + 2 * B * H * d * 2 + 2 * rec_bytes + B * H * 4
    total_ms = part_ms + merge_ms
    gbs = total_bytes / (total_ms * 1e-3) / 1e9
    part_gbs = (kv_bytes + B * H * d * 2 + rec_bytes) / (part_ms * 1e-3) / 1e9
    out = {"workload": c["name"], "splits": splits, "calls": n, "ms_per_call": total_ms,
           "partial_ms": part_ms, "merge_ms": merge_ms, "bytes_per_call": total_bytes,
           "l2": "K and V are 2 GiB each, far larger than L2",
           "roofline": {"kernel": "decode partial", "bound": "hbm", "achieved": part_gbs,
                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": part_gbs / peaks["hbm_gbs"],
                        "peak_kind": f"HBM copy ({peaks['source']})"},
           "achieved_gbs_call": gbs}
    del q, k, v, parts, o, lse
    torch.cuda.empty_cache()
    return out


def measure_varlen(args, peaks: dict) -> dict:
    """The packed benchmark batch (sequences of different lengths, no padding) through
    attn_fwd_varlen + attn_bwd_varlen, next to the same sequences padded to the longest
    one as a dense [B, H, max, d] batch through attn_fwd + attn_bwd. Both are credited
    with the same useful FLOPs (those of the real sequences). The packed calls get the host
    copies of cu_seqlens (which order the kernels' work items); the same calls without them
    are timed too."""
    import torch
    from exact_attention_tcgen05_gb300 import binding
    from exact_attention_tcgen05_gb300 import inputs as I

    w = I.VARLEN_BENCH
    q, k, v, do = (I.make_varlen_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    cu_q_host = torch.tensor(w.cu_q, dtype=torch.int32)
    cu_k_host = torch.tensor(w.cu_k, dtype=torch.int32)
    o = torch.empty_like(q)
    lse = torch.empty(w.H, w.total_q, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    ws = torch.empty_like(lse)
    # The padded batch: sequence b in rows [0, n_b) of slice b, zeros after it.
    B, H, M, d = w.B, w.H, w.max_q, w.d
    pq, pk, pv, pdo = (torch.zeros(B, H, M, d, dtype=q.dtype, device="cuda") for _ in range(4))
    for b in range(B):
        r0, r1 = w.cu_q[b], w.cu_q[b + 1]
        for src, dst in ((q, pq), (k, pk), (v, pv), (do, pdo)):
            dst[b, :, : r1 - r0] = src[r0:r1].transpose(0, 1)
    po = torch.empty_like(pq)
    plse = torch.empty(B, H, M, dtype=torch.float32, device="cuda")
    pdq, pdk, pdv = torch.empty_like(pq), torch.empty_like(pq), torch.empty_like(pq)
    pws = torch.empty_like(plse)
    stream = torch.cuda.current_stream()

    def packed(hq=cu_q_host, hk=cu_k_host):
        binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, w.max_q, w.max_k, causal=w.causal,
                                scale=w.scale, o=o, lse=lse, cu_seqlens_q_host=hq,
                                cu_seqlens_k_host=hk)
        binding.attn_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, w.max_q, w.max_k,
                                causal=w.causal, scale=w.scale, dq=dq, dk=dk, dv=dv,
                                workspace=ws, cu_seqlens_q_host=hq, cu_seqlens_k_host=hk)

    def packed_device_lengths():
        packed(None, None)

    def padded():
        binding.attn_fwd(pq, pk, pv, causal=w.causal, scale=w.scale, o=po, lse=plse)
        binding.attn_bwd(pq, pk, pv, po, plse, pdo, causal=w.causal, scale=w.scale, dq=pdq,
                         dk=pdk, dv=pdv, workspace=pws)

    n = max(10, min(args.steps, 50))
    result = {}
    for name, fn in (("packed", packed), ("packed_device_lengths", packed_device_lengths),
                     ("padded", padded)):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
        ev[0].record(stream)
        for i in range(n):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
        result[name] = ev[0].elapsed_time(ev[n]) / n
    code, where = binding.attn_last_kernel_status()
    if code != binding.ATTN_OK:
        raise RuntimeError(f"a packed-batch kernel reported status {code} (site {where:#x})")
    # useful FLOPs: forward 4*H*n^2*d per sequence (halved causal), backward 2.5x
    f_fwd = sum(4.0 * H * n_b * n_b * d for n_b in w.seqlens_q) / (2 if w.causal else 1)
    useful = 3.5 * f_fwd
    out = {"workload": w.name, "sequences": B, "lengths": list(w.seqlens_q),
           "tokens": w.total_q, "steps": n,
           "packed": {"ms_per_step": result["packed"],
                      "tflops": useful / (result["packed"] * 1e-3) / 1e12,
                      "host_cu_seqlens": True},
           "packed_device_lengths_only": {
               "ms_per_step": result["packed_device_lengths"],
               "tflops": useful / (result["packed_device_lengths"] * 1e-3) / 1e12},
           "padded": {"shape": f"B{B} H{H} N{M} d{d}", "ms_per_step": result["padded"],
                      "tflops_useful": useful / (result["padded"] * 1e-3) / 1e12},
           "speedup_vs_padded": result["padded"] / result["packed"],
           "frac_of_peak": useful / (result["packed"] * 1e-3) / 1e12 / peaks["bf16_tflops"]}
    del q, k, v, do, o, dq, dk, dv, pq, pk, pv, pdo, po, pdq, pdk, pdv
    torch.cuda.empty_cache()
    return out


def load_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this kernel
    and workload (profiles/traffic.json); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    entry = t.get(kernel, {})
    if entry.get("workload") == workload and entry.get("source_hash") == source_hash(kernel):
        return entry.get("dram_bytes_per_launch")
    return None


# The source files each kernel is compiled from (a traffic record is valid only while
# their contents match the hash stored with it).
KERNEL_SOURCES = {
    "fwd": ["fwd.cuh", "fwd_persistent.cuh", "fwd_pair.cuh", "pair.cuh", "schedule.h",
            "kernels_fwd.cu"],
    "delta": ["bwd_delta.cuh", "kernels_delta.cu"],
    "dkv": ["bwd_dkv.cuh", "bwd_dkv_persistent.cuh", "bwd_dq.cuh", "bwd_dq_persistent.cuh",
            "schedule.h", "kernels_dkv.cu"],
    "dq": ["bwd_dq.cuh", "bwd_dq_persistent.cuh", "schedule.h", "kernels_dq.cu"],
}
COMMON_SOURCES = ["common.cuh", "ptx.cuh", "launch.h", "varlen.h"]


def source_hash(kernel: str) -> str:
    """A hash of the code (comments and whitespace removed) of one kernel's sources: the
    DRAM counters in profiles/traffic.json hold only while it matches."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_tcgen05_gb300", "csrc")
    for fn in COMMON_SOURCES + KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)  # block comments
        text = re.sub(r"//[^\n]*", " ", text)                # line comments
        h.update(fn.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ------------------------------------------------------------------------------------
def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from exact_attention_tcgen05_gb300 import inputs as I
    import oracle.attention as OA
    w = workload_of(args)
    slices = I.sampled_slices(w, min(w.BH, args.steps + args.warmup))
    per_slice = (flops(w, "fwd") + flops(w, "bwd")) / w.BH
    times = []
    for i, (b, h) in enumerate(slices[: args.warmup + args.steps]):
        q, k, v, do = (I.to_f64(I.make_slice(w, b, h, t)) for t in ("q", "k", "v", "do"))
        t0 = time.perf_counter()
        OA.attention_forward(q, k, v, w.causal, w.scale)
        OA.attention_backward(q, k, v, do, w.causal, w.scale)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = per_slice * len(times) / total / 1e12
    cores = os.cpu_count() or 1
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": 1,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same generator as the CUDA arm)",
        "config": config_of(w, 1),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": f"{len(times)} (b,h) slices of {w.name}, one slice "
                                   f"forward + backward per step, fp64 numpy oracle"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--custom", default=None,
                    help="B,H,N,d,dtype,causal|full: a shape of one's own (profiling)")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--no-varlen", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
