"""Benchmark of the GB300 mixture-of-experts layer step.

One step = the whole hot path on one batch: router scoring + top-k + capacity
slotting, permute, grouped SwiGLU FFN (up and down), unpermute + combine, and
the backward (combine backward, dgrad, wgrad with fp32 accumulation, dx +
router gradient).  Default workload: the largest layer, dropless top-4 over 32
experts (T=32768, d=4096, f=1536, E=32, k=4, log-Zipf 1.3 router bias) in bf16
with an fp32 router.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own batch
(data-parallel replicas, weak scaling) and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "dropless_e32_bf16"
METRIC = "MoE-layer tokens/s fwd & fwd+bwd; grouped-GEMM % bf16 peak; permute GB/s"
PROFILE_DIR = os.path.join(ROOT, "profiles")
# source file of each kernel kind: a committed DRAM-traffic figure is used only while its source is unchanged
KERNEL_SOURCES = {
    "gemm_up_swiglu": "gemm_tc.cu", "gemm_down": "gemm_tc.cu", "gemm_dgrad_h_swiglu_bwd": "gemm_tc.cu",
    "gemm_dgrad_x": "gemm_tc.cu", "gemm_wgrad": "gemm_tc.cu", "permute": "rows.cu", "unpermute_combine": "rows.cu",
    "combine_bwd": "rows.cu", "dx_router": "rows.cu", "transpose_wr": "rows.cu", "dwr_reduce": "rows.cu",
    "router_topk": "router_tc.cu", "split_wr": "router_tc.cu", "slot_scan": "routing.cu",
    "slot_assign": "routing.cu", "dwr": "dwr_tc.cu", "split_dl": "dwr_tc.cu", "aux_loss": "aux_loss.cu",
    "aux_grad": "aux_loss.cu", "router_logit_grad": "rows.cu",
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--aux-loss-coeff", type=float, default=0.0,
                   help="auxiliary load-balancing loss coefficient (the layer configurations use none)")
    p.add_argument("--recompute", action="store_true",
                   help="keep no a, b, h between forward and backward (the backward recomputes them)")
    return p.parse_args()


# ----------------------------------------------------------------------------- #
# distributed plumbing
# ----------------------------------------------------------------------------- #
def dist_init(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- #
# clocks during the timed region
# ----------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sms, maxes, reasons, power = [], [], set(), []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms) if sms else None, "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- #
# algorithmic work per kernel (per launch)
# ----------------------------------------------------------------------------- #
def algorithmic_work(s, N: int, accumulate: bool = True, n_sms: int = 152):
    """(FLOPs, bytes) per launch of each kernel: the work the layer defines, counted on the N kept
    assignments (pad rows excluded); bytes are each operand read once and each result written once.
    The helper kernels (weight and logit-gradient splits, scans, reductions) count the bytes their
    step needs: their inputs read once and their outputs written once."""
    T, d, f, E, k = s.T, s.d_model, s.d_ff, s.E, s.k
    es = 2 if s.dtype == "bf16" else 4
    Wb = E * d * f * es  # one expert weight tensor
    grad_rw = 3 * E * d * f * 4 * (2 if accumulate else 1)
    Ep = 16 if E <= 16 else (32 if E <= 32 else (64 if E <= 64 else 128))  # experts padded for the MMA
    nb = (T + 63) // 64  # 64-token histogram blocks
    hist = E * k * nb * 4
    dwr_blocks = max(1, d // (256 if Ep <= 64 else 128))  # CTAs of the router-weight gradient along d
    dwr_ranges = max(1, min(n_sms // dwr_blocks, ((T + 63) // 64 + 1) // 2))
    # large bf16 layers take each kept row's g * dg from the dgrad h product (per row, a sum
    # of dH * h per 256-column tile), so their combine backward only scatters g * dY
    fused_dg = s.dtype == "bf16" and T * k * d * 2 >= (256 << 20)  # as the library decides
    nt = f // 256
    return {
        "split_wr": (0, d * E * 4 + 3 * Ep * d * 2),
        "router_topk": (2 * T * d * E, T * d * es + d * E * 4 + T * k * 8 + T * E * 4),
        "slot_scan": (0, 2 * hist + E * 8),
        "slot_assign": (0, T * k * 4 + hist + 2 * T * k * 4 + N * 4),
        "permute": (0, T * d * es + N * d * es),
        "gemm_up_swiglu": (4 * N * d * f, N * d * es + 2 * Wb + 3 * N * f * es),
        "gemm_down": (2 * N * f * d, N * f * es + Wb + N * d * es),
        "unpermute_combine": (0, N * d * es + T * d * es),
        "combine_bwd": (0, T * d * es + N * d * es) if fused_dg else (0, T * d * es + 2 * N * d * es + T * E * 4),
        "router_logit_grad": (0, N * nt * 4 + T * k * 12 + T * E * 4 * (2 if k == 1 else 1)),
        "aux_loss": (0, T * E * 4 + T * k * 4),
        "aux_grad": (0, 3 * T * E * 4),
        "gemm_dgrad_h_swiglu_bwd": (2 * N * d * f, N * d * es + Wb + 4 * N * f * es + (N * nt * 4 if fused_dg else 0)),
        "gemm_wgrad": (6 * N * d * f, 2 * N * d * es + 3 * N * f * es + grad_rw),
        "gemm_dgrad_x": (4 * N * f * d, 2 * N * f * es + 2 * Wb + N * d * es),
        "transpose_wr": (0, 2 * d * E * 4),
        "dx_router": (0, N * d * es + T * d * es + T * E * 4),
        "split_dl": (0, T * E * 4 + 3 * Ep * T * 2),
        "dwr": (2 * T * d * E, T * d * es + T * E * 4),
        "dwr_reduce": (0, dwr_ranges * d * E * 4 + d * E * 4 * (2 if accumulate else 1)),
    }


def binding(flops: float, nbytes: float, seconds: float, tflops_peak: float, hbm_peak: float) -> dict:
    """The roofline that binds a launch: tensor if its ideal FLOP time is the longer, else HBM."""
    t_tensor = flops / (tflops_peak * 1e12)
    t_hbm = nbytes / (hbm_peak * 1e9)
    if flops > 0 and t_tensor >= t_hbm:
        ach = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": tflops_peak, "unit": "TFLOP/s",
                "frac": round(ach / tflops_peak, 4)}
    ach = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(ach / hbm_peak, 4)}


# headers every kernel source includes (device helpers, PTX wrappers, launch declarations)
KERNEL_HEADERS = ("common.cuh", "tc_ptx.cuh", "internal.h")


def _code_only(text: str) -> str:
    """C/CUDA source with its comments removed and whitespace runs collapsed, so
    that an edit of comments alone leaves the digest unchanged."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest(name: str) -> str:
    """sha256[:16] of the code of kernel `name`: its source file and the shared headers,
    comments removed.  A committed ncu record counts only while this matches."""
    csrc = os.path.join(ROOT, "routing_permute_grouped_router_gb300", "csrc")
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES.get(name, "gemm_tc.cu"),) + KERNEL_HEADERS:
        h.update(f.encode())
        h.update(_code_only(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def committed_profile(name: str, workload: str):
    """The committed one-pass ncu record of kernel `name` on this workload
    (profiles/traffic_<workload>.json: DRAM bytes per launch and ncu duration), when it
    was taken on the current source of the kernel; None otherwise."""
    path = os.path.join(PROFILE_DIR, f"traffic_{workload}.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get("kernels", {}).get(name)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("source_sha") != source_digest(name):
        return None
    return rec


def committed_traffic(name: str, workload: str):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) from the committed
    profile of this workload, when it was taken on the current source of the kernel; None otherwise."""
    rec = committed_profile(name, workload)
    return None if rec is None else float(rec["dram_bytes_per_launch"])


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        pk = json.load(open(path))
        return pk.get("hbm_gbs", 6800.0), pk.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- #
# CPU oracle leg (a separate spawned process: numpy threads known, no fork after CUDA)
# ----------------------------------------------------------------------------- #
CPU_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle import moe_oracle as O
from routing_permute_grouped_router_gb300 import workload as W
shape = W.WORKLOADS[{name!r}].replace(T={tokens})
wl = W.make(shape, seed=0, micro_batches=1, with_dy=True)
C = O.capacity(shape.T, shape.k, shape.E, shape.capacity_factor, shape.capacity)
args = (wl.W_r, wl.bias, wl.W1.f64(), wl.W3.f64(), wl.W2.f64())
x, dy = wl.x[0].f64(), wl.dy[0].f64()
times = []
t_end = time.time() + {seconds}
for rep in range({reps}):
    t0 = time.perf_counter()
    st = O.forward(x, *args, shape.k, C)
    O.backward(dy, x, wl.W_r, args[2], args[3], args[4], st)
    times.append(time.perf_counter() - t0)
    if time.time() > t_end:
        break
print(json.dumps(dict(tokens={tokens}, times=times)))
"""


def run_oracle(name: str, tokens: int, seconds: float, reps: int, threads: int) -> dict:
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    code = CPU_SNIPPET.format(root=ROOT, name=name, tokens=tokens, seconds=seconds, reps=reps)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_baseline(name: str, T: int, seconds: float) -> dict:
    cores = len(os.sched_getaffinity(0))
    probe = run_oracle(name, min(T, 512), 0, 1, cores)
    per_tok = probe["times"][0] / probe["tokens"]
    tokens = int(max(256, min(T, (seconds / 2) / max(per_tok, 1e-9))))
    res = run_oracle(name, tokens, seconds, 50, cores)
    t = statistics.median(res["times"])
    return {"value": tokens / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 numpy oracle, forward+backward over the first {tokens} of the {T} tokens "
                      f"(capacity factor applied to the sample), median of {len(res['times'])} runs, "
                      f"BLAS threads = {cores}"}


def workload_config(name: str, s) -> dict:
    """The ``config`` of the JSON line: the same keys and values in both arms, so that the two lines
    name one workload."""
    return {"workload": name, "T": s.T, "d_model": s.d_model, "d_ff": s.d_ff, "E": s.E, "k": s.k,
            "capacity_factor": s.capacity_factor, "zipf_s": s.zipf_s, "layer_dtype": s.dtype,
            "step": "forward + backward (fp32 grad accumulate)",
            "l2": "inputs of the GPU arm exceed L2 or a 256 MB buffer is written before every timed step, "
                  "outside the step's events",
            "parallelism": "data-parallel replicas, one batch per rank"}


# ----------------------------------------------------------------------------- #
# reference arm: the oracle as it stands
# ----------------------------------------------------------------------------- #
def run_reference(args, world, rank):
    if rank != 0:
        return
    from routing_permute_grouped_router_gb300 import workload as W

    s = W.WORKLOADS[args.workload]
    cores = len(os.sched_getaffinity(0))
    probe = run_oracle(args.workload, min(s.T, 256), 0, 1, cores)
    per_tok = probe["times"][0] / probe["tokens"]
    budget = 150.0 / max(1, args.steps + args.warmup)
    tokens = int(max(16, min(s.T, budget / max(per_tok, 1e-9))))
    res = run_oracle(args.workload, tokens, 1e9, args.steps + args.warmup, cores)
    times = res["times"][args.warmup:] or res["times"]
    total = sum(times)
    value = tokens * len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args.workload, s),
        "sample_tokens": tokens,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: fp64 oracle forward+backward over the first {tokens} of {s.T} tokens"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- #
# our arm
# ----------------------------------------------------------------------------- #
def run_ours(args, world, rank, local):
    import torch

    import routing_permute_grouped_router_gb300 as pkg
    from routing_permute_grouped_router_gb300 import build as B
    from routing_permute_grouped_router_gb300 import layer
    from routing_permute_grouped_router_gb300 import workload as W

    if not os.path.exists(pkg.LIB_PATH):
        B.build()
    pkg.lib()
    dev = torch.device("cuda", local)
    s = W.WORKLOADS[args.workload]
    wl = W.make(s, seed=rank, micro_batches=1, with_dy=True)
    L = layer.from_workload(wl, str(dev), aux_loss_coeff=args.aux_loss_coeff, recompute=args.recompute)
    x = wl.x[0].torch(dev)
    dy = wl.dy[0].torch(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # 2x the 129 MB L2

    def step(accumulate=True):
        L.forward(x)
        L.backward(x, dy, accumulate=accumulate)

    for i in range(max(3, args.warmup)):
        step(accumulate=i > 0)
    torch.cuda.synchronize(dev)
    code, detail = pkg.moe_get_device_error(clear=True)
    if code != 0:
        raise RuntimeError(f"device error {code} {detail:#x}")
    N = int(L.saved["counts"].sum().item())

    # per-kernel table: an untimed pass with events around every kernel
    pkg.moe_profiler_filter(None)
    pkg.moe_profiler_enable(True)
    for _ in range(min(args.steps, 50)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    pkg.moe_profiler_enable(False)
    prof_all = pkg.moe_profiler_read()
    dom = max(prof_all.items(), key=lambda kv: kv[1][1])[0]

    # timed region: events around every step, and around the dominant kernel only
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)
    n0 = pkg.moe_launch_count()
    pkg.moe_profiler_filter(dom)
    pkg.moe_profiler_enable(True)
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    pkg.moe_profiler_enable(False)
    pkg.moe_profiler_filter(None)
    launches = pkg.moe_launch_count() - n0
    barrier(world)
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world)
    prof_dom = pkg.moe_profiler_read()

    # forward-only throughput (separate loop, same protocol)
    fs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    fe = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        fs[i].record(stream)
        L.forward(x)
        fe[i].record(stream)
    torch.cuda.synchronize(dev)
    fwd_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(fs, fe)), world)

    # inference forward (no saved state: the permuted rows and the products live
    # in the workspace, nothing is kept for a backward), same protocol
    Li = layer.from_workload(wl, str(dev), training=False)
    for _ in range(args.warmup):
        Li.forward(x)
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        flush.zero_()
        fs[i].record(stream)
        Li.forward(x)
        fe[i].record(stream)
    torch.cuda.synchronize(dev)
    inf_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(fs, fe)), world)
    del Li

    # end to end through host buffers: pinned x, dy in; y, dx out
    e2e = None
    if not args.no_e2e:
        # End to end through the public API: every step copies its x and dy in
        # from pinned host memory and its y and dx out to pinned host memory,
        # all inside the timed region.  Two buffer sets let step i+1's input
        # copy and step i-1's result copy run while step i computes, as a
        # training loop that feeds the layer would.  Each tensor moves as
        # N_COPY row chunks on N_COPY copy streams per direction, so several
        # copy engines share the host link; below 64 MB a direction one copy
        # per tensor (the extra launches and events would cost more than the
        # copies they overlap).
        N_COPY = 4 if (x.numel() + dy.numel()) * x.element_size() >= (64 << 20) else 1
        hx = x.cpu().pin_memory()
        hdy = dy.cpu().pin_memory()
        hy = torch.empty_like(L.y, device="cpu").pin_memory()
        hdx = torch.empty_like(L.dx, device="cpu").pin_memory()
        xin = [torch.empty_like(x) for _ in range(2)]
        dyin = [torch.empty_like(dy) for _ in range(2)]
        yout = [L.y, torch.empty_like(L.y)]
        dxout = [L.dx, torch.empty_like(L.dx)]
        h2d = [torch.cuda.Stream(dev) for _ in range(N_COPY)]
        d2h = [torch.cuda.Stream(dev) for _ in range(N_COPY)]

        def parts(t):
            return t.chunk(N_COPY, dim=0)

        def run(nsteps):
            ev_in = [[torch.cuda.Event() for _ in range(N_COPY)] for _ in range(nsteps)]
            ev_done = [torch.cuda.Event() for _ in range(nsteps)]
            ev_out = [[torch.cuda.Event() for _ in range(N_COPY)] for _ in range(nsteps)]
            start = torch.cuda.Event(enable_timing=True)
            stop = torch.cuda.Event(enable_timing=True)
            start.record(stream)

            def copy_in(i):
                for j, cs in enumerate(h2d):
                    with torch.cuda.stream(cs):
                        cs.wait_event(start)
                        if i >= 2:
                            cs.wait_event(ev_done[i - 2])  # step i-2 has finished reading this set
                        parts(xin[i % 2])[j].copy_(parts(hx)[j], non_blocking=True)
                        parts(dyin[i % 2])[j].copy_(parts(hdy)[j], non_blocking=True)
                        ev_in[i][j].record(cs)

            copy_in(0)
            for i in range(nsteps):
                if i + 1 < nsteps:
                    copy_in(i + 1)
                for ev in ev_in[i]:
                    stream.wait_event(ev)
                if i >= 2:
                    for ev in ev_out[i - 2]:
                        stream.wait_event(ev)  # step i-2's results have left this set
                L.y, L.dx = yout[i % 2], dxout[i % 2]
                L.forward(xin[i % 2], stream)
                L.backward(xin[i % 2], dyin[i % 2], accumulate=True, stream=stream)
                ev_done[i].record(stream)
                for j, cs in enumerate(d2h):
                    with torch.cuda.stream(cs):
                        cs.wait_event(ev_done[i])
                        parts(hy)[j].copy_(parts(yout[i % 2])[j], non_blocking=True)
                        parts(hdx)[j].copy_(parts(dxout[i % 2])[j], non_blocking=True)
                        ev_out[i][j].record(cs)
            for ev in ev_out[nsteps - 1]:
                stream.wait_event(ev)
            stop.record(stream)
            return start, stop

        run(2)
        torch.cuda.synchronize(dev)
        barrier(world)
        a, b = run(args.steps)
        torch.cuda.synchronize(dev)
        L.y, L.dx = yout[0], dxout[0]
        e2e_ms = max_over_ranks(a.elapsed_time(b), world)
        es = x.element_size()
        e2e = {"value": world * s.T * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": (x.numel() + dy.numel()) * es,
               "d2h_bytes_per_step": (L.y.numel() + L.dx.numel()) * es,
               "note": f"pinned host x, dy -> device and y, dx -> pinned host every step, {N_COPY} copy "
                       f"stream{'s' if N_COPY > 1 else ''} each way overlapping the neighbouring steps' "
                       "compute; forward + backward; no L2 flush"}

    if rank != 0:
        return
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    work = algorithmic_work(s, N, accumulate=True, n_sms=sms)
    hbm, tflops, peak_kind = peaks()
    kernels = {}
    for name, (n, ms) in prof_all.items():
        avg = ms / n
        entry = {"launches": n, "total_ms": round(ms, 4), "avg_us": round(1e3 * avg, 2),
                 "share": round(ms / sum(v[1] for v in prof_all.values()), 4)}
        if name in work:
            fl, nb = work[name]
            if fl:
                entry["tflops"] = round(fl / (avg / 1e3) / 1e12, 1)
                entry["frac_of_bf16_peak"] = round(fl / (avg / 1e3) / 1e12 / tflops, 3)
            entry["gbs"] = round(nb / (avg / 1e3) / 1e9, 1)
            entry["frac_of_hbm"] = round(nb / (avg / 1e3) / 1e9 / hbm, 3)
            entry["bound"] = binding(fl, nb, avg / 1e3, tflops, hbm)["bound"]
            # the same work over the kernel's duration in the committed ncu launch list
            # (serialised, no launch or event overhead), when taken on the current source
            rec = committed_profile(name, args.workload)
            if rec is not None and rec.get("ncu_time_us"):
                t_ncu = rec["ncu_time_us"] / 1e6
                entry["ncu_us"] = rec["ncu_time_us"]
                entry["dram_bytes_ncu"] = rec["dram_bytes_per_launch"]
                entry["frac_of_hbm_ncu"] = round(nb / t_ncu / 1e9 / hbm, 3)
                if fl:
                    entry["frac_of_bf16_peak_ncu"] = round(fl / t_ncu / 1e12 / tflops, 3)
        kernels[name] = entry
    fl, nb = work.get(dom, (0, 0))
    avg_s = prof_dom[dom][1] / prof_dom[dom][0] / 1e3
    roof = binding(fl, nb, avg_s, tflops, hbm)
    roof["algorithmic_flops_per_launch"] = fl
    roof["algorithmic_bytes_per_launch"] = nb
    roof["kernel"] = dom
    roof["launches_timed"] = prof_dom[dom][0]
    roof["traffic"] = committed_traffic(dom, args.workload)
    roof["peak_source"] = f"{peak_kind} ({'bf16_tflops_sustained' if roof['bound'] == 'tensor' else 'hbm_gbs'})"
    gemm_names = [n for n in kernels if n.startswith("gemm_")]
    gemm_flops = sum(work.get(n, (0, 0))[0] * prof_all[n][0] for n in gemm_names)  # the tail fixup adds time, no FLOPs
    gemm_ms = sum(prof_all[n][1] for n in gemm_names)
    value = world * s.T * args.steps / (total_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": s.dtype, "data": "synthetic",
        "config": workload_config(args.workload, s),
        "run": {"aux_loss_coeff": args.aux_loss_coeff, "recompute": args.recompute, "kept_assignments": N,
                "dropped_assignments": s.T * s.k - N, "replicas": world, "sms": sms,
                "l2_flush": "256 MB buffer written before every timed step, outside the step's events"},
        "fwd_tokens_per_s": world * s.T * args.steps / (fwd_ms / 1e3),
        "fwd_inference_tokens_per_s": world * s.T * args.steps / (inf_ms / 1e3),
        "grouped_gemm_frac_bf16_peak": round(gemm_flops / (gemm_ms / 1e3) / 1e12 / tflops, 4) if gemm_ms else None,
        "permute_gbs": kernels.get("permute", {}).get("gbs"),
        "roofline": roof,
        "gpu_launches": launches,
        "clocks": clk,
        "kernels": kernels,
        "kernels_note": "per-kernel CUDA events from an untimed pass of min(steps, 50) steps; the timed "
                        "region records events only around the roofline kernel; gbs = algorithmic bytes / "
                        "event time (an effective rate: reads that hit L2 count as moved); *_ncu: the same "
                        "work over the kernel's duration in the committed one-pass ncu launch list of this "
                        "workload (no launch or event overhead), present only when that list was taken on "
                        "the kernel's current source",
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline(args.workload, s.T, args.cpu_seconds)
        except Exception as exc:  # report, do not hide, a failed baseline
            line["cpu_baseline"] = {"value": None, "error": str(exc)[-300:]}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world, rank, local = dist_init(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
