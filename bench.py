"""Benchmark of the virtual-rank collectives on one GB300 (or N replicas).

Default workload (the one the headline metric is quoted on): allreduce, sum,
W = 8 virtual ranks, fp32, n = 67,108,864 elements per rank (256 MiB),
values normal(0, 1e-3).  One step = one allreduce through the library's C ABI
(one kernel launch that reads the 8 inputs once and writes the 8 outputs).
value = algorithmic bytes (2 * W * n * 4: every input read once, every output
written once) / time, in GB/s (1e9 B/s); the inputs (2 GiB) are larger than
L2, so no flush is needed between steps.

The same JSON line also carries:
  roofline      the dominant kernel's achieved GB/s (CUDA events around each
                launch on the launching stream) against the measured HBM copy
                peak, with DRAM traffic per launch from the committed ncu
                summary when the kernel sources still match it;
  e2e           the same metric with the inputs copied from pinned host memory
                and the outputs copied back inside the timed region;
  cpu_baseline  the CPU oracle, single-threaded, on a bounded sample of the
                same workload (rank 0, N = 1 only);
  ops           the other workloads and operations timed in the same run
                (reduce-scatter, allgather, ring order, bf16 avg, fusion,
                small messages) unless --no-extras.

--impl reference times the CPU oracle itself as the reference arm.
Multi-GPU (torchrun): every rank runs its own independent replica (weak
scaling, no exchange between GPUs); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import collective_reduction_virtual_gb300 as vc  # noqa: E402
from collective_reduction_virtual_gb300 import inputs as I  # noqa: E402

METRIC = "reduce-scatter/allreduce HBM GB/s (bytes read+written), % of GB300 HBM peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
# the device code of the timed kernels: DRAM traffic taken by ncu stays valid
# while these files are unchanged
KERNEL_SOURCES = ["device_common.cuh", "reduce_kernels.cuh", "reduce_f32.cu", "staged_kernels.cu"]


# ------------------------------------------------------------ distributed

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    ws, rank, _ = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return ws, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device="cpu") -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_rank_step: float, steps: int, world: int, max_seconds: float) -> float:
    """Whole-job GB/s: bytes every rank moved, over the slowest rank's time."""
    return bytes_per_rank_step * steps * world / max_seconds / 1e9


# ---------------------------------------------------------------- helpers

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "collective_reduction_virtual_gb300", "csrc")
    for name in KERNEL_SOURCES:
        p = os.path.join(csrc, name)
        if os.path.exists(p):
            with open(p, "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since it was captured."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clock and clock-event reasons during the timed region
    (NVML through ctypes; nvidia-smi as a fallback).  Read-only."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, period_s=0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            handle = ctypes.c_void_p()
            uuid = None
            try:
                uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            except Exception:
                uuid = None
            ok = False
            if uuid:
                u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                ok = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(handle)) == 0
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(handle)) == 0
            if not ok:
                raise OSError("no NVML handle")
            self._nvml, self._handle = nv, handle
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:  # 1 = SM
                self.max_mhz = mx.value
        except OSError:
            self._nvml = None

    def _poll(self):
        nv, h = self._nvml, self._handle
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        getr = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if getr(h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def _smi(self):
        cmd = ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
               "--format=csv,noheader,nounits", "-lms", "100"]
        try:
            self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, text=True)
        except OSError:
            self._proc = None
            return
        for line in self._proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                self.samples.append(int(float(parts[0])))
                self.max_mhz = int(float(parts[1]))
                self.reasons |= int(parts[2], 16)
            except (ValueError, IndexError):
                pass
            if self._stop.is_set():
                break

    def __enter__(self):
        self._thread = threading.Thread(target=self._poll if self._nvml else self._smi, daemon=True)
        self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if not self._nvml and getattr(self, "_proc", None):
            self._proc.terminate()
        self._thread.join(timeout=2)

    def summary(self):
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "samples": len(self.samples), "reasons": names,
                "source": "nvml" if self._nvml else "nvidia-smi"}


def timed_steps(step, steps, warmup, stream, per_launch=True):
    """Run warmup untimed steps, then time `steps` steps with CUDA events on
    `stream` (barrier + synchronize on both sides).  Returns (total seconds,
    median seconds per launch)."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        if per_launch:
            ev[i][0].record(stream)
        step()
        if per_launch:
            ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    total = t0.elapsed_time(t1) / 1e3
    per = (statistics.median(a.elapsed_time(b) for a, b in ev) / 1e3) if per_launch \
        else total / steps
    return total, per


# ---------------------------------------------------------------- workloads

def ar_w8_f32(n_override=None):
    W, n = 8, n_override or (1 << 26)
    return dict(name="allreduce sum, W=8 virtual ranks, fp32, n=%d per rank, normal(0,1e-3)" % n,
                W=W, n=n, kind="gradient", workload=I.AR_W8_F32, op="sum", dtype=torch.float32,
                es=4)


def shifted_copy(t, k):
    """A copy of t that starts k elements into a fresh buffer."""
    buf = torch.empty(t.numel() + 4, dtype=t.dtype, device=t.device)
    v = buf[k:k + t.numel()]
    v.copy_(t)
    return v


def fusion_pipeline_bytes(counts, es, W):
    """Algorithmic bytes and launches of the fusion-buffer pipeline: per
    batch of two or more tensors pack, allreduce and unpack (6*W*B_batch,
    3 launches), per batch of one tensor one allreduce (2*W*B, 1 launch)."""
    begin = vc.fuse_plan(counts, 0 if es == 4 else 1)
    nbytes = launches = 0
    for b in range(len(begin) - 1):
        bb = sum(counts[begin[b]:begin[b + 1]]) * es
        multi = begin[b + 1] - begin[b] > 1
        nbytes += (6 if multi else 2) * W * bb
        launches += 3 if multi else 1
    return nbytes, launches


def build_workload(args, dev, rank):
    """The timed step for --op (default: the W=8 fp32 2^26 allreduce).
    Returns a dict with the step function, its algorithmic bytes and the
    device buffers that the end-to-end measurement copies in and out."""
    vflags = {"auto": 0, "direct": vc.FLAG_DIRECT, "staged": vc.FLAG_STAGED}[args.variant]
    ring = args.order == "ring"
    red = args.reduction
    dt = torch.bfloat16 if args.dtype == "bf16" else torch.float32
    es = 2 if args.dtype == "bf16" else 4
    seed_off = 100_000 * rank  # every replica draws its own inputs
    if args.op in ("fusion", "multi"):
        W = args.W or 8
        counts = [int(c) for c in I.fusion_counts()][:args.tensors]
        g = torch.Generator(device=dev)
        tens = []
        for u in range(W):
            g.manual_seed(I.rank_seed(I.FUSION_W8, u) + seed_off)
            tens.append([torch.randn(c, generator=g, device=dev).mul_(1e-3).to(dt) for c in counts])
        outs = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
        B = sum(counts) * es
        if args.op == "fusion":
            fused = [torch.empty((64 << 20) // es, dtype=dt, device=dev) for _ in range(W)]
            step = vc.FusionBufferPlan(tens, outs, fused, op=red, ring_order=ring)
            bytes_, launches = fusion_pipeline_bytes(counts, es, W)
            desc = ("one C call: pack + in-place allreduce + unpack per 64 MiB batch (6*W*B; a "
                    "batch of one tensor is allreduced straight, 2*W*B)")
        else:
            plan = vc.FusionPlan(tens, outs, op=red, ring_order=ring)
            step = lambda: plan()  # noqa
            nb = len(vc.fuse_plan(counts, 0 if es == 4 else 1)) - 1
            launches = -(-len(counts) // min(64, 768 // W))
            bytes_ = 2 * W * B
            desc = ("64 MiB batches, read straight from the tensors and written straight to "
                    "the outputs (2*W*B), batches planned and launched in C")
        return dict(name=f"tensor-fusion allreduce {red}, W={W}, {len(counts)} {args.dtype} tensors per "
                         f"rank (log-uniform 1024..4194304 elements), {desc}",
                    W=W, n=sum(counts), step=step, bytes=bytes_, launches=launches,
                    ins=[t for row in tens for t in row], outs=[t for row in outs for t in row],
                    es=es, reduction=red, dtype=args.dtype)
    W = args.W or 8
    n = args.n or (1 << 26)
    kind = "outliers" if args.dtype == "bf16" else ("gradient" if W == 8 else "uniform")
    make = {"uniform": I.uniform, "gradient": I.gradient, "outliers": I.outliers}[kind]
    wl = {"gradient": I.AR_W8_F32, "outliers": I.AR_W8_BF16, "uniform": I.SWEEP}[kind]
    ins = [make(n, I.rank_seed(wl, u) + seed_off, dev) for u in range(W)]
    if args.misalign:  # rank u's input starts u % 4 elements past a 16-byte boundary
        ins = [shifted_copy(t, u % 4) for u, t in enumerate(ins)]
    if args.op in ("wire", "sparse", "sparse_topk"):
        outs = [torch.empty_like(t) for t in ins]
        topk = args.op == "sparse_topk"
        if args.op == "wire":
            step = lambda: vc.allreduce_wire(ins, outs, wire="f16", op=red,  # noqa
                                             ring_order=ring)
            bytes_ = 2 * W * n * 4
            what = "fp16-wire allreduce"
        else:
            acc = None if args.no_accumulation else [torch.zeros_like(t) for t in ins]
            nnz = torch.empty(W, dtype=torch.int64, device=dev)
            wsb = (vc.sparse_workspace_min_bytes(W, n, topk) if args.sparse_workspace == "min"
                   else vc.sparse_workspace_bytes(W, n, topk))
            ws = torch.empty(max(1, wsb), dtype=torch.uint8, device=dev)
            frac = args.sparsity if topk else 1e-3
            step = lambda: vc.sparse_allreduce(ins, outs, acc, frac, topk, nnz, ws)  # noqa
            bytes_ = (2 if acc is None else 4) * W * n * 4
            what = (f"sparsified allreduce, top-{frac:g} of each rank" if topk else
                    f"sparsified allreduce, threshold {frac:g}") + \
                (", without accumulations" if acc is None else ", with error feedback")
            if topk and args.sparse_workspace == "min":
                what += ", minimum workspace (no candidate lists)"
        launches = 1
        if topk:
            # 13 kernels over the whole array; 25 on the candidate path, which
            # the library takes when the lists hold 3K entries (K < n/4) or a
            # tenth of the array (a two-sided band; a second-digit sample pass
            # and its selection included), 27 when the lists also give the
            # output (an output pass, and, with accumulations, a pass that
            # restores x in them should a rank's list fail)
            K = math.ceil(frac * n)
            cap = ((n // 8 + 4096 if n // 8 + 4096 < n else n) + 3) & ~3
            wide = 4 * K < n and cap >= 3 * K  # lower bound only: output from the lists
            cand = 0 < K < n and (wide or 10 * cap >= n) and args.sparse_workspace != "min"
            launches = ((27 if acc is not None else 26) if wide else 25) if cand else 13
        return dict(name=f"{what}, W={W}, f32, n={n} per rank", W=W, n=n, step=step,
                    bytes=bytes_, launches=launches, ins=ins,
                    outs=outs, es=4, reduction=red, dtype="f32")
    if args.op == "allreduce":
        outs = [torch.empty_like(t) for t in ins]
        step = lambda: vc.allreduce(ins, outs, op=red, ring_order=ring, flags=vflags)  # noqa
        bytes_ = 2 * W * n * es
        host_step = lambda hi, ho: vc.allreduce(hi, ho, op=red, ring_order=ring,  # noqa
                                                flags=vflags)
    elif args.op == "reduce_scatter":
        outs = [torch.empty(vc.segment(n, W, j)[1], dtype=dt, device=dev) for j in range(W)]
        step = lambda: vc.reduce_scatter(ins, outs, op=red, ring_order=ring, flags=vflags)  # noqa
        bytes_ = (W + 1) * n * es
        host_step = lambda hi, ho: vc.reduce_scatter(hi, ho, op=red, ring_order=ring,  # noqa
                                                     flags=vflags)
    else:  # allgather: the inputs are the W segments
        ins = [t[:vc.segment(n, W, j)[1]].clone() for j, t in enumerate(ins)]
        outs = [torch.empty(n, dtype=dt, device=dev) for _ in range(W)]
        step = lambda: vc.allgather(ins, n, outs, flags=vflags)  # noqa
        bytes_ = (1 + W) * n * es
        host_step = lambda hi, ho: vc.allgather(hi, n, ho)  # noqa
    dist_name = {"gradient": "normal(0,1e-3)", "uniform": "uniform[-1,1]",
                 "outliers": "normal(0,1e-2) with 1% outliers x100"}[kind]
    if args.misalign:
        dist_name += ", inputs at mixed 16-byte phases (element-wise path)"
    return dict(name=f"{args.op} {red}, W={W} virtual ranks, {args.dtype}, n={n} per rank, "
                     f"{dist_name}", W=W, n=n, step=step, bytes=bytes_, launches=1, ins=ins,
                outs=outs, es=es, reduction=red, dtype=args.dtype, host_step=host_step)


def run_vcoll(args):
    world, rank = init_dist("nccl" if int(os.environ.get("WORLD_SIZE", "1")) > 1 else "gloo")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    vc.lib()
    stream = torch.cuda.current_stream()
    wl = build_workload(args, dev, rank)
    W, n, alg_bytes = wl["W"], wl["n"], wl["bytes"]

    with ClockSampler() as clocks:
        total, per_step = timed_steps(wl["step"], args.steps, args.warmup, stream)
    total_max = max_over_ranks(total, dev if world > 1 else "cpu")
    value = aggregate_gbs(alg_bytes, args.steps, world, total_max)
    achieved = alg_bytes / per_step / 1e9
    peak, peak_src = measured_peaks()
    default = args.op == "allreduce" and W == 8 and n == (1 << 26) and args.dtype == "f32"
    kernel_key = None
    if default and wl["reduction"] == "sum" and args.order == "fast":
        kernel_key = ("vc_reduce_staged<float,8,OpSum,AR,tree> W=8 n=2^26"
                      if args.variant == "staged" else
                      "vc_reduce_vec<float,8,OpSum,AR,tree> W=8 n=2^26")
    big = W * n * wl["es"] > 2 * L2_BYTES
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_max / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
        "data": "synthetic (seeded, generated on the GPU)",
        "config": {"workload": wl["name"], "op": args.op, "reduction": wl["reduction"], "W": W,
                   "n_per_rank": n, "elem": args.dtype,
                   "order": "ring" if args.order == "ring" else "fastest (pairwise tree)",
                   "variant": args.variant, "bytes_per_step": alg_bytes,
                   "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2; no flush" if big else
                         "inputs fit in L2: number is L2-warm"},
        "pct_of_peak": {"measured_copy_peak": round(100 * achieved / peak, 1),
                        "nominal_8000": round(100 * achieved / NOMINAL_HBM_GBS, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": committed_traffic(kernel_key) if kernel_key else None,
                     "kernel": kernel_key or args.op,
                     "algorithmic_bytes_per_launch": alg_bytes // wl["launches"]},
        "gpu_launches": args.steps * wl["launches"],
        "clocks": clocks.summary(),
    }
    if not args.no_e2e:
        line["e2e"] = e2e_measure(wl, args, stream, world, dev)
    if rank == 0 and world == 1 and not args.no_cpu and default:
        line["cpu_baseline"] = cpu_baseline(ar_w8_f32(), args.cpu_seconds)
    if not args.no_extras and default:
        line["ops"] = extras(args, stream, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_measure(wl, args, stream, world, dev):
    """Host buffers in, host buffers out, through the public API: the inputs
    start in pinned host memory and the results must end there.  Two ways,
    both timed with the host transfers inside the region:
      value         the collective called directly on the pinned host buffers
                    (its kernels read the inputs and write the outputs over
                    the CPU-GPU link; no staging copies);
      staged_copies H2D copies of the inputs, the collective on device
                    buffers, D2H copies of the outputs."""
    h_in = [t.cpu().pin_memory() for t in wl["ins"]]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in wl["outs"]]
    steps = max(1, min(args.steps, 10))
    bi = sum(t.numel() * t.element_size() for t in wl["ins"])
    bo = sum(t.numel() * t.element_size() for t in wl["outs"])
    out = {"unit": "GB/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": steps}
    if "host_step" in wl:
        total, _ = timed_steps(lambda: wl["host_step"](h_in, h_out), steps,
                               max(1, min(args.warmup, 2)), stream, per_launch=False)
        total = max_over_ranks(total, dev if world > 1 else "cpu")
        out["value"] = round(aggregate_gbs(wl["bytes"], steps, world, total), 1)
        out["how"] = "collective on pinned host buffers (kernel reads/writes over NVLink-C2C)"

    def step():
        for d, h in zip(wl["ins"], h_in):
            d.copy_(h, non_blocking=True)
        wl["step"]()
        for h, d in zip(h_out, wl["outs"]):
            h.copy_(d, non_blocking=True)

    total, _ = timed_steps(step, steps, max(1, min(args.warmup, 2)), stream, per_launch=False)
    total = max_over_ranks(total, dev if world > 1 else "cpu")
    staged = round(aggregate_gbs(wl["bytes"], steps, world, total), 1)
    out["staged_copies"] = staged
    if "value" not in out:
        out["value"] = staged
        out["how"] = "H2D copies, collective on device buffers, D2H copies"
    return out


def cpu_baseline(cfg, seconds):
    """The CPU oracle (single-threaded ring simulation) on a bounded sample of
    the same workload: W rank buffers of the first m elements, allreduced
    repeatedly for about `seconds` of CPU time."""
    import oracle
    W = cfg["W"]
    m = min(cfg["n"], 1 << 22)
    xs = [I.gradient(m, I.rank_seed(cfg["workload"], u)).numpy() for u in range(W)]
    t = time.perf_counter()
    oracle.allreduce(xs, "sum", oracle.F32)
    one = time.perf_counter() - t
    reps = max(1, int(round(seconds / max(one, 1e-6))))
    t = time.perf_counter()
    for _ in range(reps):
        oracle.allreduce(xs, "sum", oracle.F32)
    dt = time.perf_counter() - t
    return {"value": round(2 * W * m * cfg["es"] * reps / dt / 1e9, 3), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{reps} allreduces (sum, ring order) of W={W} fp32 buffers holding the "
                      f"first {m} elements of the workload ({dt:.1f} s on one host core)"}


# ------------------------------------------------------------------ extras

def extras(args, stream, dev):
    out = {}

    def rate(fn, nbytes, steps=20, warmup=3):
        total, per = timed_steps(fn, steps, warmup, stream)
        return {"GBps": round(nbytes / per / 1e9, 1), "ms": round(per * 1e3, 4)}

    # W=8 fp32 n=2^26: reduce-scatter, allgather, ring-order allreduce
    W, n = 8, 1 << 26
    ins = I.rank_buffers("gradient", W, n, I.AR_W8_F32, dev)
    outs = [torch.empty_like(t) for t in ins]
    segs = [torch.empty(vc.segment(n, W, j)[1], device=dev) for j in range(W)]
    out["rs_sum_w8_f32_2^26"] = rate(lambda: vc.reduce_scatter(ins, segs, op="sum"),
                                     (W + 1) * n * 4)
    out["ag_w8_f32_2^26"] = rate(lambda: vc.allgather(segs, n, outs), (1 + W) * n * 4)
    out["ag_w8_f32_2^26_tma"] = rate(lambda: vc.allgather(segs, n, outs, flags=vc.FLAG_STAGED),
                                     (1 + W) * n * 4)
    out["ar_ring_sum_w8_f32_2^26"] = rate(
        lambda: vc.allreduce(ins, outs, op="sum", ring_order=True), 2 * W * n * 4)
    out["ar_sum_w8_f32_2^26_staged"] = rate(
        lambda: vc.allreduce(ins, outs, op="sum", flags=vc.FLAG_STAGED), 2 * W * n * 4)
    out["ar_sum_w8_f32_2^26_direct"] = rate(
        lambda: vc.allreduce(ins, outs, op="sum", flags=vc.FLAG_DIRECT), 2 * W * n * 4)
    out["ar_wire_f16_sum_w8_f32_2^26"] = rate(
        lambda: vc.allreduce_wire(ins, outs, wire="f16", op="sum"), 2 * W * n * 4)
    out["rs_sum_w8_f32_2^26_staged"] = rate(
        lambda: vc.reduce_scatter(ins, segs, op="sum", flags=vc.FLAG_STAGED), (W + 1) * n * 4)
    # sparsified allreduce with error feedback (SINGA): threshold and top-1 %
    acc = [torch.zeros_like(t) for t in ins]
    nnz = torch.empty(W, dtype=torch.int64, device=dev)
    ws = torch.empty(vc.sparse_workspace_bytes(W, n, True), dtype=torch.uint8, device=dev)
    out["sparse_threshold_w8_f32_2^26"] = rate(
        lambda: vc.sparse_allreduce(ins, outs, acc, 1e-3, False, nnz), 4 * W * n * 4)
    out["sparse_topk1pct_w8_f32_2^26"] = rate(
        lambda: vc.sparse_allreduce(ins, outs, acc, 0.01, True, nnz, ws), 4 * W * n * 4)
    # without accumulations (no error feedback): reads the inputs, writes the
    # outputs
    out["sparse_topk1pct_w8_f32_2^26_noacc"] = rate(
        lambda: vc.sparse_allreduce(ins, outs, None, 0.01, True, nnz, ws), 2 * W * n * 4)
    # the same call captured in a CUDA graph (27 kernels and two memsets per
    # call: the host launch overhead is gone)
    out["sparse_topk1pct_w8_f32_2^26_graph"] = graph_rate(
        lambda s: vc.sparse_allreduce(ins, outs, acc, 0.01, True, nnz, ws, stream=s),
        4 * W * n * 4, 10)
    out["sparse_bytes_formula"] = ("4*W*n*4: read inputs and accumulations, write outputs and "
                                   "accumulations (top-K: a 1/16 to 1/128 sample, a candidate "
                                   "pass that reads both and writes x -- or, above a settled "
                                   "key, the residual -- to the accumulation, and for small K "
                                   "an output pass from the candidate lists, else the dense "
                                   "pass reading the accumulation)")
    del ins, outs, segs, acc
    torch.cuda.empty_cache()

    # W=8 bf16 avg n=2^28 with outliers
    W, n = 8, 1 << 28
    ins = I.rank_buffers("outliers", W, n, I.AR_W8_BF16, dev)
    outs = [torch.empty_like(t) for t in ins]
    out["ar_avg_w8_bf16_2^28"] = rate(lambda: vc.allreduce(ins, outs, op="avg"), 2 * W * n * 2)
    out["ar_ring_avg_w8_bf16_2^28"] = rate(
        lambda: vc.allreduce(ins, outs, op="avg", ring_order=True), 2 * W * n * 2)
    out["ar_avg_w8_bf16_2^28_staged"] = rate(
        lambda: vc.allreduce(ins, outs, op="avg", flags=vc.FLAG_STAGED), 2 * W * n * 2)
    del ins, outs
    torch.cuda.empty_cache()

    # W=4 fp32 n=2^20 reduce-scatter: hot (L2-resident) and cold.  Cold is
    # taken two ways: (a) one launch timed with events right after a kernel
    # that READS a buffer of twice L2's size (a write flush would leave L2
    # full of dirty lines that the timed kernel then pays to write back),
    # median of 20; (b) a CUDA graph cycling through 16 input sets (320 MiB,
    # more than L2), so every launch finds its inputs evicted, with no flush
    # or event between launches
    W, n = 4, 1 << 20
    ins = I.rank_buffers("uniform", W, n, I.RS_W4, dev)
    segs = [torch.empty(vc.segment(n, W, j)[1], device=dev) for j in range(W)]
    nb = (W + 1) * n * 4
    out["rs_sum_w4_f32_2^20_hot"] = graph_rate(
        lambda s: vc.reduce_scatter(ins, segs, op="sum", stream=s), nb, 200)
    flush = torch.ones(2 * L2_BYTES // 4, device=dev)
    sink = torch.empty((), device=dev)
    times = []
    for i in range(23):
        torch.sum(flush, dim=0, out=sink)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        vc.reduce_scatter(ins, segs, op="sum")
        b.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            times.append(a.elapsed_time(b) / 1e3)
    per = statistics.median(times)
    out["rs_sum_w4_f32_2^20_cold"] = {
        "GBps": round(nb / per / 1e9, 1), "ms": round(per * 1e3, 4),
        "l2": "a 258 MiB read before each launch; median of 20 event-timed launches"}
    sets = [ins] + [[t.clone() for t in ins] for _ in range(15)]
    osets = [[torch.empty_like(t) for t in segs] for _ in range(16)]
    it = iter(range(1 << 30))

    def cycle(s):
        k = next(it) % 16
        vc.reduce_scatter(sets[k], osets[k], op="sum", stream=s)

    r = graph_rate(cycle, nb, 160)
    r["l2"] = "16 input sets (320 MiB) cycled in a CUDA graph: every launch reads evicted inputs"
    out["rs_sum_w4_f32_2^20_cold_cycled"] = r
    del ins, segs, flush, sets, osets
    torch.cuda.empty_cache()

    # fusion: 200 fp32 tensors per rank, W=8, 64 MiB buffer, pack + AR avg + unpack
    W = 8
    counts = [int(c) for c in I.fusion_counts()]
    tens = I.fusion_tensors(counts, W, dev)
    fouts = [[torch.empty_like(t) for t in tens[u]] for u in range(W)]
    fused = [torch.empty((64 << 20) // 4, device=dev) for _ in range(W)]
    tot = sum(counts) * 4
    fb, _ = fusion_pipeline_bytes(counts, 4, W)
    bplan = vc.FusionBufferPlan(tens, fouts, fused, op="avg")
    out["fusion_w8_200tensors"] = rate(lambda: bplan(), fb)
    out["fusion_w8_200tensors"]["bytes_formula"] = \
        "6*W*B per batch (pack + AR + unpack in one C call; 2*W*B for a one-tensor batch)"
    plan = vc.FusionPlan(tens, fouts, op="avg")
    out["fusion_w8_200tensors_direct"] = rate(lambda: plan(), 2 * W * tot)
    out["fusion_w8_200tensors_direct"]["bytes_formula"] = \
        "2*W*B_total (one pass, no fusion buffer); same bits as the pipeline"
    del tens, fouts, fused
    torch.cuda.empty_cache()

    # small messages: latency in a CUDA graph of 1000 launches
    lat = {}
    for W in (2, 8, 16):
        for nbytes in (1 << 10, 1 << 15):
            n = nbytes // 4
            ins = I.rank_buffers("uniform", W, n, I.SWEEP, dev)
            outs = [torch.empty_like(t) for t in ins]
            r = graph_rate(lambda s: vc.allreduce(ins, outs, op="sum", stream=s), 2 * W * nbytes,
                           1000)
            lat[f"ar_sum_W{W}_{nbytes}B"] = {"us": round(r["ms"] * 1e3, 2), "GBps": r["GBps"]}
            del ins, outs
    out["small_message_graph_1000"] = lat

    # a slice of the message-size sweep (--sweep runs all 420 points): W = 8,
    # fp32 sum, per-rank sizes from the latency path to past L2, each point
    # a CUDA graph of repeated launches (bytes per op as above)
    W = 8
    sweep = {}
    for nbytes in (1 << 12, 1 << 16, 1 << 20, 1 << 23, 1 << 26):
        n = nbytes // 4
        ins = [I.uniform(n, I.rank_seed(I.SWEEP, u), dev) for u in range(W)]
        outs = [torch.empty_like(t) for t in ins]
        segs = [torch.empty(vc.segment(n, W, j)[1], device=dev) for j in range(W)]
        reps = int(max(3, min(1000, 2e9 // (2 * W * nbytes))))
        row = {}
        for name, fn, b in (
                ("rs", lambda s: vc.reduce_scatter(ins, segs, op="sum", stream=s), (W + 1) * nbytes),
                ("ag", lambda s: vc.allgather(segs, n, outs, stream=s), (1 + W) * nbytes),
                ("ar", lambda s: vc.allreduce(ins, outs, op="sum", stream=s), 2 * W * nbytes)):
            r = graph_rate(fn, b, reps)
            row[name] = {"GBps": r["GBps"], "us": round(r["ms"] * 1e3, 2)}
        sweep[f"W8_{nbytes}B_per_rank"] = row
        del ins, outs, segs
    torch.cuda.empty_cache()
    out["sweep_w8_f32_sum_graph"] = sweep
    return out


def graph_rate(launch, nbytes, reps):
    """Device time per launch of `reps` launches captured in one CUDA graph
    (no host launch overhead between them)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        launch(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(reps):
            launch(s)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    g.replay()
    b.record()
    torch.cuda.synchronize()
    per = a.elapsed_time(b) / 1e3 / reps
    del g
    return {"GBps": round(nbytes / per / 1e9, 2), "ms": round(per * 1e3, 5),
            "timing": f"CUDA graph of {reps} launches"}


# ------------------------------------------------------------------ sweep

def run_sweep(args):
    """Message-size sweep: reduce-scatter and allreduce (sum, max) and
    allgather, fp32 uniform[-1, 1], per-rank sizes 1 KiB .. 1 GiB (powers of
    two), W in {2, 4, 8, 16}.  Each point is timed as a CUDA graph of
    repeated launches (many for small sizes, a few for large ones); GB/s uses
    the algorithmic bytes of each op.  Prints one JSON line per point."""
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    vc.lib()
    sizes = [1 << k for k in range(10, 31)]
    if args.sweep_max_bytes:
        sizes = [b for b in sizes if b <= args.sweep_max_bytes]
    for W in (2, 4, 8, 16):
        for nbytes in sizes:
            n = nbytes // 4
            ins = [I.uniform(n, I.rank_seed(I.SWEEP, u), dev) for u in range(W)]
            outs = [torch.empty_like(t) for t in ins]
            segs = [torch.empty(vc.segment(n, W, j)[1], device=dev) for j in range(W)]
            reps = int(max(3, min(1000, 2e9 // (2 * W * nbytes))))
            row = {"W": W, "bytes_per_rank": nbytes, "reps": reps}
            for name, fn, b in (
                    ("rs_sum", lambda s: vc.reduce_scatter(ins, segs, op="sum", stream=s),
                     (W + 1) * nbytes),
                    ("rs_max", lambda s: vc.reduce_scatter(ins, segs, op="max", stream=s),
                     (W + 1) * nbytes),
                    ("ag", lambda s: vc.allgather(segs, n, outs, stream=s), (1 + W) * nbytes),
                    ("ar_sum", lambda s: vc.allreduce(ins, outs, op="sum", stream=s),
                     2 * W * nbytes),
                    ("ar_max", lambda s: vc.allreduce(ins, outs, op="max", stream=s),
                     2 * W * nbytes)):
                r = graph_rate(fn, b, reps)
                row[name + "_GBps"] = r["GBps"]
                row[name + "_us"] = round(r["ms"] * 1e3, 2)
            row["l2"] = "fits in L2 (warm)" if 2 * W * nbytes <= L2_BYTES else "exceeds L2"
            print(json.dumps(row), flush=True)
            del ins, outs, segs
            torch.cuda.empty_cache()


# ------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle as the reference arm: same metric, unit and config; each
    step allreduces a bounded sample of the workload on one host core."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cfg = ar_w8_f32(args.n)
    W = cfg["W"]
    m = args.ref_elems
    xs = [I.gradient(m, I.rank_seed(cfg["workload"], u)).numpy() for u in range(W)]
    for _ in range(args.warmup):
        oracle.allreduce(xs, "sum", oracle.F32)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.allreduce(xs, "sum", oracle.F32)
    dt = time.perf_counter() - t
    value = 2 * W * m * 4 * args.steps / dt / 1e9
    sample = f"allreduce sum of W={W} fp32 buffers of the first {m} elements per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded normal(0,1e-3) gradients)",
            "config": {"workload": cfg["name"], "op": "allreduce", "reduction": "sum", "W": W,
                       "n_per_rank": cfg["n"], "elem": "fp32", "order": "ring",
                       "parallelism": "host, 1 core"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["vcoll", "reference"], default="vcoll")
    ap.add_argument("--n", type=int, default=None, help="elements per rank (default 2^26)")
    ap.add_argument("--op", choices=["allreduce", "reduce_scatter", "allgather", "fusion", "multi",
                                     "wire", "sparse", "sparse_topk"], default="allreduce")
    ap.add_argument("--sparsity", type=float, default=0.01, help="top-K fraction")
    ap.add_argument("--W", type=int, default=None, help="virtual ranks (default 8)")
    ap.add_argument("--tensors", type=int, default=200, help="tensors per rank for fusion/multi")
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--reduction", choices=["sum", "max", "avg"], default=None)
    ap.add_argument("--order", choices=["fast", "ring"], default="fast")
    ap.add_argument("--no-accumulation", action="store_true",
                    help="sparsified allreduce without accumulations (no error feedback)")
    ap.add_argument("--sparse-workspace", choices=["recommended", "min"], default="recommended",
                    help="top-K workspace size: with candidate lists, or the minimum (the "
                         "passes over the whole arrays)")
    ap.add_argument("--misalign", action="store_true",
                    help="start rank u's input u %% 4 elements past a 16-byte boundary (the "
                         "element-wise kernels)")
    ap.add_argument("--variant", choices=["auto", "direct", "staged"], default="auto",
                    help="kernel variant of the timed step (identical bits)")
    ap.add_argument("--sweep", action="store_true",
                    help="run the message-size sweep (one JSON line per point) instead")
    ap.add_argument("--sweep-max-bytes", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-elems", type=int, default=1 << 22)
    args = ap.parse_args(argv)
    if args.reduction is None:
        args.reduction = "avg" if args.op in ("fusion", "multi") else "sum"
    if args.warmup < 3 and args.impl == "vcoll":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_vcoll(args)


if __name__ == "__main__":
    main()
