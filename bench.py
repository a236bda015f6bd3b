#!/usr/bin/env python3
"""Benchmark of the GB300 TT embedding bag.

One step = one pass of the whole hot path over one batch: prefix grouping,
forward contraction, bag pooling, backward into the cores and the SGD update,
on the 48M-row training workload (360x360x370 rows, D = 128 = 4x8x4,
R1 = R2 = 32, 32768 bags of U{10..30} Zipf(1.2) lookups, lr 0.01).  The
12M-row forward workload (200x240x250 rows, 32768 bags of 20 Zipf(1.2)
lookups) is timed beside it and reported under "forward".

Timing: every step is captured once as a CUDA graph and replayed; each timed
replay is bracketed by CUDA events on its stream; between timed replays a
512 MB buffer is written (L2 flush) and the cores are restored from a copy
(both outside the events).  Per-kernel durations come from the library's own
launch events (tt_emb_profile_*), recorded in a separately captured graph.
`--impl reference` times the fp64 CPU oracle on a sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "TT embedding-bag lookups/s at batch 32768 (fwd, fwd+bwd); % of roofline"
TRAIN_CFG, FWD_CFG, MULTI_CFG = 5, 3, 4
LR = 0.01
FLUSH_BYTES = 512 << 20


def peaks():
    """Measured HBM bandwidth, bf16 tensor rate and SM clock of this machine, else the
    recipe's fallback."""
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        p.update(hbm_gbs=float(d.get("hbm_gbs", p["hbm_gbs"])),
                 bf16_tflops=float(d.get("bf16_tflops", p["bf16_tflops"])),
                 sm_max_mhz=float(d.get("sm_max_mhz", p["sm_max_mhz"])), source="measured")
    return p


# Kernels whose contractions run as three-term bf16 split products on the
# tensor cores (three tensor products per fp32-level product).
TENSOR_SPLIT_KERNELS = ("k_fwd_mma", "k_fwd_mma64", "k_bwd_mma")


def kernel_sources_hash() -> str:
    """Hash of the CUDA sources, to tell whether a stored ncu capture is current."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_train_compressed_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
    `kernel` on `workload` from the committed ncu summary, or None when that
    capture was taken on other kernel sources than these."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_sources_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel \
                    and parts[1] == workload and parts[3] == src:
                return int(parts[2])
    return None


def fp32_peak_tflops(sm_count: int, mhz: float) -> float:
    """FP32 FMA peak: SMs x 128 FP32 lanes x 2 FLOP x clock."""
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


def algorithmic(x, U_12: int, U_r: int) -> dict:
    """Algorithmic FLOPs and bytes of one batch (each unique prefix and row once)."""
    n1, n2, n3 = x.n
    R1, R2 = x.R[1], x.R[2]
    D, nnz, B = x.D, x.nnz, x.num_bags
    f2 = 2 * n1 * R1 * n2 * R2
    f3 = 2 * D * R2
    return dict(
        f2=f2, f3=f3, U_12=U_12, U_r=U_r, nnz=nnz, B=B,
        fwd_contract=U_12 * f2 + U_r * f3,
        pool=nnz * D,
        bwd_contract=3 * U_12 * f2 + 2 * U_r * f3,
        s_gather=nnz * D,
        fwd_bytes=8 * nnz + 8 * (B + 1) + 4 * B * D,
    )


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs.

    Reads NVML through ctypes (read-only queries, ~1 ms polling, so even a
    timed region of a few ms gets samples); falls back to `nvidia-smi -lms 200`.
    """
    # clocks-event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: str):
        self.gpu = gpu
        self.proc = None
        self.lines = []
        self.samples = []
        self.max_mhz = None
        self.nvml = None
        self._stop = threading.Event()

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        if not self.gpu.startswith("GPU-") or \
                lib.nvmlDeviceGetHandleByUUID(self.gpu.encode(), ctypes.byref(h)) != 0:
            raise OSError("no NVML handle")
        self.nvml, self.h, self.ct = lib, h, ctypes
        mx = ctypes.c_uint(0)
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)

    def _poll(self):
        ct, lib, h = self.ct, self.nvml, self.h
        mhz, rs = ct.c_uint(0), ct.c_ulonglong(0)
        get_r = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ct.byref(mhz)) == 0 and \
                    get_r(h, ct.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        try:
            self._nvml_open()
            self.t = threading.Thread(target=self._poll, daemon=True)
            self.t.start()
            return
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.nvml is not None:
            self._stop.set()
            self.t.join(timeout=2)
            sm = [m for m, _ in self.samples]
            reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items()
                              if r & bit})
            return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": self.max_mhz,
                    "samples": len(sm), "reasons": reasons, "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons), "source": "nvidia-smi"}


def rank_max(dist, v: float) -> float:
    """Max of a per-rank time over all ranks (the slowest replica sets the step time)."""
    if dist is None:
        return float(v)
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_throughput(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job units/s: every rank processes its own batch in the max-over-ranks time."""
    return units_per_rank * world / (ms_max * 1e-3)


# ----------------------------------------------------------------------------- GPU arm


class Workload:
    """Device-resident inputs of one workload plus its captured step graphs."""

    def __init__(self, cfg: int, train: bool, torch, tte, stream, mapping=None, bags=None):
        from tensor_train_compressed_gb300.inputs import make_inputs
        self.torch, self.tte, self.stream = torch, tte, stream
        self.x = x = make_inputs(cfg, with_grad=train, mapping=mapping, num_bags=bags)
        self.train = train
        dev = torch.device("cuda")
        self.cores0 = [torch.from_numpy(c).to(dev) for c in x.cores]
        self.cores = [c.clone() for c in self.cores0]
        self.grads = [torch.zeros_like(c) for c in self.cores]
        self.idx = torch.from_numpy(x.indices).to(dev)
        self.off = torch.from_numpy(x.offsets).to(dev)
        self.out = torch.empty((x.num_bags, x.D), dtype=torch.float32, device=dev)
        self.gout = torch.from_numpy(x.grad_out).to(dev) if train else None
        ws = tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.ws_bytes = ws
        # the bf16 split of the cores is kept in the workspace: made here once
        # (as when a model is loaded), then rewritten by every SGD step
        tte.tt_emb_split(self.cores, x.m, x.n, x.R, self.ws)

    def step(self):
        """forward on the kept split of the cores, backward into the (zero) core
        gradients, SGD that also resets them and splits the updated cores"""
        t, x = self.tte, self.x
        # a training step's forward keeps the per-row lookup lists for the
        # backward; an inference call does not need them
        flags = t.TT_EMB_CORES_SPLIT | (0 if self.train else t.TT_EMB_FORWARD_ONLY)
        t.tt_emb_forward_ex(self.cores, x.m, x.n, x.R, self.idx, self.off, None, "sum", self.out,
                            self.ws, flags=flags)
        if self.train:
            t.tt_emb_backward(self.gout, self.cores, x.m, x.n, x.R, self.idx, self.off,
                              self.grads, self.ws, reuse_grouping=True)
            t.tt_emb_sgd_ex(self.cores, self.grads, x.m, x.n, x.R, LR, True, self.ws)

    def restore(self):
        """the cores of step 0 again, and their split (outside the timed region,
        before the L2 flush: cores and planes start every step cold)"""
        for c, c0 in zip(self.cores, self.cores0):
            c.copy_(c0)
        self.tte.tt_emb_split(self.cores, self.x.m, self.x.n, self.x.R, self.ws)

    def capture(self, profile: bool = False):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        if profile:
            self.tte.tt_emb_profile_start()
        with torch.cuda.graph(g, stream=self.stream, capture_error_mode="thread_local"):
            self.step()
        n = self.tte.tt_emb_profile_stop() if profile else 0
        return g, n

    def grouping(self):
        return self.tte.read_grouping(self.x.m, self.x.n, self.x.R, self.x.nnz, self.x.num_bags,
                                      self.ws)


class MultiTableWorkload(Workload):
    """The eight-table forward workload: one tt_emb_forward_tables_ex call (each
    table grouped into its own workspace, then one persistent launch of the R = 64
    tensor-core chunk kernel over all tables' chunks, then one pooling launch).
    As for the single-table inference forward, every table's cores are split
    into its workspace once, at load time, and the calls pass TT_EMB_CORES_SPLIT."""

    def __init__(self, cfg: int, torch, tte, stream, bags=None):
        from tensor_train_compressed_gb300.inputs import CONFIGS, make_inputs
        self.torch, self.tte, self.stream = torch, tte, stream
        self.train = False
        dev = torch.device("cuda")
        self.xs = [make_inputs(cfg, table=t, num_bags=bags)
                   for t in range(len(CONFIGS[cfg]["tables"]))]
        self.x = self.xs[0]
        self.tables = []
        for x in self.xs:
            ws = tte.tt_emb_workspace_bytes(x.m, x.n, x.R, x.nnz, x.num_bags)
            self.tables.append(dict(
                cores=[torch.from_numpy(c).to(dev) for c in x.cores], m=x.m, n=x.n, R=x.R,
                indices=torch.from_numpy(x.indices).to(dev),
                offsets=torch.from_numpy(x.offsets).to(dev),
                out=torch.empty((x.num_bags, x.D), dtype=torch.float32, device=dev),
                workspace=torch.empty(ws, dtype=torch.uint8, device=dev)))
        self.ws = self.tables[0]["workspace"]
        self.ws_bytes = sum(t["workspace"].numel() for t in self.tables)
        for t in self.tables:
            tte.tt_emb_split(t["cores"], t["m"], t["n"], t["R"], t["workspace"])

    def step(self):
        self.tte.tt_emb_forward_tables(self.tables, flags=self.tte.TT_EMB_CORES_SPLIT)

    def restore(self):
        pass                                # the cores never change

    def groupings(self):
        return [self.tte.read_grouping(x.m, x.n, x.R, x.nnz, x.num_bags, t["workspace"])
                for x, t in zip(self.xs, self.tables)]


def time_replays(torch, wl, graph, steps, flush, profile_n=0):
    """Per-replay device ms (events on the replay stream); flush + restore outside the events."""
    tte = wl.tte
    s = wl.stream
    times, per_kernel = [], {}
    for _ in range(steps):
        with torch.cuda.stream(s):
            wl.restore()
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            graph.replay()
            e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1))
        for i in range(profile_n):
            name, ms = tte.tt_emb_profile_read(i)
            d = per_kernel.setdefault(name, [0.0, 0])
            d[0] += ms
            d[1] += 1
    return times, per_kernel


# The workloads of one bench run: (name, config, training step, Zipf rank -> row mapping).
# "train" is the step the headline value is measured on; the others are lines beside it.
WORKLOADS = (("train", TRAIN_CFG, True, None), ("forward", FWD_CFG, False, None),
             ("forward8", MULTI_CFG, False, None), ("config1", 1, False, None),
             ("config2", 2, False, None), ("forward_permuted", FWD_CFG, False, "permuted"),
             ("train_permuted", TRAIN_CFG, True, "permuted"))


def counts_of(g, x) -> dict:
    """Unique prefixes / rows / chunks of one grouping, and the algorithmic work of the batch."""
    U_12, U_r = g["U_12"], g["U_r"]
    if g["method"] == "direct":
        # a per-lookup forward makes no grouping: the batch's unique rows and
        # (i1, i2) prefixes (row // m3) are counted here
        M = int(np.prod(x.m))
        idx = x.indices[(x.indices >= 0) & (x.indices < M)]
        U_r = int(np.unique(idx).size)
        U_12 = int(np.unique(idx // x.m[2]).size)
    a = algorithmic(x, U_12, U_r)
    a.update(n_chunks=g["n_chunks"], method=g["method"], n_valid=g["n_valid"],
             ckpt_reused=g["ckpt_reused"])
    return a


def add_counts(alls):
    tot = {}
    for a in alls:
        for k in ("U_12", "U_r", "nnz", "B", "fwd_contract", "pool", "fwd_bytes", "n_chunks"):
            tot[k] = tot.get(k, 0) + a[k]
    return tot


def kernel_work(name: str, a: dict, x, train: bool):
    """Algorithmic work of one launch of kernel `name` on a batch with counts `a`:
    ("flop", F) for the contraction kernels (each unique prefix and unique row once),
    ("bytes", B) for the others (the bytes the method itself must read and write once
    at the DRAM level), or None."""
    nnz, B, D, U_r, U_12 = a["nnz"], a["B"], x.D, a["U_r"], a["U_12"]
    nc = a.get("n_chunks", 0)
    if name in ("k_fwd_mma", "k_fwd_mma64", "k_fwd_tiled", "k_fwd_generic"):
        return "flop", a["fwd_contract"]
    if name in ("k_bwd_mma", "k_bwd_generic"):
        return "flop", a["bwd_contract"]
    if name == "k_fwd_direct":                             # every lookup's chain on its own
        n1, n2, _ = x.n
        R1, R2 = x.R[1], x.R[2]
        return "flop", 2 * nnz * (n1 * n2 * R2 * R1 + D * R2)
    if name.startswith("k_group"):
        lists = 8 * nnz + 4 * U_r if train else 0          # perm + row_start
        return "bytes", (8 * nnz + 8 * (B + 1) + 4 * nnz + lists + 8 * U_r + 12 * U_12
                         + 16 * nc)
    if name == "k_pool":
        return "bytes", 8 * (B + 1) + 4 * nnz + 4 * nnz + 4 * B * D
    if name == "k_s_gather":
        return "bytes", 12 * nnz + 4 * B * D + 4 * U_r * D
    return None


def kernel_roofline(name, per_launch_ms, a, x, train, p_fp32, pk, sms, which):
    """Achieved rate of one kernel against the peak of what bounds it."""
    work = kernel_work(name, a, x, train)
    out = {"kernel": name, "avg_launch_ms": round(per_launch_ms, 5)}
    if work is None:
        out.update(bound="hbm", achieved=None, peak=pk["hbm_gbs"], unit="GB/s", frac=None,
                   traffic=None)
        return out
    kind, amount = work
    if kind == "bytes":
        ach = amount / (per_launch_ms * 1e-3) / 1e9
        out.update(bound="hbm", achieved=round(ach, 1), peak=pk["hbm_gbs"], unit="GB/s",
                   frac=round(ach / pk["hbm_gbs"], 4), traffic=stored_traffic(name, which),
                   algorithmic_bytes_per_launch=int(amount),
                   peak_source="measured copy bandwidth (MEASURED_PEAKS.json)")
        return out
    ach = amount / (per_launch_ms * 1e-3) / 1e12
    out.update(bound="alu", achieved=round(ach, 3), peak=round(p_fp32, 2), unit="TFLOP/s",
               frac=round(ach / p_fp32, 4), traffic=stored_traffic(name, which),
               algorithmic_flop_per_launch=int(amount),
               peak_source=f"{sms} SMs x 128 FP32 lanes x 2 x {pk['sm_max_mhz']:.0f} MHz (nominal "
                           "FFMA rate; a probe on this GPU measured 115 FFMA MAC/SM/clk, 90% "
                           "of the nominal 128)")
    if name in TENSOR_SPLIT_KERNELS:
        pt = pk["bf16_tflops"] / 3.0
        out["roofline_tensor"] = {
            "bound": "tensor", "achieved": round(ach, 3), "peak": round(pt, 1), "unit": "TFLOP/s",
            "frac": round(ach / pt, 4),
            "peak_source": f"measured bf16 dense burst {pk['bf16_tflops']:.1f} TFLOP/s / 3 bf16 "
                           "products per fp32-level product (three-term split)"}
    return out


def call_roofline(a, ms, p_fp32, pk):
    """North-star roofline of a whole forward call: the larger of the unique-prefix FLOPs
    at the FP32 peak and the index + offset + output bytes at the HBM peak."""
    F = a["fwd_contract"] + a["pool"]
    t_roof = max(F / (p_fp32 * 1e12), a["fwd_bytes"] / (pk["hbm_gbs"] * 1e9))
    return {"T_roof_us": round(t_roof * 1e6, 3), "T_call_us": round(ms * 1e3, 3),
            "frac": round(t_roof / (ms * 1e-3), 4), "F_unique_flop": int(F),
            "bytes": int(a["fwd_bytes"])}


def run_ours(args, rank, world, dist):
    import torch

    import tensor_train_compressed_gb300 as tte
    from tensor_train_compressed_gb300 import build as tbuild

    tbuild.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    props = torch.cuda.get_device_properties(local)
    uuid = str(getattr(props, "uuid", ""))
    gpu_id = uuid if uuid.startswith("GPU-") else (f"GPU-{uuid}" if uuid else str(local))
    pk = peaks()
    sms = props.multi_processor_count
    p_fp32 = fp32_peak_tflops(sms, pk["sm_max_mhz"])
    stream = torch.cuda.Stream()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    result = {}
    todo = WORKLOADS
    if args.only:
        todo = tuple(t for t in todo if t[0] == args.only)
    for name, cfg, train, mapping in todo:
        main = name == "train"
        wl = (MultiTableWorkload(cfg, torch, tte, stream, args.bags) if name == "forward8"
              else Workload(cfg, train, torch, tte, stream, mapping, args.bags))
        with torch.cuda.stream(stream):
            for _ in range(2):          # eager warm-up (also settles the library's caches)
                wl.restore()
                wl.step()
        stream.synchronize()
        for w_ in ([t["workspace"] for t in wl.tables] if name == "forward8" else [wl.ws]):
            rc, bits = tte.tt_emb_get_error(w_, stream)
            if rc != 0:
                raise RuntimeError(f"device status {bits} on workload {name}")
        if name == "forward8":
            alg = add_counts([counts_of(g, x) for g, x in zip(wl.groupings(), wl.xs)])
        else:
            alg = counts_of(wl.grouping(), wl.x)
        with torch.cuda.stream(stream):   # creates the timing events before any capture
            tte.tt_emb_profile_start()
            wl.restore()
            wl.step()
            tte.tt_emb_profile_stop()
        stream.synchronize()
        graph, _ = wl.capture()
        pgraph, n_launch = wl.capture(profile=True)
        steps = args.steps if main or name in ("forward", "forward8") else max(3, args.steps // 2)
        time_replays(torch, wl, graph, max(args.warmup, 3), flush)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        clocks = ClockSampler(gpu_id)
        clocks.start()
        t0 = time.perf_counter()
        times, _ = time_replays(torch, wl, graph, steps, flush)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        clk = clocks.stop()
        if dist is not None:
            dist.barrier()
        reps = max(3, min(steps, 10))
        _, kern = time_replays(torch, wl, pgraph, reps, flush, n_launch)
        if not main:                      # the last grouping of the timed replays
            if name == "forward8":
                alg["ckpt_reused"] = 0
            else:
                alg["ckpt_reused"] = wl.grouping()["ckpt_reused"]
        result[name] = dict(wl=wl, alg=alg, ms=rank_max(dist, float(np.mean(times))),
                            times=times, wall=wall, clocks=clk, kern=kern, reps=reps,
                            n_launch=n_launch, steps=steps)

    if args.only:
        # single-workload run (profiling driver): a short report, no e2e / baseline
        r = result[args.only]
        if rank == 0:
            return {"only": args.only, "ms_per_step": round(r["ms"], 5),
                    "lookups_per_s": round(weak_throughput(r["alg"]["nnz"], world, r["ms"]), 1),
                    "kernels": {k: round(v[0] / r["reps"], 5) for k, v in r["kern"].items()}}
        return None

    # ---- end to end through the public API from pinned host buffers (training step)
    wl = result["train"]["wl"]
    x = wl.x
    # the lookups' indices go in as int32 (TT_EMB_INDICES_I32: every row number of
    # the workload fits), half the bytes of the copy the forward waits for; the
    # same loop with int64 indices is timed beside it
    assert 0 <= int(x.indices.min()) and int(x.indices.max()) < 2 ** 31
    idx_h = {torch.int32: torch.from_numpy(x.indices.astype(np.int32)).pin_memory(),
             torch.int64: torch.from_numpy(x.indices).pin_memory()}
    off_h = torch.from_numpy(x.offsets).pin_memory()
    g_h = torch.from_numpy(x.grad_out).pin_memory()
    out_h = torch.empty((x.num_bags, x.D), dtype=torch.float32).pin_memory()
    idx_d = {dt: torch.empty(x.nnz, dtype=dt, device=wl.idx.device) for dt in idx_h}
    off_d, g_d = torch.empty_like(wl.off), torch.empty_like(wl.gout)
    copy_stream = torch.cuda.Stream()
    e2e_times = {torch.int32: [], torch.int64: []}
    for it in range(max(args.warmup, 3) + args.steps):
        for dt in (torch.int32, torch.int64):
            with torch.cuda.stream(stream):
                wl.restore()
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                # one C-ABI call: copies in on the copy stream, forward, backward and
                # SGD on `stream`, the pooled output copied back during the backward
                tte.tt_emb_step_host(wl.cores, wl.grads, x.m, x.n, x.R, idx_h[dt], off_h, g_h,
                                     out_h, idx_d[dt], off_d, g_d, wl.out, LR, wl.ws,
                                     flags=tte.TT_EMB_CORES_SPLIT, stream=stream,
                                     copy_stream=copy_stream)
                e1.record(stream)
            stream.synchronize()
            if it >= max(args.warmup, 3):
                e2e_times[dt].append(e0.elapsed_time(e1))
    h2d = (idx_h[torch.int32].numel() * idx_h[torch.int32].element_size()
           + off_h.numel() * off_h.element_size() + g_h.numel() * g_h.element_size())
    d2h = out_h.numel() * 4
    ms_e2e = rank_max(dist, float(np.mean(e2e_times[torch.int32])))
    ms_e2e64 = rank_max(dist, float(np.mean(e2e_times[torch.int64])))
    if rank != 0:
        return None

    def kernels_ms(r):
        return {k: v[0] / r["reps"] for k, v in r["kern"].items()}

    def launches(r):
        return {k: v[1] / r["reps"] for k, v in r["kern"].items()}

    def dominant(r, which):
        kms = kernels_ms(r)
        dom = max(kms, key=kms.get)
        per = kms[dom] / max(1.0, launches(r)[dom])
        roof = kernel_roofline(dom, per, r["alg"], r["wl"].x, r["wl"].train, p_fp32, pk, sms,
                               which)
        roof["share"] = round(kms[dom] / sum(kms.values()), 4)
        return roof, {k: round(v, 5) for k, v in sorted(kms.items(), key=lambda kv: -kv[1])}

    def grouping_roofline(r, which):
        kms, nl = kernels_ms(r), launches(r)
        g = next((k for k in kms if k.startswith("k_group")), None)
        if g is None:
            return None
        return kernel_roofline(g, kms[g] / max(1.0, nl[g]), r["alg"], r["wl"].x, r["wl"].train,
                               p_fp32, pk, sms, which)

    def forward_line(r, workload, which):
        a = r["alg"]
        roof, kms = dominant(r, which)
        return {
            "workload": workload,
            "lookups_per_s": round(weak_throughput(a["nnz"], world, r["ms"]), 1),
            "bags_per_s": round(a["B"] * world / (r["ms"] * 1e-3), 1),
            "ms_per_call": round(r["ms"], 5), "lookups": a["nnz"],
            "unique_rows": a["U_r"], "unique_prefixes": a["U_12"], "chunks": a["n_chunks"],
            "grouping_method": a.get("method"), "prefix_partials_reused": a.get("ckpt_reused"),
            "roofline_call": call_roofline(a, r["ms"], p_fp32, pk),
            "roofline": roof, "roofline_grouping": grouping_roofline(r, which),
            "kernels_ms_per_call": kms, "clocks": r["clocks"],
        }

    tr, fw, f8 = result["train"], result["forward"], result["forward8"]
    at = tr["alg"]
    nnz_tr = tr["wl"].x.nnz
    value = weak_throughput(nnz_tr, world, tr["ms"])
    roof_tr, kms_tr = dominant(tr, "train")
    a8 = f8["alg"]
    kms_f8 = kernels_ms(f8)
    contract8 = next((k for k in ("k_fwd_mma64", "k_fwd_mma", "k_fwd_tiled", "k_fwd_generic")
                      if k in kms_f8), None)
    f8_line = {
        "workload": "8 tables of 1e5, 1e6, 4e6, 1e7, 2e7, 3e7, 4e7, 4e7 rows (3 near-equal "
                    "factors each), D=128=4x8x4, R1=R2=64, 32768 bags each of max(Poisson(20),1) "
                    "Zipf(1.4) lookups, forward, one tt_emb_forward_tables_ex call on cores "
                    "split at load time",
        "dtype": "f32 in/out; contractions as bf16x3 tensor-core products (hi/lo bf16 split, "
                 "about 4e-6 relative error per product)",
        "lookups_per_s": round(weak_throughput(a8["nnz"], world, f8["ms"]), 1),
        "bags_per_s": round(a8["B"] * world / (f8["ms"] * 1e-3), 1),
        "ms_per_batch": round(f8["ms"], 5),
        "lookups": a8["nnz"], "unique_rows": a8["U_r"], "unique_prefixes": a8["U_12"],
        "roofline_call": call_roofline(a8, f8["ms"], p_fp32, pk),
        "kernels_ms_per_batch": {k: round(v, 5) for k, v in sorted(kms_f8.items(),
                                                                     key=lambda kv: -kv[1])},
    }
    if contract8:
        ach8 = a8["fwd_contract"] / (kms_f8[contract8] * 1e-3) / 1e12
        f8_line["contraction"] = {"kernel": contract8, "bound": "alu", "achieved": round(ach8, 3),
                                  "peak": round(p_fp32, 2), "unit": "TFLOP/s",
                                  "frac": round(ach8 / p_fp32, 4),
                                  "traffic": stored_traffic(contract8, "forward8")}
        if contract8 in TENSOR_SPLIT_KERNELS:
            pt = pk["bf16_tflops"] / 3.0
            f8_line["contraction"]["roofline_tensor"] = {
                "bound": "tensor", "achieved": round(ach8, 3), "peak": round(pt, 1),
                "unit": "TFLOP/s", "frac": round(ach8 / pt, 4)}
    small = {}
    for nm, cfg in (("config1", 1), ("config2", 2)):
        r = result[nm]
        ln = forward_line(r, CONFIG_NAMES[cfg] + ", forward only", nm)
        ln["dtype"] = ("f32 (FP32 FFMA, one warp per bag forming each lookup's row on its own: "
                       "a forward-only batch this small is not grouped)"
                       if r["alg"].get("method") == "direct" else "f32 (FP32 FFMA chunk kernel)")
        small[nm] = ln
    sens = {}
    for nm, base in (("forward_permuted", fw), ("train_permuted", tr)):
        r = result[nm]
        a = r["alg"]
        ln = {"workload": CONFIG_NAMES[r["wl"].x.cfg] + ", Zipf ranks mapped to rows through a "
                          "seeded random permutation",
              "lookups_per_s": round(weak_throughput(a["nnz"], world, r["ms"]), 1),
              "ms_per_step": round(r["ms"], 5), "unique_rows": a["U_r"],
              "unique_prefixes": a["U_12"], "grouping_method": a.get("method"),
              "F_unique_flop": int(a["fwd_contract"] + a["pool"]),
              "vs_identity_mapping_time": round(r["ms"] / base["ms"], 3),
              "kernels_ms": {k: round(v, 5) for k, v in sorted(kernels_ms(r).items(),
                                                                 key=lambda kv: -kv[1])}}
        if nm == "forward_permuted":
            ln["roofline_call"] = call_roofline(a, r["ms"], p_fp32, pk)
        sens[nm] = ln
    cpu = cpu_baseline(args) if (world == 1 and not args.no_cpu_baseline) else None
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "lookups/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(tr["ms"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 in/out; contractions as bf16x3 tensor-core products (hi/lo bf16 split, "
                 "fp32 accumulate, ~4e-6 relative error per product)",
        "data": "synthetic (seeded cores, Zipf indices, Gaussian grad_out)",
        "gpu_launches": tr["n_launch"] * args.steps,
        "config": {
            "workload": "training step: 47,952,000 rows = 360x360x370, D=128=4x8x4, "
                        "R1=R2=32, 32768 bags of U{10..30} Zipf(1.2) lookups, "
                        "forward + backward + SGD(lr=0.01) that also rewrites the kept "
                        "bf16 split of the cores",
            "global_batch": 32768 * world, "lookups_per_gpu": nnz_tr,
            "unique_rows": at["U_r"], "unique_prefixes": at["U_12"],
            "grouping_method": at.get("method"),
            "parallelism": f"replicas x{world}",
            "l2": "flushed between timed steps (512 MB write outside the timed events, "
                  "after the cores and their split are restored)",
            "timing": "one CUDA graph replay per step, CUDA events on its stream",
        },
        "bags_per_s": round(32768 * world / (tr["ms"] * 1e-3), 1),
        "roofline": roof_tr,
        "roofline_grouping": grouping_roofline(tr, "train"),
        "kernels_ms_per_step": kms_tr,
        "forward": forward_line(fw, CONFIG_NAMES[FWD_CFG] + ", forward only (inference: "
                                "TT_EMB_FORWARD_ONLY), on the bf16 split of the cores made "
                                "once when they were loaded", "forward"),
        "forward_8_tables": f8_line,
        "forward_small": small,
        "sensitivity_permuted_zipf": sens,
        "e2e": {"value": round(nnz_tr * world / (ms_e2e * 1e-3), 1), "unit": "lookups/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 5),
                "path": "one tt_emb_step_host call per step: pinned host int32 indices "
                        "(TT_EMB_INDICES_I32), int64 offsets and grad_out -> device (indices "
                        "and offsets on the compute stream, grad_out on a copy stream), "
                        "forward on the kept core split as soon as the lookups are in, "
                        "backward, SGD + split; the pooled output -> pinned host while the "
                        "backward runs; from its second call with the same arguments the "
                        "library replays a CUDA graph of that work (same copies and kernels)",
                "int64_indices": {"value": round(nnz_tr * world / (ms_e2e64 * 1e-3), 1),
                                  "ms_per_step": round(ms_e2e64, 5),
                                  "h2d_bytes_per_step": h2d + 4 * int(x.nnz)}},
        "clocks": tr["clocks"],
        "workspace_bytes": tr["wl"].ws_bytes,
        "wall_s_timed_region": round(tr["wall"], 4),
        "peaks": pk,
    }
    line["forward"]["dtype"] = line["dtype"]
    if cpu is not None:
        line["cpu_baseline"] = cpu
        if not args.no_oracle_matrix:
            line["oracle_matrix"] = oracle_matrix()
    return line


CONFIG_NAMES = {
    1: "1000 rows = 10x10x10, D=16=2x4x2, R1=R2=4, 64 bags of U{1..4} uniform lookups",
    2: "1,000,000 rows = 100^3, D=64=4x4x4, R1=R2=16, 4096 bags of 1 Zipf(1.05) lookup "
       "over a random row permutation (a pure gather)",
    3: "12,000,000 rows = 200x240x250, D=128=4x8x4, R1=R2=32, 32768 bags x 20 Zipf(1.2) lookups",
    4: "8 tables, D=128, R1=R2=64, 32768 bags each of max(Poisson(20),1) Zipf(1.4) lookups",
    5: "47,952,000 rows = 360x360x370, D=128=4x8x4, R1=R2=32, 32768 bags of U{10..30} "
       "Zipf(1.2) lookups",
}


# ----------------------------------------------------------------------------- CPU oracle arm


def _oracle_sample(bags: int, cfg: int = TRAIN_CFG, table: int = 0):
    from tensor_train_compressed_gb300.inputs import make_inputs
    x = make_inputs(cfg, table=table, with_grad=cfg == TRAIN_CFG)
    bags = min(bags, x.num_bags)
    idx = x.indices[:x.offsets[bags]]
    off = x.offsets[:bags + 1]
    g = x.grad_out[:bags] if x.grad_out is not None else None
    return x, idx, off, g


def oracle_step(x, idx, off, g, threads):
    import oracle
    oracle.forward(x.cores, x.m, x.n, x.R, idx, off, threads=threads)
    if g is not None:
        dG = oracle.backward(g, x.cores, x.m, x.n, x.R, idx, off, threads=threads)
        for k in range(3):
            oracle.sgd(x.cores[k], dG[k], LR)


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(args, target_s: float = 10.0) -> dict:
    """The oracle, as it stands, on a bounded sample of the training workload."""
    import oracle
    oracle.build()
    threads = cpu_threads()
    bags = 2048
    x, idx, off, g = _oracle_sample(bags)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_step(x, idx, off, g, threads)
        n += 1
        if time.perf_counter() - t0 >= target_s or n >= 50:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": round(len(idx) / dt, 1), "unit": "lookups/s", "cores": threads,
            "kind": "oracle",
            "sample": f"first {bags} bags ({len(idx)} lookups) of the training workload, "
                      f"fp64 forward + backward + SGD, {n} repetitions"}


def oracle_rate(cfg: int, threads: int, target_s: float, table: int = 0) -> dict:
    """Lookups/s of the oracle on the first bags of a workload, the sample grown until one
    pass takes about target_s (forward; forward + backward + SGD for the training step)."""
    bags = 16
    while True:
        x, idx, off, g = _oracle_sample(bags, cfg, table)
        t0 = time.perf_counter()
        oracle_step(x, idx, off, g, threads)
        dt = time.perf_counter() - t0
        full = x.offsets.shape[0] - 1
        if dt >= target_s or bags >= full:
            return {"lookups_per_s": round(len(idx) / dt, 1),
                    "sample": f"first {min(bags, full)} bags ({len(idx)} lookups)"}
        bags = min(full, max(bags * 2, int(bags * target_s / max(dt, 1e-4) * 1.1)))


def oracle_matrix(target_s: float = 1.0) -> dict:
    """The oracle at 1 thread and at every host thread on each workload (config 4: its
    1e7-row table), forward; forward + backward + SGD for the training step."""
    import oracle
    oracle.build()
    allt = cpu_threads()
    res = {"cores": allt}
    for cfg in (1, 2, 3, 4, 5):
        table = 3 if cfg == 4 else 0
        one = oracle_rate(cfg, 1, target_s, table)
        many = oracle_rate(cfg, allt, target_s, table)
        res[f"config{cfg}"] = {
            "pass": "forward + backward + SGD" if cfg == TRAIN_CFG else "forward",
            "threads_1": one["lookups_per_s"], f"threads_{allt}": many["lookups_per_s"],
            "sample_threads_1": one["sample"], f"sample_threads_{allt}": many["sample"]}
    return res


def run_reference(args):
    import oracle
    oracle.build()
    threads = cpu_threads()
    bags = 1024
    x, idx, off, g = _oracle_sample(bags)
    for _ in range(args.warmup):
        oracle_step(x, idx, off, g, threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(x, idx, off, g, threads)
        times.append(time.perf_counter() - t0)
    ms = float(np.mean(times)) * 1e3
    value = len(idx) / (ms * 1e-3)
    sample = (f"first {bags} bags ({len(idx)} lookups) of the training workload per step, "
              "fp64 forward + backward + SGD")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "lookups/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "training step: 47,952,000 rows = 360x360x370, D=128=4x8x4, "
                               "R1=R2=32, U{10..30} Zipf(1.2) bags, forward + backward + SGD",
                   "sample_bags_per_step": bags},
        "cpu_baseline": {"value": round(value, 1), "unit": "lookups/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "lookups/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-oracle-matrix", action="store_true",
                    help="skip the per-workload oracle timings (1 thread / all threads)")
    ap.add_argument("--only", choices=[w[0] for w in WORKLOADS], default=None,
                    help="time one workload only (short report; used to drive ncu captures)")
    ap.add_argument("--bags", type=int, default=None,
                    help="with --only: that many bags per table instead of the workload's "
                         "(a smaller case of the same shapes and distributions, for captures)")
    args = ap.parse_args(argv)
    if args.bags is not None and not args.only:
        ap.error("--bags needs --only")
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist_mod.init_process_group("gloo")
        dist = dist_mod
    line = run_ours(args, rank, world, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
