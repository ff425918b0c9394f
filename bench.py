#!/usr/bin/env python
"""Benchmark of the block-sparse masked attention forward on GB300.

One step = the whole hot path over one batch of synthetic input: the device
mask-info build (2 launches; 3 above 2^20 block cells) and the forward
kernel (1 launch, after a 4-byte reset of its work counter), through the
C ABI.  Throughput is counted in unmasked
FLOPs (4*D per visible (q, k) pair) per second.  Inputs are resident in
HBM before timing; L2 is flushed (a 256 MiB write) between timed steps,
outside the step's events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) the heads are partitioned over the ranks, one rank
per GPU, with no data-path collective (the forward of one head never needs
another head's data).  By default the job grows with N (weak scaling): the
N-GPU problem has N*H heads, and rank r owns heads [r*H, (r+1)*H), each rank
holding only its own heads' q/k/v.  With ``--strong`` the workload's H heads
are split over the ranks instead (rank r owns heads [r*H/N, (r+1)*H/N)).
Rank 0 prints one JSON line with the max step time over ranks.
``--impl reference`` times the fp64 CPU oracle instead (rank 0 only).
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_sparse_masked_build_gb300 import workloads as wl  # noqa: E402
from block_sparse_masked_build_gb300 import flops as fl  # noqa: E402

METRIC = ("masked-attn fwd TFLOP/s (unmasked FLOPs) and % of GB300 bf16 "
          "tensor peak")
UNIT = "TFLOP/s"
FLUSH_BYTES = 256 << 20
FWD_SOURCES = ["block_sparse_masked_build_gb300/csrc/bsm_fwd.cu",
               "block_sparse_masked_build_gb300/csrc/bsm_ptx.cuh",
               "block_sparse_masked_build_gb300/csrc/bsm_internal.h"]


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=wl.HEADLINE, choices=list(wl.WORKLOADS))
    p.add_argument("--all", action="store_true",
                   help="one line per workload (diagnostics)")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--bwd", action="store_true",
                   help="time the backward (dQ, dK, dV) instead (diagnostic)")
    p.add_argument("--strong", action="store_true",
                   help="split the workload's heads over the ranks "
                   "(default: each rank owns a block of H heads)")
    return p.parse_args(argv)


# ------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a host scalar over ranks (gloo or nccl process group)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def head_partition(H: int, world: int, rank: int, group: int = 1):
    """Heads [h0, h1) of `rank` when H heads are split over `world` ranks in
    whole groups of `group` query heads (the heads that share one K/V head),
    as evenly as possible; the ranges of all ranks partition [0, H)."""
    if H % group:
        raise ValueError("H must be a multiple of the group size")
    ng = H // group
    g0 = rank * ng // world
    g1 = (rank + 1) * ng // world
    return g0 * group, g1 * group


def rank_seed(w, rank: int) -> int:
    """Seed of the q/k/v draw of head block `rank` in weak scaling (block 0
    is the single-GPU workload itself)."""
    return w.seed + 1000 * rank


def rank_workload(w, world: int, rank: int, strong: bool):
    """(workload of this rank's share, h0, h1, global H).  Weak: the N-GPU
    problem has world*H heads and rank r owns [r*H, (r+1)*H), drawn with
    its own seed.  Strong: the workload's H heads are partitioned."""
    if strong:
        g = w.H // w.Hkv_  # query heads per K/V head stay together
        h0, h1 = head_partition(w.H, world, rank, g)
        return (w.with_(H=h1 - h0, Hkv=(h1 - h0) // g), h0, h1, w.H)
    h0, h1 = head_partition(world * w.H, world, rank)
    return w.with_(seed=rank_seed(w, rank)), h0, h1, world * w.H


# ------------------------------------------------------------------ peaks

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]),
                "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def fwd_source_hash() -> str:
    h = hashlib.sha256()
    for rel in FWD_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the forward kernel from the committed ncu
    summary, if it was taken on the current kernel source for this
    workload; else None."""
    prof = os.path.join(ROOT, "profiles")
    if not os.path.isdir(prof):
        return None
    want = fwd_source_hash()
    for name in sorted(os.listdir(prof)):
        if not name.endswith((".md", ".txt")):
            continue
        with open(os.path.join(prof, name)) as f:
            for line in f:
                m = re.match(r"\s*TRAFFIC_JSON:\s*(\{.*\})\s*$", line)
                if not m:
                    continue
                try:
                    d = json.loads(m.group(1))
                except ValueError:
                    continue
                if d.get("src") == want and d.get("workload") == workload:
                    return float(d["dram_bytes_per_launch"])
    return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.err = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:  # pragma: no cover
            self.gpu_id = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="bsm_clocks_", suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except OSError as e:
            self.err = str(e)

    def stop(self):
        if self.proc is None:
            return {"error": self.err or "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) != 8:
                    continue
                try:
                    rows.append((float(parts[0]), float(parts[1]),
                                 float(parts[2]), float(parts[3]), parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"error": "no samples"}
        load = [r for r in rows if r[3] >= 50.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, s in enumerate(r[4])
                          if s.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "samples_under_load": len([r for r in rows if r[3] >= 50.0])}


# ------------------------------------------------------------- workloads

def mask_name(flags, window):
    parts = []
    if flags & wl.MASK_CAUSAL:
        parts.append("causal")
    if flags & wl.MASK_LOCAL:
        parts.append(f"|q-k|<{window}" if flags & wl.MASK_BAND
                     else f"q-k<{window}")
    if flags & wl.MASK_SEGMENT:
        parts.append("same-segment")
    if flags & wl.MASK_DENSE:
        parts.append("arbitrary-mask")
    return "&".join(parts) or "full"


def workload_flops(w, seg):
    return fl.unmasked_flops(w.flags, w.window, w.B, w.H, w.Sq, w.Skv_, w.D,
                             dense=wl.make_dense_mask(w), q_seg=seg, kv_seg=seg)


def config_block(w, seg, flops):
    return {"workload": w.name, "B": w.B, "H": w.H, "H_kv": w.Hkv_,
            "S": w.S, "D": w.D,
            "mask": mask_name(w.flags, w.window),
            "score": "softmax" if w.score == wl.SCORE_SOFTMAX
            else "hstu_pointwise",
            "scale": w.scale, "block_q": w.block_q, "block_kv": w.block_kv,
            "unmasked_flops_per_step": flops,
            "l2": "flushed between timed steps (256 MiB write)"}


# --------------------------------------------------------------- our arm

def run_ours(args, w, world, rank, local):
    import block_sparse_masked_build_gb300 as bsm

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wfull = w
    # this rank's heads; segment ids and any arbitrary mask are per batch
    # row, shared by every head, so every rank uses the same ones
    w, h0, h1, H_global = rank_workload(wfull, world, rank, args.strong)
    if args.strong:
        g = wfull.H // wfull.Hkv_
        qf, kf, vf = wl.make_qkv(wfull)
        q = qf[:, h0:h1].contiguous()
        k, v = (t[:, h0 // g:h1 // g].contiguous() for t in (kf, vf))
    else:
        q, k, v = wl.make_qkv(w)
    seg = wl.make_segment_ids(w)
    flops = workload_flops(w, seg) if w.H > 0 else 0
    # unmasked FLOPs of the whole N-GPU problem (every head sees the same
    # mask, so each rank's share is proportional to its heads)
    job_flops = (workload_flops(wfull, seg) if args.strong
                 else world * flops)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    segd = None if seg is None else torch.from_numpy(seg).to(dev)
    dm = wl.make_dense_mask(w)
    densed = (None if dm is None else
              torch.from_numpy(wl.pack_dense_mask(dm).view(np.int32)).to(dev))
    nbytes = bsm.bsm_mask_info_bytes(w.flags, w.window, w.B, w.Sq, w.Skv_,
                                     w.block_q, w.block_kv)
    mibuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.H, w.Sq, w.D), dtype=torch.bfloat16, device=dev)
    lse = (torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
           if w.score == wl.SCORE_SOFTMAX else None)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        info = bsm.bsm_build_mask_info(w.flags, w.window, segd, segd, w.B,
                                       w.Sq, w.Skv_, w.block_q, w.block_kv,
                                       mibuf, stream, dense_bits=densed)
        if ev is not None:
            ev[1].record(stream)
        bsm.bsm_splash_fwd(qd, kd, vd, info, segd, segd, w.scale, w.score,
                           out, lse, stream)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    st, detail = bsm.bsm_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")

    info0 = bsm.bsm_build_mask_info(w.flags, w.window, segd, segd, w.B, w.Sq,
                                    w.Skv_, w.block_q, w.block_kv, mibuf,
                                    stream, dense_bits=densed)
    mi_bytes = mask_info_bytes(w, info0)
    mi_launches = mask_info_launches(info0)
    executed_flops = executed_mma_flops(w, info0)
    K = args.steps
    if K is None:  # about 1.5 s of timed work so the clock samples mean something
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(5):
            flush.zero_()
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        per = e0.elapsed_time(e1) / 5
        K = int(min(20000, max(20, 1500.0 / max(per, 1e-3))))

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(K)]
    sampler = ClockSampler(local)
    torch.cuda.synchronize(dev)
    barrier(world)
    sampler.start()
    t_wall0 = time.perf_counter()
    for i in range(K):
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize(dev)
    t_wall1 = time.perf_counter()
    barrier(world)
    clocks = sampler.stop()
    st, detail = bsm.bsm_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")

    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    mi_ms = [e[0].elapsed_time(e[1]) for e in evs]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    ms_step = statistics.fmean(step_ms)
    ms_step_max = reduce_max(ms_step, world, dev)
    value = job_flops / (ms_step_max * 1e-3) / 1e12
    fwd_mean = statistics.fmean(fwd_ms)
    peaks = load_peaks()
    achieved = flops / (fwd_mean * 1e-3) / 1e12
    traffic = recorded_traffic(w.name)
    roof = forward_roofline(w, flops, fwd_mean, peaks, traffic)
    roof["executed_mma_flops"] = executed_flops

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, q, k, v, seg, flops, dev)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": max(3, args.warmup),
        "ms_per_step": round(ms_step_max, 5), "higher_is_better": True,
        "scaling": "strong" if args.strong else "weak", "vs_baseline": None,
        "dtype": "bf16",
        "data": ("synthetic: seeded bf16 normal q/k/v; segment lengths "
                 "uniform in [256, 2048] from a seeded generator"),
        "config": dict(config_block(wfull, seg, job_flops),
                       H=H_global,
                       parallelism=(f"heads sharded over {world} GPUs (rank "
                                    f"r owns {h1 - h0} of {H_global} heads, "
                                    "no collective on the data path)"
                                    if world > 1 else "single GPU")),
        "step_ms": {"mean": round(ms_step, 5), "min": round(min(step_ms), 5),
                    "median": round(statistics.median(step_ms), 5),
                    "max": round(max(step_ms), 5)},
        "pct_of_bf16_peak": round(100.0 * value / world / peaks["bf16_tflops"],
                                  2),
        "roofline": roof,
        "mask_info": mask_info_line(w, mi_bytes, statistics.fmean(mi_ms),
                                    peaks, mi_launches),
        "gpu_launches": (1 + mi_launches) * K,
        "clocks": clocks,
        "wall_s_timed": round(t_wall1 - t_wall0, 3),
    }
    if e2e is not None:
        line["e2e"] = e2e
    return line


def run_bwd(args, w, dev):
    """Backward diagnostic: dQ, dK, dV of the workload (single GPU), timed
    per launch set with CUDA events, L2 flushed between steps.  FLOPs count
    the five products per visible (q, k) pair (q.k, dO.v, P^T dO, dS^T Q,
    dS K): 10 * D each, 2.5 times the forward's."""
    import block_sparse_masked_build_gb300 as bsm

    q, k, v = wl.make_qkv(w)
    g = torch.Generator().manual_seed(w.seed + 7)
    do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
    seg = wl.make_segment_ids(w)
    fwd_flops = workload_flops(w, seg)
    flops = fwd_flops * 10 // 4
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    segd = None if seg is None else torch.from_numpy(seg).to(dev)
    dm = wl.make_dense_mask(w)
    densed = (None if dm is None else
              torch.from_numpy(wl.pack_dense_mask(dm).view(np.int32)).to(dev))
    info = bsm.build_mask_info(w.flags, w.B, w.Sq, w.Skv_, w.block_q,
                               w.block_kv, w.window, segd, segd, device=dev,
                               dense_bits=densed)
    out, lse = bsm.splash_attention(qd, kd, vd, mask_flags=w.flags,
                                    window=w.window, q_segment_ids=segd,
                                    kv_segment_ids=segd, scale=w.scale,
                                    score=w.score, mask_info=info)
    dq, dk, dv = (torch.empty_like(t) for t in (qd, kd, vd))
    ws_n = bsm.bsm_splash_bwd_workspace_bytes(w.B, w.H, w.Sq, w.score)
    ws = torch.empty(max(ws_n, 256), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sm = w.score == wl.SCORE_SOFTMAX

    def step():
        bsm.bsm_splash_bwd(qd, kd, vd, out if sm else None,
                           lse if sm else None, dod, info, segd, segd,
                           w.scale, w.score, dq, dk, dv, stream, ws)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    K = args.steps or 20
    ms = []
    for _ in range(K):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    st, detail = bsm.bsm_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} {detail}")
    mean = statistics.fmean(ms)
    peaks = load_peaks()
    tf = flops / (mean * 1e-3) / 1e12
    nnz = int(info.row_ptr[-1].item())
    per_table = w.H if info.struct.num_tables > 1 else w.B * w.H
    executed = nnz * w.block_q * w.block_kv * 2 * w.D * 7 * per_table
    return {
        "metric": "masked-attn bwd TFLOP/s (unmasked FLOPs, 5 products per "
                  "visible pair)",
        "value": round(tf, 2), "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": max(3, args.warmup), "ms_per_step": round(mean, 5),
        "higher_is_better": True, "dtype": "bf16",
        "config": dict(config_block(w, seg, flops), parallelism="single GPU"),
        "roofline": {"kernel": "splash_bwd_kernel (dK/dV, dQ) + D_q",
                     "bound": "tensor", "achieved": round(tf, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(tf / peaks["bf16_tflops"], 4),
                     "executed_mma_flops": executed},
        "gpu_launches": 3 * K if sm else 2 * K,
    }


def mask_info_bytes(w, info):
    """Algorithmic HBM bytes of one mask-info build: segment ids read once,
    every table written once (block classes, next-block table, CSR offsets,
    the nonzero lists, segment ranges, longest-first order)."""
    s = info.struct
    T, nq, nk = s.num_tables, s.nq, s.nk
    cells = T * nq * nk
    nnz = int(info.row_ptr[-1].item())
    seg = bool(w.flags & wl.MASK_SEGMENT)
    read = 4 * w.B * (w.Sq + w.Skv_) if seg else 0
    if s.dense_bits:
        read += 4 * w.Sq * s.dense_row_words
    written = (cells + 4 * cells + 4 * (T * nq + 1) + 5 * nnz
               + (8 * w.B * w.Sq + 4 if seg else 0)
               + (4 * T * s.num_super if s.super_order else 0))
    return read + written


def mask_info_launches(info):
    """Kernels one mask-info build launches: classify and copy for masks of
    at most 2^20 block cells (and fewer than 2^24 block rows), else
    classify, offsets and compaction."""
    s = info.struct
    rows = s.num_tables * s.nq
    return 2 if rows < (1 << 24) and rows * s.nk <= (1 << 20) else 3


def mask_info_line(w, nbytes, ms, peaks, launches):
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 5),
            "launches": launches,
            "bound": f"latency ({launches} small launches)",
            "algorithmic_bytes": nbytes, "achieved": round(gbs, 2),
            "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 5)}


def executed_mma_flops(w, info):
    """Block-level MMA work of one forward: nonempty mask blocks x
    block_q x block_kv x 4 D, over every (batch, head) the tables cover."""
    s = info.struct
    nnz = int(info.row_ptr[-1].item())
    per_table = w.H if s.num_tables > 1 else w.B * w.H
    return nnz * w.block_q * w.block_kv * 4 * w.D * per_table


def forward_roofline(w, flops, fwd_ms, peaks, traffic):
    """Roofline of the forward kernel: tensor-bound when the unmasked
    FLOPs per algorithmic byte reach the measured ridge (peak FLOP/s over
    peak HBM B/s), else HBM-bound and reported in GB/s."""
    nbytes = algorithmic_bytes(w)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    # at head dim 128 without an arbitrary mask, segment-id masks and masks
    # of fewer than 4096 keys run the kernel with decoupled query tiles
    dt = not (w.flags & wl.MASK_DENSE) and w.D == 128 and \
        ((w.flags & wl.MASK_SEGMENT) or w.Skv_ < 4096)
    common = {"kernel": "splash_fwd_dt_kernel" if dt else "splash_fwd_kernel",
              "traffic": traffic,
              "algorithmic_bytes": nbytes,
              "flop_per_byte": round(flops / nbytes, 1),
              "ridge_flop_per_byte": round(ridge, 1),
              "fwd_ms": round(fwd_ms, 5)}
    if flops / nbytes >= ridge:
        achieved = flops / (fwd_ms * 1e-3) / 1e12
        return dict(common, bound="tensor", achieved=round(achieved, 2),
                    peak=peaks["bf16_tflops"], unit="TFLOP/s",
                    frac=round(achieved / peaks["bf16_tflops"], 4),
                    peak_source=f"{peaks['source']} (burst bf16 GEMM)")
    gbs = nbytes / (fwd_ms * 1e-3) / 1e9
    return dict(common, bound="hbm", achieved=round(gbs, 2),
                peak=peaks["hbm_gbs"], unit="GB/s",
                frac=round(gbs / peaks["hbm_gbs"], 5),
                peak_source=f"{peaks['source']} (STREAM-style copy)",
                tflops=round(flops / (fwd_ms * 1e-3) / 1e12, 3))


def algorithmic_bytes(w):
    """q, k, v, out once each (bf16) plus lse (f32)."""
    qo = 2 * w.B * w.H * w.Sq * w.D * 2
    kv = 2 * w.B * w.Hkv_ * w.Skv_ * w.D * 2
    lse = 4 * w.B * w.H * w.Sq if w.score == wl.SCORE_SOFTMAX else 0
    return qo + kv + lse


def run_e2e(args, w, q, k, v, seg, flops, dev):
    """Same metric through the public API with pinned host buffers: every
    step copies q/k/v/segment ids host->device and out/lse device->host."""
    import block_sparse_masked_build_gb300 as bsm

    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    sh = None if seg is None else torch.from_numpy(seg).pin_memory()
    dm = wl.make_dense_mask(w)
    dh = None if dm is None else torch.from_numpy(dm).pin_memory()
    oh = torch.empty((w.B, w.H, w.Sq, w.D), dtype=torch.bfloat16,
                     pin_memory=True)
    lh = (torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, pin_memory=True)
          if w.score == wl.SCORE_SOFTMAX else None)
    stream = torch.cuda.current_stream(dev)

    def call():
        bsm.splash_attention(qh, kh, vh, mask_flags=w.flags, window=w.window,
                             q_segment_ids=sh, kv_segment_ids=sh,
                             scale=w.scale, score=w.score, block_q=w.block_q,
                             block_kv=w.block_kv, out=oh, lse=lh,
                             dense_mask=dh)

    for _ in range(2):
        call()
    times = []
    for _ in range(args.e2e_steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.fmean(times)
    h2d = (qh.nbytes + kh.nbytes + vh.nbytes
           + (0 if sh is None else 2 * sh.nbytes)
           + (0 if dh is None else dh.nbytes))
    d2h = oh.nbytes + (0 if lh is None else lh.nbytes)
    via = ("splash_attention -> bsm_splash_fwd_host (pinned host tensors)"
           if dh is None else
           "splash_attention (pinned host tensors; mask packed on the GPU)")
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": args.e2e_steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "call": via}


# ----------------------------------------------------- oracle (CPU) arm

def oracle_head(w, q, k, v, seg, b, h):
    """Run the fp64 oracle on every row of one (batch, head)."""
    import oracle

    if k.shape[1] != q.shape[1]:  # grouped K/V heads: the oracle takes one
        g = q.shape[1] // k.shape[1]  # K/V head per query head
        k, v = k.repeat_interleave(g, dim=1), v.repeat_interleave(g, dim=1)

    rows = [(b, h, r) for r in range(w.Sq)]
    dm = wl.make_dense_mask(w)
    if w.score == wl.SCORE_SOFTMAX:
        oracle.softmax_attention(q, k, v, w.flags, w.window, seg, seg,
                                 w.scale, rows=rows, dense=dm)
    else:
        oracle.pointwise_attention(q, k, v, w.flags, w.window, seg, seg,
                                   w.scale, rows=rows, dense=dm)


def head_flops(w, seg, b):
    sb = None if seg is None else seg[b:b + 1]
    return fl.unmasked_flops(w.flags, w.window, 1, 1, w.Sq, w.Skv_, w.D, sb,
                             sb, dense=wl.make_dense_mask(w))


def cpu_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def cpu_baseline(args, w):
    """The oracle as it stands on the host cores, on whole heads of the
    workload until about ``--cpu-seconds`` of CPU work is done."""
    q, k, v = wl.make_qkv(w)
    seg = wl.make_segment_ids(w)
    done_flops, heads = 0, 0
    t0 = time.perf_counter()
    for idx in range(w.B * w.H):
        b, h = divmod(idx, w.H)
        oracle_head(w, q, k, v, seg, b, h)
        done_flops += head_flops(w, seg, b)
        heads += 1
        if time.perf_counter() - t0 >= args.cpu_seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(done_flops / el / 1e12, 6), "unit": UNIT,
            "cores": cpu_threads(), "kind": "oracle",
            "sample": (f"all {w.Sq} rows of the first {heads} of {w.B * w.H} "
                       f"(batch, head) pairs of {w.name}, fp64 numpy "
                       f"(materialised scores, two-pass), {el:.1f} s"),
            "seconds": round(el, 2)}


def run_reference(args, w):
    """Reference arm: the fp64 oracle, each step one whole (batch, head)."""
    q, k, v = wl.make_qkv(w)
    seg = wl.make_segment_ids(w)
    K = args.steps if args.steps is not None else 5
    W = args.warmup if args.warmup is not None else 1
    nheads = w.B * w.H
    for i in range(W):
        b, h = divmod(i % nheads, w.H)
        oracle_head(w, q, k, v, seg, b, h)
    times, fls = [], []
    for i in range(K):
        b, h = divmod((W + i) % nheads, w.H)
        t0 = time.perf_counter()
        oracle_head(w, q, k, v, seg, b, h)
        times.append(time.perf_counter() - t0)
        fls.append(head_flops(w, seg, b))
    el = sum(times)
    value = sum(fls) / el / 1e12
    sample = (f"each step: all {w.Sq} rows of one (batch, head) of {w.name}, "
              f"fp64 numpy oracle")
    return {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "impl": "reference", "n_gpus": 0, "steps": K, "warmup": W,
        "ms_per_step": round(1e3 * el / K, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (same seeded inputs as the CUDA arm)",
        "config": dict(config_block(w, seg, workload_flops(w, seg)),
                       parallelism="host cores"),
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT,
                         "cores": cpu_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT,
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    args = parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl.WORKLOADS[args.workload])),
                  flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    names = list(wl.WORKLOADS) if args.all else [args.workload]
    if args.bwd:
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        for name in names:
            if rank == 0:
                print(json.dumps(run_bwd(args, wl.WORKLOADS[name], dev)),
                      flush=True)
        return 0
    for name in names:
        w = wl.WORKLOADS[name]
        line = run_ours(args, w, world, rank, local)
        if rank == 0 and world == 1 and not args.no_cpu_baseline \
                and not args.all:
            line["cpu_baseline"] = cpu_baseline(args, w)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
