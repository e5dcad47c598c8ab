#!/usr/bin/env python
"""Benchmark of the hot path on one GB300 (or N independent replicas under torchrun).

A step is one pass of the convolution hot path over the 64,000-atom / ~2.56M-edge workload
(128x0e+128x1o+128x2e, SH l<=3, outputs l<=3, fp32): spherical harmonics of the edge
vectors, the fused convolution forward, and the sender-major convolution backward
(dx, dy, dw). value = edges processed per second by all ranks (the "conv fwd+bwd edges/s"
half of the metric). The tensor product on the 200,000-row workload is timed in the same
run (forward and backward, own timed loops) and reported under "tp" (the "TP fwd achieved
HBM GB/s" half). Inputs are resident in HBM; the edge weights alone (31.5 GB) exceed L2
(129 MB), so no flush is needed between steps. "e2e" measures the same step through the
public API with host buffers: pinned host -> device copies of the step's inputs and
device -> host copies of all outputs inside the timed region (consecutive steps overlap their
copies and compute on three streams with two device buffer sets).

Profiling options shrink single parts of the run (--atoms for the main step, --tp-rows, --coo-rows,
--workload-atoms for every conv workload's box, --dbwd-atoms, --workloads to pick timings).

Throughput accounting follows "e3j ...", Sec. 3 Eq. (9): (bytes of inputs + outputs) /
runtime, backward counting input primals, output cotangents and input cotangents.

--impl reference times the float64 CPU oracle on the same workload (a bounded sample of
receivers per step) on the host cores; rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "conv fwd+bwd edges/s and TP fwd achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "edges/s"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# the sources each traffic entry's kernel is compiled and launched from
KERNEL_SOURCES = {
    "conv_fwd": ("conv_pipe.cuh", "kernels.cuh", "cg_table.hpp", "configs.def", "instances.cu"),
    "conv_bwd": ("conv_pipe.cuh", "kernels.cuh", "cg_table.hpp", "configs.def", "instances.cu"),
    "tp_fwd": ("kernels.cuh", "cg_table.hpp", "configs.def", "instances.cu"),
}


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the kernel's sources (all of csrc/ when the kernel has no entry above)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "message_passing_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(d))
    for n in names:
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, units: float):
    """Per-launch DRAM bytes of `kernel` from profiles/traffic.json, scaled to `units`
    (edges or rows) of one launch; None when absent or taken on other kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            tr = json.load(f)
    except Exception:
        return None
    ent = tr.get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return float(ent["bytes_per_unit"]) * units


# ---------------------------------------------------------------------------------------
# algorithmic bytes (Eq. 9)
# ---------------------------------------------------------------------------------------
def conv_bytes(N, E, d1, d2, P, D, Nq, s):
    """s = bytes per stored input element; outputs are fp32."""
    fwd = N * d1 * Nq * s + E * d2 * s + E * P * Nq * s + (N + 1) * 4 + E * 4 + N * D * Nq * 4
    bwd = (N * d1 * Nq * s + E * d2 * s + E * P * Nq * s + N * D * Nq * s      # x, y, w, dm
           + (N + 1) * 4 + 2 * E * 4                                           # sender-major index
           + (N * d1 * Nq + E * d2 + E * P * Nq) * 4)                          # dx, dy, dw
    return fwd, bwd


def sh_bytes(E, d2, s):
    return E * 12 + E * d2 * s


def tp_bytes(R, d1, d2, P, D, Nq, s):
    fwd = R * (d1 * Nq + d2 + P * Nq + D * Nq) * s
    bwd = R * (d1 * Nq + d2 + P * Nq + D * Nq + d1 * Nq + d2 + P * Nq) * s
    return fwd, bwd


def max_over_ranks(seconds: float, device=None) -> float:
    """The slowest rank's time (all_reduce MAX); the local time when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, seconds: float) -> float:
    """Units processed by all ranks per second of the slowest rank (weak scaling)."""
    return units_per_rank_step * steps * world / seconds


# ---------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        import torch
        cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200"]
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------------------
def oracle_conv_sample(w, g, ot, x, y, wfetch, dm, scale, n_recv, seed=0):
    """Oracle conv fwd + bwd on the edges of n_recv receivers; returns (edges, seconds)."""
    import oracle
    rng = np.random.default_rng(seed)
    recv = np.sort(rng.choice(g.n_nodes, size=n_recv, replace=False))
    cnt = np.diff(g.rowptr)[recv]
    edges = np.concatenate([np.arange(g.rowptr[r], g.rowptr[r + 1]) for r in recv]) if n_recv else np.zeros(0, int)
    t0 = time.perf_counter()
    oracle.conv_forward(ot, g.rowptr, g.sender, x, y, wfetch, scale, receivers=recv)
    oracle.conv_backward_edges(ot, g.rowptr, g.sender, x, y, wfetch, dm, scale, edges=edges)
    oracle.conv_backward_dx(ot, g.rowptr, g.sender, y, wfetch, dm, scale, senders=recv, Nq=w.mul)
    return int(cnt.sum()), time.perf_counter() - t0


def cpu_inputs(w, g, ot):
    import oracle
    from synth import workloads as W
    x, _ = W.make_conv(w, g, ot.n_paths, edge_ids=np.zeros(0, np.int64))
    y = oracle.sh(g.vec.astype(np.float32).astype(np.float64), w.sh_lmax)
    return x.astype(np.float64), y


def run_reference(args):
    """The oracle as it stands, timed on the host cores, on the benchmark workload."""
    import oracle
    from synth import STREAM_GRAD
    from synth import workloads as W
    if int(os.environ.get("RANK", "0")) != 0:
        return
    oracle.build()
    w = W.WORKLOADS[4]
    ot = oracle.table(w.blocks, w.sh_lmax, w.out_lmax)
    g = W.make_graph(w, n_atoms=args.atoms, order=args.order)
    scale = g.n_nodes / g.n_edges
    wfetch = lambda ids: W.make_conv(w, g, ot.n_paths, edge_ids=np.asarray(ids, np.int64))[1]
    x, y = cpu_inputs(w, g, ot)
    dm = W.make_grad(w, g.n_nodes, ot.D).astype(np.float64)
    n_recv = args.ref_receivers
    for _ in range(args.warmup):
        oracle_conv_sample(w, g, ot, x, y, wfetch, dm, scale, n_recv, seed=1)
    tot_e, tot_t = 0, 0.0
    for k in range(args.steps):
        e, t = oracle_conv_sample(w, g, ot, x, y, wfetch, dm, scale, n_recv, seed=100 + k)
        tot_e += e
        tot_t += t
    v = tot_e / tot_t
    cores = oracle.num_threads()
    sample = f"{n_recv} random receivers per step ({tot_e / args.steps:.0f} edges): conv fwd + dy/dw of their edges + dx of {n_recv} senders"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, g, args),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _median(xs):
    return float(statistics.median(xs))


def time_conv_workload(wl, dt, dev, stream, reps: int, hbm_peak: float, order: str = "cell",
                       pad_frac: float = 0.0, n_atoms=None):
    """Per-kernel device times of SH, conv forward and conv backward on one conv workload.
    pad_frac > 0: the same graph plus one padding node holding that fraction of all edge slots
    (mostly pad -> pad, 2% pad -> real receivers, 1% real senders -> pad), with NaN inputs on
    every padding row, run with pad_node set; rates count the real edges. n_atoms: a smaller box
    of the same density and degree (profiling)."""
    import torch

    import message_passing_gb300 as e3
    import synth
    from synth import STREAM_GRAD, STREAM_W, device_normal
    from synth import workloads as W
    s = 2 if dt == torch.bfloat16 else 4
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=n_atoms, order=order)
    E_real, pad = g.n_edges, -1
    x_np, _ = W.make_conv(wl, g, t.n_paths, edge_ids=np.zeros(0, np.int64))
    if pad_frac > 0:
        n_pad = int(round(E_real * pad_frac / (1 - pad_frac)))
        n_out, n_in = n_pad // 50, n_pad // 100
        g, pad, orig = synth.padded_graph(g, n_pad - n_out - n_in, n_out, n_in, (wl.wid, 9))
        x_np = np.concatenate([x_np, np.full((1,) + x_np.shape[1:], np.nan, x_np.dtype)])
    N, E, Nq, P, D = g.n_nodes, g.n_edges, wl.mul, t.n_paths, t.D
    scale = N / E
    xd = torch.from_numpy(x_np).to(dev).to(dt)
    vec = torch.from_numpy(g.vec.astype(np.float32)).to(dev)
    rp = torch.from_numpy(g.rowptr).to(dev)
    sd = torch.from_numpy(g.sender).to(dev)
    wd = device_normal((E, P, Nq), (wl.wid, STREAM_W), W.weight_scale(wl, P), device=dev, dtype=dt)
    dmd = device_normal((N, D, Nq), (wl.wid, STREAM_GRAD), device=dev, dtype=dt)
    if pad >= 0:   # padding rows hold NaN: the kernels must not read them
        wd.index_fill_(0, torch.from_numpy(np.nonzero(orig < 0)[0]).to(dev), float("nan"))
        dmd[pad] = float("nan")
    y = torch.empty((E, t.d2), device=dev, dtype=dt)
    f32 = dict(dtype=torch.float32)
    m = torch.empty((N, D, Nq), device=dev, **f32)
    dx, dy, dw = torch.empty_like(xd, **f32), torch.empty_like(y, **f32), torch.empty_like(wd, **f32)
    csc = e3.graph_prepare(rp, sd, N)
    # the sender-major index (once per graph, so outside the step): its own timed loop
    gws = torch.empty(e3.graph_prepare_workspace_bytes(N, E), dtype=torch.uint8, device=dev)
    evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(reps + 2)]
    for k in range(reps + 2):
        evg[k][0].record(stream)
        e3.graph_prepare(rp, sd, N, out=csc, workspace=gws, stream=stream)
        evg[k][1].record(stream)
    torch.cuda.synchronize()
    tgp = _median([e[0].elapsed_time(e[1]) for e in evg[2:]]) / 1e3
    del gws
    dvec = torch.empty_like(vec)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(reps + 2)]
    for k in range(reps + 2):
        ev[k][0].record(stream)
        e3.sh_forward(vec, wl.sh_lmax, out=y, stream=stream)
        ev[k][1].record(stream)
        e3.conv_forward(t, rp, sd, xd, y, wd, scale, out=m, stream=stream, pad_node=pad)
        ev[k][2].record(stream)
        e3.conv_backward(t, csc, xd, y, wd, dmd, scale, out=(dx, dy, dw), stream=stream, pad_node=pad)
        ev[k][3].record(stream)
        e3.sh_backward(vec, dy, wl.sh_lmax, out=dvec, stream=stream)   # forces through the harmonics
        ev[k][4].record(stream)
    torch.cuda.synchronize()
    e3.check_device_status()
    if pad >= 0:
        assert bool(torch.isfinite(m).all()) and bool(torch.isfinite(dw).all()), "padding leaked into outputs"
    tsh = _median([e[0].elapsed_time(e[1]) for e in ev[2:]]) / 1e3
    tf = _median([e[1].elapsed_time(e[2]) for e in ev[2:]]) / 1e3
    tb = _median([e[2].elapsed_time(e[3]) for e in ev[2:]]) / 1e3
    tshb = _median([e[3].elapsed_time(e[4]) for e in ev[2:]]) / 1e3
    # algorithmic bytes of the real graph; with padding the backward also writes the padding
    # edges' zero dy, dw rows and scans the sender-major receiver ids
    bf, bb = conv_bytes(N, E_real, t.d1, t.d2, P, D, Nq, s)
    bb += (E - E_real) * (t.d2 + P * Nq) * 4 + (E * 4 if pad >= 0 else 0)
    bshb = E * (12 + t.d2 * 4 + 12)   # vec, dy (fp32 from the backward), dvec
    E = E_real
    name = wl.name if pad < 0 else f"{wl.name} + {pad_frac:.0%} padding edge slots on one padding node"
    out = {"workload": name, "dtype": "bf16" if s == 2 else "f32", "atoms": N, "edges": E,
           "sh_ms": tsh * 1e3, "graph_prepare_ms": tgp * 1e3,
           "sh_backward": {"ms": tshb * 1e3, "alg_GBps": bshb / tshb / 1e9, "frac": bshb / tshb / 1e9 / hbm_peak},
           "fwd": {"ms": tf * 1e3, "edges_per_s": E / tf, "alg_GBps": bf / tf / 1e9, "frac": bf / tf / 1e9 / hbm_peak},
           "bwd": {"ms": tb * 1e3, "edges_per_s": E / tb, "alg_GBps": bb / tb / 1e9, "frac": bb / tb / 1e9 / hbm_peak},
           "fwd_bwd_edges_per_s": E / (tf + tb + tsh)}
    del xd, wd, dmd, y, m, dx, dy, dw, dvec
    torch.cuda.empty_cache()
    return out


def dbwd_bytes(N, E, d1, d2, P, D, Nq, s):
    """Algorithmic bytes of the double backward (Eq. 9 accounting): primals x, y, w, dm and
    the variations ddx, ddy, ddw in; delta_x, delta_y, delta_w, delta_dm out (fp32); both
    graph indices."""
    return (2 * (N * d1 * Nq + E * d2 + E * P * Nq) * s + N * D * Nq * s
            + 2 * (N + 1) * 4 + 3 * E * 4
            + (N * d1 * Nq + E * d2 + E * P * Nq + N * D * Nq) * 4)


def time_double_backward(wl, dev, stream, reps: int, hbm_peak: float, n_atoms=None):
    """Device time of the fused double backward (Eq. 17-18) on a conv workload, and of the
    pages' formulation beside it: three conv and three conv_bwd calls (their three output
    additions not counted)."""
    import torch

    import message_passing_gb300 as e3
    from synth import STREAM_GRAD, STREAM_W, device_normal
    from synth import workloads as W
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=n_atoms)
    N, E, Nq, P, D = g.n_nodes, g.n_edges, wl.mul, t.n_paths, t.D
    scale = N / E
    x_np, _ = W.make_conv(wl, g, P, edge_ids=np.zeros(0, np.int64))
    xd = torch.from_numpy(x_np).to(dev)
    ddx = torch.from_numpy(np.ascontiguousarray(x_np[::-1])).to(dev)
    rp = torch.from_numpy(g.rowptr).to(dev)
    sd = torch.from_numpy(g.sender).to(dev)
    y = e3.sh_forward(torch.from_numpy(g.vec.astype(np.float32)).to(dev), wl.sh_lmax)
    ddy = torch.flip(y, dims=(0,)).contiguous()
    wd = device_normal((E, P, Nq), (wl.wid, STREAM_W), W.weight_scale(wl, P), device=dev)
    ddw = device_normal((E, P, Nq), (wl.wid, STREAM_W, 1), W.weight_scale(wl, P), device=dev)
    dmd = device_normal((N, D, Nq), (wl.wid, STREAM_GRAD), device=dev)
    csc = e3.graph_prepare(rp, sd, N)
    f32 = dict(dtype=torch.float32)
    out = (torch.empty_like(xd), torch.empty_like(y), torch.empty_like(wd), torch.empty_like(dmd))
    tmp_m = torch.empty((N, D, Nq), device=dev, **f32)
    tmp_b = (torch.empty_like(xd), torch.empty_like(y), torch.empty_like(wd))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps + 2)]
    for k in range(reps + 2):
        ev[k][0].record(stream)
        e3.conv_double_backward(t, rp, sd, csc, xd, y, wd, dmd, ddx, ddy, ddw, scale, out=out, stream=stream)
        ev[k][1].record(stream)
        for a_, b_, c_ in ((ddx, y, wd), (xd, ddy, wd), (xd, y, ddw)):
            e3.conv_forward(t, rp, sd, a_, b_, c_, scale, out=tmp_m, stream=stream)
            e3.conv_backward(t, csc, a_, b_, c_, dmd, scale, out=tmp_b, stream=stream)
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    e3.check_device_status()
    tf = _median([e[0].elapsed_time(e[1]) for e in ev[2:]]) / 1e3
    tc = _median([e[1].elapsed_time(e[2]) for e in ev[2:]]) / 1e3
    bb = dbwd_bytes(N, E, t.d1, t.d2, P, D, Nq, 4)
    res = {"workload": wl.name, "dtype": "f32", "atoms": N, "edges": E,
           "fused": {"ms": tf * 1e3, "edges_per_s": E / tf, "alg_GBps": bb / tf / 1e9, "frac": bb / tf / 1e9 / hbm_peak},
           "composition_six_calls": {"ms": tc * 1e3, "edges_per_s": E / tc},
           "speedup_vs_composition": tc / tf}
    del xd, ddx, y, ddy, wd, ddw, dmd, out, tmp_m, tmp_b
    torch.cuda.empty_cache()
    return res


# FP32 FMA peak of a GB300 derived from its unit counts and the maximum SM clock: 152 SMs x
# 128 FP32 lanes x 2 flop x 2.07 GHz (the roofline of the arithmetic-bound radial kernels)
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def radial_flops(E, nnz, P, D, Nq, H):
    """Algorithmic flops per pass: the convolution's 2 Nq (nnz + D) per edge (the coupling
    entries applied to the channels, and the weighted sums) plus the output layer of the radial
    network formed in the kernel, 2 H P Nq per edge; the backward does the weights once, their
    cotangent once and about twice the forward's convolution work."""
    conv = 2.0 * Nq * (nnz + D) * E
    wts = 2.0 * H * P * Nq * E
    return conv + wts, 2.0 * conv + 2.0 * wts


def time_hub_workload(wl, dev, stream, reps: int, hbm_peak: float, n_atoms=None, hub_edges: int = 200_000):
    """A heavy real receiver: the conv workload's graph plus one more node that receives
    hub_edges edges from random senders. Conv forward device times: the split forward on that
    graph (the hub cut into 256-edge pieces), the plain forward on the workload's own graph,
    and one launch of the plain forward on the hub graph (one warp sums the hub's edges)."""
    import torch

    import message_passing_gb300 as e3
    from synth import STREAM_W, device_normal
    from synth import workloads as W
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=n_atoms)
    x_np, _ = W.make_conv(wl, g, t.n_paths, edge_ids=np.zeros(0, np.int64))
    N0, E0 = g.n_nodes, g.n_edges
    rng = np.random.default_rng([wl.wid, 11])
    hub_send = np.sort(rng.integers(0, N0, hub_edges)).astype(np.int32)
    rowptr = np.concatenate([g.rowptr, [E0 + hub_edges]]).astype(np.int32)
    sender = np.concatenate([g.sender, hub_send]).astype(np.int32)
    x_np = np.concatenate([x_np, rng.standard_normal((1,) + x_np.shape[1:]).astype(x_np.dtype)])
    vec = np.concatenate([g.vec, rng.standard_normal((hub_edges, 3))]).astype(np.float32)
    N, E, Nq, P, D = N0 + 1, E0 + hub_edges, wl.mul, t.n_paths, t.D
    xd = torch.from_numpy(x_np).to(dev)
    rp, sd = torch.from_numpy(rowptr).to(dev), torch.from_numpy(sender).to(dev)
    y = e3.sh_forward(torch.from_numpy(vec).to(dev), wl.sh_lmax)
    wd = device_normal((E, P, Nq), (wl.wid, STREAM_W), W.weight_scale(wl, P), device=dev)
    m = torch.empty((N, D, Nq), device=dev)
    chunk = 256
    ws = torch.empty(e3.load().e3gb_conv_forward_split_workspace_bytes(t.handle, N, E, 64), dtype=torch.uint8,
                     device=dev)
    scale = N / E

    def timed(fn, n):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for k in range(n):
            ev[k][0].record(stream)
            fn()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
        return _median([e[0].elapsed_time(e[1]) for e in ev[min(2, n - 1):]])

    sweep = {c: timed(lambda: e3.conv_forward_split(t, rp, sd, xd, y, wd, scale, chunk=c, out=m, workspace=ws,
                                                    stream=stream), reps + 2) for c in (64, 1024)}
    t_split = timed(lambda: e3.conv_forward_split(t, rp, sd, xd, y, wd, scale, chunk=chunk, out=m, workspace=ws,
                                                  stream=stream), reps + 2)
    m_split = m.clone()
    t_plain_hub = timed(lambda: e3.conv_forward(t, rp, sd, xd, y, wd, scale, out=m, stream=stream), 1)
    e3.check_device_status()
    same_light = bool(torch.equal(m_split[:N0], m[:N0]))
    rp0, sd0 = rp[:N0 + 1], sd[:E0]
    m0 = torch.empty((N0, D, Nq), device=dev)
    t_base = timed(lambda: e3.conv_forward(t, rp0, sd0, xd[:N0], y[:E0], wd[:E0], scale, out=m0, stream=stream),
                   reps + 2)
    e3.check_device_status()
    del xd, wd, y, m, m0, ws, m_split
    torch.cuda.empty_cache()
    return {"workload": f"{wl.name} + one hub receiver of {hub_edges} edges (split forward, chunk {chunk})",
            "dtype": "f32", "atoms": N0, "edges": E, "hub_edges": hub_edges,
            "fwd_split_ms": t_split, "fwd_split_ms_by_chunk": {"64": sweep[64], "256": t_split, "1024": sweep[1024]},
            "fwd_plain_ms_on_hub_graph": t_plain_hub,
            "fwd_plain_ms_without_hub": t_base, "light_receivers_bitwise_equal": same_light,
            "edges_per_s_split": E / (t_split / 1e3)}


def time_radial_workload(wl, dev, stream, reps: int, hbm_peak: float, n_atoms=None):
    """The radial form of the convolution step (e3j App. E.1, the edge scalars produced by a
    radial network; App. A.3 "Linear mixing" fused into message passing): SH + the radial
    hidden layer + conv forward and backward with the weights formed in the kernels (w and dw
    never reach memory) + forces (SH backward plus the radial backward)."""
    import torch

    import message_passing_gb300 as e3
    from synth import STREAM_GRAD, device_normal
    from synth import workloads as W
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    g = W.make_graph(wl, n_atoms=n_atoms)
    N, E, Nq, P, D = g.n_nodes, g.n_edges, wl.mul, t.n_paths, t.D
    H = e3.RADIAL_HIDDEN
    scale = N / E
    rc = float(g.cutoff)
    x_np, _ = W.make_conv(wl, g, P, edge_ids=np.zeros(0, np.int64))
    W1, W2 = W.make_radial(wl, P, hidden=H)
    xd = torch.from_numpy(x_np).to(dev)
    vec = torch.from_numpy(g.vec.astype(np.float32)).to(dev)
    rp = torch.from_numpy(g.rowptr).to(dev)
    sd = torch.from_numpy(g.sender).to(dev)
    W1d, W2d = torch.from_numpy(W1).to(dev), torch.from_numpy(W2).to(dev)
    dmd = device_normal((N, D, Nq), (wl.wid, STREAM_GRAD), device=dev)
    csc = e3.graph_prepare(rp, sd, N)
    y = torch.empty((E, t.d2), device=dev)
    h = torch.empty((E, H), device=dev)
    m = torch.empty((N, D, Nq), device=dev)
    dx, dy, dh = torch.empty_like(xd), torch.empty_like(y), torch.empty_like(h)
    dvec = torch.empty_like(vec)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(reps + 2)]
    for k in range(reps + 2):
        ev[k][0].record(stream)
        e3.sh_forward(vec, wl.sh_lmax, out=y, stream=stream)
        e3.radial_hidden(vec, W1d, rc, out=h, stream=stream)
        ev[k][1].record(stream)
        e3.conv_forward_radial(t, rp, sd, xd, y, h, W2d, scale, out=m, stream=stream)
        ev[k][2].record(stream)
        e3.conv_backward_radial(t, csc, xd, y, h, W2d, dmd, scale, out=(dx, dy, dh), stream=stream)
        ev[k][3].record(stream)
        e3.sh_backward(vec, dy, wl.sh_lmax, out=dvec, stream=stream)
        e3.radial_backward(vec, W1d, rc, dh, out=dvec, accumulate=True, stream=stream)
        ev[k][4].record(stream)
    torch.cuda.synchronize()
    e3.check_device_status()
    med = lambda i, j: _median([e[i].elapsed_time(e[j]) for e in ev[2:]]) / 1e3
    tpre, tf, tb, tforce = med(0, 1), med(1, 2), med(2, 3), med(3, 4)
    ff, fb = radial_flops(E, t.nnz, P, D, Nq, H)
    # bytes the fused kernels move (no w, no dw): x and m (dx, dm) once per node, y, h, the
    # indices and dy, dh once per edge, W2 once
    bf = 4 * (N * (t.d1 + D) * Nq + E * (t.d2 + H + 1) + N + 1 + H * P * Nq)
    bb = 4 * (N * (2 * t.d1 + D) * Nq + E * (2 * t.d2 + 2 * H + 2) + N + 1 + H * P * Nq)
    res = {"workload": wl.name + " (radial edge scalars: Bessel basis x8, SiLU hidden layer of 8, weights formed in the kernels)",
           "dtype": "f32", "atoms": N, "edges": E, "hidden": H, "sh_and_hidden_ms": tpre * 1e3,
           "fwd": {"ms": tf * 1e3, "edges_per_s": E / tf, "alg_GBps": bf / tf / 1e9,
                   "TFLOPs": ff / tf / 1e12, "frac_fp32_peak": ff / tf / 1e12 / FP32_PEAK_TFLOPS},
           "bwd": {"ms": tb * 1e3, "edges_per_s": E / tb, "alg_GBps": bb / tb / 1e9,
                   "TFLOPs": fb / tb / 1e12, "frac_fp32_peak": fb / tb / 1e12 / FP32_PEAK_TFLOPS},
           "forces_ms": tforce * 1e3,
           "step_edges_per_s": E / (tpre + tf + tb + tforce),
           "fp32_peak_TFLOPs": FP32_PEAK_TFLOPS}
    del xd, vec, dmd, y, h, m, dx, dy, dh, dvec, W1d, W2d
    torch.cuda.empty_cache()
    return res


def time_coo_tp(wl, dev, stream, reps: int, hbm_peak: float, rows=None):
    """The generic COO-coefficient tensor product with the table's CG records, beside the
    compile-time kernels, on a row workload (fp32); rows: fewer rows (profiling)."""
    import torch

    import message_passing_gb300 as e3
    from synth import workloads as W
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    rec, coef = t.coo_records()
    rec_d, coef_d = torch.from_numpy(rec).to(dev), torch.from_numpy(coef).to(dev)
    u, x, ww = W.make_tp(wl, t.n_paths, rows=rows)
    R = x.shape[0]
    xd, wd = torch.from_numpy(x).to(dev), torch.from_numpy(ww).to(dev)
    y = e3.sh_forward(torch.from_numpy(u.astype(np.float32)).to(dev), wl.sh_lmax)
    dz = torch.from_numpy(W.make_grad(wl, R, t.D)).to(dev)
    z = torch.empty((R, t.D, wl.mul), device=dev)
    gx, gy, gw = torch.empty_like(xd), torch.empty_like(y), torch.empty_like(wd)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(reps + 2)]
    for k in range(reps + 2):
        ev[k][0].record(stream)
        e3.coo_tp_forward(rec_d, coef_d, xd, y, wd, t.D, out=z, stream=stream)
        ev[k][1].record(stream)
        e3.coo_tp_backward(rec_d, coef_d, xd, y, wd, dz, out=(gx, gy, gw), stream=stream)
        ev[k][2].record(stream)
        e3.tp_forward(t, xd, y, wd, out=z, stream=stream)
        ev[k][3].record(stream)
        e3.tp_backward(t, xd, y, wd, dz, out=(gx, gy, gw), stream=stream)
        ev[k][4].record(stream)
    torch.cuda.synchronize()
    e3.check_device_status()
    tms = [_median([e[i].elapsed_time(e[i + 1]) for e in ev[2:]]) / 1e3 for i in range(4)]
    bf, bb = tp_bytes(R, t.d1, t.d2, t.n_paths, t.D, wl.mul, 4)
    res = {"workload": wl.name + " (generic COO records)", "dtype": "f32", "rows": R, "records": int(len(rec)),
           "fwd": {"ms": tms[0] * 1e3, "alg_GBps": bf / tms[0] / 1e9, "frac": bf / tms[0] / 1e9 / hbm_peak},
           "bwd": {"ms": tms[1] * 1e3, "alg_GBps": bb / tms[1] / 1e9, "frac": bb / tms[1] / 1e9 / hbm_peak},
           "compile_time_tables": {"fwd_ms": tms[2] * 1e3, "bwd_ms": tms[3] * 1e3}}
    del xd, wd, y, dz, z, gx, gy, gw
    torch.cuda.empty_cache()
    return res


def time_tp_workload(wl, dev, stream, reps: int, hbm_peak: float):
    """Per-kernel device times of TP forward and backward on a row workload (fp32)."""
    import torch

    import message_passing_gb300 as e3
    from synth import workloads as W
    t = e3.Table.create(wl.blocks, wl.mul, wl.sh_lmax, wl.out_lmax)
    u, x, ww = W.make_tp(wl, t.n_paths)
    R = x.shape[0]
    xd, wd = torch.from_numpy(x).to(dev), torch.from_numpy(ww).to(dev)
    y = e3.sh_forward(torch.from_numpy(u.astype(np.float32)).to(dev), wl.sh_lmax)
    dz = torch.from_numpy(W.make_grad(wl, R, t.D)).to(dev)
    z = torch.empty((R, t.D, wl.mul), device=dev)
    gx, gy, gw = torch.empty_like(xd), torch.empty_like(y), torch.empty_like(wd)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps + 2)]
    for k in range(reps + 2):
        ev[k][0].record(stream)
        e3.tp_forward(t, xd, y, wd, out=z, stream=stream)
        ev[k][1].record(stream)
        e3.tp_backward(t, xd, y, wd, dz, out=(gx, gy, gw), stream=stream)
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    tf = _median([e[0].elapsed_time(e[1]) for e in ev[2:]]) / 1e3
    tb = _median([e[1].elapsed_time(e[2]) for e in ev[2:]]) / 1e3
    btf, btb = tp_bytes(R, t.d1, t.d2, t.n_paths, t.D, wl.mul, 4)
    return {"workload": wl.name, "dtype": "f32", "rows": R,
            "fwd": {"ms": tf * 1e3, "rows_per_s": R / tf, "alg_GBps": btf / tf / 1e9, "frac": btf / tf / 1e9 / hbm_peak},
            "bwd": {"ms": tb * 1e3, "rows_per_s": R / tb, "alg_GBps": btb / tb / 1e9, "frac": btb / tb / 1e9 / hbm_peak}}


def workload_config(w, g, args):
    return {"workload": f"{w.name} ({args.dtype})", "atoms": g.n_nodes, "edges": g.n_edges,
            "atom_order": args.order, "parallelism": "replicas" if args.gpus > 1 else "single",
            "l2": "inputs larger than L2 (edge weights alone exceed 129 MB)",
            "tp_workload": "tp-batched: 200000 rows, 128x0e+128x1o+128x2e, SH l<=3, out l<=3 (fp32)"}


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    import message_passing_gb300 as e3
    from message_passing_gb300 import build as libbuild
    from synth import STREAM_GRAD, STREAM_W, device_normal
    from synth import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(e3.LIB_PATH):
        libbuild.build()
    if world > 1:
        dist.barrier()
    e3.load()
    bf16 = args.dtype == "bf16"
    dt = torch.bfloat16 if bf16 else torch.float32
    s = 2 if bf16 else 4
    hbm_peak, peak_kind = peaks()

    # ---- conv workload
    w = W.WORKLOADS[4]
    t = e3.Table.create(w.blocks, w.mul, w.sh_lmax, w.out_lmax)
    g = W.make_graph(w, n_atoms=args.atoms, order=args.order)
    N, E, Nq, P, D = g.n_nodes, g.n_edges, w.mul, t.n_paths, t.D
    scale = N / E
    x_np, _ = W.make_conv(w, g, P, edge_ids=np.zeros(0, np.int64))
    vec = torch.from_numpy(g.vec.astype(np.float32)).to(dev)
    rp = torch.from_numpy(g.rowptr).to(dev)
    sd = torch.from_numpy(g.sender).to(dev)
    xd = torch.from_numpy(x_np).to(dev).to(dt)
    wd = device_normal((E, P, Nq), (w.wid, STREAM_W), W.weight_scale(w, P), device=dev, dtype=dt)
    dmd = device_normal((N, D, Nq), (w.wid, STREAM_GRAD), device=dev, dtype=dt)
    y = torch.empty((E, t.d2), device=dev, dtype=dt)
    m = torch.empty((N, D, Nq), device=dev, dtype=torch.float32)
    f32 = dict(dtype=torch.float32)
    dx, dy, dw = torch.empty_like(xd, **f32), torch.empty_like(y, **f32), torch.empty_like(wd, **f32)
    csc = e3.graph_prepare(rp, sd, N)
    e3.check_device_status()
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev: ev[0].record(stream)
        e3.sh_forward(vec, w.sh_lmax, out=y, stream=stream)
        if ev: ev[1].record(stream)
        e3.conv_forward(t, rp, sd, xd, y, wd, scale, out=m, stream=stream)
        if ev: ev[2].record(stream)
        e3.conv_backward(t, csc, xd, y, wd, dmd, scale, out=(dx, dy, dw), stream=stream)
        if ev: ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    e3.check_device_status()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = Clocks(local) if rank == 0 else None
    if clocks: clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, dev)
    ksh = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) / 1e3
    kfw = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) / 1e3
    kbw = statistics.mean(e[2].elapsed_time(e[3]) for e in evs) / 1e3
    e3.check_device_status()
    bf, bb = conv_bytes(N, E, t.d1, t.d2, P, D, Nq, s)
    bsh = sh_bytes(E, t.d2, s)
    rows = {
        "sh": {"ms": ksh * 1e3, "alg_GBps": bsh / ksh / 1e9, "frac": bsh / ksh / 1e9 / hbm_peak},
        "conv_fwd": {"ms": kfw * 1e3, "alg_GBps": bf / kfw / 1e9, "frac": bf / kfw / 1e9 / hbm_peak,
                     "edges_per_s": E / kfw},
        "conv_bwd": {"ms": kbw * 1e3, "alg_GBps": bb / kbw / 1e9, "frac": bb / kbw / 1e9 / hbm_peak,
                     "edges_per_s": E / kbw},
    }
    dom = max(("conv_fwd", kfw, bf), ("conv_bwd", kbw, bb), key=lambda r: r[1])
    traffic = ncu_traffic(dom[0], E)
    roofline = {"kernel": dom[0], "bound": "hbm", "achieved": dom[2] / dom[1] / 1e9, "peak": hbm_peak,
                "unit": "GB/s", "frac": dom[2] / dom[1] / 1e9 / hbm_peak, "traffic": traffic,
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback"}

    # ---- TP rows
    tp = None
    if not args.no_tp:
        del dw, dy, dx
        torch.cuda.empty_cache()
        w2 = W.WORKLOADS[2]
        t2 = e3.Table.create(w2.blocks, w2.mul, w2.sh_lmax, w2.out_lmax)
        R = w2.rows if args.tp_rows is None else args.tp_rows
        u, x2, ww2 = W.make_tp(w2, t2.n_paths, rows=R)
        v2 = torch.from_numpy(u.astype(np.float32)).to(dev)
        x2d = torch.from_numpy(x2).to(dev)
        w2d = torch.from_numpy(ww2).to(dev)
        dz = device_normal((R, t2.D, w2.mul), (w2.wid, STREAM_GRAD), device=dev)
        y2 = e3.sh_forward(v2, w2.sh_lmax)
        z = torch.empty((R, t2.D, w2.mul), device=dev)
        gx, gy, gw = torch.empty_like(x2d), torch.empty_like(y2), torch.empty_like(w2d)
        reps = max(args.steps, 5)
        for _ in range(args.warmup):
            e3.tp_forward(t2, x2d, y2, w2d, out=z, stream=stream)
            e3.tp_backward(t2, x2d, y2, w2d, dz, out=(gx, gy, gw), stream=stream)
        torch.cuda.synchronize()
        ef = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
        for k in range(reps):
            ef[k][0].record(stream)
            e3.tp_forward(t2, x2d, y2, w2d, out=z, stream=stream)
            ef[k][1].record(stream)
            e3.tp_backward(t2, x2d, y2, w2d, dz, out=(gx, gy, gw), stream=stream)
            ef[k][2].record(stream)
        torch.cuda.synchronize()
        tf = statistics.mean(e[0].elapsed_time(e[1]) for e in ef) / 1e3
        tb = statistics.mean(e[1].elapsed_time(e[2]) for e in ef) / 1e3
        btf, btb = tp_bytes(R, t2.d1, t2.d2, t2.n_paths, t2.D, w2.mul, 4)
        tp = {"rows": R, "fwd": {"ms": tf * 1e3, "alg_GBps": btf / tf / 1e9, "frac": btf / tf / 1e9 / hbm_peak,
                                 "rows_per_s": R / tf, "traffic": ncu_traffic("tp_fwd", R)},
              "bwd": {"ms": tb * 1e3, "alg_GBps": btb / tb / 1e9, "frac": btb / tb / 1e9 / hbm_peak,
                      "rows_per_s": R / tb}}
        del x2d, w2d, dz, y2, z, gx, gy, gw
        torch.cuda.empty_cache()
        dx, dy, dw = torch.empty_like(xd, **f32), torch.empty_like(y, **f32), torch.empty_like(wd, **f32)

    # ---- end to end through the API with host buffers
    e2e = None
    if not args.no_e2e:
        pin = lambda tns: torch.empty(tns.shape, dtype=tns.dtype, pin_memory=True).copy_(tns)
        h_vec, h_rp, h_sd, h_x = pin(vec.cpu()), pin(rp.cpu()), pin(sd.cpu()), pin(xd.cpu())
        h_w = torch.empty(wd.shape, dtype=wd.dtype, pin_memory=True)
        h_w.copy_(wd)
        h_dm = pin(dmd.cpu())
        o_m = torch.empty(m.shape, dtype=torch.float32, pin_memory=True)
        o_dx = torch.empty(xd.shape, dtype=torch.float32, pin_memory=True)
        o_dy = torch.empty(y.shape, dtype=torch.float32, pin_memory=True)
        o_dw = torch.empty(wd.shape, dtype=torch.float32, pin_memory=True)
        h2d = sum(a.numel() * a.element_size() for a in (h_vec, h_rp, h_sd, h_x, h_w, h_dm))
        d2h = sum(a.numel() * a.element_size() for a in (o_m, o_dx, o_dy, o_dw))

        # Two device buffer sets, three streams: the H2D copies of step i (stream s_in) overlap
        # the compute of step i-1 (s_comp) and the D2H copies of step i-2 (s_out).
        # Events keep a set's inputs until its compute is done and its outputs until they are
        # copied out. Every step's own copies are inside the timed region.
        def dev_set(first):
            if first:
                ts = dict(vec=vec, rp=rp, sd=sd, x=xd, w=wd, dm=dmd, y=y, m=m, dx=dx, dy=dy, dw=dw, csc=csc)
            else:
                ts = {k: torch.empty_like(v) for k, v in
                      dict(vec=vec, rp=rp, sd=sd, x=xd, w=wd, dm=dmd, y=y, m=m, dx=dx, dy=dy, dw=dw).items()}
                ts["csc"] = tuple(torch.empty_like(c) for c in csc)
            ts["ws"] = torch.empty(e3.graph_prepare_workspace_bytes(N, E), dtype=torch.uint8, device=dev)
            return ts
        sets = [dev_set(True), dev_set(False)]
        # (non-blocking streams: work on the legacy default stream would serialise with the copies)
        s_in, s_comp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        used = [False, False]

        def e2e_step(i):
            j = i % 2
            b = sets[j]
            with torch.cuda.stream(s_in):
                if used[j]:
                    s_in.wait_event(ev_comp[j])        # step i-2 is done reading these inputs
                for k, h in (("vec", h_vec), ("rp", h_rp), ("sd", h_sd), ("x", h_x), ("w", h_w), ("dm", h_dm)):
                    b[k].copy_(h, non_blocking=True)
                ev_in[j].record(s_in)
            s_comp.wait_event(ev_in[j])
            if used[j]:
                s_comp.wait_event(ev_out[j])           # step i-2's outputs are copied out
            e3.sh_forward(b["vec"], w.sh_lmax, out=b["y"], stream=s_comp)
            c = e3.graph_prepare(b["rp"], b["sd"], N, out=b["csc"], workspace=b["ws"], stream=s_comp)
            e3.conv_forward(t, b["rp"], b["sd"], b["x"], b["y"], b["w"], scale, out=b["m"], stream=s_comp)
            e3.conv_backward(t, c, b["x"], b["y"], b["w"], b["dm"], scale, out=(b["dx"], b["dy"], b["dw"]),
                             stream=s_comp)
            ev_comp[j].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[j])
                for o, k in ((o_m, "m"), (o_dx, "dx"), (o_dy, "dy"), (o_dw, "dw")):
                    o.copy_(b[k], non_blocking=True)
                ev_out[j].record(s_out)
            used[j] = True

        e2e_step(0)
        e2e_step(1)
        torch.cuda.synchronize()
        ke = max(1, min(max(args.steps, 2), args.e2e_steps))
        if world > 1:
            dist.barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(s_in)
        for i in range(ke):
            e2e_step(i)
        a1.record(s_out)
        torch.cuda.synchronize()
        te = max_over_ranks(a0.elapsed_time(a1) / 1e3, dev)
        e3.check_device_status()
        e2e = {"value": whole_job_rate(E, ke, world, te), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": ke, "ms_per_step": te / ke * 1e3,
               "includes": ("pinned H2D of vec, rowptr, sender, x, w, dm; SH; graph_prepare; conv fwd; conv bwd; "
                            "D2H of m, dx, dy, dw; H2D, compute and D2H of consecutive steps overlap on three "
                            "streams with two device buffer sets (the first H2D and the last D2H are not hidden)")}
        del sets
        del h_w, o_dw
    # ---- the other workloads (kernel times only; rank 0)
    others = double_bwd = None
    if rank == 0 and not args.no_workloads:
        del wd, dmd, dx, dy, dw, xd, y, m
        torch.cuda.empty_cache()
        want = set(args.workloads.split(","))
        na = args.workload_atoms   # a smaller box of every conv workload (profiling)
        jobs = [("tp1", lambda: time_tp_workload(W.WORKLOADS[1], dev, stream, 20, hbm_peak)),
                ("conv4", lambda: time_conv_workload(W.WORKLOADS[4], torch.float32, dev, stream, 5, hbm_peak,
                                                     n_atoms=na)),
                ("conv3", lambda: time_conv_workload(W.WORKLOADS[3], torch.float32, dev, stream, 5, hbm_peak,
                                                     n_atoms=na)),
                ("conv4bf16", lambda: time_conv_workload(W.WORKLOADS[4], torch.bfloat16, dev, stream, 5, hbm_peak,
                                                         n_atoms=na)),
                ("conv5", lambda: time_conv_workload(W.WORKLOADS[5], torch.float32, dev, stream, 5, hbm_peak,
                                                     n_atoms=na)),
                ("pad", lambda: time_conv_workload(W.WORKLOADS[4], torch.float32, dev, stream, 5, hbm_peak,
                                                   pad_frac=0.25, n_atoms=na)),
                ("coo", lambda: time_coo_tp(W.WORKLOADS[2], dev, stream, 5, hbm_peak, rows=args.coo_rows)),
                ("radial4", lambda: time_radial_workload(W.WORKLOADS[4], dev, stream, 5, hbm_peak, n_atoms=na)),
                ("hub", lambda: time_hub_workload(W.WORKLOADS[4], dev, stream, 5, hbm_peak, n_atoms=na))]
        others = [f() for k, f in jobs if "all" in want or k in want]
        if "all" in want or "dbwd" in want:
            double_bwd = time_double_backward(W.WORKLOADS[4], dev, stream, 3, hbm_peak, n_atoms=args.dbwd_atoms)

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        from synth import STREAM_GRAD as SG
        ot = oracle.table(w.blocks, w.sh_lmax, w.out_lmax)
        P = t.n_paths
        wfetch = lambda ids: W.make_conv(w, g, P, edge_ids=np.asarray(ids, np.int64))[1].astype(np.float64)
        xo, yo = cpu_inputs(w, g, ot)
        dmo = W.make_grad(w, N, t.D).astype(np.float64)
        n_recv = 8
        e_cnt, secs = oracle_conv_sample(w, g, ot, xo, yo, wfetch, dmo, scale, n_recv, seed=5)
        # grow the sample to about 10 s of CPU work
        n_recv = int(min(N, max(8, n_recv * 10.0 / max(secs, 1e-3))))
        e_cnt, secs = oracle_conv_sample(w, g, ot, xo, yo, wfetch, dmo, scale, n_recv, seed=6)
        cpu = {"value": e_cnt / secs, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": f"{n_recv} random receivers ({e_cnt} edges): oracle conv fwd + dy/dw of those edges + dx of {n_recv} senders, f64, {secs:.1f} s"}

    if rank == 0:
        line = {"metric": METRIC, "value": whole_job_rate(E, args.steps, world, elapsed), "unit": UNIT,
                "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if bf16 else "f32", "data": "synthetic", "config": workload_config(w, g, args),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 3 * args.steps,
                "clocks": clk, "rows": rows, "tp": tp, "workloads": others,
                "double_backward": double_bwd}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--order", choices=["cell", "draw"], default="cell")
    ap.add_argument("--atoms", type=int, default=None, help="smaller conv workload (profiling)")
    ap.add_argument("--tp-rows", type=int, default=None, help="smaller TP workload (profiling)")
    ap.add_argument("--coo-rows", type=int, default=None, help="smaller COO workload (profiling)")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--ref-receivers", type=int, default=24)
    ap.add_argument("--no-tp", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload kernel timings")
    ap.add_argument("--workloads", default="all",
                    help="comma list of per-workload timings: tp1,conv4,conv3,conv4bf16,conv5,pad,coo,radial4,hub,dbwd "
                         "(or all)")
    ap.add_argument("--dbwd-atoms", type=int, default=None, help="smaller double-backward case (profiling)")
    ap.add_argument("--workload-atoms", type=int, default=None,
                    help="smaller box for every conv workload's timing (profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
