#!/usr/bin/env python
"""Benchmark of the ternary (TQ2_0-style) matvec on GB300.

Workload (one "step"): the whole MiniCPM4-8B-shaped ternary stack streamed
once at M=1 -- 32 layers x {q,o: 4096->4096; k,v: 4096->256; gate,up:
4096->16384; down: 16384->4096} = 224 linears, 7.58e9 weights, 1.96 GB of
packed codes + scales per step (more than 15x the 129 MB L2, so every step
reads its weights from HBM).  Synthetic seeded inputs (codes P(1)=1/2,
P(0)=P(2)=1/4; d ~ U[0.005,0.05] fp16; x ~ N(0,1) fp16), packed on the GPU
with tq2_pack.  The 224 tq2_matvec calls are captured once in a CUDA graph
(programmatic dependent launches between them) and replayed.

Metric: HBM GB/s of algorithmic bytes (N*K/4 + 2*N*K/256 + 2*M*K + 4*M*N per
linear) and the decode-equivalent tok/s (one step = one token).

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on the
host cores instead (the reference arm of this comparison).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYER = [("q", 4096, 4096), ("k", 256, 4096), ("v", 256, 4096), ("o", 4096, 4096),
         ("gate", 16384, 4096), ("up", 16384, 4096), ("down", 4096, 16384)]
N_LAYERS = 32
SEED = 1
METRIC = "ternary matvec HBM GB/s (% of GB300 peak) and 8B-stack decode-equivalent tok/s"
WORKLOAD = ("MiniCPM4-8B ternary stack: 224 linears (32 x q,k,v,o,gate,up,down), M=1, "
            "fp16 x, fp32 y, TQ2_0 2-bit codes + fp16 per-256 scales")


def linear_bytes(M, N, K, ybytes=4):
    return N * K // 4 + 2 * N * (K // 256) + 2 * M * K + ybytes * M * N


def stack_linears():
    return [(L, *LAYER[L % 7]) for L in range(N_LAYERS * 7)]


STACK_BYTES = sum(linear_bytes(1, N, K) for _, _, N, K in stack_linears())


def max_over_ranks(value, device=None):
    """The largest `value` over all ranks of the default process group (the
    value itself when no group is initialised): the slowest replica sets the
    step time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world, bytes_per_step, ms_per_step):
    """Whole-job throughput: every replica streams bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def _peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy, burst)"
    except Exception:
        return 6800.0, "fallback (6.8 TB/s, one earlier GB300 copy measurement)"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the GPU is loaded."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index_or_uuid):
        self.ident = str(device_index_or_uuid)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm
def build_stack(torch, tq2, syn, dev, with_prologue_scales=True):
    """Generate and pack the 224 linears on the device (seeded)."""
    lin = stack_linears()
    qs, ds = [], []
    x_off, y_off = [], []
    xo = yo = 0
    for L, name, N, K in lin:
        bits = torch.from_numpy(syn.code_bits(SEED, syn.tensor_id(L, syn.SLOT_CODE_BITS),
                                              N * K // 4)).to(dev)
        codes = syn.codes_from_bits_torch(bits, N, K)
        del bits
        qs.append(tq2.pack(codes))
        del codes
        ds.append(torch.from_numpy(syn.scales(SEED, N, K // 256, linear=L)).to(dev))
        x_off.append(xo)
        y_off.append(yo)
        xo += K
        yo += N
    x_host = torch.empty(xo, dtype=torch.float16).pin_memory()
    import numpy as np
    xh = x_host.numpy()
    for (L, name, N, K), o in zip(lin, x_off):
        xh[o:o + K] = syn.activations(SEED, 1, K, linear=L)[0]
    X = x_host.to(dev)
    Y = torch.zeros(yo, dtype=torch.float32, device=dev)
    y_host = torch.empty(yo, dtype=torch.float32).pin_memory()
    scales = [syn.act_scale(SEED, linear=L) for L, *_ in lin] if with_prologue_scales else None
    out_scales = [syn.out_scale(SEED, linear=L) for L, *_ in lin] if with_prologue_scales else None
    torch.cuda.synchronize()
    return dict(lin=lin, qs=qs, d=ds, x_off=x_off, y_off=y_off, X=X, Y=Y, x_host=x_host,
                y_host=y_host, scales=scales, out_scales=out_scales)


def capture(torch, tq2, st, calls, stream):
    """calls: list of (x view, qs, d, y view, act_scale, impl, out_scale) -> CUDA graph."""
    with torch.cuda.stream(stream):
        for x, qs, d, y, s, impl, so in calls:  # eager warm-up (kernel attributes, module load)
            tq2.matvec(x, qs, d, y=y, act_scale=s, impl=impl, out_scale=so)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for x, qs, d, y, s, impl, so in calls:
                tq2.matvec(x, qs, d, y=y, act_scale=s, impl=impl, out_scale=so)
    stream.synchronize()
    return g


def stack_calls(st, prologue=False, impl=0, requant=False):
    calls = []
    for i, (L, name, N, K) in enumerate(st["lin"]):
        x = st["X"][st["x_off"][i]:st["x_off"][i] + K].view(1, K)
        y = st["Y"][st["y_off"][i]:st["y_off"][i] + N].view(1, N)
        calls.append((x, st["qs"][i], st["d"][i], y, st["scales"][i] if prologue else 0.0, impl,
                      st["out_scales"][i] if requant else 0.0))
    return calls


def grouped_stack(st):
    """The stack as a decoder would run it with shared inputs: per layer
    q,k,v as one tq2_matvec_grouped call on q's x, o, gate,up as one grouped
    call on gate's x, down -- 4 launches per layer.  Returns (calls, bytes):
    each call is (x view, [qs], [d], [y views]); bytes count x once per call."""
    calls, nbytes = [], 0
    lin = st["lin"]
    i = 0
    while i < len(lin):
        name = lin[i][1]
        n = 3 if name == "q" else (2 if name == "gate" else 1)  # q,k,v / gate,up / single
        idx = list(range(i, i + n))
        K = lin[i][3]
        x = st["X"][st["x_off"][i]:st["x_off"][i] + K].view(1, K)
        ys = [st["Y"][st["y_off"][j]:st["y_off"][j] + lin[j][2]].view(1, lin[j][2]) for j in idx]
        calls.append((x, [st["qs"][j] for j in idx], [st["d"][j] for j in idx], ys))
        nbytes += 2 * K + sum(linear_bytes(1, lin[j][2], K) - 2 * K for j in idx)
        i += len(idx)
    return calls, nbytes


def capture_grouped(torch, tq2, calls, stream, act_scale=0.0, workspace=None):
    with torch.cuda.stream(stream):
        for x, qs, d, ys in calls:  # eager warm-up
            tq2.matvec_grouped(x, qs, d, y_list=ys, act_scale=act_scale, workspace=workspace)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for x, qs, d, ys in calls:
                tq2.matvec_grouped(x, qs, d, y_list=ys, act_scale=act_scale, workspace=workspace)
    stream.synchronize()
    return g


def time_graph(torch, g, stream, steps, warmup, barrier=None):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("tq2_timed")
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    return e0.elapsed_time(e1) / steps  # ms per replay


SHAPE_GROUPS = {"qo_4096x4096": ("q", "o"), "kv_256x4096": ("k", "v"),
                "gateup_16384x4096": ("gate", "up"), "down_4096x16384": ("down",)}


L2_BYTES = 129 * 1024 * 1024  # GB300 L2


def shape_pool(torch, st, names, min_bytes=4 * L2_BYTES):
    """Distinct (qs, d) pairs of one shape totalling at least min_bytes: the
    stack's own tensors first, then copies of them (new allocations), so
    that back-to-back calls read their weights from HBM, not L2."""
    idx = [i for i, (L, n, N, K) in enumerate(st["lin"]) if n in names]
    N, K = st["lin"][idx[0]][2], st["lin"][idx[0]][3]
    per = N * K // 4 + 2 * N * (K // 256)
    need = max(len(idx), -(-min_bytes // per))
    pool = [(st["qs"][i], st["d"][i]) for i in idx]
    j = 0
    while len(pool) < need:
        q, d = pool[j % len(idx)]
        pool.append((q.clone(), d.clone()))
        j += 1
    return pool, N, K


def shape_graphs(torch, tq2, st, stream, M_list=(1,), impl=0, groups=None, heavy=False, prologue=False,
                 repeats=21):
    """Back-to-back calls of one shape over distinct weight sets totalling at
    least 4x L2 (q/o 120 sets, 520 MB; k/v 1,844 sets, 516 MB; gate/up and
    down 30 sets, 521 MB), one CUDA graph per shape and M replayed `repeats`
    times: us per call as the median and the 95th percentile over the
    replays; optionally heavy-tailed x (1 % of entries x50) and the int8
    prologue with each linear's act_scale."""
    out = {}
    dev = st["X"].device
    import tq2_synth as syn
    for gname, names in SHAPE_GROUPS.items():
        if groups is not None and gname not in groups:
            continue
        pool, N, K = shape_pool(torch, st, names)
        sc = [st["scales"][i] for i, (L, n, N_, K_) in enumerate(st["lin"]) if n in names]
        for M in M_list:
            x = torch.from_numpy(syn.activations(SEED + 7, M, K, linear=0, heavy=heavy)).to(dev)
            ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in pool]
            calls = [(x, q, d, y, sc[j % len(sc)] if prologue else 0.0, impl, 0.0)
                     for j, ((q, d), y) in enumerate(zip(pool, ys))]
            g = capture(torch, tq2, st, calls, stream)
            time_graph(torch, g, stream, 2, 1)
            per_rep = [1e3 * time_graph(torch, g, stream, 1, 1 if r == 0 else 0) / len(pool)
                       for r in range(repeats)]
            per_rep.sort()
            med = statistics.median(per_rep)
            p95 = per_rep[min(len(per_rep) - 1, int(round(0.95 * (len(per_rep) - 1))))]
            nbytes = linear_bytes(M, N, K)
            out[(gname, M)] = dict(us_per_call=med, us_p95=p95,
                                   gbs=nbytes / (med * 1e-6) / 1e9,
                                   distinct_weight_sets=len(pool),
                                   distinct_bytes=len(pool) * (N * K // 4 + 2 * N * (K // 256)),
                                   repeats=repeats)
            del g, ys
        del pool
    return out


def grouped_sweep(torch, tq2, st, stream, M_list=(2, 4, 8, 9, 12, 16), repeats=11):
    """tq2_matvec_grouped on q/k/v and on gate/up at M activation rows, back
    to back over distinct weight groups totalling at least 4x L2 (the stack's
    own, then copies), with and without the int8 prologue (one shared
    workspace: x converted once per group where the group runs as
    consecutive calls).  us per group (median of the replays) and GB/s of
    the group's algorithmic bytes."""
    import tq2_synth as syn
    out = {}
    dev = st["X"].device
    K = 4096
    for gname, names in (("qkv", ("q", "k", "v")), ("gateup", ("gate", "up"))):
        by_layer = {}  # the stack's seven linears per layer, in order
        for i, (L, n, N, K_) in enumerate(st["lin"]):
            by_layer.setdefault(i // 7, {})[n] = i
        groups = [[(st["qs"][lay[n]], st["d"][lay[n]]) for n in names] for lay in by_layer.values()]
        Ns = [st["lin"][by_layer[0][n]][2] for n in names]
        per = sum(N * K // 4 + 2 * N * (K // 256) for N in Ns)
        j = 0
        while len(groups) * per < 4 * L2_BYTES:
            groups.append([(q.clone(), d.clone()) for q, d in groups[j]])
            j += 1
        s_act = float(syn.act_scale(SEED, linear=0))
        for M in M_list:
            x = torch.from_numpy(syn.activations(SEED + 13, M, K, linear=0, heavy=True)).to(dev)
            ys = [[torch.empty((M, N), dtype=torch.float32, device=dev) for N in Ns] for _ in groups]
            calls = [(x, [q for q, _ in g], [d for _, d in g], y) for g, y in zip(groups, ys)]
            ws = torch.empty(2 * M * K, dtype=torch.uint8, device=dev)
            nbytes = sum(linear_bytes(M, N, K) for N in Ns)
            for tag, s, w in (("", 0.0, None), ("_prologue", s_act, ws)):
                g = capture_grouped(torch, tq2, calls, stream, act_scale=s, workspace=w)
                time_graph(torch, g, stream, 2, 1)
                per_rep = sorted(1e3 * time_graph(torch, g, stream, 1, 0) / len(groups) for _ in range(repeats))
                med = statistics.median(per_rep)
                out[f"{gname}_M{M}{tag}"] = dict(us_per_group=med, gbs=nbytes / (med * 1e-6) / 1e9,
                                                 distinct_groups=len(groups))
                del g
            del ys, calls, ws
        del groups
    return out


def _bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops: cuBLAS bf16, burst)"
    except Exception:
        return 1900.0, "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 measurement)"


def prefill_gemm(torch, tq2, st, stream, M_list=(512, 2048)):
    """tq2_gemm (tcgen05) on the layer shapes with M activation rows (a prompt
    chunk): us per call and TFLOP/s (2 M N K), against the measured dense
    bf16 tensor peak (fp16 runs at the same rate).  Also with the int8
    prologue, run as a pass of its own into a workspace ("_prologue") and
    inside every weight tile with no workspace ("_prologue_in_tile")."""
    import tq2_synth as syn
    peak, src = _bf16_peak()
    out = {"peak_tflops": peak, "peak_source": src}
    dev = st["X"].device
    s_act = float(syn.act_scale(SEED, linear=0))
    for gname, names in SHAPE_GROUPS.items():
        i = [j for j, (L, n, N, K) in enumerate(st["lin"]) if n in names][0]
        N, K = st["lin"][i][2], st["lin"][i][3]
        for M in M_list:
            x = torch.from_numpy(syn.activations(SEED + 11, M, K, linear=0)).to(dev)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            ws = torch.empty(tq2.gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            for tag, kw in (("", dict(workspace=None)), ("_prologue", dict(act_scale=s_act, workspace=ws)),
                            ("_prologue_in_tile", dict(act_scale=s_act, workspace=None))):
                with torch.cuda.stream(stream):
                    for _ in range(3):
                        tq2.gemm(x, st["qs"][i], st["d"][i], y=y, **kw)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    reps = 20
                    e0.record(stream)
                    for _ in range(reps):
                        tq2.gemm(x, st["qs"][i], st["d"][i], y=y, **kw)
                    e1.record(stream)
                stream.synchronize()
                us = e0.elapsed_time(e1) * 1e3 / reps
                tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
                out[f"{gname}_M{M}{tag}"] = dict(us_per_call=us, tflops=tf, frac_of_peak=tf / peak)
            del x, y, ws
    return out


def affine4_bytes(M, N, K, G):
    """Algorithmic bytes of one affine-int4 call: 4-bit codes, fp16 s and z
    per group, fp16 x, fp32 y."""
    return N * K // 2 + 4 * N * (K // G) + 2 * M * K + 4 * M * N


def affine4_shapes(torch, tq2, stream, groups=(64, 128, 256)):
    """tq2_affine4_matvec at M = 1 on the layer shapes: back-to-back calls
    over distinct weight copies (>= 4x L2 in total, so weights stream from
    HBM), us per call, GB/s and the fraction of the measured HBM peak."""
    import tq2_synth as syn
    peak, _ = _peak()
    dev = torch.device("cuda", torch.cuda.current_device())
    out = {}
    for gname, (N, K) in (("qo_4096x4096", (4096, 4096)), ("gateup_16384x4096", (16384, 4096)),
                          ("down_4096x16384", (4096, 16384))):
        for G in groups:
            qs, sc, z = syn.affine4_weights(SEED + 13, N, K, G)
            one = [torch.from_numpy(a).to(dev) for a in (qs, sc, z)]
            copies = max(2, int(4 * 129e6 // affine4_bytes(1, N, K, G)) + 1)
            ws = [one] + [[t.clone() for t in one] for _ in range(copies - 1)]
            x = torch.from_numpy(syn.activations(SEED + 13, 1, K)).to(dev)
            ys = [torch.empty((1, N), dtype=torch.float32, device=dev) for _ in ws]
            with torch.cuda.stream(stream):
                for (q, a, b), y in zip(ws, ys):
                    tq2.affine4_matvec(x, q, a, b, G, y=y)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for (q, a, b), y in zip(ws, ys):
                        tq2.affine4_matvec(x, q, a, b, G, y=y)
            once = time_graph(torch, g, stream, 2, 1)
            ms = time_graph(torch, g, stream, max(3, int(0.3 / max(once * 1e-3, 1e-6))), 3)
            us = 1e3 * ms / len(ws)
            gbs = affine4_bytes(1, N, K, G) / (us * 1e-6) / 1e9
            out[f"{gname}_G{G}"] = dict(us_per_call=us, gbs=gbs, frac_of_hbm_peak=gbs / peak,
                                        distinct_tensors=len(ws))
            del g, ws, ys, one
    return out


def cpu_info():
    """(cores in this process's affinity mask, CPU model string)."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for ln in open("/proc/cpuinfo"):
                if ln.lower().startswith(("model name", "cpu part")):
                    model = ln.split(":", 1)[1].strip()
                    break
        except Exception:
            model = "unknown"
    return cores, model


def run_manifest(torch, st):
    """What produced this line: the source tree and input hashes, the seed,
    the GPU, driver, toolkit and library versions, and the host CPU."""
    import glob
    import hashlib
    import platform

    def run(cmd):
        try:
            return subprocess.run(cmd, capture_output=True, text=True, timeout=20, cwd=ROOT).stdout.strip()
        except Exception:
            return None

    src = hashlib.sha256()
    pkg = os.path.join(ROOT, "quantized_gemv_tq2_gb300")
    files = sorted(glob.glob(os.path.join(pkg, "csrc", "*")) + [os.path.join(ROOT, "include", "tq2.h"),
                   os.path.join(pkg, "__init__.py"), os.path.join(pkg, "build.py"), os.path.abspath(__file__)])
    for f in files:
        src.update(os.path.relpath(f, ROOT).encode())
        src.update(open(f, "rb").read())
    # inputs: the packed weights, scales and x of layer 0 (seeded; the other
    # layers come from the same generator with their own linear index)
    inp = hashlib.sha256()
    for i, (L, name, N, K) in enumerate(st["lin"]):
        if L != 0:
            break
        inp.update(st["qs"][i].cpu().numpy().tobytes())
        inp.update(st["d"][i].cpu().numpy().tobytes())
        xh = st["x_host"].numpy()
        inp.update(xh[st["x_off"][i]:st["x_off"][i] + K].tobytes())
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    nvcc = run([os.environ.get("NVCC", "nvcc"), "--version"])
    smi = run(["nvidia-smi", "--query-gpu=driver_version,name", "--format=csv,noheader"])
    cores, model = cpu_info()
    return {
        "source_sha256": src.hexdigest(),
        "git_sha": run(["git", "rev-parse", "HEAD"]) or None,
        "seed": SEED,
        "input_sha256_layer0": inp.hexdigest(),
        "gpu": props.name,
        "sm_count": props.multi_processor_count,
        "compute_capability": f"{props.major}.{props.minor}",
        "memory_bytes": props.total_memory,
        "driver": smi.splitlines()[0].split(",")[0].strip() if smi else None,
        "nvcc": nvcc.splitlines()[-1].strip() if nvcc else None,
        "torch": torch.__version__,
        "torch_cuda": torch.version.cuda,
        "python": platform.python_version(),
        "host": f"{platform.machine()}, {model}, {cores} cores in the affinity mask",
    }


def cpu_baseline_oracle(budget_s=10.0, stack_host=None):
    """The CPU oracle (plain C, fp64, as it stands) timed on the host: one
    thread on layer 0 of the stack, and every core of the process's affinity
    mask (rows split in contiguous ranges, one oracle call per range) on the
    PR1 linear, one q/o linear, layer 0 and -- when the stack's weights are
    given (copied from the device) -- the whole 224-linear stack once.  The
    headline value is the whole stack on all cores."""
    import numpy as np
    import oracle
    import tq2_synth as syn
    cores, model = cpu_info()
    layer = []
    for L, name, N, K in stack_linears()[:7]:
        codes = syn.codes(SEED, N, K, linear=L)
        qs, _ = oracle.pack(codes)
        layer.append((syn.activations(SEED, 1, K, linear=L), qs, syn.scales(SEED, N, K // 256, linear=L), N, K))

    def run(items, threads):
        t0 = time.perf_counter()
        nbytes = 0
        for x, qs, d, N, K in items:
            oracle.matvec_threads(x, qs, d, K, threads=threads)
            nbytes += linear_bytes(1, N, K)
        return nbytes, time.perf_counter() - t0

    b1, t1 = run(layer, 1)
    out = dict(kind="oracle", unit="GB/s", cores=cores, cpu_model=model,
               one_thread_layer0=dict(gbs=b1 / t1 / 1e9, seconds=t1))
    # PR1: one 32 x 512 linear, many calls (latency-bound at this size, one thread)
    c = syn.codes(0, 32, 512)
    q1, _ = oracle.pack(c)
    pr1 = [(syn.activations(0, 1, 512), q1, syn.scales(0, 32, 2), 32, 512)] * 2000
    bp, tp = run(pr1, 1)
    out["pr1_one_thread"] = dict(us_per_call=1e6 * tp / len(pr1), gbs=bp / tp / 1e9)
    bq, tq = run(layer[:1], cores)
    out["qo_all_cores"] = dict(gbs=bq / tq / 1e9, seconds=tq)
    bl, tl = run(layer, cores)
    out["layer0_all_cores"] = dict(gbs=bl / tl / 1e9, seconds=tl)
    if stack_host is not None:
        bs, ts = run(stack_host, cores)
        out["stack_all_cores"] = dict(gbs=bs / ts / 1e9, seconds=ts, tok_s=1.0 / ts)
        out["value"] = bs / ts / 1e9
        out["sample"] = (f"the whole 224-linear stack once (the device's packed weights copied to the host, "
                         f"{bs} algorithmic bytes), plain C fp64 oracle, {cores} threads over row ranges "
                         f"({model}), {ts:.2f} s; also one thread on layer 0, all cores on PR1 / q/o / layer 0")
    else:
        out["value"] = bl / tl / 1e9
        out["sample"] = (f"layer 0 of the stack (7 linears, {bl} algorithmic bytes), plain C fp64 oracle, "
                         f"{cores} threads over row ranges ({model}), {tl:.2f} s")
    out["tok_s"] = out["value"] * 1e9 / STACK_BYTES
    return out


def read_profile_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources (sha256 of both kernels of the step and of
    the device header they include match); else None."""
    import hashlib
    csrc = os.path.join(ROOT, "quantized_gemv_tq2_gb300", "csrc")
    prof = os.path.join(ROOT, "profiles", "tq2_matvec_mma_stack_m1.md")
    try:
        sha = {key: hashlib.sha256(open(os.path.join(csrc, f), "rb").read()).hexdigest()
               for key, f in (("kernel_source_sha256", "tq2_matvec_mma.cu"),
                              ("smalln_source_sha256", "tq2_matvec_smalln.cu"),
                              ("device_header_sha256", "tq2_device.cuh"))}
        vals = {}
        for line in open(prof):
            if ":" in line and line.strip().startswith("- `"):
                k, v = line.strip()[3:].split("`:", 1)
                vals[k.strip()] = v.strip().strip("`")
        if any(vals.get(k) != v for k, v in sha.items()):
            return None
        return float(vals["traffic_bytes_per_launch_avg"])
    except Exception:
        return None


def run_gpu(args):
    import torch
    import quantized_gemv_tq2_gb300 as tq2
    import tq2_synth as syn

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    barrier = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        barrier = dist.barrier
    tq2.load()

    st = build_stack(torch, tq2, syn, dev)
    stream = torch.cuda.Stream(device=dev)
    g = capture(torch, tq2, st, stack_calls(st), stream)
    launches_per_step = len(st["lin"])

    # clocks: soak ~1 s under the same load, then the timed region, sampled throughout
    props = torch.cuda.get_device_properties(dev)
    ident = getattr(props, "uuid", None)
    ident = f"GPU-{ident}" if ident is not None and not str(ident).startswith("GPU-") else (ident or local)
    sampler = ClockSampler(ident)
    if not args.no_clocks:
        sampler.start()
        soak = time_graph(torch, g, stream, 1, 0)
        time_graph(torch, g, stream, max(1, int(1.0 / max(soak * 1e-3, 1e-6))), 0)
    ms = time_graph(torch, g, stream, args.steps, args.warmup, barrier)
    clocks = sampler.stop() if not args.no_clocks else {"skipped": True}
    ms = max_over_ranks(ms, dev)

    # e2e: every step copies its x from pinned host memory and its y back to
    # pinned host memory, inside the timed region; two buffer sets (one
    # graph each) and a copy stream let step i+1's input copy and step i-1's
    # result copy overlap step i's compute, as a serving loop would.
    e2e_steps = max(3, min(args.steps, 300))
    st2 = dict(st)
    st2["X"] = torch.empty_like(st["X"])
    st2["Y"] = torch.zeros_like(st["Y"])
    st2["x_host"] = torch.empty_like(st["x_host"]).pin_memory()
    st2["x_host"].copy_(st["x_host"])
    st2["y_host"] = torch.empty_like(st["y_host"]).pin_memory()
    bufs = [st, st2]
    graphs = [g, capture(torch, tq2, st2, stack_calls(st2), stream)]
    copy = torch.cuda.Stream()

    def e2e_run(n):
        h2d = [torch.cuda.Event() for _ in bufs]
        done = [torch.cuda.Event() for _ in bufs]
        d2h = [torch.cuda.Event() for _ in bufs]

        def put(i):  # x of step i -> device (after step i-2 has read buffer i % 2)
            b = i % 2
            with torch.cuda.stream(copy):
                if i >= 2:
                    copy.wait_event(done[b])
                bufs[b]["X"].copy_(bufs[b]["x_host"], non_blocking=True)
                h2d[b].record(copy)

        put(0)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(stream):
                stream.wait_event(h2d[b])
                if i >= 2:
                    stream.wait_event(d2h[b])  # step i-2's y is on the host
                graphs[b].replay()
                done[b].record(stream)
            if i + 1 < n:
                put(i + 1)  # queued before this step's result copy: overlaps this step
            with torch.cuda.stream(copy):
                copy.wait_event(done[b])
                bufs[b]["y_host"].copy_(bufs[b]["Y"], non_blocking=True)
                d2h[b].record(copy)

    e2e_run(4)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(copy)
    e2e_run(e2e_steps)
    e1.record(copy)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dev)
    del graphs, st2, bufs

    # per-shape back-to-back calls (>= 4x L2 of distinct weights per shape):
    # the roofline of each call shape, in the headline line
    per_shape = {}
    if rank == 0:
        peak0, _ = _peak()
        for (gname, M), v in shape_graphs(torch, tq2, st, stream, M_list=(1,)).items():
            per_shape[gname] = dict(us_per_call=round(v["us_per_call"], 4), us_p95=round(v["us_p95"], 4),
                                    gbs=round(v["gbs"], 1), frac=round(v["gbs"] / peak0, 4),
                                    distinct_weight_sets=v["distinct_weight_sets"],
                                    distinct_bytes=v["distinct_bytes"], repeats=v["repeats"])

    extras = {}
    if not args.quick and rank == 0:
        gp = capture(torch, tq2, st, stack_calls(st, prologue=True), stream)
        ms_p = time_graph(torch, gp, stream, max(3, min(args.steps, 2000)), 5)
        extras["stack_with_prologue"] = dict(ms_per_step=ms_p, gbs=STACK_BYTES / (ms_p * 1e-3) / 1e9,
                                             tok_s=1e3 / ms_p)
        del gp
        gq = capture(torch, tq2, st, stack_calls(st, prologue=True, requant=True), stream)
        ms_q = time_graph(torch, gq, stream, max(3, min(args.steps, 2000)), 5)
        extras["stack_wna8o8"] = dict(
            ms_per_step=ms_q, gbs=STACK_BYTES / (ms_q * 1e-3) / 1e9, tok_s=1e3 / ms_q,
            how="int8 fake-quant of x on load (per-linear act_scale) and requantisation of y "
                "at store (per-linear out_scale, tq2_matvec_requant), both U[0.01, 0.1]")
        del gq
        gcalls, gbytes = grouped_stack(st)
        gg = capture_grouped(torch, tq2, gcalls, stream)
        ms_g = time_graph(torch, gg, stream, max(3, min(args.steps, 2000)), 5)
        extras["stack_grouped"] = dict(
            ms_per_step=ms_g, gbs=gbytes / (ms_g * 1e-3) / 1e9, tok_s=1e3 / ms_g,
            launches_per_step=len(gcalls), bytes_per_step=gbytes,
            how="per layer q,k,v as one tq2_matvec_grouped launch on a shared x, o, gate,up as one "
                "grouped launch on a shared x, down: 4 launches per layer, the same 224 weight sets")
        del gg
        simt = shape_graphs(torch, tq2, st, stream, M_list=(1,), impl=2)
        extras["shapes_m1_cuda_core_impl"] = {k[0]: v for k, v in simt.items()}
        pre = shape_graphs(torch, tq2, st, stream, M_list=(1, 2), impl=4)
        extras["shapes_prescaled_impl"] = {f"{k[0]}_M{k[1]}": v for k, v in pre.items()}
        sweep = shape_graphs(torch, tq2, st, stream, M_list=(2, 4, 8, 16),
                             groups=("gateup_16384x4096", "down_4096x16384"))
        extras["m_sweep"] = {f"{k[0]}_M{k[1]}": v for k, v in sweep.items()}
        sweep_h = shape_graphs(torch, tq2, st, stream, M_list=(1, 2, 4, 8, 16),
                               groups=("gateup_16384x4096", "down_4096x16384"), heavy=True, prologue=True)
        extras["m_sweep_heavy_prologue"] = {f"{k[0]}_M{k[1]}": v for k, v in sweep_h.items()}
        extras["grouped_m_sweep"] = grouped_sweep(torch, tq2, st, stream)
        extras["prefill_gemm"] = prefill_gemm(torch, tq2, st, stream)
        extras["affine4_m1"] = affine4_shapes(torch, tq2, stream)

    peak, peak_src = _peak()
    value = job_gbs(world, STACK_BYTES, ms)
    per_gpu = STACK_BYTES / (ms * 1e-3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic (seeded; MiniCPM4-8B shapes, no trained weights)",
        "config": {
            "workload": WORKLOAD,
            "linears": len(st["lin"]),
            "bytes_per_step": STACK_BYTES,
            "M": 1,
            "prologue": False,
            "parallelism": "replicas" if world > 1 else "single-gpu",
            "l2": "inputs larger than L2 (1.96 GB of weights per step vs 129 MB L2)",
            "launch": "CUDA graph of 224 tq2_matvec calls with programmatic dependent launch",
        },
        "tok_s": round(world * 1e3 / ms, 2),
        "pct_of_peak": round(100 * per_gpu / peak, 2),
        "roofline": {
            "bound": "hbm",
            "kernel": "tq2::matvec_mma_kernel<1, 1, 1, false> (q, o, gate, up, down: 160 launches) and "
                      "tq2::matvec_smalln_kernel<1,1> (k, v: 64 launches): all 224 launches of a step",
            "achieved": round(per_gpu, 2),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(per_gpu / peak, 4),
            "traffic": read_profile_traffic(),
            "peak_source": peak_src,
            "per_launch": f"avg algorithmic bytes {STACK_BYTES / launches_per_step:.0f} / "
                          f"avg launch time {1e3 * ms / launches_per_step:.3f} us",
            "per_shape": per_shape,
            "per_shape_how": "M = 1, back-to-back tq2_matvec calls in a CUDA graph over distinct weight "
                             "sets totalling >= 4x L2; median and 95th percentile of 21 replays; "
                             "frac = GB/s / peak",
        },
        "e2e": {
            "value": round(job_gbs(world, STACK_BYTES, e2e_ms), 2),
            "unit": "GB/s",
            "ms_per_step": round(e2e_ms, 5),
            "h2d_bytes_per_step": st["X"].numel() * 2,
            "d2h_bytes_per_step": st["Y"].numel() * 4,
            "path": "every step: pinned host x -> device, graph replay of the 224 tq2_matvec calls, "
                    "y -> pinned host; two buffer sets and a copy stream overlap step i+1's input "
                    "copy and step i-1's result copy with step i's compute",
        },
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "manifest": run_manifest(torch, st),
    }
    if extras:
        line["extras"] = extras
    if world == 1 and not args.no_cpu_baseline:
        stack_host = None
        if not args.quick:  # the device's stack, copied to the host once
            xh = st["x_host"].numpy()
            stack_host = [(xh[st["x_off"][i]:st["x_off"][i] + K].reshape(1, K), st["qs"][i].cpu().numpy(),
                           st["d"][i].cpu().numpy(), N, K) for i, (L, n, N, K) in enumerate(st["lin"])]
        line["cpu_baseline"] = cpu_baseline_oracle(args.cpu_seconds, stack_host)
        del stack_host
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ profiling case
CASES = {"gateup": (16384, 4096), "down": (4096, 16384), "qo": (4096, 4096), "kv": (256, 4096)}


def run_case(args):
    """A small case for ncu: `copies` distinct weight sets of one shape (more
    than L2 in total for the big shapes), `launches` eager tq2_matvec calls
    (tq2_gemm when M > 16) round-robin over them, with the int8 prologue when
    --act-scale > 0 (and a workspace: its pass where that pays).  Prints the
    mean wall time per call (not a bench value: the calls are eager and may
    run under a profiler)."""
    import torch
    import quantized_gemv_tq2_gb300 as tq2
    import tq2_synth as syn
    N, K = CASES[args.case]
    dev = torch.device("cuda", 0)
    tq2.load()
    if args.affine4_group:  # the affine-int4 sibling: distinct copies of one weight set
        G = args.affine4_group
        one = [torch.from_numpy(a).to(dev) for a in syn.affine4_weights(SEED, N, K, G)]
        ws4 = [one] + [[t.clone() for t in one] for _ in range(args.copies - 1)]
        x = torch.from_numpy(syn.activations(SEED, args.M, K)).to(dev)
        y = torch.empty((args.M, N), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.launches):
            q, sc, z = ws4[i % len(ws4)]
            tq2.affine4_matvec(x, q, sc, z, G, y=y)
        torch.cuda.synchronize()
        dt = (time.perf_counter() - t0) / args.launches
        print(json.dumps({"case": args.case, "affine4_group": G, "N": N, "K": K, "M": args.M,
                          "copies": args.copies, "launches": args.launches,
                          "wall_us_per_call_eager": round(dt * 1e6, 2)}))
        return
    ws = []
    for c in range(args.copies):
        bits = torch.from_numpy(syn.code_bits(SEED, syn.tensor_id(c, syn.SLOT_CODE_BITS),
                                              N * K // 4)).to(dev)
        ws.append((tq2.pack(syn.codes_from_bits_torch(bits, N, K)),
                   torch.from_numpy(syn.scales(SEED, N, K // 256, linear=c)).to(dev)))
    x = torch.from_numpy(syn.activations(SEED, args.M, K)).to(dev)
    y = torch.empty((args.M, N), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.launches):
        qs, d = ws[i % len(ws)]
        if args.M > 16:  # prefill-sized M: tq2_gemm
            tq2.gemm(x, qs, d, y=y, act_scale=args.act_scale)
        else:
            tq2.matvec(x, qs, d, y=y, impl=args.case_impl, act_scale=args.act_scale)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / args.launches
    print(json.dumps({"case": args.case, "N": N, "K": K, "M": args.M, "copies": args.copies,
                      "launches": args.launches, "impl": args.case_impl, "act_scale": args.act_scale,
                      "wall_us_per_call_eager": round(dt * 1e6, 2)}))


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The CPU oracle timed on the host cores, on this workload's metric."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    import tq2_synth as syn
    # one step = the oracle's matvec of one k/v-shaped linear of the stack
    # (4096 -> 256, 1.05e6 weights): a bounded sample of the stack workload
    L, name, N, K = stack_linears()[1]
    codes = syn.codes(SEED, N, K, linear=L)
    qs, _ = oracle.pack(codes)
    d = syn.scales(SEED, N, K // 256, linear=L)
    x = syn.activations(SEED, 1, K, linear=L)
    cores, model = cpu_info()
    for _ in range(args.warmup):
        oracle.matvec_threads(x, qs, d, K, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.matvec_threads(x, qs, d, K, threads=cores)
    dt = (time.perf_counter() - t0) / args.steps
    nbytes = linear_bytes(1, N, K)
    v = nbytes / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; MiniCPM4-8B shapes)",
        "config": {"workload": WORKLOAD, "step_sample": "the k linear of layer 0 (4096->256)"},
        "tok_s": round(v * 1e9 / STACK_BYTES, 4),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "cpu_model": model,
                         "sample": f"one 4096->256 linear of the stack per step, plain C fp64 oracle, "
                                   f"{cores} threads over row ranges"},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PHASES = ("entry", "wait returned", "x staged", "first stage read", "stage loop done", "y stored",
          "producer done")


def run_phases(args):
    """Where one call's time goes, in the steady state: back-to-back
    tq2_matvec calls (the class-column kernel) of one shape over distinct
    weight sets totalling >= 4x L2, replayed in a CUDA graph, on the trace
    build (TQ2_TRACE=1: globaltimer stamps per CTA at each phase).  Prints
    one JSON line: for the last call, each phase's time after the previous
    call's last y store (median / min / max over its CTAs), the per-CTA
    phase lengths, and the call time of the replay (the stamps make calls
    ~0.3 us slower: not a bench value)."""
    import numpy as np
    import torch
    import quantized_gemv_tq2_gb300 as tq2
    assert tq2.traced(), "--phases needs the trace build: run with TQ2_TRACE=1"
    N, K = CASES[args.phases]
    M = args.M
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(SEED)
    per = N * K // 4 + 2 * N * (K // 256)
    copies = max(4, int(4 * L2_BYTES // per) + 1)
    def packed():  # valid codes {0, 1, 2}, four per byte
        c = torch.randint(0, 3, (N, K // 4, 4), dtype=torch.uint8, device=dev, generator=g)
        return (c[..., 0] + 4 * c[..., 1] + 16 * c[..., 2] + 64 * c[..., 3]).contiguous()

    qs = [packed() for _ in range(copies)]
    d = [(torch.rand(N, K // 256, device=dev, generator=g) * 0.045 + 0.005).half() for _ in range(copies)]
    x = torch.randn(M, K, device=dev, generator=g).half()
    ys = [torch.empty(M, N, device=dev) for _ in range(copies)]
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for q, dd, y in zip(qs, d, ys):
            tq2.matvec(x, q, dd, y=y, impl=tq2.IMPL_MMA)
        st.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=st):
            for q, dd, y in zip(qs, d, ys):
                tq2.matvec(x, q, dd, y=y, impl=tq2.IMPL_MMA)
        for _ in range(3):
            graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        graph.replay()
        e1.record(st)
        e1.synchronize()
    us_call = e0.elapsed_time(e1) * 1e3 / copies
    tr = tq2.trace_read().astype(np.int64)
    ctas = int((tr[0, :, 0] > 0).sum())
    tr = tr[:, :ctas]
    last = 0 if tr[0, :, 5].max() > tr[1, :, 5].max() else 1  # the last call of the replay
    cur, prev = tr[last], tr[1 - last]
    t0 = prev[:, 5].max()  # the previous call's last y store

    def stats(v):
        return {"median_us": round(float(np.median(v)) / 1e3, 3), "min_us": round(float(v.min()) / 1e3, 3),
                "max_us": round(float(v.max()) / 1e3, 3)}

    stamped = [bool((cur[:, i] > 0).all()) for i in range(7)]

    out = {
        "phases": args.phases, "N": N, "K": K, "M": M, "ctas": ctas, "weight_sets": copies,
        "us_per_call_trace_build": round(us_call, 3),
        "after_previous_y_store": {PHASES[i]: stats(cur[:, i] - t0) if stamped[i] else None for i in range(7)},
        "per_cta": {
            name: stats(cur[:, j] - cur[:, i]) if stamped[i] and stamped[j] else None
            for name, i, j in (("wait -> x staged", 1, 2), ("x staged -> first stage read", 2, 3),
                               ("first stage read -> loop done", 3, 4), ("loop done -> y stored", 4, 5))
        },
        "call_span_us": round(float(cur[:, 5].max() - t0) / 1e3, 3),
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only, no extras")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true",
                    help="no clock sampling / soak (for runs under a profiler)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--case", choices=sorted(CASES), help="profiling case instead of the bench")
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--copies", type=int, default=8)
    ap.add_argument("--launches", type=int, default=8)
    ap.add_argument("--case-impl", type=int, default=0)
    ap.add_argument("--act-scale", type=float, default=0.0,
                    help="with --case: the int8 prologue's scale (0: none)")
    ap.add_argument("--affine4-group", type=int, default=0,
                    help="with --case: run tq2_affine4_matvec with this group size instead")
    ap.add_argument("--phases", choices=sorted(CASES),
                    help="per-phase time budget of back-to-back calls of this shape (trace build: TQ2_TRACE=1)")
    args = ap.parse_args()
    if args.phases:
        return run_phases(args)
    if args.case:
        return run_case(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
