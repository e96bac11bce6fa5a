"""Throughput benchmark of the GB300 affine group-quantized GEMV / small-M GEMM
library (libgai4.so).

One "step" is one pass over the whole hot path on seeded synthetic inputs
resident in HBM:
  * qmv, 4-bit, group size 64, bf16: (N, K) = 4096x4096, 5120x5120,
    14336x5120, 5120x14336, 27648x5120
  * qmm_t, 4-bit, group size 64, bf16, split-K: (K x N, M) = 2048x2048/22,
    4096x4096/16, 10752x2048/85, 14336x4096/33, 17408x5120/56, 5120x17408/28,
    256x4096/40, and 4096x4096/8
  * Q8_0 and Q4_K GEMV (f32 activations): 4096x4096 and 14336x5120
The metric is effective GB/s = algorithmic bytes (packed weights + scales +
biases + activations + outputs; blocks + activations + outputs for Q8_0/Q4_K)
per unit time. Each kernel family of the step is one CUDA graph, bracketed by
CUDA events on the launching stream; the step's weights (~0.5 GB) exceed the
129 MB L2 many times, so every call streams its weights from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU
("replicas only": the path has no exchange step); rank 0 prints one JSON line.
`--impl reference` times the CPU oracle on a bounded sample of the same work.
"""
from __future__ import annotations

import argparse
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "qmv/qmm_t effective HBM GB/s (% of GB300 peak), 4-bit gs64 bf16, M=1..85"
UNIT = "GB/s"

QMV_SHAPES = [(4096, 4096), (5120, 5120), (14336, 5120), (5120, 14336), (27648, 5120)]   # (N, K)
QMM_SHAPES = [(2048, 2048, 22), (4096, 4096, 16), (10752, 2048, 85), (14336, 4096, 33),  # (K, N, M)
              (17408, 5120, 56), (5120, 17408, 28), (256, 4096, 40), (4096, 4096, 8)]
BLOCKQ_SHAPES = [(4096, 4096), (14336, 5120)]                                              # (N, K)
BITS, GS = 4, 64

# sources whose kernels run in each family's calls (a recorded ncu traffic
# figure is used only while these files are unchanged)
_CSRC = "gemm_affine_int4_gb300/csrc/"
KERNEL_SOURCES = {
    "qmv": [_CSRC + f for f in ("qmv4.cu", "pipeline.cuh", "common.cuh", "api.cu")],
    "qmm_t": [_CSRC + f for f in ("qmm_tc.cu", "pipeline.cuh", "common.cuh", "api.cu")],
    "q8_0": [_CSRC + f for f in ("blockq_tma.cu", "blockq.cu", "pipeline.cuh", "common.cuh", "api.cu")],
    "q4_k": [_CSRC + f for f in ("blockq_tma.cu", "blockq.cu", "pipeline.cuh", "common.cuh", "api.cu")],
}


def affine_bytes(M, N, K, tbytes=2):
    return N * K * BITS // 8 + 2 * N * (K // GS) * tbytes + M * K * tbytes + M * N * tbytes


def q8_bytes(N, K):
    return N * (K // 32) * 36 + K * 4 + N * 4


def q4k_bytes(N, K):
    return N * (K // 256) * 144 + K * 4 + N * 4


def step_bytes():
    fam = {
        "qmv": sum(affine_bytes(1, N, K) for N, K in QMV_SHAPES),
        "qmm_t": sum(affine_bytes(M, N, K) for K, N, M in QMM_SHAPES),
        "q8_0": sum(q8_bytes(N, K) for N, K in BLOCKQ_SHAPES),
        "q4_k": sum(q4k_bytes(N, K) for N, K in BLOCKQ_SHAPES),
    }
    return fam


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        h.update(open(os.path.join(ROOT, p), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(family, algorithmic_bytes):
    """DRAM bytes per step of a family from the committed ncu summary, if the
    summary was taken on the current kernel source and on this workload (the
    same algorithmic bytes per step: a run restricted by --only is not)."""
    path = os.path.join(ROOT, "profiles", f"{family}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != source_hash(KERNEL_SOURCES[family]):
        return None
    try:
        if int(vals["algorithmic_bytes_per_step"]) != int(algorithmic_bytes):
            return None
        return float(vals["dram_bytes_per_step"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def selected(only, fam, idx):
    """--only FAMILY[:INDEX] restricts the workload (profiling runs)."""
    if not only:
        return True
    f, _, i = only.partition(":")
    return f == fam and (i == "" or int(i) == idx)


# batched / strided qmm_t, measured beside the step (not part of it):
# (batch, K, N, M): stacked weights [batch, N, K], activations a strided,
# odd-offset view (rows K + 8 apart, one element in), so the call gathers them
BATCHED_SHAPES = [(4, 4096, 4096, 16), (8, 2048, 2048, 22)]


def batched_bytes(B, M, N, K):
    return B * affine_bytes(M, N, K)


def build_batched(torch, g4, dev, seed=7):
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    bf = torch.bfloat16
    out = []
    for (B, K, N, M) in BATCHED_SHAPES:
        w = torch.randn((B * N, K), generator=gen, device=dev, dtype=torch.float32) * 0.02
        p, s, b = g4.gai4_quantize(w, BITS, GS, bf)
        del w
        p, s, b = p.view(B, N, -1), s.view(B, N, -1), b.view(B, N, -1)
        base = torch.randn((B * M * (K + 8) + 16,), generator=gen, device=dev).to(bf)
        x = torch.as_strided(base, (B, M, K), (M * (K + 8), K + 8, 1), 1)
        ws_n = g4.gai4_qmm_t_batched_workspace_bytes(B, M, N, K, BITS, GS, bf, 0)
        ws = torch.empty(max(ws_n, 16) // 4 + 64, dtype=torch.float32, device=dev)
        out.append(dict(kind="qmm_t_batched", p=p, s=s, b=b, x=x, out=torch.empty((B, M, N), dtype=bf, device=dev),
                        ws=ws, B=B, M=M, N=N, K=K, bytes=batched_bytes(B, M, N, K)))
    torch.cuda.synchronize()
    return out


# large-M (prefill) qmm_t, measured beside the step (not part of it): (K, N, M);
# 4096x4096 at M=512 is tensor-bound (about 400 flop per byte), 14336x4096 at
# M=2048 more so
PREFILL_SHAPES = [(4096, 4096, 512), (4096, 14336, 2048)]


def build_prefill(torch, g4, dev, seed=11):
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    bf = torch.bfloat16
    out = []
    for (K, N, M) in PREFILL_SHAPES:
        w = torch.randn((N, K), generator=gen, device=dev, dtype=torch.float32) * 0.02
        p, s, b = g4.gai4_quantize(w, BITS, GS, bf)
        del w
        x = torch.randn((M, K), generator=gen, device=dev).to(bf)
        ws = g4.gai4_qmm_t_workspace_bytes(M, N, K, BITS, GS, bf, 0)
        wsp = torch.empty(max(ws, 16) // 4 + 4, dtype=torch.float32, device=dev)
        out.append(dict(kind="qmm_t", p=p, s=s, b=b, x=x, out=torch.empty((M, N), dtype=bf, device=dev), ws=wsp,
                        M=M, N=N, K=K, bytes=affine_bytes(M, N, K)))
    torch.cuda.synchronize()
    return out


def q8_i8_bytes(N, K):
    return N * (K // 32) * 36 + K + (K // 32) * 4 + N * 4


def build_q8_i8(torch, g4, dev):
    """Q8_0 with integer activations (x quantized on the GPU once, outside the timing)."""
    import synth
    out = []
    for i, (N, K) in enumerate(BLOCKQ_SHAPES):
        blk = torch.from_numpy(synth.q8_0_blocks(N, K, 300 + i).view(np.int32)).to(dev)
        xq, xd = g4.gai4_quantize_x_q8(torch.from_numpy(synth.f32_vector(K, 301 + i)).to(dev))
        out.append(dict(kind="q8_0_i8", blocks=blk, xq=xq, xd=xd, out=torch.empty(N, device=dev), N=N, K=K,
                        bytes=q8_i8_bytes(N, K)))
    torch.cuda.synchronize()
    return out


def gguf_bytes(kind, N, K):
    blk = N * (K // 32) * 34 if kind == "q8_0_34b" else N * (K // 256) * 210
    return blk + 4 * K + 4 * N


def build_gguf(torch, g4, dev):
    """GGUF's 34-byte Q8_0 blocks and Q6_K super-blocks (f32 activations),
    measured beside the step at the Q8_0 / Q4_K shapes."""
    import synth
    out = []
    for i, (N, K) in enumerate(BLOCKQ_SHAPES):
        x = torch.from_numpy(synth.f32_vector(K, 311 + i)).to(dev)
        for kind, gen in (("q8_0_34b", synth.q8_0_34b_blocks), ("q6_k", synth.q6_k_blocks)):
            blk = torch.from_numpy(gen(N, K, 312 + i)).to(dev)
            out.append(dict(kind=kind, blocks=blk, x=x, out=torch.empty(N, device=dev), N=N, K=K,
                            bytes=gguf_bytes(kind, N, K)))
    torch.cuda.synchronize()
    return out


# the other activation dtypes of the qmv shapes, and the bit-width / group-size
# / M sweep at 4096^2: measured per call beside the step (not part of it)
SWEEP_QMV_SHAPES = [(5120, 5120), (14336, 5120), (5120, 14336), (27648, 5120)]   # (N, K)
SWEEP_BITS, SWEEP_GS, SWEEP_M = [2, 3, 4, 6, 8], [32, 64, 128], [1, 8, 64]


def affine_bytes_g(M, N, K, bits, gs, tbytes):
    return N * K * bits // 8 + 2 * N * (K // gs) * tbytes + M * K * tbytes + M * N * tbytes


def build_sweep(torch, g4, dev, seed=13):
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    calls = []

    def add(M, N, K, bits, gs, T, tag):
        w = torch.randn((N, K), generator=gen, device=dev, dtype=torch.float32) * 0.02
        p, s, b = g4.gai4_quantize(w, bits, gs, T)
        del w
        tb = torch.empty((), dtype=T).element_size()
        x = torch.randn((K,) if M == 1 else (M, K), generator=gen, device=dev).to(T)
        c = dict(kind="qmv" if M == 1 else "qmm_t", p=p, s=s, b=b, x=x,
                 out=torch.empty((N,) if M == 1 else (M, N), dtype=T, device=dev), M=M, N=N, K=K, bits=bits, gs=gs,
                 dtype=str(T).replace("torch.", ""), tag=tag, bytes=affine_bytes_g(M, N, K, bits, gs, tb))
        if M > 1:
            ws = g4.gai4_qmm_t_workspace_bytes(M, N, K, bits, gs, T, 0)
            c["ws"] = torch.empty(max(ws, 16) // 4 + 4, dtype=torch.float32, device=dev)
        calls.append(c)

    for T in (torch.float16, torch.float32):
        for (N, K) in SWEEP_QMV_SHAPES:
            add(1, N, K, BITS, GS, T, "qmv dtypes")
    for bits in SWEEP_BITS:
        for gs in SWEEP_GS:
            for M in SWEEP_M:
                add(M, 4096, 4096, bits, gs, torch.bfloat16, "bits x group size x M, 4096^2")
    torch.cuda.synchronize()
    return calls


def time_sweep(torch, g4, dev, stream):
    calls = build_sweep(torch, g4, dev)
    with torch.cuda.stream(stream):   # one eager call each: first-use kernel set-up outside graph capture
        for c in calls:
            issue(g4, c)
    stream.synchronize()
    recs = time_per_call(torch, g4, {"sweep": calls}, stream, ["sweep"])
    for r, c in zip(recs, calls):
        r.update({"set": c["tag"], "dtype": c["dtype"], "bits": c["bits"], "gs": c["gs"], "M": c["M"]})
    del calls
    return recs


def build_workload(torch, g4, dev, seed=0, only=None):
    """Seeded synthetic inputs on the device: W ~ N(0, 0.02) quantized on the
    GPU (4-bit, gs 64, bf16 scales/biases), x ~ N(0, 1) bf16, Q8_0 / Q4_K
    blocks from the shared seeded generators."""
    import synth
    # profiling runs of the calls measured beside the step: --only
    # prefill|gguf|q8_0_i8|batched|sweep[:INDEX]
    extra = {"prefill": build_prefill, "gguf": build_gguf, "q8_0_i8": build_q8_i8, "batched": build_batched,
             "sweep": build_sweep}
    if only and only.partition(":")[0] in extra:
        fam, _, idx = only.partition(":")
        cs = extra[fam](torch, g4, dev)
        return {fam: cs if idx == "" else [cs[int(idx)]]}
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    bf = torch.bfloat16
    calls = {"qmv": [], "qmm_t": [], "q8_0": [], "q4_k": []}

    def qweights(N, K):
        w = torch.randn((N, K), generator=gen, device=dev, dtype=torch.float32) * 0.02
        p, s, b = g4.gai4_quantize(w, BITS, GS, bf)
        del w
        return p, s, b

    for i, (N, K) in enumerate(QMV_SHAPES):
        if not selected(only, "qmv", i):
            continue
        p, s, b = qweights(N, K)
        x = torch.randn((K,), generator=gen, device=dev).to(bf)
        out = torch.empty((N,), dtype=bf, device=dev)
        calls["qmv"].append(dict(kind="qmv", p=p, s=s, b=b, x=x, out=out, M=1, N=N, K=K,
                                 bytes=affine_bytes(1, N, K)))
    for i, (K, N, M) in enumerate(QMM_SHAPES):
        if not selected(only, "qmm_t", i):
            continue
        p, s, b = qweights(N, K)
        x = torch.randn((M, K), generator=gen, device=dev).to(bf)
        out = torch.empty((M, N), dtype=bf, device=dev)
        ws = g4.gai4_qmm_t_workspace_bytes(M, N, K, BITS, GS, bf, 0)
        wsp = torch.empty(max(ws, 16) // 4 + 4, dtype=torch.float32, device=dev)
        calls["qmm_t"].append(dict(kind="qmm_t", p=p, s=s, b=b, x=x, out=out, ws=wsp, M=M, N=N, K=K,
                                   bytes=affine_bytes(M, N, K)))
    for i, (N, K) in enumerate(BLOCKQ_SHAPES):
        if selected(only, "q8_0", i):
            blk8 = torch.from_numpy(synth.q8_0_blocks(N, K, 300 + i).view(np.int32)).to(dev)
            x8 = torch.from_numpy(synth.f32_vector(K, 301 + i)).to(dev)
            calls["q8_0"].append(dict(kind="q8_0", blocks=blk8, x=x8, out=torch.empty(N, device=dev), N=N, K=K,
                                      bytes=q8_bytes(N, K)))
        if selected(only, "q4_k", i):
            blk4 = torch.from_numpy(synth.q4_k_blocks(N, K, 302 + i)).to(dev)
            x4 = torch.from_numpy(synth.f32_vector(K, 303 + i)).to(dev)
            calls["q4_k"].append(dict(kind="q4_k", blocks=blk4, x=x4, out=torch.empty(N, device=dev), N=N, K=K,
                                      bytes=q4k_bytes(N, K)))
    torch.cuda.synchronize()
    return {f: cs for f, cs in calls.items() if cs}


def issue(g4, c):
    k = c["kind"]
    if k == "qmv":
        g4.gai4_qmv(c["p"], c["s"], c["b"], c["x"], out=c["out"], bits=c.get("bits", BITS),
                    group_size=c.get("gs", GS))
    elif k == "qmm_t":
        g4.gai4_qmm_t(c["p"], c["s"], c["b"], c["x"], out=c["out"], bits=c.get("bits", BITS),
                      group_size=c.get("gs", GS), split_k=0, workspace=c["ws"])
    elif k == "qmm_t_batched":
        g4.gai4_qmm_t_batched(c["p"], c["s"], c["b"], c["x"], out=c["out"], bits=BITS, group_size=GS, split_k=0,
                              workspace=c["ws"])
    elif k == "q8_0_i8":
        g4.gai4_q8_0_gemv_i8(c["blocks"], c["xq"], c["xd"], out=c["out"])
    elif k == "q8_0":
        g4.gai4_q8_0_gemv(c["blocks"], c["x"], out=c["out"])
    elif k == "q8_0_34b":
        g4.gai4_q8_0_34b_gemv(c["blocks"], c["x"], out=c["out"])
    elif k == "q6_k":
        g4.gai4_q6_k_gemv(c["blocks"], c["x"], out=c["out"])
    else:
        g4.gai4_q4_k_gemv(c["blocks"], c["x"], out=c["out"])


def kernel_launches_per_step(g4, calls, torch):
    n = 0
    for fam, cs in calls.items():
        for c in cs:
            if fam == "qmm_t":
                path, splits = g4.gai4_qmm_t_plan(c["M"], c["N"], c["K"], BITS, GS, torch.bfloat16, 0,
                                                  c["ws"].numel() * 4)
                n += 2 if splits > 1 else 1
            else:
                n += 1
    return n


def inner_reps(torch, stream, one_step, K, args):
    """Replays of the step per timed step: --inner if given, else enough that
    the K timed steps span at least --min-timed-s seconds (estimated from a few
    untimed replays), so that the clock sampler sees the timed region."""
    if args.inner > 0:
        return args.inner
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n = 10
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n):
            one_step()
        e1.record(stream)
    stream.synchronize()
    step_ms = max(e0.elapsed_time(e1) / n, 1e-3)
    return max(1, int(math.ceil(args.min_timed_s * 1e3 / (max(K, 1) * step_ms))))


def max_over_ranks(torch, dist, x, device):
    """The slowest rank's value (every rank gets it): the job's step time."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, bytes_per_rank_step, ms_per_step):
    """Whole-job GB/s: every replica moves the same step bytes (weak scaling),
    and the job's step takes the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def run_gpu(args, rank, world, local_rank):
    import torch
    import gemm_affine_int4_gb300 as g4

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    g4.lib()
    calls = build_workload(torch, g4, dev, only=args.only)
    fam_bytes = {f: sum(c["bytes"] for c in cs) for f, cs in calls.items()}
    total_bytes = sum(fam_bytes.values())
    stream = torch.cuda.Stream(device=dev)

    # eager warm-up (lazy library set-up happens outside any capture)
    with torch.cuda.stream(stream):
        for cs in calls.values():
            for c in cs:
                issue(g4, c)
    stream.synchronize()
    st = g4.gai4_last_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    # one CUDA graph per kernel family
    graphs = {}
    for fam, cs in calls.items():
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for c in cs:
                issue(g4, c)
        graphs[fam] = gr
    fams = list(calls)
    # the step: every call of every family, in order, in one CUDA graph (the
    # timed unit; kernels of consecutive calls overlap launch and set-up)
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=stream):
        for fam in fams:
            for c in calls[fam]:
                issue(g4, c)

    def one_step():
        step_graph.replay()

    def family_pass(evs):
        # the per-family breakdown: each family's graph between two events
        for i, fam in enumerate(fams):
            evs[i][0].record(stream)
            graphs[fam].replay()
            evs[i][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
            family_pass([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                         for _ in fams])
    stream.synchronize()

    dist = None
    if world > 1:
        import torch.distributed as dist
    K = args.steps
    reps = inner_reps(torch, stream, one_step, K, args)
    if world > 1:   # every rank replays the same number of steps
        reps = int(max_over_ranks(torch, dist, reps, dev))
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in fams]
          for _ in range(K)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else str(local_rank))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for k in range(K):
            for _ in range(reps):
                one_step()
        t1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    steps_total = K * reps
    # per-family breakdown, after the timed region (same inputs, same number of passes)
    with torch.cuda.stream(stream):
        for k in range(K):
            family_pass(ev[k])
    stream.synchronize()
    fam_ms = {fam: sum(ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(K)) / K for i, fam in enumerate(fams)}
    st = g4.gai4_last_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")

    per_call = None if args.no_per_call else time_per_call(torch, g4, calls, stream, fams)
    # batched / strided qmm_t beside the step (same cold-L2 per-call timing)
    extra = extra_i8 = extra_pf = extra_gg = None
    if not args.no_per_call and not args.only:
        bcalls = build_batched(torch, g4, dev)
        extra = time_per_call(torch, g4, {"qmm_t_batched": bcalls}, stream, ["qmm_t_batched"])
        icalls = build_q8_i8(torch, g4, dev)
        extra_i8 = time_per_call(torch, g4, {"q8_0_i8": icalls}, stream, ["q8_0_i8"])
        gcalls = build_gguf(torch, g4, dev)
        extra_gg = time_per_call(torch, g4, {"gguf": gcalls}, stream, ["gguf"])
        del gcalls
        pcalls = build_prefill(torch, g4, dev)
        extra_pf = time_per_call(torch, g4, {"prefill": pcalls}, stream, ["prefill"])
        del pcalls

    # end to end through the public API: per step, H2D of every call's
    # activations from pinned host memory, the calls, D2H of every output
    e2e = None if args.no_e2e else run_e2e(torch, g4, calls, stream, args)

    ms_per_step = elapsed_ms / steps_total
    if world > 1:
        ms_per_step = max_over_ranks(torch, dist, ms_per_step, dev)
    value = job_throughput(world, total_bytes, ms_per_step)

    hbm, tflops, peak_src = load_peaks()
    dom = max(fam_ms, key=fam_ms.get)
    dom_ms = fam_ms[dom]
    n_launch = len(calls[dom])
    achieved = fam_bytes[dom] / (dom_ms * 1e-3) / 1e9
    traffic = recorded_traffic(dom, fam_bytes[dom])
    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 activations, 4-bit weights, fp32 accumulate (f32 activations for Q8_0/Q4_K)",
        "data": "synthetic (seeded; W~N(0,0.02) quantized on the GPU, x~N(0,1))",
        "config": {
            "workload": "one pass of the hot path: qmv 4-bit gs64 bf16 x5 shapes (4096^2..27648x5120); "
                        "qmm_t 4-bit gs64 bf16 split-K (KxN,M) 2048x2048/22, 4096x4096/16, 10752x2048/85, "
                        "14336x4096/33, 17408x5120/56, 5120x17408/28, 256x4096/40, 4096x4096/8; "
                        "Q8_0 and Q4_K GEMV 4096x4096 and 14336x5120 (f32 x)",
            "bytes_per_step": total_bytes, "calls_per_step": sum(len(v) for v in calls.values()),
            "l2": "no flush: %.0f MB of distinct weights per step > 129 MB L2" % (total_bytes / 1e6),
            "timing": "the step is one CUDA graph (kernels chained by programmatic dependent launch), "
                      "CUDA events on the launching stream; the breakdown replays one graph per family",
            "replays_per_timed_step": reps, "timed_region_s": round(elapsed_ms / 1e3, 3),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "breakdown": {fam: {"ms": round(fam_ms[fam], 5), "GB/s": round(fam_bytes[fam] / (fam_ms[fam] * 1e-3) / 1e9, 1),
                            "frac_of_hbm": round(fam_bytes[fam] / (fam_ms[fam] * 1e-3) / 1e9 / hbm, 3),
                            "bytes": fam_bytes[fam]} for fam in fams},
        "roofline": {"kernel": {"qmv": "qmv4_kernel (qmv, M=1)",
                                "qmm_t": "qmm_t family (qmm_tc_kernel + splitk_reduce)",
                                "q8_0": "q8_0_tma_kernel", "q4_k": "q4_k_tma_kernel"}.get(dom, dom),
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": f"{peak_src} hbm_gbs",
                     "launches_per_step": n_launch,
                     "algorithmic_bytes_per_launch": round(fam_bytes[dom] / n_launch),
                     "avg_launch_us": round(dom_ms * 1e3 / n_launch, 3),
                     "traffic": None if traffic is None else round(traffic / n_launch)},
        "per_call_cold_l2": per_call,
        "batched_cold_l2": extra,
        "q8_0_int8_activations_cold_l2": extra_i8,
        "prefill_qmm_t_cold_l2": extra_pf,
        "gguf_blocks_cold_l2": extra_gg,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": kernel_launches_per_step(g4, calls, torch) * steps_total,
    }
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if not args.no_per_call and not args.only:
        # last, and guarded: a measurement beside the step never costs the step's line
        try:
            res["sweep_cold_l2"] = time_sweep(torch, g4, dev, stream)
        except Exception as e:
            res["sweep_cold_l2"] = {"error": f"{type(e).__name__}: {e}"[:300]}
    return res


def call_name(c):
    if c["kind"] == "q8_0_i8":
        return f"q8_0 int8 activations N{c['N']}xK{c['K']}"
    if c["kind"] == "qmm_t_batched":
        return f"qmm_t batched {c['B']}x (K{c['K']}xN{c['N']} M={c['M']}), strided odd-offset x"
    if c["kind"] == "qmm_t":
        return f"qmm_t K{c['K']}xN{c['N']} M={c['M']}"
    return f"{c['kind']} N{c['N']}xK{c['K']}"


def time_per_call(torch, g4, calls, stream, fams, reps=8):
    """Each call alone with a cold L2: a graph of `reps` x [overwrite a 256 MB
    buffer, the call] minus a graph of `reps` x [overwrite] (the same flushes),
    divided by `reps`: the call's own time, without graph-launch latency.
    Reported beside the step timing."""
    hbm, tflops, _ = load_peaks()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=stream.device)

    def graph_us(body):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for r in range(reps):
                body(r)
        best = None
        with torch.cuda.stream(stream):
            gr.replay()
        for _ in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                gr.replay()
                e1.record(stream)
            stream.synchronize()
            t = e0.elapsed_time(e1) * 1e3
            best = t if best is None else min(best, t)
        return best

    flush_only = graph_us(lambda r: flush.fill_(float(r)))
    out = []
    for fam in fams:
        for c in calls[fam]:
            def body(r, c=c):
                flush.fill_(float(r))
                issue(g4, c)
            us = max((graph_us(body) - flush_only) / reps, 1e-3)
            gbs = c["bytes"] / (us * 1e-6) / 1e9
            rec = {"call": call_name(c), "us": round(us, 3), "GB/s": round(gbs, 1),
                   "frac_of_hbm": round(gbs / hbm, 3)}
            if c["kind"] in ("qmm_t", "qmm_t_batched"):
                # min(HBM, tensor) roofline: the call cannot beat the larger of
                # its byte time and its bf16 tensor-core time
                flops = 2.0 * c.get("B", 1) * c["M"] * c["N"] * c["K"]
                hbm_us, tc_us = c["bytes"] / (hbm * 1e9) * 1e6, flops / (tflops * 1e12) * 1e6
                rec.update({"TFLOP/s": round(flops / (us * 1e-6) / 1e12, 2),
                            "bound": "tensor" if tc_us > hbm_us else "hbm",
                            "frac_of_roofline": round(max(hbm_us, tc_us) / us, 3)})
            out.append(rec)
    del flush
    return out


def run_e2e(torch, g4, calls, stream, args):
    """Same workload through the public calls with host buffers. Every call's
    activations sit in one pinned host buffer and its output lands in another
    (256-byte aligned views, in call order). The first family's activations
    are copied in first; the rest follow in one copy on a copy stream while
    the first family runs (joined before its last call), and each family's
    outputs are copied back on a second copy stream as soon as the family is
    done. Copies and calls are
    captured in one CUDA graph (the copy streams forked from and joined back
    into the launching stream), replayed per step, inside the timed region."""
    order = [c for cs in calls.values() for c in cs]
    dev = order[0]["x"].device

    def layout(ts, align=256):   # 256-byte aligned offsets in a packed buffer
        offs, off = [], 0
        for t in ts:
            offs.append(off)
            off += (t.numel() * t.element_size() + align - 1) // align * align
        return offs, off

    in_offs, in_total = layout([c["x"] for c in order])
    out_offs, out_total = layout([c["out"] for c in order])
    dev_in = torch.empty(in_total, dtype=torch.uint8, device=dev)
    dev_out = torch.empty(out_total, dtype=torch.uint8, device=dev)
    host_in = torch.zeros(in_total, dtype=torch.uint8, pin_memory=True)
    host_out = torch.empty(out_total, dtype=torch.uint8, pin_memory=True)

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    packed_calls = []
    for c, oi, oo in zip(order, in_offs, out_offs):
        view(host_in, oi, c["x"]).copy_(c["x"].cpu())
        packed_calls.append(dict(c, x=view(dev_in, oi, c["x"]), out=view(dev_out, oo, c["out"])))
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    fam_of = [f for f, cs in calls.items() for _ in cs]
    n_first = fam_of.count(fam_of[0])          # calls of the first family
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream):
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        ready = []
        with torch.cuda.stream(s_in):
            for lo, hi in ((0, n_first), (n_first, len(order))):
                if lo < hi:
                    a, b = in_offs[lo], (in_offs[hi] if hi < len(order) else in_total)
                    dev_in[a:b].copy_(host_in[a:b], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(s_in)
                ready.append(ev)
        first_out = 0
        # the later families' activations are joined before the first
        # family's last call (its completion, which the next call waits for,
        # then covers the copy), so that the kernel-to-kernel edge into the
        # second family stays a programmatic one
        join_rest = n_first - 1 if n_first > 1 else n_first
        for i, c in enumerate(packed_calls):
            if i == 0:
                stream.wait_event(ready[0])
            if i == join_rest and n_first < len(order):
                stream.wait_event(ready[1])
            issue(g4, c)
            last_of_family = i + 1 == len(order) or fam_of[i + 1] != fam_of[i]
            if last_of_family:
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                a, b = out_offs[first_out], (out_offs[i + 1] if i + 1 < len(order) else out_total)
                with torch.cuda.stream(s_out):
                    host_out[a:b].copy_(dev_out[a:b], non_blocking=True)
                first_out = i + 1
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)
    with torch.cuda.stream(stream):
        for _ in range(3):
            gr.replay()
    stream.synchronize()
    K = max(args.steps, 1)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(K):
            gr.replay()
        t1.record(stream)
    stream.synchronize()
    ms = t0.elapsed_time(t1) / K
    total = sum(c["bytes"] for c in order)
    # the step's outputs came back: compare one against the device result
    c0, o0 = order[-1], out_offs[-1]
    if not torch.equal(view(host_out, o0, c0["out"]), packed_calls[-1]["out"].cpu()):
        raise RuntimeError("end-to-end output copy does not match the device result")
    return {"value": round(total / (ms * 1e-3) / 1e9, 1), "unit": UNIT, "h2d_bytes_per_step": in_total,
            "d2h_bytes_per_step": out_total, "ms_per_step": round(ms, 5),
            "copies_per_step": 2 + len(calls),
            "copy_overlap": "input copies ahead of the calls on one copy stream, family outputs back on another"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def _oracle_work(fraction):
    """The oracle on a sample of the step: every call of the step, restricted
    to a deterministic subset of its output rows (all x rows). Each item is
    (oracle call, rows, bytes, the plain binary32 loop on the same inputs)."""
    import oracle
    import synth
    items = []
    for i, (N, K) in enumerate(QMV_SHAPES):
        items.append(("affine", 1, N, K, i))
    for i, (K, N, M) in enumerate(QMM_SHAPES):
        items.append(("affine", M, N, K, 100 + i))
    for i, (N, K) in enumerate(BLOCKQ_SHAPES):
        items.append(("q8_0", 1, N, K, 300 + i))
        items.append(("q4_k", 1, N, K, 302 + i))
    prepared = []
    for kind, M, N, K, seed in items:
        nr = max(8, int(round(N * fraction)))
        rows = np.linspace(0, N - 1, nr).astype(np.int64)
        if kind == "affine":
            W = synth.affine_weights(nr, K, seed)      # the sampled rows' weights
            packed, s, b = oracle.quantize(W, BITS, GS, "bf16")
            x = synth.activations(M, K, "bf16", seed + 1)

            def f64(rows, p=packed, s_=s, b_=b, x_=x):
                return oracle.qmm(p, s_, b_, x_, BITS, GS, "bf16", rows=rows)

            def f32(rows, p=packed, s_=s, b_=b, x_=x):
                return oracle.qmm_f32loop(p, s_, b_, x_, BITS, GS, "bf16", rows=rows)
            prepared.append((f64, nr, affine_bytes(M, N, K) * nr / N, f32))
        else:
            gen = synth.q8_0_blocks if kind == "q8_0" else synth.q4_k_blocks
            ref = oracle.q8_0_gemv if kind == "q8_0" else oracle.q4_k_gemv
            loop = oracle.q8_0_gemv_f32loop if kind == "q8_0" else oracle.q4_k_gemv_f32loop
            blk = gen(nr, K, seed)
            x = synth.f32_vector(K, seed + 1)

            def f64(rows, b_=blk, x_=x, f=ref):
                return f(b_, x_, rows=rows)

            def f32(rows, b_=blk, x_=x, f=loop):
                return f(b_, x_, rows=rows)
            byt = (q8_bytes(N, K) if kind == "q8_0" else q4k_bytes(N, K)) * nr / N
            prepared.append((f64, nr, byt, f32))
    return prepared


def _run_work(work, threads):
    """Run every sampled call once: on one thread, or split into row ranges
    over `threads` host threads (the C oracle releases the GIL while it runs)."""
    if threads <= 1:
        for w in work:
            w[0](None)
        return
    from concurrent.futures import ThreadPoolExecutor
    tasks = []
    for w in work:
        fn, nr = w[0], w[1]
        chunk = max(1, -(-nr // (4 * threads)))
        for a in range(0, nr, chunk):
            tasks.append((fn, np.arange(a, min(nr, a + chunk), dtype=np.int64)))
    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(lambda t: t[0](t[1]), tasks))


def _timed_sample(target_s, threads, max_frac=1.0):
    """A sample of the step sized to about target_s seconds on `threads`
    threads (at most max_frac of the rows: preparing the sample's inputs costs
    more than running it): (bytes, seconds, fraction of output rows, work)."""
    frac = 1.0 / 512
    for _ in range(4):   # grow the sample until it takes at least half the target time
        work = _oracle_work(frac)
        byt = sum(w[2] for w in work)
        t = time.perf_counter()
        _run_work(work, threads)
        dt = time.perf_counter() - t
        if dt >= 0.5 * target_s or frac >= max_frac:
            break
        frac = min(max_frac, frac * min(16.0, max(1.5, target_s / max(dt, 1e-3))))
    return byt, dt, frac, work


def host_threads():
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))


def cpu_baseline(target_s=12.0):
    """Time the oracle (binary64, as it stands) on a bounded sample of the
    step, on all host cores (row ranges over threads) and on one thread."""
    threads = host_threads()
    # one sample, sized for a single thread, timed on one thread and on all
    byt, dt1, frac, work = _timed_sample(target_s * 0.7, 1)
    t = time.perf_counter()
    _run_work(work, threads)
    dt = time.perf_counter() - t
    # the plain binary32 loops on the same rows (the "reasonable CPU" number)
    work32 = [(w[3], w[1], w[2]) for w in work]
    t = time.perf_counter()
    _run_work(work32, threads)
    dt32 = time.perf_counter() - t
    return {"value": round(byt / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"every call of the step on {frac:.4%} of its output rows (all x rows), binary64 C oracle, "
                      f"row ranges over {threads} threads, {dt:.1f} s",
            "single_thread": {"value": round(byt / dt1 / 1e9, 4), "cores": 1, "sample": f"the same rows, {dt1:.1f} s"},
            "fp32_loop": {"value": round(byt / dt32 / 1e9, 4), "cores": threads, "kind": "plain binary32 C loops",
                          "sample": f"the same rows, row ranges over {threads} threads, {dt32:.1f} s"}}


def run_reference(args):
    """The reference arm: the oracle, as it stands, on the step (a bounded
    sample of every call's output rows), on all host cores."""
    threads = host_threads()
    target = max(2.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    _, _, frac, work = _timed_sample(target, threads, max_frac=0.25)
    byt = sum(w[2] for w in work)
    steps, byt_total, t_total = [], 0.0, 0.0
    for i in range(args.warmup + args.steps):
        t = time.perf_counter()
        _run_work(work, threads)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            steps.append(dt)
            byt_total += byt
            t_total += dt
    value = byt_total / t_total / 1e9
    ms = 1e3 * t_total / max(1, len(steps))
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded)",
            "config": {"workload": "the same step as the GPU arm, each call restricted to "
                                   f"{frac:.4%} of its output rows"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{frac:.4%} of output rows of every call, row ranges over {threads} threads"},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--inner", type=int, default=0,
                    help="step replays per timed step (0: enough for --min-timed-s seconds in all)")
    ap.add_argument("--min-timed-s", type=float, default=1.0)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", default=None, help="FAMILY[:INDEX]: time one kernel family / call (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-call", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
