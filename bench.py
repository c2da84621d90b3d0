"""Benchmark of the MXFP4 linear layer (fused bf16 -> MXFP4 quantize + GEMM).

One step = one call of the fused entry (mxfp4_quant_gemm) on one activation
batch: A bf16 [M, K] quantized in-kernel, times a pre-packed MXFP4 weight
[N, K], bf16 C [M, N] out.  The headline workload is M=32, N=4096, K=512.

Timing: a CUDA graph of R calls, call i on copy i % R of both A and the packed
weight, with R chosen so that the copies exceed twice the L2 cache (every call
streams its operands from HBM); the graph is replayed until exactly K steps
ran, bracketed by CUDA events on the replay stream, with an L2-sized write
enqueued just before the start event.  Per shape, beside this pipelined
figure: the same calls without overlap between consecutive calls (a lone
call's latency) and the per-layer time of a dependent chain of layers.
Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "µs/call and % of roofline (HBM GB/s or FP4 TFLOPS) per MXFP4 GEMM shape"
UNIT = "us/call"
# The pages' published per-call time for the headline shape (MI355X, end to end
# including Python dispatch; submission 733989's benchmark table).
PAGES_US = {"m32_n4096_k512": 10.6, "m4_n2880_k512": 9.7, "m16_n2112_k7168": 20.9,
            "m32_n2880_k512": 11.3, "m64_n7168_k2048": 17.5, "m256_n3072_k1536": 16.2}
DENSE_FP4_TFLOPS_NOMINAL = 13500.0  # GB300 dense FP4 (no sparsity), nominal


# ----------------------------------------------------------------------------- helpers
def algorithmic_bytes(M: int, N: int, K: int, fused: bool = True) -> int:
    """Each operand once: A (bf16 for the fused entry, codes+scales otherwise),
    weight codes + scales, bf16 C."""
    a = 2 * M * K if fused else M * K // 2 + M * K // 32
    return a + N * K // 2 + N * K // 32 + 2 * M * N


def flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def source_hash() -> str:
    """Hash of the CUDA sources' code: comments and whitespace are left out, so
    a comment edit does not void counters taken on the same code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_scaled_mxfp4_activation_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            code = re.sub(r"/\*.*?\*/", " ", fh.read(), flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(f.encode() + " ".join(code.split()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch of the GEMM kernel from the committed ncu summary,
    or None when the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- our arm
ALL_WORKLOADS = {**workloads.WORKLOADS, **workloads.EXTRA_WORKLOADS}

L2_METHOD = ("each timed pass streams rotating copies of A and the packed weight totalling more than 2x L2, and an "
             "L2-sized write precedes the timed region")


def bench_config(w: workloads.Workload) -> dict:
    """The `config` of both arms' JSON lines for one workload (one dict, so the
    two arms' lines compare equal)."""
    return {"workload": f"{w.name}: fused bf16->MXFP4 quantize + block-scaled MXFP4 GEMM, bf16 out, {w.label}",
            "M": w.M, "N": w.N, "K": w.K, "seed": w.seed, "l2": L2_METHOD}


class Problem:
    """R rotating copies of A and of the packed weight for one workload."""

    def __init__(self, w: workloads.Workload, device: torch.device, copies: int | None = None):
        import block_scaled_mxfp4_activation_gb300 as mx

        self.mx, self.w = mx, w
        A, B = workloads.make_inputs(w)
        W0 = mx.quantize_weights(B.to(device))
        per_copy = W0.data.numel() + 2 * w.M * w.K + 2 * w.M * w.N
        l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20))
        self.copies = copies or max(2, math.ceil(2 * l2 / per_copy))
        self.W = [W0] + [mx.PackedWeight(W0.data.clone(), w.N, w.K) for _ in range(self.copies - 1)]
        A_dev = A.to(device)
        self.A = [A_dev] + [A_dev.clone() for _ in range(self.copies - 1)]
        self.C = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device) for _ in range(self.copies)]
        # one workspace for every call: calls on a stream are ordered, and the
        # quantize pass of a call waits for the previous GEMM before writing it
        self.ws = torch.empty(max(mx.workspace_bytes(w.M, w.N, w.K), 1), dtype=torch.uint8, device=device)
        self.rotating_bytes = per_copy * self.copies
        self.l2 = l2
        self.launches_per_call = 2 if mx.gemm_plan(w.M, w.N, w.K, fused=True)["two_pass"] else 1
        self.flush = torch.empty(2 * l2, dtype=torch.uint8, device=device)

    def call(self, i: int):
        j = i % self.copies
        self.mx.quant_gemm(self.A[j], self.W[j], out=self.C[j], workspace=self.ws)

    def graph(self, n: int, stream: torch.cuda.Stream, first: int = 0, rotate: bool = True) -> torch.cuda.CUDAGraph:
        """n calls on copies first, first + 1, ... (or all on copy 0)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    self.call(first + i if rotate else 0)
        return g


class Chain:
    """A dependent chain of layers at one workload's shape: layer 2i maps
    [M, K] -> [M, N] with a weight [N, K], layer 2i+1 maps [M, N] -> [M, K]
    with a weight [K, N] (an up- and a down-projection), each layer's output
    the next layer's activation.  Every layer has its own weight copy, enough
    that the weights of one pass exceed 2x L2; weights ~ N(0, 1/fan_in) keep
    the activations' magnitude steady along the chain."""

    def __init__(self, w: workloads.Workload, device: torch.device):
        import block_scaled_mxfp4_activation_gb300 as mx

        self.mx, self.w = mx, w
        g = torch.Generator().manual_seed(w.seed + 77)
        up = (torch.randn((w.N, w.K), generator=g) / math.sqrt(w.K)).to(torch.bfloat16).to(device)
        down = (torch.randn((w.K, w.N), generator=g) / math.sqrt(w.N)).to(torch.bfloat16).to(device)
        Wu, Wd = mx.quantize_weights(up), mx.quantize_weights(down)
        l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 128 << 20))
        pairs = max(2, math.ceil(2 * l2 / (Wu.data.numel() + Wd.data.numel())))
        self.layers = []
        for _ in range(pairs):
            self.layers.append(mx.PackedWeight(Wu.data.clone(), w.N, w.K))
            self.layers.append(mx.PackedWeight(Wd.data.clone(), w.K, w.N))
        A = workloads.make_inputs(w)[0].to(device)
        self.x = A.clone()
        self.y = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
        nbytes = max(mx.workspace_bytes(w.M, w.N, w.K), mx.workspace_bytes(w.M, w.K, w.N), 1)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.flush = torch.empty(2 * l2, dtype=torch.uint8, device=device)

    def graph(self, stream: torch.cuda.Stream) -> torch.cuda.CUDAGraph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i, W in enumerate(self.layers):
                    src, dst = (self.x, self.y) if i % 2 == 0 else (self.y, self.x)
                    self.mx.quant_gemm(src, W, out=dst, workspace=self.ws)
        return g


class MultiLayer:
    """The same chain of layers as Chain, run through the multi-layer entry
    (mxfp4_quant_gemm_chain): launches of `per_launch` layers each, launch j's
    input the previous launch's last output."""

    def __init__(self, chain: Chain, per_launch: int = 16):
        mx, w = chain.mx, chain.w
        self.chain, self.mx = chain, mx
        L = chain.layers
        self.groups = [L[i:i + per_launch] for i in range(0, len(L) - len(L) % per_launch, per_launch)]
        Ns = [W.N for W in self.groups[0]]
        dev = chain.x.device
        self.outs = [torch.empty((w.M, n), dtype=torch.bfloat16, device=dev) for n in Ns]
        self.ws = torch.zeros(mx.chain_workspace_bytes(w.M, w.K, Ns), dtype=torch.uint8, device=dev)
        self.layers = per_launch * len(self.groups)

    def calls(self, stream):
        return [self.mx.prepare_quant_gemm_chain(self.chain.x if j == 0 else self.outs[-1], g, outs=self.outs,
                                                 workspace=self.ws, stream=stream)
                for j, g in enumerate(self.groups)]


def time_multilayer(ml: MultiLayer, stream: torch.cuda.Stream, reps: int = 3) -> tuple[float, float]:
    """(µs per layer graph-replayed, µs per layer with every launch issued from
    the host) of the multi-layer entry."""
    calls = ml.calls(stream)
    for c in calls:
        c()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c()
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    graphed = float(np.median([_timed(g.replay, ml.chain.flush, stream) for _ in range(reps)])) * 1e3 / ml.layers

    def eager():
        for c in calls:
            c()

    eager_us = float(np.median([_timed(eager, ml.chain.flush, stream) for _ in range(reps)])) * 1e3 / ml.layers
    return graphed, eager_us


def time_chain_eager(chain: Chain, stream: torch.cuda.Stream, reps: int = 3) -> float:
    """µs per layer of the dependent chain with every per-layer call issued from
    the host (prepared calls, no graph)."""
    calls = []
    for i, W in enumerate(chain.layers):
        src, dst = (chain.x, chain.y) if i % 2 == 0 else (chain.y, chain.x)
        calls.append(chain.mx.prepare_quant_gemm(src, W, out=dst, workspace=chain.ws, stream=stream))

    def eager():
        for c in calls:
            c()

    eager()
    torch.cuda.synchronize()
    return float(np.median([_timed(eager, chain.flush, stream) for _ in range(reps)])) * 1e3 / len(calls)


def aggregate_over_ranks(ms_local: float, steps: int, world: int) -> tuple[float, float]:
    """The job's time is the slowest rank's (all_reduce MAX over the process
    group when world > 1); the whole-job value is that time per call over all
    ranks' calls (every rank runs `steps` independent calls: replicas, weak
    scaling).  Returns (max ms, us per call for the whole job)."""
    times = torch.tensor([ms_local], dtype=torch.float64)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(times, op=dist.ReduceOp.MAX)
    ms_max = float(times[0])
    return ms_max, ms_max * 1e3 / (steps * world)


def _timed(replays, flush: torch.Tensor, stream: torch.cuda.Stream, barrier=None) -> float:
    """ms of `replays()` (graph replays enqueued on `stream`) between CUDA events
    on that stream.  An L2-sized write goes first: it leaves L2 holding none of
    the operands, and it keeps the GPU busy while the host enqueues the events
    and replays, so the timed region starts on the device with work queued."""
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    with torch.cuda.stream(stream):
        flush.fill_(1)
        start.record(stream)
        replays()
        end.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(end)


def time_graph_steps(prob: Problem, steps: int, warmup: int, stream: torch.cuda.Stream, rotate: bool = True,
                     barrier=None) -> float:
    """Exactly `steps` calls (graph replays), after `warmup` untimed calls on
    copies the timed calls do not start with (the last ones); returns ms."""
    R = prob.copies if rotate else 1
    chunk = min(steps, max(R, 256))
    full, rest = divmod(steps, chunk)
    g_full = prob.graph(chunk, stream, rotate=rotate)
    g_rest = prob.graph(rest, stream, first=chunk, rotate=rotate) if rest else None
    w = max(warmup, 1)
    g_warm = prob.graph(w, stream, first=R - (w % R) if rotate else 0, rotate=rotate)
    with torch.cuda.stream(stream):
        g_warm.replay()
    torch.cuda.synchronize()

    def replays():
        for _ in range(full):
            g_full.replay()
        if g_rest is not None:
            g_rest.replay()

    return _timed(replays, prob.flush, stream, barrier)


def time_chain(chain: Chain, stream: torch.cuda.Stream, reps: int = 3) -> float:
    """µs per layer of the dependent chain (median of `reps` timed passes after
    one untimed pass)."""
    g = chain.graph(stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    times = [_timed(g.replay, chain.flush, stream) for _ in range(reps)]
    return float(np.median(times)) * 1e3 / len(chain.layers)


def time_e2e(prob: Problem, steps: int, warmup: int, stream: torch.cuda.Stream, via: str = "c_abi") -> float:
    """Per step, one call of the host-buffer entry mxfp4_quant_gemm_host: pinned
    host A -> device, the fused layer, C -> pinned host (and C_dev).  Eager
    launches, no graph.  via="c_abi": the exported C function itself, called
    through ctypes with the step's arguments prepared once (the call a C or C++
    user makes); via="prepared": the Python wrapper's prepared call
    (prepare_quant_gemm_host, arguments checked once); via="python": the Python
    wrapper, which checks and marshals torch tensors on every call.  Returns ms."""
    w = prob.w
    hostA = prob.A[0].cpu().pin_memory()
    hostC = torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory()
    devA = torch.empty_like(prob.A[0])
    devC = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=devA.device)
    mx = prob.mx
    if via == "c_abi":
        fn = mx.load_library().mxfp4_quant_gemm_host
        args = [(hostA.data_ptr(), w.K, devA.data_ptr(), w.K, prob.W[j].data.data_ptr(), devC.data_ptr(),
                 hostC.data_ptr(), w.M, w.N, w.K, prob.ws.data_ptr(), prob.ws.numel(), int(stream.cuda_stream))
                for j in range(prob.copies)]

        def step(i):
            status = fn(*args[i % prob.copies])
            if status:
                raise mx.MXFP4Error(status, "mxfp4_quant_gemm_host")
    elif via == "prepared":
        calls = [mx.prepare_quant_gemm_host(hostA, prob.W[j], devA, devC, hostC, workspace=prob.ws, stream=stream)
                 for j in range(prob.copies)]

        def step(i):
            calls[i % prob.copies]()
    else:
        def step(i):
            mx.quant_gemm_host(hostA, prob.W[i % prob.copies], devA, devC, hostC, workspace=prob.ws, stream=stream)

    # warm-up: every copy once (the steady state of a loop that reuses its
    # buffers: each call's tensor maps come from the library's host-side cache)
    for i in range(max(warmup, prob.copies)):
        step(prob.copies - 1 - (i % prob.copies))
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def shape_report(name: str, us: float, peaks: dict, fused: bool = True) -> dict:
    w = ALL_WORKLOADS[name]
    b = algorithmic_bytes(w.M, w.N, w.K, fused)
    gbs = b / (us * 1e-6) / 1e9
    tflops = flops(w.M, w.N, w.K) / (us * 1e-6) / 1e12
    return {"us_per_call": round(us, 4), "bytes": b, "gbs": round(gbs, 1),
            "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "fp4_tflops": round(tflops, 2),
            "fp4_frac_nominal": round(tflops / DENSE_FP4_TFLOPS_NOMINAL, 5), "bound": "hbm"}


def cpu_baseline(name: str, budget_s: float = 12.0) -> dict:
    """The oracle (plain C, one thread, fp64) on a bounded sample of one call:
    the whole activation is quantized, then a fixed set of output elements is
    summed; the per-call time is scaled from the sampled elements to M*N."""
    import oracle

    w = workloads.WORKLOADS[name]
    A, B = workloads.make_inputs(w)
    bq, bs = oracle.quantize(B)
    rng = np.random.default_rng(0)
    t0 = time.perf_counter()
    aq, as_ = oracle.quantize(A)
    t_quant = time.perf_counter() - t0
    n_sample, spent, done = 256, 0.0, 0
    while spent < budget_s:
        ms = rng.integers(0, w.M, n_sample)
        ns = rng.integers(0, w.N, n_sample)
        t0 = time.perf_counter()
        oracle.gemm_sampled(aq, as_, bq, bs, ms, ns)
        spent += time.perf_counter() - t0
        done += n_sample
        n_sample = min(n_sample * 2, 1 << 16)
    per_elem = spent / done
    us = (t_quant + per_elem * w.M * w.N) * 1e6
    return {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle", "elements": done,
            "sample": f"{name}: one full A quantization + {done} randomly sampled output elements "
                      f"(of {w.M * w.N} per call; fp64, ascending k) in {spent:.1f} s, scaled to M*N"}


def _oracle_sampled_chunk(args) -> float:
    """Worker of cpu_baseline_all_cores: the oracle's sampled sum over one chunk
    of output elements (a separate process with its own copy of the oracle)."""
    aq, as_, bq, bs, ms, ns = args
    import oracle

    t0 = time.perf_counter()
    oracle.gemm_sampled(aq, as_, bq, bs, ms, ns)
    return time.perf_counter() - t0


def cpu_baseline_all_cores(name: str, per_core_elems: int, cores: int | None = None) -> dict:
    """The same oracle on every host core: one process per core (spawned, so
    none inherits the parent's CUDA state), each summing its own chunk of
    randomly sampled output elements; wall time scaled to M*N (plus the one
    activation quantization, which stays on one core)."""
    import multiprocessing as mp

    import oracle

    cores = cores or os.cpu_count() or 1
    w = workloads.WORKLOADS[name]
    A, B = workloads.make_inputs(w)
    bq, bs = oracle.quantize(B)
    t0 = time.perf_counter()
    aq, as_ = oracle.quantize(A)
    t_quant = time.perf_counter() - t0
    rng = np.random.default_rng(1)
    chunks = [(aq, as_, bq, bs, rng.integers(0, w.M, per_core_elems), rng.integers(0, w.N, per_core_elems))
              for _ in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        pool.map(_oracle_sampled_chunk, [(aq, as_, bq, bs, c[4][:16], c[5][:16]) for c in chunks])  # start-up
        t0 = time.perf_counter()
        pool.map(_oracle_sampled_chunk, chunks, chunksize=1)
        wall = time.perf_counter() - t0
    done = per_core_elems * cores
    us = (t_quant + wall * w.M * w.N / done) * 1e6
    return {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{name}: one full A quantization + {done} randomly sampled output elements in {cores} "
                      f"processes ({wall:.1f} s wall), scaled to M*N"}


def latency_report(w: workloads.Workload, prob: Problem, stream: torch.cuda.Stream, warmup: int, n: int) -> dict:
    """Beside the pipelined figure (independent calls, each overlapping the one
    before it): the same calls with no overlap (programmatic launch off: every
    call starts once the previous one has finished, the latency of a lone
    call), and the per-layer time of a dependent chain (each layer's output is
    the next layer's input), with overlap on and off."""
    mx = prob.mx
    out = {}
    try:
        mx.set_programmatic_launch(0)
        out["us_per_call_no_overlap"] = round(time_graph_steps(prob, n, warmup, stream) * 1e3 / n, 4)
        chain = Chain(w, prob.A[0].device)
        out["chain_us_per_layer_no_overlap"] = round(time_chain(chain, stream), 4)
        mx.set_programmatic_launch(3)
        out["chain_us_per_layer"] = round(time_chain(chain, stream), 4)
        out["chain_layers"] = len(chain.layers)
        out["chain_how"] = (f"a CUDA graph of {len(chain.layers)} dependent layers alternating [M,K]->[M,N] and "
                            f"[M,N]->[M,K], each with its own weight copy; µs per layer")
        out["chain_eager_us_per_layer"] = round(time_chain_eager(chain, stream), 4)
        ml = MultiLayer(chain)
        graphed, eager = time_multilayer(ml, stream)
        out["multilayer_us_per_layer"] = round(graphed, 4)
        out["multilayer_eager_us_per_layer"] = round(eager, 4)
        out["multilayer_how"] = (f"the same layers through mxfp4_quant_gemm_chain, {len(ml.groups)} launches of "
                                 f"{len(ml.groups[0])} layers; graph-replayed, and issued from the host per launch "
                                 f"(the eager figure beside chain_eager_us_per_layer: one host call per layer)")
        del chain, ml
    finally:
        mx.set_programmatic_launch(3)
    return out


def run_ours(args) -> dict:
    import block_scaled_mxfp4_activation_gb300 as mx

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    barrier = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("gloo")
        barrier = dist.barrier
    mx.load_library()
    mx.set_programmatic_launch(3)
    peaks = measured_peaks()
    stream = torch.cuda.Stream(device)
    warmup = max(args.warmup, 3)

    name = args.workload
    w = ALL_WORKLOADS[name]
    prob = Problem(w, device)
    plan = mx.gemm_plan(w.M, w.N, w.K, fused=True)
    assert mx.device_error(reset=True) == 0

    with ClockSampler(local) as clk:
        ms = time_graph_steps(prob, args.steps, warmup, stream, barrier=barrier)
    clocks = clk.summary()
    ms_total, value = aggregate_over_ranks(ms, args.steps, world)

    ms_warm = time_graph_steps(prob, min(args.steps, 2000), warmup, stream, rotate=False)
    us_warm = ms_warm * 1e3 / min(args.steps, 2000)
    e2e_steps = min(max(args.steps, 200), 500)
    ms_e2e = time_e2e(prob, e2e_steps, warmup, stream, via="c_abi")
    us_e2e = ms_e2e * 1e3 / e2e_steps
    us_e2e_py = time_e2e(prob, e2e_steps, warmup, stream, via="python") * 1e3 / e2e_steps
    us_e2e_prep = time_e2e(prob, e2e_steps, warmup, stream, via="prepared") * 1e3 / e2e_steps
    err = mx.device_error(reset=True)
    if err:
        raise RuntimeError(f"device error word {err:#x} after timing")

    us_call = ms_total * 1e3 / args.steps
    rep = shape_report(name, us_call, peaks)
    traffic = committed_traffic(name)
    out = {
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": warmup, "ms_per_step": round(ms_total / args.steps, 7), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": round(value / PAGES_US[name], 4) if name in PAGES_US else None,
        "vs_baseline_note": "pages' figure is end-to-end per call on MI355X incl. Python dispatch (context)",
        "dtype": "mxfp4", "data": "synthetic",
        "config": bench_config(w),
        "timing": {"how": "a CUDA graph of calls replayed until exactly `steps` calls ran, CUDA events on the "
                          "replay stream; call i on rotating copy i of A and of the packed weight; programmatic "
                          "launch mode 3 (each call overlaps the one before it)",
                   "copies": prob.copies, "rotating_mib": round(prob.rotating_bytes / 2**20, 1),
                   "l2_mib": round(prob.l2 / 2**20, 1)},
        "plan": plan,
        "roofline": {"bound": "hbm", "achieved": rep["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": rep["hbm_frac"], "traffic": traffic,
                     "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": rep["bytes"], "kernel": "mxfp4_gemm_kernel<fused>"},
        "fp4": {"tflops": rep["fp4_tflops"], "frac_of_nominal_dense": rep["fp4_frac_nominal"]},
        "warm_l2_us_per_call": round(us_warm, 4),
        "e2e": {"value": round(us_e2e, 3), "unit": UNIT, "h2d_bytes_per_step": 2 * w.M * w.K,
                "d2h_bytes_per_step": 2 * w.M * w.N,
                "how": "the C-ABI call mxfp4_quant_gemm_host per step (through ctypes, arguments prepared once): "
                       "pinned host A -> device, fused layer, C -> pinned host; eager launches; "
                       f"{e2e_steps} steps over the rotating copies after one warm-up call on each",
                "python_api_value": round(us_e2e_py, 3),
                "python_api_how": "the same step through the Python wrapper quant_gemm_host (tensor checks and "
                                  "marshalling on every call)",
                "python_prepared_value": round(us_e2e_prep, 3),
                "python_prepared_how": "the same step through prepare_quant_gemm_host (arguments checked once, then "
                                       "one call per step)"},
        "gpu_launches": args.steps * prob.launches_per_call,
        "clocks": clocks,
    }
    if args.all_shapes:
        shapes = {}
        names = list(workloads.WORKLOADS) + list(workloads.EXTRA_WORKLOADS)
        for other in names:
            wo = ALL_WORKLOADS[other]
            p = prob if other == name else Problem(wo, device)
            n = min(max(args.steps, 1000), 4000)
            t = time_graph_steps(p, n, warmup, stream)
            r = shape_report(other, t * 1e3 / n, peaks)
            if other in workloads.WORKLOADS:
                r.update(latency_report(wo, p, stream, warmup, n))
            r["plan"] = mx.gemm_plan(wo.M, wo.N, wo.K, fused=True)
            r["pages_us_mi355x"] = PAGES_US.get(other)
            shapes[other] = r
            if p is not prob:
                del p
                torch.cuda.empty_cache()
        out["per_shape"] = shapes
        head = shapes[name]
        out["latency"] = {k: head[k] for k in ("us_per_call_no_overlap", "chain_us_per_layer",
                                               "chain_us_per_layer_no_overlap", "chain_eager_us_per_layer",
                                               "multilayer_us_per_layer", "multilayer_eager_us_per_layer")
                          if k in head}
        err = mx.device_error(reset=True)
        if err:
            raise RuntimeError(f"device error word {err:#x} after the per-shape timings")
    if rank == 0 and world == 1 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(name)
        # all host cores, each process on half as many elements as the one-core run summed
        per_core = max(256, out["cpu_baseline"]["elements"] // 2)
        out["cpu_baseline_all_cores"] = cpu_baseline_all_cores(name, per_core)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return out if rank == 0 else None


def run_multilayer_only(args) -> dict:
    """The multi-layer entry alone on the workload's chain of up/down layers
    (graph-replayed and host-issued µs per layer); no headline line."""
    import block_scaled_mxfp4_activation_gb300 as mx

    torch.cuda.set_device(0)
    mx.load_library()
    stream = torch.cuda.Stream()
    w = ALL_WORKLOADS[args.workload]
    ml = MultiLayer(Chain(w, torch.device("cuda", 0)))
    graphed, eager = time_multilayer(ml, stream)
    err = mx.device_error(reset=True)
    if err:
        raise RuntimeError(f"device error word {err:#x}")
    return {"workload": args.workload, "layers": ml.layers, "multilayer_us_per_layer": round(graphed, 4),
            "multilayer_eager_us_per_layer": round(eager, 4)}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args) -> dict | None:
    """The oracle timed on the host cores, on a bounded sample per step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle

    oracle.build()
    name = args.workload
    w = ALL_WORKLOADS[name]
    A, B = workloads.make_inputs(w)
    bq, bs = oracle.quantize(B)
    warmup = max(args.warmup, 3)
    per_step_budget = max(0.05, min(2.0, 150.0 / (args.steps + warmup)))
    # calibrate the sample size of one step
    aq, as_ = oracle.quantize(A)
    rng = np.random.default_rng(1)
    t0 = time.perf_counter()
    oracle.gemm_sampled(aq, as_, bq, bs, rng.integers(0, w.M, 64), rng.integers(0, w.N, 64))
    per_elem = (time.perf_counter() - t0) / 64
    n_sample = int(max(16, min(w.M * w.N, per_step_budget / per_elem)))
    times = []
    for i in range(warmup + args.steps):
        ms = rng.integers(0, w.M, n_sample)
        ns = rng.integers(0, w.N, n_sample)
        t0 = time.perf_counter()
        aq, as_ = oracle.quantize(A)
        tq = time.perf_counter() - t0
        t1 = time.perf_counter()
        oracle.gemm_sampled(aq, as_, bq, bs, ms, ns)
        tg = time.perf_counter() - t1
        if i >= warmup:
            times.append((tq + tg * (w.M * w.N) / n_sample) * 1e6)
    us = float(np.mean(times))
    sample = f"{name}: per step, full A quantization + {n_sample} of {w.M * w.N} outputs, scaled to M*N"
    return {
        "impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": warmup, "ms_per_step": round(us / 1e3, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w),
        "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=sorted(ALL_WORKLOADS))
    ap.add_argument("--all-shapes", dest="all_shapes", action="store_true", default=True)
    ap.add_argument("--headline-only", dest="all_shapes", action="store_false")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    ap.add_argument("--multilayer-only", action="store_true",
                    help="time only the multi-layer entry on the workload's up/down chain (a profiling target)")
    args = ap.parse_args(argv)
    if args.multilayer_only:
        out = run_multilayer_only(args)
    else:
        out = run_reference(args) if args.impl == "reference" else run_ours(args)
    if out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
