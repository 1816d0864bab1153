"""Benchmark of the batch-invariant output head on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--workload pr1|sweep|spec|logprob|int8|int8f|gated|sample|verify]
                    [--impl ours|reference]

Prints ONE JSON line. A step is one pass of the whole hot path over one batch
of synthetic input:

* pr1 (default): the greedy-decode workload -- 16 independent hidden rows,
  each a B=1 call on the bf16 head d=2048, V=32000 (TinyLlama-1.1B shape),
  returning fp32 logits, the token and the top-2 gap;
* sweep: the same head with 8 planted near-tie rows, 64 rows evaluated at
  B = 1, 2, 3, 8, 17, 64;
* spec: speculative-verify block, bf16 d=3584, V=152064, B=256, with logits;
* logprob: trainer scoring, bf16 d=1536, V=151936, 8192 rows, target logp;
* int8: the integer head d=4096, V=128256 at --batch rows (default 512);
* int8f: the integer head fed by bf16 rows at --batch rows: the per-token
  int8 quantization kernel, then the int8 call;
* gated: the pr1 calls through the margin-gated greedy call (tau = 0.001),
  adding the rounded head's token and its top-two margin per row;
* sample: the pr1 calls through the seeded sampling call (T = 1, one seed
  and position per row), returning the drawn token and its score gap;
* verify: the spec block through the speculative-verify call, 16 requests
  x 16 drafted positions, adding the accepted length per request.

value = rows/s for the whole job (all ranks); inputs resident in HBM. Several
copies of W rotate so that every call streams W from HBM (their total is
larger than L2). The timed region runs the calls back to back; after it, a
separate loop brackets the projection kernel of every call with CUDA events
on the call's stream (at least --kernel-launches launches) and the roofline
figure uses the median. `e2e` is the same metric through the host-buffer
entry point (pinned host memory, copies inside the timed region).
`cpu_baseline` times the CPU oracle on a bounded sample and compares its
decisions with the GPU's on the sampled rows.
With --gpus N > 1 the script starts N ranks itself (torch.distributed.run on
127.0.0.1) unless it already runs under a launcher; each rank runs the same
per-GPU workload (weak scaling, no collective on the data path) and the
timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("lm-head rows/s & HBM GB/s (B=1) or TFLOP/s (B≥256) vs roofline, "
          "bit-stable")

WORKLOADS = {
    "pr1": dict(desc="PR1 greedy decode: bf16 head d=2048 V=32000, 16 independent B=1 "
                     "rows, fp32 logits + token + top-2 gap",
                fmt="bf16", V=32000, d=2048, mode="greedy", bound="hbm"),
    "sweep": dict(desc="batch-invariance sweep: bf16 head d=2048 V=32000, 64 rows (8 planted "
                       "near ties) at B in {1,2,3,8,17,64}, logits + token + gap",
                  fmt="bf16", V=32000, d=2048, mode="greedy", bound="hbm"),
    "spec": dict(desc="speculative verify: bf16 head d=3584 V=152064, B=256 (16x16), "
                      "logits + token + gap", fmt="bf16", V=152064, d=3584, B=256,
                 mode="greedy", bound="tensor"),
    "logprob": dict(desc="trainer log-prob scoring: bf16 head d=1536 V=151936, 8x1024 rows, "
                         "target logp", fmt="bf16", V=151936, d=1536, B=8192,
                    mode="logprob", bound="tensor"),
    "int8": dict(desc="integer-only head: int8 d=4096 V=128256, exact int32 logits + token",
                 fmt="int8", V=128256, d=4096, mode="greedy", bound="hbm"),
    "int8f": dict(desc="integer head fed by float rows: bf16 rows quantized per token (dyadic "
                       "multiplier), int8 d=4096 V=128256, exact int32 logits + token",
                  fmt="int8", V=128256, d=4096, mode="int8f", bound="hbm"),
    "gated": dict(desc="margin-gated greedy decode (tau=0.001): bf16 head d=2048 V=32000, "
                       "16 independent B=1 rows, fp32 logits + token + gap + bf16-head token "
                       "+ margin", fmt="bf16", V=32000, d=2048, mode="gated", bound="hbm"),
    "sample": dict(desc="seeded Gumbel-max sampling (T=1): bf16 head d=2048 V=32000, 16 "
                        "independent B=1 rows, fp32 logits + sampled token + score gap",
                   fmt="bf16", V=32000, d=2048, mode="sample", bound="hbm"),
    "verify": dict(desc="greedy speculative verify: bf16 head d=3584 V=152064, 16 requests x "
                        "16 drafted positions, logits + token + gap + accepted length",
                   fmt="bf16", V=152064, d=3584, B=256, mode="verify", bound="tensor"),
}
GATE_TAU = 0.001
SAMPLE_T = 1.0
SEED_DRAFTS = 3103


# ------------------------------------------------------------------ helpers

def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained",
                                                     d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _code_only(text: str) -> str:
    """Source text without comments and blank lines (string literals in
    these files hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


# The source files that make up each projection kernel and its launch: a
# change elsewhere leaves that kernel's profile summary valid.
KERNEL_SOURCES = {
    "head_gemm_kernel": ("detlm_head.cu", "head_kernels.cuh", "ptx.cuh"),
    "head_rows_kernel": ("detlm_head.cu", "head_kernels.cuh", "ptx.cuh", "rows_kernels.cuh"),
    "int8_gemm_kernel": ("detlm_head.cu", "head_kernels.cuh", "int8_kernels.cuh", "ptx.cuh"),
    "head_pair_kernel": ("detlm_head.cu", "head_kernels.cuh", "pair_kernels.cuh", "ptx.cuh",
                         "rows_kernels.cuh"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments and blank lines ignored) of the files that
    make up `kernel`: its profile summary applies while this matches the
    value recorded with the capture."""
    src = os.path.join(ROOT, "invariant_output_head_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(src, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def projection_kernel(workload: str, batch: int) -> str:
    """Name of the call's projection kernel (the one the roofline covers): the
    integer head's streaming kernel below 256 rows; the log-prob kernel; the
    pair kernel for greedy calls (plain, verify, integer) of more than 128
    rows; the one-CTA kernel otherwise (and for the gated and sampling
    calls)."""
    spec = WORKLOADS[workload]
    if spec["fmt"] == "int8":
        return "int8_gemm_kernel" if batch < 256 else "head_pair_kernel"
    if spec["mode"] == "logprob":
        return "head_rows_kernel"
    # --batch sets the integer workloads' rows only; the decode workloads make
    # calls of one row (the sweep: at most 64)
    rows = spec.get("B", 1)
    if spec["mode"] in ("greedy", "verify") and rows > 128:
        return "head_pair_kernel"
    return "head_gemm_kernel"


def profiled_traffic(workload: str, batch: int):
    """DRAM bytes per launch of the projection kernel from a committed ncu
    summary (profiles/<kernel>_<workload>[_b<batch>].md), only while the
    kernel sources still hash to the value recorded with the capture."""
    kernel = projection_kernel(workload, batch)
    kern = kernel.replace("_kernel", "")
    path = None
    for name in (f"{kern}_{workload}_b{batch}.md", f"{kern}_{workload}.md"):
        cand = os.path.join(ROOT, "profiles", name)
        if os.path.exists(cand):
            path = cand
            break
    if path is None:
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256_16") != kernel_source_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                n += 1
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def instruction_peaks(dev, n_sms: int) -> dict:
    """What the integer head's wide path is measured against beside the bf16
    peak: the dense rate of the instruction it runs on (tcgen05 kind::f16,
    fp16 operands, M = 128, N = 256; the library's probe kernel, one CTA per
    SM, no loads), and torch._int_mm on 8192^3 int8 as the library
    reference for an int8 x int8 -> int32 product."""
    import ctypes
    import torch
    out = {}
    lib_path = os.path.join(ROOT, "invariant_output_head_gb300", "_lib", "libdetlm_peak.so")
    try:
        lib = ctypes.CDLL(lib_path)
        lib.detlm_mma_f16_peak.restype = ctypes.c_int
        lib.detlm_mma_f16_peak.argtypes = [ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_double)]
        vals = []
        for _ in range(3):
            tf = ctypes.c_double()
            if lib.detlm_mma_f16_peak(n_sms, 40000, ctypes.byref(tf)) == 0:
                vals.append(tf.value)
        out["mma_f16_dense_tflops"] = round(max(vals), 1) if vals else None
    except OSError as e:
        out["mma_f16_dense_tflops"] = None
        out["mma_f16_note"] = f"probe library not loaded: {e}"
    try:
        n = 8192
        a = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
        b = torch.randint(-127, 128, (n, n), dtype=torch.int8, device=dev)
        torch._int_mm(a, b)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            torch._int_mm(a, b)
        e1.record()
        torch.cuda.synchronize()
        sec = e0.elapsed_time(e1) / 1e3 / 10
        out["torch_int_mm_8192_tops"] = round(2.0 * n ** 3 / sec / 1e12, 1)
        del a, b
    except Exception as e:   # noqa: BLE001 - a reference figure, reported either way
        out["torch_int_mm_8192_tops"] = None
        out["torch_int_mm_note"] = f"{type(e).__name__}: {str(e)[:160]}"
    return out


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host scalar over all ranks (NCCL on GPUs, gloo on CPUs)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = (torch.device("cuda", torch.cuda.current_device())
           if dist.get_backend() == "nccl" else torch.device("cpu"))
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_step: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Whole-job throughput: every rank runs the same per-GPU workload (weak
    scaling), timed by the slowest rank."""
    return rows_per_step * steps * world / (elapsed_ms / 1e3)


# ------------------------------------------------------------- workloads

def launches_per_call(mode: str, fmt: str, B: int) -> int:
    """Kernels one call launches: projection + merge; the int8 head at
    B >= 256 first converts the rows to fp16; the float-fed int8 call first
    quantizes them."""
    n = 2
    if fmt == "int8" and B >= 256:
        n += 1
    if mode == "int8f":
        n += 1
    return n


def mode_of(name: str) -> str:
    return WORKLOADS[name]["mode"]


def make_inputs(name: str, batch: int):
    import synth
    if name in ("pr1", "gated", "sample"):
        c = synth.pr1()
        c["calls"] = [(r, 1) for r in range(c["h"].shape[0])]
        if name == "sample":
            rk = np.random.default_rng(SEED_DRAFTS + 2)
            c["seeds"] = rk.integers(0, 2 ** 63, size=16).astype(np.int64)
            c["positions"] = rk.integers(0, 4096, size=16).astype(np.int64)
    elif name == "sweep":
        c = synth.sweep()
        calls = []
        for B in (1, 2, 3, 8, 17, 64):
            for r0 in range(0, 64, B):
                calls.append((r0, min(B, 64 - r0)))
        c["calls"] = calls
    elif name in ("spec", "verify"):
        c = synth.spec_verify()
        c["calls"] = [(0, 256)]
        if name == "verify":
            # drafts planted on a seeded stand-in sequence (acceptance does not
            # change the work of the call)
            seq = np.random.default_rng(SEED_DRAFTS).integers(0, c["V"], size=(16, 16))
            c["drafts"], _ = synth.plant_drafts(seq, c["V"], seed=SEED_DRAFTS + 1)
    elif name == "logprob":
        c = synth.logprob()
        c["calls"] = [(0, c["h"].shape[0])]
    elif name in ("int8", "int8f"):
        c = synth.int8_head(B=batch)
        c["calls"] = [(0, batch)]
        if name == "int8f":
            c["x"] = synth.float_rows(SEED_DRAFTS + 3, batch, c["d"], "bf16", special=False)
    else:
        raise SystemExit(f"unknown workload {name}")
    return c


def algorithmic(name, c, B):
    """Algorithmic bytes and flops of one call with B rows."""
    V, d = c["V"], c["d"]
    eb = 1 if c["dtype"] == "int8" else 2
    by = V * d * eb + B * d * eb
    mode = WORKLOADS[name]["mode"]
    if mode == "logprob":
        by += B * 8                      # targets + logp
    else:
        by += B * V * 4 + B * 8          # logits + token + gap
    if mode == "gated":
        by += B * 8                      # rounded head's token + margin
    if mode == "verify":
        by += B * 4 + (B // 16) * 4      # drafts + accepted
    if mode == "sample":
        by += B * 16                     # seeds + positions
    if mode == "int8f":
        by += B * d * 2 + B * d + B * 8  # bf16 rows read, int8 rows written, M and S
    return by, 2.0 * B * V * d


L2_NOTE = ("inputs larger than L2: the GPU arm rotates over copies of W totalling more "
           "than twice the L2")


def workload_config(name, c, calls, world):
    """The `config` object of the JSON line: the same on both arms."""
    return {"workload": WORKLOADS[name]["desc"], "name": name, "V": c["V"], "d": c["d"],
            "rows_per_step": sum(B for _, B in calls), "calls_per_step": len(calls),
            "l2": L2_NOTE, "parallelism": f"replicas x{world}"}


# ------------------------------------------------------------------ our arm

def graph_steady(torch, stream, step, k, n_calls, n_copies, steps, heads, snapshot, first):
    """The step's calls captured once into a CUDA graph (as many steps as make
    the rotation over the W copies repeat) and replayed: the steady state
    without host launch costs. Returns per-call time and bit stability, or
    the capture error."""
    reps_per_graph = n_copies // math.gcd(n_calls, n_copies)
    k[0] = 0                       # the captured calls start on the first copy
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream().cuda_stream
            for _ in range(reps_per_graph):
                step(stream_ptr=cs)
    except Exception as e:          # reported, not fatal: the eager figures stand
        return {"error": f"{type(e).__name__}: {e}"[:300]}
    g.replay()
    torch.cuda.synchronize()
    replays = max(1, -(-steps // reps_per_graph))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(replays):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    for hd in heads:
        assert hd.check() == 0, "device error in the graph replays"
    last = snapshot()
    stable = all(
        all(torch.equal(x.view(torch.int32), y.view(torch.int32)) for x, y in zip(p, q))
        if isinstance(p, tuple) else torch.equal(p.view(torch.int32), q.view(torch.int32))
        for p, q in zip(first, last))
    calls = replays * reps_per_graph * n_calls
    return {"us_per_call": round(a.elapsed_time(b) * 1e3 / calls, 2),
            "calls_per_graph": reps_per_graph * n_calls, "replays": replays,
            "bit_stable": bool(stable),
            "note": "one graph of the step's calls, replayed back to back; frac against "
                    "the sustained peak for tensor-bound workloads"}


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import invariant_output_head_gb300 as ioh
    from invariant_output_head_gb300 import binding as bd

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    spec = dict(WORKLOADS[args.workload])
    if args.workload in ("int8", "int8f") and args.batch >= 256:
        spec["bound"] = "tensor"     # fp16-rate tensor-core path, compute-bound
    c = make_inputs(args.workload, args.batch)
    fmt, V, d = c["dtype"], c["V"], c["d"]
    tdt = {"bf16": torch.bfloat16, "fp16": torch.float16, "int8": torch.int8}[fmt]

    def to_dev(a):
        a = np.ascontiguousarray(a)
        t = torch.from_numpy(a.view(np.int16) if fmt != "int8" else a)
        return t.to(dev).view(tdt) if fmt != "int8" else t.to(dev)

    W0 = to_dev(c["W"])
    wbytes = W0.numel() * W0.element_size()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_copies = args.copies or max(2, int(np.ceil(2 * l2 / wbytes)) + 1)
    Ws = [W0] + [W0.clone() for _ in range(n_copies - 1)]
    heads = [ioh.Head(W, fmt) for W in Ws]
    h_all = to_dev(c["h"])
    if mode_of(args.workload) == "int8f":
        x_all = torch.from_numpy(c["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    rows = h_all.shape[0]
    calls = c["calls"]
    maxB = max(B for _, B in calls)
    for hd in heads:
        bd.detlm_head_reserve(hd.handle, maxB)
    mode = spec["mode"]
    greedy = mode != "logprob"
    gdt = torch.int32 if fmt == "int8" else torch.float32
    outs = []
    for r0, B in calls:
        if greedy:
            o = [torch.empty(B, dtype=torch.int32, device=dev),
                 torch.empty(B, dtype=gdt, device=dev),
                 torch.empty((B, V), dtype=gdt, device=dev)]
            if mode == "gated":
                o += [torch.empty(B, dtype=torch.int32, device=dev),
                      torch.empty(B, dtype=torch.float32, device=dev)]
            if mode == "verify":
                o += [torch.empty(B // 16, dtype=torch.int32, device=dev)]
            outs.append(tuple(o))
        else:
            outs.append(torch.empty(B, dtype=torch.float32, device=dev))
    targets = torch.from_numpy(c["targets"]).to(dev) if not greedy else None
    drafts = torch.from_numpy(c["drafts"]).to(dev) if mode == "verify" else None
    if mode == "sample":
        seeds_d = torch.from_numpy(c["seeds"]).to(dev)
        pos_d = torch.from_numpy(c["positions"]).to(dev)
    stream = torch.cuda.current_stream(dev)
    n_calls = len(calls)
    k = [0]

    def step(ev=None, stream_ptr=None):
        sp = stream.cuda_stream if stream_ptr is None else stream_ptr
        for j, (r0, B) in enumerate(calls):
            hd = heads[k[0] % n_copies]
            k[0] += 1
            if ev is not None and ev[j] is not None:
                bd.detlm_head_time_next(hd.handle, ev[j][0].cuda_event, ev[j][1].cuda_event)
            hv = h_all[r0:r0 + B]
            if mode == "greedy":
                tok, gap, lg = outs[j]
                bd.detlm_head_greedy(hd.handle, hv.data_ptr(), B, tok.data_ptr(),
                                     gap.data_ptr(), lg.data_ptr(), sp)
            elif mode == "gated":
                tok, gap, lg, base, margin = outs[j]
                bd.detlm_head_greedy_gated(hd.handle, hv.data_ptr(), B, GATE_TAU, tok.data_ptr(),
                                           gap.data_ptr(), lg.data_ptr(), base.data_ptr(),
                                           margin.data_ptr(), sp)
            elif mode == "int8f":
                tok, gap, lg = outs[j]
                bd.detlm_head_greedy_from_float(hd.handle, x_all[r0:r0 + B].data_ptr(),
                                                bd.DETLM_BF16, B, tok.data_ptr(), gap.data_ptr(),
                                                lg.data_ptr(), None, None, sp)
            elif mode == "sample":
                tok, gap, lg = outs[j]
                bd.detlm_head_sample(hd.handle, hv.data_ptr(), B, SAMPLE_T,
                                     seeds_d[r0:r0 + B].data_ptr(), pos_d[r0:r0 + B].data_ptr(),
                                     tok.data_ptr(), gap.data_ptr(), lg.data_ptr(), sp)
            elif mode == "verify":
                tok, gap, lg, acc = outs[j]
                bd.detlm_head_verify(hd.handle, hv.data_ptr(), B // 16, 16, drafts.data_ptr(),
                                     tok.data_ptr(), gap.data_ptr(), lg.data_ptr(),
                                     acc.data_ptr(), sp)
            else:
                bd.detlm_head_logprob(hd.handle, hv.data_ptr(), targets[r0:r0 + B].data_ptr(),
                                      B, outs[j].data_ptr(), sp)

    def snapshot():
        if greedy:
            return [tuple(t.clone() for t in o) for o in outs]
        return [o.clone() for o in outs]

    # warm-up, and the reference outputs for the bit-stability check
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    first = snapshot()
    for hd in heads:
        assert hd.check() == 0, "device error after warm-up"

    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)
    for hd in heads:
        assert hd.check() == 0, "device error in the timed region"

    # bit stability: last step's outputs equal the warm-up outputs bit for bit
    last = snapshot()
    stable = all(
        all(torch.equal(a.view(torch.int32) if a.dtype != torch.int32 else a,
                        b.view(torch.int32) if b.dtype != torch.int32 else b)
            for a, b in zip(x, y)) if greedy else torch.equal(x.view(torch.int32),
                                                                y.view(torch.int32))
        for x, y in zip(first, last))

    # The projection kernel alone: a separate loop after the timed region in
    # which every call's projection kernel is bracketed by CUDA events on the
    # call's stream (an event between two kernels keeps the next call from
    # starting early, so the timed region itself carries none). The median
    # over at least `kernel_launches` launches does not depend on --steps.
    kl_steps = max(1, -(-args.kernel_launches // n_calls))
    ev = []
    for _ in range(kl_steps):
        row = []
        for _ in range(n_calls):
            pair = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            pair[0].record(stream)      # torch creates an event at its first record
            pair[1].record(stream)
            row.append(pair)
        ev.append(row)
    torch.cuda.synchronize()
    for s in range(kl_steps):
        step(ev[s])
    torch.cuda.synchronize()
    graph = graph_steady(torch, stream, step, k, n_calls, n_copies, args.steps, heads,
                         snapshot, first)
    clocks = sampler.stop() if rank == 0 else None
    for hd in heads:
        assert hd.check() == 0, "device error in the kernel-timing loop"
    kus = np.array([[e[0].elapsed_time(e[1]) * 1e3 for e in row] for row in ev])  # [step, call]

    rows_per_step = sum(B for _, B in calls)
    by, fl = 0.0, 0.0
    by_call = []
    for _, B in calls:
        b_, f_ = algorithmic(args.workload, c, B)
        by += b_
        fl += f_
        by_call.append(b_)
    by_launch, fl_launch = by / n_calls, fl / n_calls
    # median duration of each call of the step, then the step's kernel time
    med_call_us = np.median(kus, axis=0)
    kernel_s = float(med_call_us.sum()) / 1e6 / n_calls     # per launch
    peaks = measured_peaks()
    spec_hbm = 8000.0                    # the nominal HBM3e figure (~8 TB/s)
    hbm_achieved = by_launch / kernel_s / 1e9
    if spec["bound"] == "hbm":
        achieved = hbm_achieved
        peak, unit, peak_key = peaks["hbm_gbs"], "GB/s", "hbm_gbs"
    else:
        # timed alone (one launch between two events): the burst peak applies
        achieved = fl_launch / kernel_s / 1e12
        peak, unit, peak_key = peaks["bf16_tflops"], "TFLOP/s", "bf16_tflops"
    steady_call_s = elapsed_ms / 1e3 / (args.steps * n_calls)
    if spec["bound"] == "hbm":
        steady_frac = by_launch / steady_call_s / 1e9 / peaks["hbm_gbs"]
    else:
        # back to back over the whole timed region: the sustained peak applies
        steady_frac = fl_launch / steady_call_s / 1e12 / peaks["bf16_tflops_sustained"]
    traffic = profiled_traffic(args.workload, args.batch)
    per_B = {}
    for j, (_, B) in enumerate(calls):
        per_B.setdefault(B, []).append(j)
    by_B = None
    if len(per_B) > 1:
        by_B = {}
        for B, js in sorted(per_B.items()):
            us = float(np.median(kus[:, js]))
            by_B[str(B)] = {"kernel_us": round(us, 2),
                            "gbs": round(by_call[js[0]] / (us / 1e6) / 1e9, 1),
                            "frac": round(by_call[js[0]] / (us / 1e6) / 1e9 / peaks["hbm_gbs"], 4),
                            "launches": int(kus[:, js].size)}

    value = job_rows_per_s(rows_per_step, args.steps, world, elapsed_ms)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int8" if fmt == "int8" else fmt, "data": "synthetic",
        "config": workload_config(args.workload, c, calls, world),
        "l2_rotation": f"{n_copies} rotating copies of W ({n_copies * wbytes / 1e6:.0f} MB) "
                       f"> 2x L2 ({l2 / 1e6:.0f} MB)",
        "roofline": {"bound": spec["bound"], "achieved": round(achieved, 1),
                     "peak": peak, "unit": unit, "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "kernel": projection_kernel(args.workload, args.batch),
                     "kernel_us_per_launch": round(kernel_s * 1e6, 2),
                     "kernel_us_stat": "median",
                     "timed_launches": int(kus.size),
                     "hbm_achieved_gbs": round(hbm_achieved, 1),
                     "hbm_frac_of_measured": round(hbm_achieved / peaks["hbm_gbs"], 4),
                     "hbm_frac_of_spec_8tbs": round(hbm_achieved / spec_hbm, 4),
                     # the launch's lower bounds: its algorithmic bytes at the
                     # measured copy bandwidth, its flops at the burst tensor
                     # peak; the larger one is the binding roofline
                     "roofline_us": {"hbm": round(by_launch / (peaks["hbm_gbs"] * 1e9) * 1e6, 2),
                                     "tensor": round(fl_launch / (peaks["bf16_tflops"] * 1e12) * 1e6, 2)},
                     "binding": "hbm" if by_launch / peaks["hbm_gbs"] >= fl_launch / (peaks["bf16_tflops"] * 1e3)
                                else "tensor",
                     "frac_of_binding_roofline": round(
                         max(by_launch / (peaks["hbm_gbs"] * 1e9),
                             fl_launch / (peaks["bf16_tflops"] * 1e12)) / kernel_s, 4),
                     "steady_us_per_call": round(steady_call_s * 1e6, 2),
                     "steady_frac": round(steady_frac, 4),
                     "note": "achieved/frac: the projection kernel alone, median over a "
                             "separate loop in which every launch is bracketed by CUDA "
                             "events, against the burst peak; steady_*: all calls of the "
                             "timed region back to back (both kernels, overlapped), against "
                             "the sustained peak for tensor-bound workloads",
                     "algorithmic_bytes_per_launch": int(by_launch),
                     "algorithmic_flops_per_launch": fl_launch,
                     "peak_source": f"MEASURED_PEAKS.json ({peaks['source']}, {peak_key})"},
        "bit_stable": bool(stable),
        "gpu_launches": args.steps * sum(launches_per_call(mode, fmt, B) for _, B in calls),
        "clocks": clocks,
    }
    if by_B is not None:
        res["roofline"]["per_B"] = by_B
    if "us_per_call" in graph:
        graph["frac"] = round((by_launch / (graph["us_per_call"] * 1e-6) / 1e9 / peaks["hbm_gbs"])
                              if spec["bound"] == "hbm" else
                              (fl_launch / (graph["us_per_call"] * 1e-6) / 1e12
                               / peaks["bf16_tflops_sustained"]), 4)
    res["roofline"]["graph_replay"] = graph
    if fmt == "int8" and spec["bound"] == "tensor" and rank == 0:
        ip = instruction_peaks(dev, torch.cuda.get_device_properties(dev).multi_processor_count)
        if ip.get("mma_f16_dense_tflops"):
            ip["frac_of_mma_f16_dense"] = round(achieved / ip["mma_f16_dense_tflops"], 4)
        res["roofline"]["instruction_peaks"] = ip
    if rank == 0 and not args.profile:
        res["e2e"] = run_e2e(args, c, heads, calls, mode, rows_per_step, dev, stream)
        res["cpu_baseline"] = cpu_baseline(args.workload, c, budget_s=args.cpu_seconds,
                                           gpu_rows=gpu_row_decisions(first, calls, mode))
    if args.profile:
        res["profile_run"] = "e2e and cpu_baseline legs skipped (--profile)"
    return res


def gpu_row_decisions(snap, calls, mode):
    """Row -> the GPU's decision (token, or logp) from one step's outputs; the
    first call that holds a row decides it."""
    rows = {}
    for (r0, B), o in zip(calls, snap):
        vals = (o if mode == "logprob" else o[0]).cpu().numpy()
        for k in range(B):
            rows.setdefault(r0 + k, vals[k].item())
    return rows


def run_e2e(args, c, heads, calls, mode, rows_per_step, dev, stream):
    """Same metric end to end: pinned host inputs are copied in and the
    results copied out on every call, and every step ends when its results
    are in host memory. The greedy and log-prob calls go through their
    asynchronous host-buffer entry points (one pinned result buffer set per
    call; the step ends with detlm_head_check on each head it used); the
    other calls, which have no host-buffer form, through their device entry
    points with their inputs copied in on the same stream and their outputs
    written by the kernels straight into pinned host buffers (one set per
    call), the step ending with a stream synchronization."""
    import torch
    from invariant_output_head_gb300 import binding as bd
    fmt, V = c["dtype"], c["V"]
    greedy = mode != "logprob"
    h_host = torch.from_numpy(np.ascontiguousarray(
        c["h"].view(np.int16) if fmt != "int8" else c["h"])).pin_memory()
    esz = h_host.element_size()
    d = c["d"]
    maxB = max(B for _, B in calls)
    # the asynchronous calls: a result buffer set of their own per call
    res_bufs = []
    if mode in ("greedy", "logprob"):
        for _, B in calls:
            if mode == "greedy":
                res_bufs.append((torch.empty(B, dtype=torch.int32).pin_memory(),
                                 torch.empty(B, dtype=torch.int32).pin_memory(),
                                 torch.empty((B, V), dtype=torch.int32).pin_memory()))
            else:
                res_bufs.append((torch.empty(B, dtype=torch.float32).pin_memory(),))
    tg = torch.from_numpy(c["targets"]).pin_memory() if not greedy else None
    sp = stream.cuda_stream
    steps = max(3, min(args.steps, int(args.e2e_seconds / 0.002)))
    if mode == "int8f":
        x_host = torch.from_numpy(np.ascontiguousarray(c["x"].view(np.int16))).pin_memory()
        x_dev = torch.empty((maxB, d), dtype=torch.int16, device=dev)
        o8 = [(torch.empty(B, dtype=torch.int32).pin_memory(),
               torch.empty(B, dtype=torch.int32).pin_memory(),
               torch.empty((B, V), dtype=torch.int32).pin_memory()) for _, B in calls]
    if mode in ("gated", "verify", "sample"):
        tdt = {"bf16": torch.bfloat16, "fp16": torch.float16}[fmt]
        h_dev = torch.empty((maxB, d), dtype=tdt, device=dev)
        # per call: token, gap, logits, and the gate's base token + margin or
        # the accepted lengths, all pinned host memory the kernels write
        o_pin = [(torch.empty(B, dtype=torch.int32).pin_memory(),
                  torch.empty(B, dtype=torch.float32).pin_memory(),
                  torch.empty((B, V), dtype=torch.float32).pin_memory(),
                  torch.empty(2 * B, dtype=torch.int32).pin_memory()) for _, B in calls]
        dr_host = (torch.from_numpy(c["drafts"]).pin_memory() if mode == "verify" else None)
        dr_dev = torch.empty(maxB, dtype=torch.int32, device=dev)
        if mode == "sample":
            seed_host = torch.from_numpy(np.ascontiguousarray(c["seeds"])).pin_memory()
            pos_host = torch.from_numpy(np.ascontiguousarray(c["positions"])).pin_memory()
            seed_dev = torch.empty_like(seed_host, device=dev)
            pos_dev = torch.empty_like(pos_host, device=dev)

    def one_step(i):
        used = {}
        for j, (r0, B) in enumerate(calls):
            hd = heads[(i * len(calls) + j) % len(heads)]
            used[id(hd)] = hd
            hp = h_host.data_ptr() + r0 * d * esz
            if mode == "greedy":
                rt, rg, rl = res_bufs[j]
                bd.detlm_head_greedy_host_async(hd.handle, hp, B, rt.data_ptr(), rg.data_ptr(),
                                                rl.data_ptr(), sp)
            elif mode == "logprob":
                bd.detlm_head_logprob_host_async(hd.handle, hp, tg.data_ptr() + r0 * 4, B,
                                                 res_bufs[j][0].data_ptr(), sp)
            elif mode == "int8f":
                ot, og, ol = o8[j]
                with torch.cuda.stream(stream):
                    x_dev[:B].copy_(x_host[r0:r0 + B], non_blocking=True)
                    bd.detlm_head_greedy_from_float(hd.handle, x_dev.data_ptr(), bd.DETLM_BF16, B,
                                                    ot.data_ptr(), og.data_ptr(), ol.data_ptr(),
                                                    None, None, sp)
            else:
                ot, og, ol, ox = o_pin[j]
                with torch.cuda.stream(stream):
                    h_dev[:B].view(torch.int16).copy_(h_host[r0:r0 + B], non_blocking=True)
                    if mode == "gated":
                        bd.detlm_head_greedy_gated(
                            hd.handle, h_dev.data_ptr(), B, GATE_TAU, ot.data_ptr(),
                            og.data_ptr(), ol.data_ptr(), ox.data_ptr(), ox.data_ptr() + 4 * B, sp)
                    elif mode == "sample":
                        seed_dev[r0:r0 + B].copy_(seed_host[r0:r0 + B], non_blocking=True)
                        pos_dev[r0:r0 + B].copy_(pos_host[r0:r0 + B], non_blocking=True)
                        bd.detlm_head_sample(
                            hd.handle, h_dev.data_ptr(), B, SAMPLE_T,
                            seed_dev[r0:r0 + B].data_ptr(), pos_dev[r0:r0 + B].data_ptr(),
                            ot.data_ptr(), og.data_ptr(), ol.data_ptr(), sp)
                    else:
                        dr_dev[:B].copy_(dr_host.view(-1)[:B], non_blocking=True)
                        bd.detlm_head_verify(
                            hd.handle, h_dev.data_ptr(), B // 16, 16, dr_dev.data_ptr(),
                            ot.data_ptr(), og.data_ptr(), ol.data_ptr(), ox.data_ptr(), sp)
        # the step's results are in host memory when the step ends
        if mode in ("greedy", "logprob"):
            for hd in used.values():
                assert hd.check() == 0
        else:
            stream.synchronize()
    for i in range(3):
        one_step(i)
    torch.cuda.synchronize()
    t = time.perf_counter()
    for i in range(steps):
        one_step(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t
    if mode == "int8f":
        esz = 2                          # the bf16 rows are what is copied in
    h2d = sum(B * d * esz + (4 * B if mode in ("logprob", "verify") else 0)
              + (16 * B if mode == "sample" else 0) for _, B in calls)
    d2h = sum(4 * B if mode == "logprob" else 8 * B + 4 * B * V for _, B in calls)
    d2h += sum(8 * B if mode == "gated" else (4 * (B // 16) if mode == "verify" else 0)
               for _, B in calls)
    api = {"greedy": "detlm_head_greedy_host_async (+ detlm_head_check per step)",
           "logprob": "detlm_head_logprob_host_async (+ detlm_head_check per step)",
           "gated": "detlm_head_greedy_gated, inputs copied in on the call's stream, "
                    "outputs written by the kernels into pinned host buffers",
           "verify": "detlm_head_verify, inputs copied in on the call's stream, "
                     "outputs written by the kernels into pinned host buffers",
           "sample": "detlm_head_sample, inputs copied in on the call's stream, "
                     "outputs written by the kernels into pinned host buffers",
           "int8f": "detlm_head_greedy_from_float, rows copied in on the call's stream, "
                    "outputs written by the kernels into pinned host buffers"}[mode]
    return {"value": round(rows_per_step * steps / dt, 2), "unit": "rows/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps, "api": api}


# ---------------------------------------------------------------- CPU oracle

def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_rows_per_s(name, c, budget_s, max_rows=None):
    """Time the oracle as it stands on rows of the workload, one call at a time
    (each call decodes W and computes every logit and the decision)."""
    import oracle
    fmt = c["dtype"]
    h = c["h"]
    n = 0
    t0 = time.perf_counter()
    while True:
        r = n % h.shape[0]
        oracle_row(name, c, r)
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or (max_rows is not None and n >= max_rows):
            return n / dt, n, dt


def oracle_row(name, c, r):
    """The oracle on row r of the workload: what one row of the call computes."""
    import oracle
    fmt, h, mode = c["dtype"], c["h"], WORKLOADS[name]["mode"]
    if mode == "logprob":
        return oracle.head_logprob(c["W"], h[r:r + 1], c["targets"][r:r + 1], fmt)
    if mode == "int8f":
        q, _, _ = oracle.quantize_rows(oracle.decode(c["x"][r:r + 1], "bf16"))
        return oracle.head_greedy(c["W"], q, "int8")
    out = oracle.head_greedy(c["W"], h[r:r + 1], fmt)
    if mode == "gated":
        out["gate"] = oracle.gated_greedy(out["logits"], GATE_TAU, fmt)
    if mode == "sample":
        out["sample"] = oracle.sample(out["logits"], SAMPLE_T, c["seeds"][r:r + 1],
                                      c["positions"][r:r + 1])
    if mode == "verify":
        # the row's comparison with its draft (the request's accepted length
        # is a prefix scan over its 16 rows)
        out["accept"] = oracle.verify_accept(out["token"].reshape(1, 1),
                                             c["drafts"].reshape(-1, 1)[r:r + 1])
    return out


def cpu_baseline(name, c, budget_s, gpu_rows=None):
    """The oracle timed on a bounded sample of the workload's rows; with the
    GPU's decisions for those rows (gpu_rows[r] = token or logp of row r), the
    sampled rows are also compared and every disagreement is listed: a token
    that differs inside the tolerance of the logits is a near-tie exception,
    one outside it a mismatch; both are listed, never dropped."""
    v, n, dt = oracle_rows_per_s(name, c, budget_s)
    res = {"value": round(v, 4), "unit": "rows/s", "cores": cpu_cores(), "kind": "oracle",
           "sample": f"{n} hidden rows of the {name} workload, one oracle call per row "
                     f"(exact decode of W, float64/int64 logits, decision), {dt:.1f} s"}
    if gpu_rows:
        res["parity_sample"] = compare_sample(name, c, gpu_rows, min(n, c["h"].shape[0]))
    return res


def compare_sample(name, c, gpu_rows, n_rows):
    """Compare the oracle with the GPU decisions on rows 0 .. n_rows-1 (outside
    any timed region)."""
    mode = WORKLOADS[name]["mode"]
    listed, mismatches, max_dlogp = [], 0, 0.0
    for r in range(n_rows):
        if r not in gpu_rows:
            continue
        out = oracle_row(name, c, r)
        g = gpu_rows[r]
        if mode == "logprob":
            max_dlogp = max(max_dlogp, abs(float(out["logp"][0]) - float(g)))
            continue
        if mode == "sample":
            t = int(out["sample"]["token"][0])
        else:
            t = int(out["token"][0])
        if int(g) == t:
            continue
        if "A" in out and mode != "sample":
            z, e = out["logits"][0], 1e-6 * out["A"][0]
            near = bool(z[t] - z[int(g)] <= e[t] + e[int(g)])
        else:
            near = False
        if near:
            listed.append({"row": r, "oracle": t, "gpu": int(g),
                           "gap_ulp": float(out["gap"][0])})
        else:
            mismatches += 1
    res = {"rows_compared": n_rows, "token_mismatches": mismatches,
           "near_tie_exceptions": listed}
    if mode == "logprob":
        res = {"rows_compared": n_rows, "max_abs_logp_diff": max_dlogp}
    return res


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step one row of the workload."""
    if rank != 0:
        return None
    c = make_inputs(args.workload, args.batch)
    fmt = c["dtype"]
    h = c["h"]

    def one(i):
        oracle_row(args.workload, c, i % h.shape[0])
    for i in range(args.warmup):
        one(i)
    # bound the timed work to a few minutes of CPU time
    t0 = time.perf_counter()
    one(0)
    per = time.perf_counter() - t0
    steps = max(1, min(args.steps, int(args.ref_seconds / max(per, 1e-6))))
    t0 = time.perf_counter()
    for i in range(steps):
        one(i)
    dt = time.perf_counter() - t0
    value = steps / dt
    sample = (f"{steps} of {args.steps} requested steps, each one hidden row of the "
              f"{args.workload} workload through the CPU oracle (B=1 call)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "rows/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": round(dt / steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64" if fmt != "int8" else "int64",
            "data": "synthetic",
            "config": workload_config(args.workload, c, c["calls"], world),
            "cpu_baseline": {"value": round(value, 4), "unit": "rows/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def free_port() -> int:
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def relaunch_ranks(n: int):
    """Start n ranks of this same command (one per GPU) and exit with their
    status: `python bench.py --gpus n` behaves like the torchrun launch."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={free_port()}",
           os.path.abspath(__file__), *sys.argv[1:]]
    raise SystemExit(subprocess.call(cmd))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="pr1", choices=sorted(WORKLOADS))
    ap.add_argument("--batch", type=int, default=512, help="rows per call (int8 workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-seconds", type=float, default=3.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--kernel-launches", type=int, default=512,
                    help="projection-kernel launches bracketed by CUDA events in the "
                         "separate kernel-timing loop (median reported)")
    ap.add_argument("--copies", type=int, default=0,
                    help="copies of W to rotate (default: enough to exceed 2x L2)")
    ap.add_argument("--profile", action="store_true",
                    help="GPU leg only (no e2e, no CPU baseline): for profiler runs")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local_rank = env_rank()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        relaunch_ranks(args.gpus)
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: start one rank per GPU")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
