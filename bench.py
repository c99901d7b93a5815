#!/usr/bin/env python3
"""Benchmark of the Q8_0 x Q8_0 matmul on GB300.

One step = one pass of the decode hot path over the decode projection sweep
workload (attn_q_b shape: W 32768 x 1024 Q8_0, activations fp32 with 1% of
values scaled x20): for n_tok = 1, 4 and 16, quantise the activations and
multiply (q8_matmul).  Metric: weight GB/s (34 bytes per 32 weights read per
call); prefill int8-equivalent TOPS and routed-expert GB/s are reported in
the same JSON line under "secondary".

Timing: W >= 3 warm-up steps, then exactly K steps replayed as CUDA graphs
(each holding several consecutive steps, as an engine's graph holds a whole
forward pass; the remainder of K as one-step graphs), bracketed by a barrier and a device synchronise, CUDA events on the launching
stream, max over ranks.  Inputs larger than L2: every call of a step reads its
own copy of the weights, rotating through copies totalling more than 4x L2.
SM clocks are sampled with nvidia-smi during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (test infrastructure, the only other
place this file runs it) on the host cores on a bounded sample of the same
workload.  Under torchrun each rank runs its own replica (weak scaling).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import inputs  # noqa: E402

QK, QB = 32, 34
METRIC = "Q8_0 matmul weight GB/s (n_tok≤16) & int8 TOPS (prefill), % of roofline"
IN_DIM, OUT_DIM, N_TOKS = 1024, 32768, (1, 4, 16)
W_BYTES = OUT_DIM * IN_DIM // QK * QB
WORKLOAD = ("decode projection sweep (attn_q_b shape): in_dim=1024, out_dim=32768, n_tok in {1,4,16}; "
            "Q8_0 weights q~U[-127,127], d~U[1e-3,1e-2] fp16; x~N(0,1) with 1% x20 outliers; seed 0")
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--profile-case", choices=("decode1", "decode4", "decode16", "prefill", "prefill_long", "moe",
                                               "moe_zipf", "moe_zipf_small", "moe_ffn", "rmsnorm", "kq_moe_q4k",
                                               "kq_moe_q2k"),
                    help="run one workload's call a few times without timing (for ncu captures)")
    a = ap.parse_args()
    a.warmup = max(a.warmup, 3)
    return a


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend: str = "nccl"):
    """One process group over the ranks (NCCL for the bench; gloo runs the same plumbing on CPU)."""
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend)
    return dist


def max_over_ranks(dist, v: float) -> float:
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="q8clk", suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except (OSError, FileNotFoundError):
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
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ peaks and traffic
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


GEMV_FILES = ("q8_gemv.cu", "q8_common.cuh", "q8_quant.cuh")


def kernel_source_hash(files=GEMV_FILES) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "q8_quantized_matmul_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged since."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("source_hash") != kernel_source_hash(tuple(e.get("files", GEMV_FILES))):
            return None
        return e
    except (OSError, KeyError, ValueError):
        return None


# ------------------------------------------------------------------ GPU arm
def weight_copies(torch, dev, host_w, total_bytes_min):
    n = max(1, math.ceil(total_bytes_min / host_w.nbytes))
    t = torch.from_numpy(host_w).to(dev)
    return [t] + [t.clone() for _ in range(n - 1)]


def graph_replays(torch, stream, graphs, steps):
    """Replay graphs[i % len] for i in range(steps) on `stream`; returns elapsed ms (CUDA events)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def run_ours(args, rank, world, local, dist):
    import torch
    import q8_quantized_matmul_gb300 as q8
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    stream = torch.cuda.Stream(device=dev)

    # ---- inputs (seeded, synthetic; weights resident in HBM before timing)
    Wh = inputs.weights(OUT_DIM, IN_DIM, seed=0)
    n_calls = len(N_TOKS)
    copies = weight_copies(torch, dev, Wh, 4 * l2)
    while len(copies) % n_calls:
        copies.append(copies[0].clone())
    xs = {n: torch.from_numpy(inputs.normal((n, IN_DIM), seed=0, p_out=0.01, out_scale=20.0)).to(dev) for n in N_TOKS}
    outs = {n: torch.empty((n, OUT_DIM), dtype=torch.float32, device=dev) for n in N_TOKS}
    n_graphs = len(copies) // n_calls

    def call(n, W):
        rc = q8.q8_matmul(outs[n], W, IN_DIM, OUT_DIM, xs[n], n, stream)
        if rc:
            raise q8.Q8Error(rc, "q8_matmul")

    # warm-up eagerly (sizes the scratch, sets kernel attributes), then capture
    with torch.cuda.stream(stream):
        for g in range(n_graphs):
            for c, n in enumerate(N_TOKS):
                call(n, copies[g * n_calls + c])
    stream.synchronize()
    assert q8.q8_last_error(stream) == 0
    def capture(groups):
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            for g in groups:
                for c, n in enumerate(N_TOKS):
                    call(n, copies[g * n_calls + c])
        return cg
    # A decode engine captures a token's whole forward pass (many projections)
    # in one graph, so consecutive steps run back to back: one graph holds
    # n_graphs steps, each step on its own weight copies; the K % n_graphs
    # steps left over replay one-step graphs, so exactly K steps are timed.
    multi = capture(range(n_graphs))
    singles = [capture([g]) for g in range(n_graphs)]
    n_multi, n_rest = divmod(args.steps, n_graphs)
    graph_replays(torch, stream, [multi], max(1, -(-args.warmup // n_graphs)))
    graph_replays(torch, stream, singles, n_graphs)   # every graph runs at least once
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local if world > 1 else (torch.cuda.current_device())) as clk:
        ms = graph_replays(torch, stream, [multi] * n_multi + singles[:n_rest], n_multi + n_rest)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms = max_over_ranks(dist, ms)
    assert q8.q8_last_error(stream) == 0

    # Kernel-level timing: per token count, a graph of back-to-back calls, each on
    # its own weight copy, replayed; per-call time = replay time / calls.  For
    # n_tok <= 8 a call is one GEMV launch (it quantises the activations itself);
    # for n_tok = 16 it is the quantiser kernel plus the GEMV behind it (PDL).
    per_call = {}
    for n in N_TOKS:
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            for c in copies:
                call(n, c)
        graph_replays(torch, stream, [cg], 2)
        reps = 8
        per_call[n] = graph_replays(torch, stream, [cg], reps) / (reps * len(copies))
        del cg
    assert q8.q8_last_error(stream) == 0

    ms_step = ms / args.steps
    step_bytes = W_BYTES * n_calls
    value = world * step_bytes / (ms_step * 1e-3) / 1e9
    tokens_per_s = world * sum(N_TOKS) / (ms_step * 1e-3)

    # algorithmic bytes of one call: weights, fp32 activations, fp32 outputs, and
    # for 16 tokens the activation planes written by the quantiser and read back
    def kbytes(n):
        b = W_BYTES + n * IN_DIM * 4 + n * OUT_DIM * 4
        if n > 8:
            npad = (n + 15) // 16 * 16
            b += 2 * (npad * IN_DIM + npad * (IN_DIM // QK) * 4)
        return b
    tot_bytes = sum(kbytes(n) for n in N_TOKS)
    tot_ms = sum(per_call.values())
    peak, peak_kind = hbm_peak()
    achieved = tot_bytes / (tot_ms * 1e-3) / 1e9
    tr = committed_traffic("k_gemv decode sweep")
    roofline = {"bound": "hbm", "kernel": "q8::k_gemv", "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "algorithmic_bytes_per_launch": round(tot_bytes / n_calls),
                "timing": "graph of back-to-back calls per token count, CUDA events around the replays",
                "per_n": {str(n): {"us_per_call": round(per_call[n] * 1e3, 2),
                                   "launches_per_call": 1 if n <= 8 else 2,
                                   "weight_gbs": round(W_BYTES / (per_call[n] * 1e-3) / 1e9, 1),
                                   "frac_of_peak": round(kbytes(n) / (per_call[n] * 1e-3) / 1e9 / peak, 4)}
                          for n in N_TOKS}}

    # ---- end to end through the public API with pinned host buffers
    xh = {n: xs[n].cpu().pin_memory() for n in N_TOKS}
    oh = {n: torch.empty((n, OUT_DIM), dtype=torch.float32).pin_memory() for n in N_TOKS}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_step(i):
        for c, n in enumerate(N_TOKS):
            rc = q8.q8_matmul_host(oh[n], copies[(i * n_calls + c) % len(copies)], IN_DIM, OUT_DIM, xh[n], n,
                                   stream)
            if rc:
                raise q8.Q8Error(rc, "q8_matmul_host")
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            e2e_step(i)
        stream.synchronize()
        barrier(dist)
        e0.record(stream)
        for i in range(args.steps):
            e2e_step(i)
        e1.record(stream)
    e1.synchronize()
    assert q8.q8_last_error(stream) == 0
    for n in N_TOKS:
        # every weight copy holds the same bytes.  With 3 or more tokens the host-result
        # call splits each CTA's rows in two items (partial sums added in another
        # order), so it agrees with the device-result call to rounding, not bitwise
        ref = outs[n].cpu()
        err = (oh[n] - ref).abs().max().item()
        assert err <= 1e-4 * ref.abs().max().item(), f"host-buffer result differs from the device one ({err})"
    e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / args.steps
    e2e = {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
           "ms_per_step": round(e2e_ms, 4),
           "h2d_bytes_per_step": sum(n * IN_DIM * 4 for n in N_TOKS),
           "d2h_bytes_per_step": sum(n * OUT_DIM * 4 for n in N_TOKS),
           "path": "q8_matmul_host via the C ABI, one eager call per matmul: the kernels read the pinned "
                   "host x and write the pinned host result directly over the GPU's host link (no staging "
                   "copies); bytes counted are those x and result buffers"}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "s8", "data": "synthetic",
        "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {len(copies)} weight copies ({len(copies) * W_BYTES / 2 ** 20:.0f} MiB) "
                         f"rotated, each call reads its own copy (L2 {l2 / 2 ** 20:.0f} MiB)",
                   "launch": f"CUDA graphs of {n_graphs} consecutive steps each (the last K mod {n_graphs} "
                             "steps one-step graphs); per call n_tok 1 and 4: one fused GEMV kernel each; "
                             "n_tok 16: quantiser + GEMV",
                   "tokens_per_s": round(tokens_per_s, 1)},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": args.steps * sum(1 if n <= 8 else 2 for n in N_TOKS),
        "clocks": clk.summary(),
    }
    del copies, multi, singles
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_secondary:
        result["secondary"] = secondary(args, torch, q8, dev, stream, l2)
    return result


def timed_eager(torch, stream, fn, iters, warm=2):
    with torch.cuda.stream(stream):
        for i in range(warm):
            fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(iters):
            fn(i)
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / iters


def secondary(args, torch, q8, dev, stream, l2):
    """Other workloads, one line each (kernel timing through the library's event hook)."""
    out = []
    tflops, tflops_sus, tkind = tensor_peak()
    hbm, hkind = hbm_peak()

    def prof_mean(npairs):
        v = [q8.q8_profile_read(i) for i in range(npairs)]
        return statistics.mean(v)

    # single matvec (attn_q_a shape)
    W = inputs.weights(1024, 4096, seed=0)
    copies = weight_copies(torch, dev, W, 4 * l2)
    x = torch.from_numpy(inputs.normal((1, 4096), seed=0)).to(dev)
    o = torch.empty((1, 1024), device=dev)
    with torch.cuda.stream(stream):
        for c in copies:
            q8.q8_matmul(o, c, 4096, 1024, x, 1, stream)
    stream.synchronize()
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cg, stream=stream):
        for c in copies:
            q8.q8_matmul(o, c, 4096, 1024, x, 1, stream)
    graph_replays(torch, stream, [cg], 3)
    ms = graph_replays(torch, stream, [cg], 20) / (20 * len(copies))
    wb = W.nbytes
    out.append({"workload": "single matvec (attn_q_a shape) in 4096 -> out 1024, n_tok 1",
                "ms_per_call": round(ms, 5), "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 1),
                "launches_per_call": 1,
                "frac_of_hbm_peak": round(wb / (ms * 1e-3) / 1e9 / hbm, 4),
                "timing": "graph of back-to-back calls, each on its own weight copy"})
    del copies, cg

    # RMSNorm feeding the quantiser at the long-prefill input (4096 tokens x 4096): reads x,
    # writes the Q8_0 rows; each call on its own copy of x (copies > 4x L2)
    n, dim = 4096, 4096
    xh = inputs.normal((n, dim), seed=6)
    xcopies = weight_copies(torch, dev, xh, 4 * l2)
    gamma = torch.from_numpy((1.0 + 0.1 * np.random.default_rng(6).standard_normal(dim)).astype(np.float32)).to(dev)
    xq = torch.empty((n, dim // QK * QB), dtype=torch.uint8, device=dev)
    cg = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in xcopies:
            q8.q8_rmsnorm_quantize(xq, None, c, gamma, dim, n, 1e-6, stream)
    stream.synchronize()
    with torch.cuda.graph(cg, stream=stream):
        for c in xcopies:
            q8.q8_rmsnorm_quantize(xq, None, c, gamma, dim, n, 1e-6, stream)
    graph_replays(torch, stream, [cg], 3)
    ms = graph_replays(torch, stream, [cg], 10) / (10 * len(xcopies))
    nbytes = n * dim * 4 + n * dim // QK * QB + dim * 4
    out.append({"workload": f"RMSNorm + Q8_0 quantiser, {n} tokens x {dim} (long-prefill q_a input)",
                "ms_per_call": round(ms, 4), "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                "frac_of_hbm_peak": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
                "bytes_per_call": nbytes,
                "timing": "graph of back-to-back calls, each on its own copy of x"})
    assert q8.q8_last_error(stream) == 0
    del xcopies, cg

    # prefill GEMMs (attn_output_a and shared-expert shapes) at n_tok = 512; every call reads its own
    # copy of the weights and of the activations (each set of copies larger than L2)
    for in_dim, out_dim in ((32768, 1024), (4096, 2048), (2048, 4096)):
        n = 512
        W = inputs.weights(out_dim, in_dim, seed=1)
        copies = weight_copies(torch, dev, W, 2 * l2)
        xcopies = weight_copies(torch, dev, inputs.normal((n, in_dim), seed=1), 2 * l2)
        o = torch.empty((n, out_dim), device=dev)
        q8.q8_profile_arm(8)
        ms = timed_eager(torch, stream, lambda i: q8.q8_matmul(o, copies[i % len(copies)], in_dim, out_dim,
                                                                xcopies[i % len(xcopies)], n, stream), 8)
        kms = prof_mean(8)
        q8.q8_profile_arm(0)
        ops = 2.0 * in_dim * out_dim * n
        out.append({"workload": f"prefill GEMM in {in_dim} -> out {out_dim}, n_tok {n}",
                    "ms_per_call": round(ms, 4), "tops": round(ops / (ms * 1e-3) / 1e12, 2),
                    "kernel_ms": round(kms, 4), "kernel_tops": round(ops / (kms * 1e-3) / 1e12, 2),
                    "kernel_frac_of_bf16_peak": round(ops / (kms * 1e-3) / 1e12 / tflops, 4),
                    "peak_note": f"int8-equivalent ops vs {tkind} dense bf16 tensor peak {tflops} TFLOP/s "
                                 "(no int8 MMA instruction on sm_103a)",
                    "timing": "eager calls, each on its own copy of the weights and of x (both > L2)"})
        del copies, xcopies

    # the same GEMM on weights repacked once into the tensor-core operand layout (no per-call
    # expansion above 2048 tokens); eager calls, each on its own copy of the packed weights
    for in_dim, out_dim, n in ((32768, 1024, 512), (1024, 32768, 4096)):
        W = inputs.weights(out_dim, in_dim, seed=1)
        Wd = torch.from_numpy(W).to(dev)
        pk = [q8.repack(Wd, in_dim, out_dim, q8.Q8_LAYOUT_TC)]
        pk += [pk[0].clone() for _ in range(max(1, int(2 * l2 // pk[0].numel())))]
        copies = [Wd] + [Wd.clone() for _ in range(max(1, int(2 * l2 // Wd.numel())))]
        xcopies = weight_copies(torch, dev, inputs.normal((n, in_dim), seed=1), 2 * l2)
        o = torch.empty((n, out_dim), device=dev)
        ms_raw = timed_eager(torch, stream, lambda i: q8.q8_matmul(o, copies[i % len(copies)], in_dim, out_dim,
                                                                    xcopies[i % len(xcopies)], n, stream), 6)
        ms_pk = timed_eager(torch, stream, lambda i: q8.q8_matmul_packed(o, pk[i % len(pk)], q8.Q8_LAYOUT_TC, in_dim,
                                                                          out_dim, xcopies[i % len(xcopies)], n,
                                                                          stream), 6)
        ops = 2.0 * in_dim * out_dim * n
        out.append({"workload": f"prefill in {in_dim} -> out {out_dim}, n_tok {n}: weights packed once in the "
                                "tensor-core layout (q8_matmul_packed) against raw Q8_0 rows (q8_matmul)",
                    "ms_per_call_packed": round(ms_pk, 4), "tops_packed": round(ops / (ms_pk * 1e-3) / 1e12, 2),
                    "ms_per_call_raw": round(ms_raw, 4), "tops_raw": round(ops / (ms_raw * 1e-3) / 1e12, 2),
                    "frac_of_bf16_peak_packed": round(ops / (ms_pk * 1e-3) / 1e12 / tflops, 4)})
        del pk, copies, Wd, xcopies
    torch.cuda.empty_cache()

    # routed experts: gate/up (x per token) and down (x per pair), 256 experts, 64 tokens, uniform top-6
    n_exp, n_tok, k = 256, 64, 6
    ids = inputs.route_uniform(n_tok, k, n_exp, seed=0)
    touched = len(np.unique(ids))
    idsd = torch.from_numpy(ids).to(dev)
    for name, in_dim, out_dim, per_pair in (("gate/up", 4096, 2048, 0), ("down", 2048, 4096, 1)):
        W = torch.from_numpy(inputs.weights(n_exp * out_dim, in_dim, seed=2)).to(dev)
        stride = out_dim * in_dim // QK * QB
        x = torch.from_numpy(inputs.normal((n_tok * k if per_pair else n_tok, in_dim), seed=2)).to(dev)
        o = torch.empty((n_tok * k, out_dim), device=dev)
        q8.q8_profile_arm(6)
        ms = timed_eager(torch, stream, lambda i: q8.q8_moe_matmul(o, W, n_exp, stride, idsd, k, in_dim, out_dim, x,
                                                                    per_pair, n_tok, stream), 6)
        kms = prof_mean(6)
        q8.q8_profile_arm(0)
        wb = touched * stride
        out.append({"workload": f"routed MoE {name}: 256 experts [{out_dim}x{in_dim}], n_tok 64, uniform top-6 "
                                f"({touched} experts touched)",
                    "ms_per_call": round(ms, 4), "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 1),
                    "kernel_ms": round(kms, 4), "kernel_weight_gbs": round(wb / (kms * 1e-3) / 1e9, 1),
                    "kernel_frac_of_hbm_peak": round(wb / (kms * 1e-3) / 1e9 / hbm, 4)})
        del W
    assert q8.q8_last_error(stream) == 0
    torch.cuda.empty_cache()

    # the second weight format on the same routing: Q4_K and Q2_K experts against Q8_K activations
    for fmt, fname in ((q8.Q8_KQ_Q4_K, "Q4_K"), (q8.Q8_KQ_Q2_K, "Q2_K")):
        for name, in_dim, out_dim, per_pair in (("gate/up", 4096, 2048, 0), ("down", 2048, 4096, 1)):
            stride = out_dim * q8.q8_kq_row_bytes(in_dim, fmt)
            W = torch.from_numpy(inputs.kq_weights(n_exp * out_dim, in_dim, fmt, seed=2).reshape(-1)).to(dev)
            x = torch.from_numpy(inputs.normal((n_tok * k if per_pair else n_tok, in_dim), seed=2)).to(dev)
            o = torch.empty((n_tok * k, out_dim), device=dev)
            q8.q8_profile_arm(6)
            ms = timed_eager(torch, stream, lambda i: q8.q8_kq_moe_matmul(o, W, fmt, n_exp, stride, idsd, k, in_dim,
                                                                           out_dim, x, per_pair, n_tok, stream), 6)
            kms = prof_mean(6)
            q8.q8_profile_arm(0)
            wb = touched * stride
            out.append({"workload": f"routed {fname} experts {name}: 256 experts [{out_dim}x{in_dim}], Q8_K "
                                    f"activations, n_tok 64, uniform top-6 ({touched} experts touched)",
                        "ms_per_call": round(ms, 4), "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 1),
                        "kernel_ms": round(kms, 4), "kernel_weight_gbs": round(wb / (kms * 1e-3) / 1e9, 1),
                        "kernel_frac_of_hbm_peak": round(wb / (kms * 1e-3) / 1e9 / hbm, 4)})
            del W
    assert q8.q8_last_error(stream) == 0
    torch.cuda.empty_cache()

    # the routed expert FFN on the same routing: gate and up (one routing, one quantisation
    # of x), SwiGLU with clamp 10, down on the re-quantised mid, weighted sum of the 6 experts
    in_dim, mid_dim = 4096, 2048
    Wg, Wu = (torch.from_numpy(inputs.weights(n_exp * mid_dim, in_dim, seed=s)).to(dev) for s in (2, 4))
    Wd = torch.from_numpy(inputs.weights(n_exp * in_dim, mid_dim, seed=5)).to(dev)
    gu_stride, d_stride = mid_dim * in_dim // QK * QB, in_dim * mid_dim // QK * QB
    wts = torch.from_numpy(np.random.default_rng(0).random((n_tok, k)).astype(np.float32)).to(dev)
    x = torch.from_numpy(inputs.normal((n_tok, in_dim), seed=2)).to(dev)
    o = torch.empty((n_tok, in_dim), device=dev)
    reps = 6
    q8.q8_profile_arm(2 * reps)          # two timed launch groups per call: the gate/up pair, down
    ms = timed_eager(torch, stream, lambda i: q8.q8_moe_ffn(o, Wg, Wu, Wd, n_exp, gu_stride, d_stride, idsd, wts, k,
                                                             in_dim, mid_dim, in_dim, 10.0, x, n_tok, stream), reps)
    kms = sum(q8.q8_profile_read(i) for i in range(2 * reps)) / reps
    q8.q8_profile_arm(0)
    assert q8.q8_last_error(stream) == 0
    wb = touched * (2 * gu_stride + d_stride)
    out.append({"workload": "routed MoE FFN: 256 experts, gate/up [2048x4096], down [4096x2048], n_tok 64, "
                            f"uniform top-6 ({touched} experts touched), SwiGLU clamp 10, weighted sum",
                "ms_per_call": round(ms, 4), "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 1),
                "frac_of_hbm_peak": round(wb / (ms * 1e-3) / 1e9 / hbm, 4),
                "matmul_kernels_ms": round(kms, 4),
                "matmul_kernel_weight_gbs": round(wb / (kms * 1e-3) / 1e9, 1),
                "launches_per_call": "3 routing + 1 quantiser + gate/up pair GEMVs (SwiGLU in their epilogue) + "
                                     "3 routing + 1 quantiser + down GEMVs + weighted sum"})
    del Wg, Wu, Wd
    torch.cuda.empty_cache()

    # long prefill layer slice: 4096 tokens through q_a, q_b, output_a, output_b, then routed
    # gate/up and down over 256 experts with Zipf(1.1) top-6 routing
    n = 4096
    rows = []
    total_ops, total_ms = 0.0, 0.0
    for in_dim, out_dim in ((4096, 1024), (1024, 32768), (32768, 1024), (1024, 4096)):
        W = torch.from_numpy(inputs.weights(out_dim, in_dim, seed=3)).to(dev)
        x = torch.from_numpy(inputs.normal((n, in_dim), seed=3)).to(dev)
        o = torch.empty((n, out_dim), device=dev)
        ms = timed_eager(torch, stream, lambda i: q8.q8_matmul(o, W, in_dim, out_dim, x, n, stream), 3, warm=1)
        ops = 2.0 * in_dim * out_dim * n
        total_ops += ops
        total_ms += ms
        rows.append(f"{in_dim}->{out_dim}: {ms:.3f} ms, {ops / (ms * 1e-3) / 1e12:.0f} TOPS")
        del W, x, o
    ids = torch.from_numpy(inputs.route_zipf(n, 6, 256, s=1.1, seed=0)).to(dev)
    for name, in_dim, out_dim, per_pair in (("gate/up", 4096, 2048, 0), ("down", 2048, 4096, 1)):
        W = torch.from_numpy(inputs.weights(256 * out_dim, in_dim, seed=2)).to(dev)
        stride = out_dim * in_dim // QK * QB
        x = torch.from_numpy(inputs.normal((n * 6 if per_pair else n, in_dim), seed=2)).to(dev)
        o = torch.empty((n * 6, out_dim), device=dev)
        ms = timed_eager(torch, stream, lambda i: q8.q8_moe_matmul(o, W, 256, stride, ids, 6, in_dim, out_dim, x,
                                                                    per_pair, n, stream), 3, warm=1)
        ops = 2.0 * in_dim * out_dim * n * 6
        total_ops += ops
        total_ms += ms
        rows.append(f"MoE {name}: {ms:.3f} ms, {ops / (ms * 1e-3) / 1e12:.0f} TOPS")
        del W, x, o
    assert q8.q8_last_error(stream) == 0
    out.append({"workload": "long prefill layer slice, n_tok 4096: q_a 4096->1024, q_b 1024->32768, "
                            "output_a 32768->1024, output_b 1024->4096, routed gate/up and down over 256 experts "
                            "(Zipf(1.1) top-6)",
                "ms_per_slice": round(total_ms, 3), "tops": round(total_ops / (total_ms * 1e-3) / 1e12, 1),
                "frac_of_bf16_peak": round(total_ops / (total_ms * 1e-3) / 1e12 / tflops, 4),
                "per_call": rows,
                "timing": "eager calls (quantise + expand + GEMM each), CUDA events, mean of 3"})
    torch.cuda.empty_cache()
    # every line also as tokens per second: the tokens a call (or the slice) processes over its time
    for d in out:
        m = re.search(r"n_tok (\d+)|(\d+) tokens", d["workload"])
        ms = d.get("ms_per_call", d.get("ms_per_slice", d.get("ms_per_call_packed")))
        if m and ms:
            d["tokens_per_s"] = round(int(m.group(1) or m.group(2)) / (ms * 1e-3), 1)
    return out


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)
def host_cores() -> int:
    """Cores this process may run on (the baseline uses one thread per core)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleRunner:
    """Runs the CPU oracle, as it stands, on slices of a workload from `threads` threads.

    The oracle's C functions are called through ctypes, which releases the GIL for
    the duration of each call, so the slices run on separate cores.  Nothing here
    changes the oracle's arithmetic: the quantiser is cut into ranges of tokens, a
    dense product into contiguous ranges of weight rows (one q8o_matmul call each),
    a routed product into ranges of sampled (pair, row) outputs (one q8o_moe_sample
    call each)."""

    def __init__(self, threads: int):
        import concurrent.futures as cf
        import oracle
        self.o = oracle.get()
        self.threads = threads
        self.pool = cf.ThreadPoolExecutor(max_workers=threads) if threads > 1 else None

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()

    def _run(self, fns):
        if self.pool is None:
            for f in fns:
                f()
        else:
            for fut in [self.pool.submit(f) for f in fns]:
                fut.result()

    def _cuts(self, n):
        k = max(1, min(self.threads, n))
        return [(i * n // k, (i + 1) * n // k) for i in range(k)]

    def quantize(self, x):
        n_tok, in_dim = x.shape
        rb = in_dim // QK * QB
        xq = np.empty((n_tok, rb), np.uint8)

        def part(a, b):
            assert self.o.lib.q8o_quantize(xq.ctypes.data + a * rb, x.ctypes.data + a * in_dim * 4, in_dim,
                                           b - a) == 0
        self._run([(lambda a=a, b=b: part(a, b)) for a, b in self._cuts(n_tok)])
        return xq

    def dense(self, W, xq, in_dim, n_tok, rows):
        """out = W[:rows] x from quantised activations (outputs [n_tok][slice] per slice)."""
        o = self.o
        row_bytes = in_dim // QK * QB

        def part(r0, r1):
            out = np.empty((n_tok, r1 - r0), np.float32)
            assert o.lib.q8o_matmul(out.ctypes.data, None, W.ctypes.data + r0 * row_bytes, in_dim, r1 - r0,
                                    xq.ctypes.data, n_tok) == 0
        self._run([(lambda a=a, b=b: part(a, b)) for a, b in self._cuts(rows)])

    def moe_outputs(self, W, n_exp, stride, ids, in_dim, out_dim, xq, per_pair, pair, row):
        o = self.o
        n_tok = ids.shape[0]

        def part(a, b):
            out = np.empty(b - a, np.float32)
            assert o.lib.q8o_moe_sample(out.ctypes.data, None, W.ctypes.data, n_exp, stride, ids.ctypes.data,
                                        ids.shape[1], in_dim, out_dim, xq.ctypes.data, int(per_pair), n_tok,
                                        pair[a:].ctypes.data, row[a:].ctypes.data, b - a) >= 0
        self._run([(lambda a=a, b=b: part(a, b)) for a, b in self._cuts(pair.size)])


def _timed(fn, target_s):
    """Runs fn() until about target_s has passed (at least once); returns seconds per run."""
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    reps = max(0, int(target_s / max(dt, 1e-6)) - 1)
    t0 = time.perf_counter()
    for _ in range(reps):
        fn()
    return (time.perf_counter() - t0) / reps if reps else dt


def _rows_for(runner, W, xq, in_dim, n_tok, rows_max, target_s):
    """Weight rows of a dense sample that take about target_s on one core (at least 8)."""
    probe = min(rows_max, 8)
    t0 = time.perf_counter()
    runner.dense(W, xq, in_dim, n_tok, probe)
    per_row = (time.perf_counter() - t0) / probe
    return int(min(rows_max, max(8, target_s / max(per_row, 1e-9))))


def cpu_baseline_configs(target_s: float = 1.0, threads: int | None = None):
    """The oracle on each of the five workloads, single-threaded and on every host core.

    Each workload is timed as quantise (all activations) + products.  Large
    products are a bounded sample, the same one for both thread counts, scaled to
    the whole workload: dense products take their first weight rows (rows are
    independent, and the time per row does not depend on which), routed products a
    seeded sample of (pair, row) outputs on the real expert shape (16 experts held
    on the host; the time per output does not depend on the expert).  Units follow
    the GPU lines: weight GB/s where the GPU reports weight GB/s, int8-equivalent
    TOPS where it reports TOPS."""
    threads = threads or host_cores()
    runners = (OracleRunner(1), OracleRunner(threads))
    res = []

    def both(fn, t=target_s):
        """seconds per run of fn(runner) on one core and on all cores"""
        return [_timed(lambda: fn(r), t / (1 if r.threads == 1 else 2)) for r in runners]

    def dense_time(W, x, in_dim, out_dim, t):
        """(1-core, n-core) seconds for quantise + the whole product, from a row sample"""
        n_tok = x.shape[0]
        tq = both(lambda r: r.quantize(x), t / 4)
        xq = runners[0].quantize(x)
        rows = _rows_for(runners[0], W, xq, in_dim, n_tok, out_dim, t)
        tm = both(lambda r: r.dense(W, xq, in_dim, n_tok, rows), t)
        return [q + m * out_dim / rows for q, m in zip(tq, tm)], rows

    # 1. single matvec 4096 -> 1024, one token: weight GB/s
    W = inputs.weights(1024, 4096, seed=0)
    (t1, tn), _ = dense_time(W, inputs.normal((1, 4096), seed=0), 4096, 1024, target_s)
    res.append(("single matvec (attn_q_a) in 4096 -> out 1024, n_tok 1", "GB/s", W.nbytes / t1 / 1e9,
                W.nbytes / tn / 1e9, "whole workload"))
    # 2. decode projection sweep 1024 -> 32768, n_tok 1, 4, 16: weight GB/s
    W = inputs.weights(OUT_DIM, IN_DIM, seed=0)
    t1 = tn = 0.0
    rows = []
    for n in N_TOKS:
        (a, c), r = dense_time(W, inputs.normal((n, IN_DIM), seed=0, p_out=0.01, out_scale=20.0), IN_DIM, OUT_DIM,
                               target_s / 3)
        t1, tn = t1 + a, tn + c
        rows.append(r)
    b = len(N_TOKS) * W.nbytes
    res.append(("decode projection sweep in 1024 -> out 32768, n_tok 1, 4, 16", "GB/s", b / t1 / 1e9, b / tn / 1e9,
                "first " + "/".join(map(str, rows)) + f" of {OUT_DIM} weight rows for n_tok 1/4/16, scaled to all"))
    # 3. prefill at 512 tokens: out_a 32768 -> 1024, shared expert 4096 -> 2048 and 2048 -> 4096: TOPS
    ops = t1 = tn = 0.0
    notes = []
    for in_dim, out_dim in ((32768, 1024), (4096, 2048), (2048, 4096)):
        (a, c), r = dense_time(inputs.weights(out_dim, in_dim, seed=1), inputs.normal((512, in_dim), seed=1),
                               in_dim, out_dim, target_s / 3)
        t1, tn = t1 + a, tn + c
        ops += 2.0 * in_dim * out_dim * 512
        notes.append(f"{r}/{out_dim}")
    res.append(("prefill GEMMs at 512 tokens (32768->1024, 4096->2048, 2048->4096)", "TOPS", ops / t1 / 1e12,
                ops / tn / 1e12, "first " + ", ".join(notes) + " weight rows, scaled to all"))
    g = np.random.default_rng(0)

    def moe_time(ids_full, in_dim, out_dim, per_pair, t):
        n_tok, k = ids_full.shape
        ne = 16
        ids = np.ascontiguousarray(ids_full % ne, dtype=np.int32)   # same shapes and loop, 16 experts held
        Wm = inputs.weights(ne * out_dim, in_dim, seed=2)
        stride = out_dim * in_dim // QK * QB
        x = inputs.normal((n_tok * k if per_pair else n_tok, in_dim), seed=2)
        tq = both(lambda r: r.quantize(x), t / 4)
        xq = runners[0].quantize(x)
        n_sample = 64
        t0 = time.perf_counter()
        runners[0].moe_outputs(Wm, ne, stride, ids, in_dim, out_dim, xq, per_pair,
                               g.integers(0, n_tok * k, n_sample).astype(np.int64),
                               g.integers(0, out_dim, n_sample).astype(np.int64))
        per = (time.perf_counter() - t0) / n_sample
        n_sample = int(max(256, min(200000, t / max(per, 1e-9))))
        pair = g.integers(0, n_tok * k, n_sample).astype(np.int64)
        row = g.integers(0, out_dim, n_sample).astype(np.int64)
        tm = both(lambda r: r.moe_outputs(Wm, ne, stride, ids, in_dim, out_dim, xq, per_pair, pair, row), t)
        total = n_tok * k * out_dim
        return [q + m * total / n_sample for q, m in zip(tq, tm)], n_sample

    # 4. routed experts, 64 tokens, uniform top-6 over 256: gate/up and down, weight GB/s of touched experts
    ids4 = inputs.route_uniform(64, 6, 256, seed=0)
    touched = len(np.unique(ids4))
    t1 = tn = 0.0
    wb = 0
    notes = []
    for in_dim, out_dim, per_pair in ((4096, 2048, 0), (2048, 4096, 1)):
        (a, c), ns = moe_time(ids4, in_dim, out_dim, per_pair, target_s / 2)
        t1, tn, wb = t1 + a, tn + c, wb + touched * out_dim * in_dim // QK * QB
        notes.append(str(ns))
    res.append((f"routed MoE gate/up + down, 256 experts, 64 tokens, uniform top-6 ({touched} touched)", "GB/s",
                wb / t1 / 1e9, wb / tn / 1e9, " and ".join(notes) + " sampled outputs of the gate/up and down "
                "matrices, scaled to all 384 pair rows"))
    # 5. long-prefill layer slice, 4096 tokens: four dense projections and routed gate/up + down (Zipf top-6)
    ops = t1 = tn = 0.0
    for in_dim, out_dim in ((4096, 1024), (1024, 32768), (32768, 1024), (1024, 4096)):
        (a, c), _ = dense_time(inputs.weights(out_dim, in_dim, seed=3), inputs.normal((4096, in_dim), seed=3),
                               in_dim, out_dim, target_s / 6)
        t1, tn = t1 + a, tn + c
        ops += 2.0 * in_dim * out_dim * 4096
    idsz = inputs.route_zipf(4096, 6, 256, s=1.1, seed=0)
    for in_dim, out_dim, per_pair in ((4096, 2048, 0), (2048, 4096, 1)):
        (a, c), _ = moe_time(idsz, in_dim, out_dim, per_pair, target_s / 6)
        t1, tn = t1 + a, tn + c
        ops += 2.0 * in_dim * out_dim * 4096 * 6
    res.append(("long-prefill layer slice, 4096 tokens (q_a, q_b, output_a, output_b, routed gate/up + down)",
                "TOPS", ops / t1 / 1e12, ops / tn / 1e12,
                "all activations quantised; first weight rows of each projection and sampled routed outputs, "
                "scaled to the whole slice"))
    for r in runners:
        r.close()
    return [{"workload": w, "unit": u, "single_core": float(f"{v1:.4g}"), "all_cores": float(f"{vn:.4g}"),
             "threads": threads, "sample": smp} for w, u, v1, vn, smp in res], threads


def cpu_baseline(target_s: float = 1.0):
    """cpu_baseline object of the bench line: the decode sweep on every host core, plus every config."""
    per, threads = cpu_baseline_configs(target_s)
    head = per[1]
    return {"value": head["all_cores"], "unit": "GB/s", "cores": threads, "kind": "oracle",
            "host_cores_online": os.sysconf("SC_NPROCESSORS_ONLN") if hasattr(os, "sysconf") else None,
            "single_core_value": head["single_core"],
            "sample": f"decode projection sweep: {head['sample']} x n_tok 1, 4, 16 (quantise + matmul), "
                      f"oracle on {threads} threads (one per core, ctypes releases the GIL)",
            "per_config": per}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    threads = host_cores()
    runner = OracleRunner(threads)
    Wh = inputs.weights(OUT_DIM, IN_DIM, seed=0)
    xs = {n: inputs.normal((n, IN_DIM), seed=0, p_out=0.01, out_scale=20.0) for n in N_TOKS}
    probe = 512

    def step_rows(rows):
        for n in N_TOKS:
            runner.dense(Wh, runner.quantize(xs[n]), IN_DIM, n, rows)
    t0 = time.perf_counter()
    step_rows(probe)
    per_row = (time.perf_counter() - t0) / probe
    budget = 120.0 / (args.steps + args.warmup)          # whole run within about two minutes
    rows = int(min(OUT_DIM, max(64, budget / max(per_row, 1e-9))))

    def step():
        step_rows(rows)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    runner.close()
    bytes_ = rows * IN_DIM // QK * QB * len(N_TOKS)
    v = bytes_ / dt / 1e9
    sample = (f"each step: first {rows} of {OUT_DIM} weight rows, n_tok 1, 4, 16 (quantise + matmul), "
              f"plain C oracle on {threads} threads (one per core)")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_case(case: str):
    """A small, fixed case for profiler captures: 2 warm-up calls then 3 profiled calls."""
    import torch
    import q8_quantized_matmul_gb300 as q8
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if case in ("decode1", "decode4", "decode16"):
        n = int(case[len("decode"):])
        W = torch.from_numpy(inputs.weights(OUT_DIM, IN_DIM, seed=0)).to(dev)
        x = torch.from_numpy(inputs.normal((n, IN_DIM), seed=0, p_out=0.01, out_scale=20.0)).to(dev)
        fn = lambda: q8.matmul(W, x, OUT_DIM)
    elif case == "prefill":
        W = torch.from_numpy(inputs.weights(1024, 32768, seed=1)).to(dev)
        x = torch.from_numpy(inputs.normal((512, 32768), seed=1)).to(dev)
        fn = lambda: q8.matmul(W, x, 1024)
    elif case == "prefill_long":   # long-prefill shape: the weights go through the fp16 plane
        W = torch.from_numpy(inputs.weights(32768, 1024, seed=3)).to(dev)
        x = torch.from_numpy(inputs.normal((4096, 1024), seed=3)).to(dev)
        fn = lambda: q8.matmul(W, x, 32768)
    elif case == "moe":
        ids = torch.from_numpy(inputs.route_uniform(64, 6, 256, seed=0)).to(dev)
        W = torch.from_numpy(inputs.weights(256 * 2048, 4096, seed=2)).to(dev)
        x = torch.from_numpy(inputs.normal((64, 4096), seed=2)).to(dev)
        fn = lambda: q8.moe_matmul(W, 256, 2048 * 128 * QB, ids, x, False, 2048)
    elif case in ("kq_moe_q4k", "kq_moe_q2k"):   # routed K-quant experts, gate/up shape, 64 tokens, top-6
        fmt = q8.Q8_KQ_Q4_K if case.endswith("q4k") else q8.Q8_KQ_Q2_K
        ids = torch.from_numpy(inputs.route_uniform(64, 6, 256, seed=0)).to(dev)
        W = torch.from_numpy(inputs.kq_weights(256 * 2048, 4096, fmt, seed=2).reshape(-1)).to(dev)
        x = torch.from_numpy(inputs.normal((64, 4096), seed=2)).to(dev)
        stride = 2048 * q8.q8_kq_row_bytes(4096, fmt)
        fn = lambda: q8.kq_moe_matmul(W, fmt, 256, stride, ids, x, False, 2048)
    elif case == "rmsnorm":   # RMSNorm feeding the quantiser at the long-prefill input, 4096 x 4096
        x = torch.from_numpy(inputs.normal((4096, 4096), seed=6)).to(dev)
        gamma = torch.from_numpy((1.0 + 0.1 * np.random.default_rng(6).standard_normal(4096)).astype(np.float32)).to(dev)
        fn = lambda: q8.rmsnorm_quantize(x, gamma, 1e-6)
    elif case == "moe_ffn":   # the routed expert FFN at the decode size (256 experts, 64 tokens, top-6)
        ids = torch.from_numpy(inputs.route_uniform(64, 6, 256, seed=0)).to(dev)
        Wg, Wu = (torch.from_numpy(inputs.weights(256 * 2048, 4096, seed=s)).to(dev) for s in (2, 4))
        Wd = torch.from_numpy(inputs.weights(256 * 4096, 2048, seed=5)).to(dev)
        wts = torch.from_numpy(np.random.default_rng(0).random((64, 6)).astype(np.float32)).to(dev)
        x = torch.from_numpy(inputs.normal((64, 4096), seed=2)).to(dev)
        fn = lambda: q8.moe_ffn(Wg, Wu, Wd, 256, 2048 * 128 * QB, 4096 * 64 * QB, ids, wts, x, 2048, 4096, 10.0)
    else:   # routed gate/up with Zipf(1.1) top-6: the layer slice's (moe_zipf) or 1024 tokens over 64 experts
        n, ne = (4096, 256) if case == "moe_zipf" else (1024, 64)
        ids = torch.from_numpy(inputs.route_zipf(n, 6, ne, s=1.1, seed=0)).to(dev)
        W = torch.from_numpy(inputs.weights(ne * 2048, 4096, seed=2)).to(dev)
        x = torch.from_numpy(inputs.normal((n, 4096), seed=2)).to(dev)
        fn = lambda: q8.moe_matmul(W, ne, 2048 * 128 * QB, ids, x, False, 2048)
    for _ in range(5):
        fn()
    torch.cuda.synchronize()
    assert q8.q8_last_error() == 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.profile_case:
        profile_case(args.profile_case)
        return 0
    if args.impl == "reference":
        r = run_reference(args, rank, world)
        if r is not None:
            print(json.dumps(r))
        return 0
    dist = dist_init(world)
    res = run_ours(args, rank, world, local, dist)
    if rank == 0:
        if not args.no_cpu:
            res["cpu_baseline"] = cpu_baseline(target_s=1.0)
        print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
