#!/usr/bin/env python3
"""Throughput of the In-Place TTT fast-weight layer on B300.

A step is one pass of the whole hot path -- gated up-projection, chunk-padded
conv + target projection, and the chunk-wise apply / residual / update loop --
over one batch of synthetic input, through ``ipttt_layer_forward``.  The
default workload is the 4B-scale layer: d=2560, d_ff=9728, L=131072 tokens,
chunk B=1024, MSE rule, batch 1, bf16 activations with an fp32 fast weight.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own
sequences (different seeds); nothing is exchanged on the data path
("scaling": "weak"); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from chunked_weight_mlp_place_b300 import inputs  # noqa: E402

METRIC = "fast-weight layer tokens/s and % roofline at d=2560,d_ff=9728,L=128k,B=1024"
METRIC_DOCS = "packed-document fast-weight layer tokens/s and % roofline at d=2560,d_ff=9728,128k tokens,B=1024"
METRIC_LAYERS = "multi-layer fast-weight MLP (token x layer)/s and % roofline, one call per step for all layers"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_SOURCES = {  # source files whose change invalidates a stored ncu traffic figure
    "gate_up": ["gemm_tc.cu", "common.cuh", "gemm.h"],
    "proj": ["gemm_tc.cu", "common.cuh", "gemm.h"],
    "apply": ["gemm_tc.cu", "common.cuh", "gemm.h"],
    "update": ["gemm_tc.cu", "common.cuh", "gemm.h"],
    "engine": ["gemm_tc.cu", "engine_tc.cuh", "common.cuh", "gemm.h"],
    "residual": ["elementwise.cu", "common.cuh"],
    "conv": ["elementwise.cu", "common.cuh"],
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="4b", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--B", type=int, default=None, help="chunk size override (the 4b_sweep points)")
    ap.add_argument("--L", type=int, default=None, help="sequence length override (small profiling cases)")
    ap.add_argument("--rule", choices=["mse", "add", "add_blockcausal"], default="mse")
    ap.add_argument("--layers", type=int, default=0,
                    help="this many layers' fast-weight MLPs in one call per step (0: one layer)")
    ap.add_argument("--docs", default=None, choices=sorted(inputs.DOC_MIXES),
                    help="pack the tokens as documents of this length mix (fast weight reset per document)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle work for the CPU baseline")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def flops_per_token(w):
    return 8 * w.d * w.d_ff + 2 * w.d * w.d


def chunk_counts(w, cu=None):
    """Chunks of every sequence (or packed document): the fast-weight updates a step makes."""
    if cu is None:
        return np.full(w.batch, w.L // w.B, dtype=np.int64)
    return (np.diff(np.asarray(cu, np.int64)) + w.B - 1) // w.B


def window_tokens(w, rule="mse", cu=None):
    """Tokens of the windows the library runs the MSE rule in (bf16, whole sequences, chunks
    below 1024 tokens): the largest of 1024, 768, 512, 256 holding at least two chunks and
    dividing L, with d and d_ff multiples of 256, where d (m - 1) >= 2 W for its m = W / B
    chunks; 0 where the chunks run one by one."""
    if rule != "mse" or cu is not None or w.dtype != "bf16" or w.d % 256 or w.d_ff % 256:
        return 0
    for W in (1024, 768, 512, 256):
        if W % (2 * w.B) == 0 and w.L % W == 0:
            return W if w.d * (W // w.B - 1) >= 2 * W else 0
    return 0


def window_flops(w):
    """FLOPs of the window GEMMs of a step: the masked Gram (kept pairs), the rows of the
    inverse, Zt = X^T Z and the output X Y (dense W x W operands)."""
    W = window_tokens(w)
    if not W:
        return 0.0
    m, B = W // w.B, w.B
    nwin = w.batch * (w.L // W)
    gram = 2.0 * w.d_ff * B * B * m * (m - 1) / 2
    inv = sum(2.0 * B * (j * B) * (j * B) for j in range(1, m))
    return nwin * (gram + inv + 2.0 * W * W * w.d_ff + 2.0 * W * W * w.d)


def roofline_tokens_per_s(w, peaks, cu=None):
    """The layer's roofline: the slower of all GEMM FLOPs at the dense bf16 peak
    and one fp32 read + write of W_o per chunk at the HBM bandwidth (per layer:
    several layers scale both terms alike)."""
    T = w.batch * w.L
    t_flop = flops_per_token(w) * T / (peaks["bf16_tflops"] * 1e12)
    t_hbm = int(chunk_counts(w, cu).sum()) * 2 * w.d_ff * w.d * 4 / (peaks["hbm_gbs"] * 1e9)
    return T / max(t_flop, t_hbm), ("tensor" if t_flop >= t_hbm else "hbm")


def kernel_work(w, name, cu=None, layers=1, rule="mse"):
    """Algorithmic FLOPs and bytes of ONE launch of kernel `name` in a step (with
    packed documents, the step's total over its launches of that kernel; with
    several layers, every launch covers all of them)."""
    if rule == "add_blockcausal" and name in ("scores", "apply", "group_sum"):
        # the quadratic form: kept (query, key) pairs per sequence = B^2 K (K-1) / 2
        K = w.L // w.B
        pairs = w.batch * w.B * w.B * K * (K - 1) / 2
        T = w.batch * w.L
        fl = {"scores": 2.0 * w.d_ff * pairs, "apply": 2.0 * T * w.d * w.d_ff + 2.0 * w.d * pairs,
              "group_sum": 2.0 * T * w.d * w.d_ff}[name]
        return fl * layers, 0.0
    fl, by = _kernel_work_one(w, name, cu)
    return fl * layers, by * layers


def _kernel_work_one(w, name, cu=None):
    T = w.batch * w.L
    n_chunks = chunk_counts(w, cu)
    steps = int(n_chunks.max())  # launches of the chunk kernels per step
    w_bytes = int(n_chunks.sum()) * 2.0 * w.d_ff * w.d * 4
    if name == "gate_up":
        return 4.0 * w.d * w.d_ff * T, 0.0
    if name == "proj":
        return 2.0 * w.d * w.d * T, 0.0
    if name == "apply":
        return 2.0 * w.d * w.d_ff * T / steps, 0.0
    if name == "update":
        return 2.0 * w.d * w.d_ff * T / steps, w_bytes / steps
    if name == "engine":  # the whole chunk loop (apply and update of every chunk) in one launch
        W = window_tokens(w, cu=cu)
        if W:  # windows of chunks: the fast weight is read and written once per window
            w_bytes = w.batch * (w.L // W) * 2.0 * w.d_ff * w.d * 4
        return 4.0 * w.d * w.d_ff * T, w_bytes
    if name == "window":
        return window_flops(w), 0.0
    if name == "conv":
        return 0.0, 2.0 * T * w.d * 2
    if name == "residual":
        return 0.0, T * w.d * (4 + 4 + 2 + 2 + 2) / steps
    return 0.0, 0.0


def source_sha(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "chunked_weight_mlp_place_b300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel, workload_key):
    """Per-launch DRAM bytes from the committed ncu summary, if the kernel's
    sources have not changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or kernel not in KERNEL_SOURCES:
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload_key, {}).get(kernel)
    if not e or e.get("source_sha") != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_id)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def nvidia_smi_id(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return dev


# ------------------------------------------------------------- CPU baseline
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(w, seconds):
    """Time the float64 oracle on the first chunks of sequence 0 of workload w.
    Returns (tokens/s, description, cores)."""
    from oracle import ipttt_oracle as orc  # test infrastructure: the CPU baseline only
    one = w.replace(batch=1)
    t0 = time.perf_counter()
    a = inputs.generate(one, seed=0, n_tokens=min(one.L, 64 * one.B))
    gen_s = time.perf_counter() - t0
    del gen_s

    def run(n):
        s = time.perf_counter()
        orc.layer_forward(a["X"][:n * one.B], a["E"][:n * one.B], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"],
                          a["P"], n * one.B, one.B, one.eta, "mse" if "mse" in one.rules else one.rules[0])
        return time.perf_counter() - s

    t1 = run(1)
    n = int(max(1, min(one.K, 64, round(seconds / max(t1, 1e-3)))))
    tn = run(n) if n > 1 else t1
    desc = (f"float64 oracle, first {n} of {one.K} chunks ({n * one.B} tokens) of one sequence of the "
            f"{w.name} workload (d={w.d}, d_ff={w.d_ff}, B={w.B})")
    return n * one.B / tn, desc, blas_threads(), n * one.B


def oracle_sample_docs(w, cu, seconds):
    """Time the float64 oracle on whole documents of the packed workload,
    shortest first, until about `seconds` of work.  Returns (tokens/s, description, cores)."""
    from oracle import ipttt_oracle as orc  # test infrastructure: the CPU baseline only
    lens = np.diff(cu)
    order = np.argsort(lens, kind="stable")
    a = inputs.generate(w.replace(batch=1), seed=0)
    done, tok, el = 0, 0, 0.0
    for i in order:
        r = slice(int(cu[i]), int(cu[i + 1]))
        s = time.perf_counter()
        orc.layer_forward_varlen(a["X"][r], a["E"][r], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"],
                                 [0, int(lens[i])], w.B, w.eta, "mse")
        el += time.perf_counter() - s
        tok += int(lens[i])
        done += 1
        if el >= seconds:
            break
    desc = (f"float64 oracle over the {done} shortest of {len(lens)} packed documents ({tok} tokens) of the "
            f"{w.name} workload (d={w.d}, d_ff={w.d_ff}, B={w.B})")
    return tok / el, desc, blas_threads()


# ------------------------------------------------------------------ ranks
def rank_seed(rank):
    """Seed of the inputs rank `rank` draws: every rank runs its own sequences
    (weak scaling, no data shared between ranks and no collective on the path)."""
    return 1000 + rank


def max_over_ranks(value, dist, device):
    """The largest `value` over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ reference arm
def run_reference(args, w, rank, world):
    if rank != 0:
        return
    from oracle import ipttt_oracle as orc  # the reference arm is the oracle, on the host
    one = w.replace(batch=1)
    a = inputs.generate(one, seed=0, n_tokens=one.B)
    rule = "mse" if args.rule == "mse" else "add"  # the block-causal form has the additive rule's outputs

    def step():
        if args.docs:  # one document of one chunk through the packed-document oracle
            orc.layer_forward_varlen(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"],
                                     [0, one.B], one.B, one.eta, rule)
        else:
            orc.layer_forward(a["X"], a["E"], a["W_g"], a["W_u"], a["W_o0"], a["conv_w"], a["P"], one.B, one.B,
                              one.eta, rule)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    tok = args.steps * one.B
    val = tok / el
    unit = "(token x layer)/s" if args.layers else "tokens/s"  # one layer of one chunk per step
    sample = f"one chunk ({one.B} tokens) of the {w.name} workload per step, float64 oracle"
    print(json.dumps({
        "impl": "reference", "metric": metric_of(args), "value": val, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, args, world,
                            inputs.doc_boundaries(w.batch * w.L, seed=0, mix=args.docs) if args.docs else None),
        "cpu_baseline": {"value": val, "unit": unit, "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def metric_of(args):
    return METRIC_LAYERS if args.layers else (METRIC_DOCS if args.docs else METRIC)


def config_of(w, args, world, cu=None):
    docs = ""
    if cu is not None:
        lens = np.diff(cu)
        docs = (f" packed as {len(lens)} documents of {int(lens.min())}..{int(lens.max())} tokens "
                f"({args.docs} mix), fast weight reset per document;")
    if args.layers:
        docs += f" {args.layers} layers (own weights and hidden states each, shared token embeddings);"
    return {"workload": f"{w.name}: batch={w.batch} L={w.L} B={w.B} d={w.d} d_ff={w.d_ff} rule={args.rule} "
                        f"eta={w.eta}{docs} bf16 activations, fp32 fast weight",
            "batch_per_gpu": w.batch, "L": w.L, "B": w.B, "d": w.d, "d_ff": w.d_ff, "rule": args.rule,
            "parallelism": f"sequence-sharded x{world} (no collective)",
            "l2": "inputs (X, E, Z: >=0.6 GB each) exceed the 126 MB L2; no flush"}


# ---------------------------------------------------------------------- main
def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = inputs.workload(args.workload)
    if args.B:
        w = w.replace(B=args.B)
    if args.L:
        w = w.replace(L=args.L)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import chunked_weight_mlp_place_b300 as ip
    from chunked_weight_mlp_place_b300.build import build

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0 or not os.path.exists(ip._lib.LIB_PATH):
        build()
    if dist:
        dist.barrier()
    ip.lib()

    peaks, peaks_kind = load_peaks()
    nl = max(0, args.layers)
    a = inputs.generate(w, seed=rank_seed(rank))
    if nl:  # each layer its own hidden states and weights, drawn from seeds of their own
        per = [a] + [inputs.generate(w, seed=rank_seed(rank) + 7919 * l, want=("X", "W_g", "W_u", "W_o0", "conv_w", "P"))
                     for l in range(1, nl)]
        for k in ("X", "W_g", "W_u", "W_o0", "conv_w", "P"):
            a[k] = np.stack([q[k] for q in per])
        del per
    bf = torch.bfloat16
    dev = torch.device("cuda", local_rank)
    h = {k: torch.from_numpy(a[k]) for k in ("X", "E", "W_g", "W_u", "P")}
    h = {k: v.to(bf) for k, v in h.items()}
    h["W_o0"] = torch.from_numpy(a["W_o0"])
    h["conv_w"] = torch.from_numpy(a["conv_w"])
    del a
    d = {k: v.to(dev) for k, v in h.items()}
    T = w.batch * w.L
    O = torch.empty(((nl,) if nl else ()) + (T, w.d), dtype=bf, device=dev)
    Wf = torch.empty(((nl,) if nl else ()) + (w.batch, w.d_ff, w.d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    cu = inputs.doc_boundaries(T, seed=rank, mix=args.docs) if args.docs else None
    if cu is not None:
        Wf = torch.empty(len(cu) - 1, w.d_ff, w.d, dtype=torch.float32, device=dev)

    def step():
        if nl:
            ip.layers_forward(d["X"], d["E"], d["W_g"], d["W_u"], d["W_o0"], d["conv_w"], d["P"], w.L, w.B, w.eta,
                              args.rule, O, Wf, stream=stream)
        elif cu is not None:
            ip.layer_forward_varlen(d["X"], d["E"], d["W_g"], d["W_u"], d["W_o0"], d["conv_w"], d["P"], cu, w.B,
                                    w.eta, args.rule, O, Wf, stream=stream)
        else:
            ip.layer_forward(d["X"], d["E"], d["W_g"], d["W_u"], d["W_o0"], d["conv_w"], d["P"], w.L, w.B, w.eta,
                             args.rule, O, Wf, stream=stream)

    for _ in range(max(args.warmup, 1)):
        step()
    if ip.sync_status(stream) != 0:
        raise RuntimeError("device error during warm-up")
    launches_per_step = ip.last_launch_count()

    # ---- timed region: K plain steps (no per-launch events), CUDA events on the launching stream
    sampler = ClockSampler(nvidia_smi_id(torch, dev)) if rank == 0 else None
    if sampler:
        sampler.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    elapsed_ms = e0.elapsed_time(e1)
    if ip.sync_status(stream) != 0:
        raise RuntimeError("device error in the timed region")
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)
    tokens = world * T * args.steps * max(1, nl)
    value = tokens / (elapsed_ms / 1e3)

    # ---- a second, instrumented pass: every launch bracketed by CUDA events on its stream
    # (the per-kernel times of the roofline block; the headline above has no such events)
    n_kt = max(1, min(args.steps, 10))
    ip.kernel_timing(True)
    e0.record(stream)
    for _ in range(n_kt):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ip.kernel_timing(False)
    kt_ms_per_step = e0.elapsed_time(e1) / n_kt
    if ip.sync_status(stream) != 0:
        raise RuntimeError("device error in the instrumented pass")
    kt = ip.kernel_timing_read()

    # ---- several layers: the same layers as one call each, for comparison
    sequential = None
    if nl:
        def step_seq():
            for l in range(nl):
                ip.layer_forward(d["X"][l], d["E"], d["W_g"][l], d["W_u"][l], d["W_o0"][l], d["conv_w"][l],
                                 d["P"][l], w.L, w.B, w.eta, args.rule, O[l], Wf[l], stream=stream)

        step_seq()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step_seq()
        e1.record(stream)
        torch.cuda.synchronize()
        t_seq = max_over_ranks(e0.elapsed_time(e1), dist, dev)
        sequential = {"value": world * T * nl * args.steps / (t_seq / 1e3), "unit": "(token x layer)/s",
                      "ms_per_step": t_seq / args.steps, "launches_per_step": ip.last_launch_count() * nl}

    # ---- end to end: pinned host inputs in, O and W_final out, every step
    e2e = None
    if not args.no_e2e:
        hp = {k: v.pin_memory() for k, v in h.items()}
        O_h = torch.empty(O.shape, dtype=bf).pin_memory()
        W_h = torch.empty(Wf.shape, dtype=torch.float32).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in hp.values())
        d2h = O_h.numel() * 2 + W_h.numel() * 4

        def e2e_step():
            for k, v in hp.items():
                d[k].copy_(v, non_blocking=True)
            step()
            O_h.copy_(O, non_blocking=True)
            W_h.copy_(Wf, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(1, min(args.steps, 5))
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        t_e2e = e0.elapsed_time(e1)
        t_e2e = max_over_ranks(t_e2e, dist, dev)
        e2e = {"value": world * T * max(1, nl) * n_e2e / (t_e2e / 1e3),
               "unit": "(token x layer)/s" if nl else "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e}

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel
    dom = max(kt, key=lambda k: kt[k][1]) if kt else None
    roof = None
    if dom:
        n_launch, total_ms = kt[dom]
        avg_s = total_ms / n_launch / 1e3
        fl, by = kernel_work(w, dom, cu, max(1, nl), args.rule)
        t_f = fl / (peaks["bf16_tflops_sustained"] * 1e12) if fl else 0.0
        t_b = by / (peaks["hbm_gbs"] * 1e9) if by else 0.0
        wk = f"{w.name}-B{w.B}-{args.rule}" + (f"-docs-{args.docs}" if args.docs else "")
        if t_f >= t_b:
            roof = {"bound": "tensor", "kernel": dom, "achieved": fl / avg_s / 1e12,
                    "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                    "peak_kind": f"{peaks_kind} sustained dense bf16 (kernel timed inside a long step)"}
        else:
            roof = {"bound": "hbm", "kernel": dom, "achieved": by / avg_s / 1e9, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "peak_kind": f"{peaks_kind} copy bandwidth"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["traffic"] = stored_traffic(dom, wk)
        roof["avg_launch_ms"] = avg_s * 1e3
        roof["launches"] = n_launch
        roof["timing"] = (f"per-launch CUDA events in a separate pass of {n_kt} steps "
                          f"({kt_ms_per_step:.3f} ms/step there, against {elapsed_ms / args.steps:.3f} without events)")
    kernels = {k: {"launches": n, "total_ms": round(ms, 4), "avg_us": round(ms / n * 1e3, 2),
                   "share": round(ms / max(1e-9, sum(x[1] for x in kt.values())), 4)} for k, (n, ms) in kt.items()}

    roof_tps, layer_bound = roofline_tokens_per_s(w, peaks, cu)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        if cu is not None:
            v, desc, cores = oracle_sample_docs(w, cu, args.cpu_seconds)
        else:
            v, desc, cores, _ = oracle_sample(w, args.cpu_seconds)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
    ms_step = elapsed_ms / args.steps
    out = {
        "metric": metric_of(args), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, args, world, cu),
        "pct_roofline": 100.0 * value / world / roof_tps,
        "layer_roofline": {"tokens_per_s": roof_tps, "bound": layer_bound,
                           "tflops_achieved": flops_per_token(w) * value / 1e12,
                           "peaks": f"{peaks_kind}: {peaks['bf16_tflops']} TFLOP/s bf16 burst, "
                                    f"{peaks['hbm_gbs']} GB/s"},
        "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
    }
    W = window_tokens(w, args.rule, cu)
    if W and not nl:
        # the windowed form's own bound: its FLOPs (the window GEMMs added) at the tensor peak,
        # and the fast weight read and written once per window
        t_f = (flops_per_token(w) * T + window_flops(w)) / (peaks["bf16_tflops"] * 1e12)
        t_b = w.batch * (w.L // W) * 2 * w.d_ff * w.d * 4 / (peaks["hbm_gbs"] * 1e9)
        out["window_form"] = {"window_tokens": W, "chunks_per_window": W // w.B,
                              "roofline_tokens_per_s": T / max(t_f, t_b),
                              "pct_roofline": 100.0 * value / world / (T / max(t_f, t_b))}
    if nl:
        out["unit"] = "(token x layer)/s"
        out["one_call_per_layer"] = sequential
    print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
