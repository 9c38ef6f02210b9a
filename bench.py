#!/usr/bin/env python
"""Throughput of the streamed-layer training step on one GB300 (per rank).

One step = one mt_train_step of the decoder workload: stream every unit's
bf16 weights host->device through two buffers, forward with checkpoints,
fused head + cross entropy, segment recompute + backward, K-slab gradient
offload, host accumulate + Adam on the FP32 master (all through libmt.so).

The default workload is the 7B decoder (2 x 4096 tokens, C = 4, K = 12);
``--config`` picks another. Prints one JSON line (rank 0):
  value  tokens/s over all ranks, token/label arrays already in device memory,
         timed with per-launch profiling off
  e2e    the same through mt_train_step with host token/label arrays
  roofline  the dominant kernel (the tcgen05 GEMM): algorithmic FLOPs of its
         launches / their CUDA-event device time, over a separate profiled
         pass of the same steps
  step_roofline  model FLOPs at the bf16 peak vs weight + gradient bytes over
         the measured host link, whichever is slower
  cpu_baseline  the oracle on this host's cores on a bounded sample
``--impl reference`` times the oracle (plain numpy CPU restatement) instead.
``--kernel gemm --shape M,N,K`` runs one GEMM shape (for profiler captures).
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

import synth  # noqa: E402

METRIC = "train tokens/s & model TFLOPS on 1 GB300 vs min(TC peak, host-link) roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def model_flops(shape, B, s):
    """6 * N_mm + 6 * L * s * H * hd per token (causal attention), times B*s."""
    d, f, V = shape.d_model, shape.ffn_dim, shape.vocab
    qkv = (shape.n_heads + 2 * shape.n_kv_heads) * shape.head_dim
    hq = shape.n_heads * shape.head_dim
    n_mm = shape.n_layers * (qkv * d + d * hq + 2 * f * d + d * f) + V * d
    per_tok = 6.0 * n_mm + 6.0 * shape.n_layers * s * shape.n_heads * shape.head_dim
    return per_tok * B * s


def workload_desc(shape):
    return (f"{shape.name} decoder: {shape.n_layers} layers, d={shape.d_model}, {shape.n_heads}x{shape.head_dim} "
            f"heads ({shape.n_kv_heads} KV), ffn={shape.ffn_dim}, vocab={shape.vocab}, batch={shape.batch}, "
            f"seq={shape.seq}, ckpt_interval={shape.ckpt_interval}, slabs={shape.n_slabs}")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.device)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

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
        self.t.join(timeout=2)
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


# --------------------------------------------------------------- host link
def host_link_probe(torch, dev, nbytes=1 << 30, reps=5):
    """Pinned cudaMemcpyAsync bandwidth: H2D alone, D2H alone, both at once."""
    n = nbytes // 2
    hs = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    hd = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    d1 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    d2 = torch.empty(n, dtype=torch.bfloat16, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        best = 1e30
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            best = min(best, time.perf_counter() - t0)
        return best

    def h2d():
        with torch.cuda.stream(s1):
            d1.copy_(hs, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            hd.copy_(d2, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_h, t_d, t_b = timed(h2d), timed(d2h), timed(both)
    gb = nbytes / 1e9
    return {"h2d_gbs": gb / t_h, "d2h_gbs": gb / t_d, "bidir_h2d_gbs": gb / t_b, "bidir_d2h_gbs": gb / t_b}


def host_adam_probe(mt, n=44_044_288, reps=4, threads=0, keep_grads=False):
    """Rate of the library's per-unit host pass (bf16 slab in, FP32 grad out
    if kept, Adam, bf16 emit) on one 1.1B-layer-sized slice, in GB/s at the
    pass's algorithmic bytes (32 B/param with the grad array, 28 without)."""
    rng = np.random.default_rng(0)
    w = rng.standard_normal(n).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    g = np.empty(n, np.float32)
    slab = mt.host_to_bf16(w * 1e-3)
    store = np.empty(n, np.uint16)
    best = 1e30
    for t in range(1, reps + 1):
        t0 = time.perf_counter()
        mt.host_adam_slab(w, m, v, slab, t, 1e-3, 0.9, 0.999, 1e-8, grad_out=g if keep_grads else None,
                          store=store, threads=threads)
        best = min(best, time.perf_counter() - t0)
    return host_bytes_per_param(keep_grads) * n / best / 1e9


def host_bytes_per_param(keep_grads):
    """Host DRAM bytes of the per-unit pass: bf16 gradient in (2), master, m,
    v read and written (24), bf16 store out (2), FP32 gradient out (4) if kept."""
    return 32.0 if keep_grads else 28.0


def _union(iv):
    """Merge [start, end) intervals; returns the sorted disjoint list."""
    out = []
    for a, b in sorted(iv):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return out


def _overlap(iv, cover):
    """Total length of the intervals `iv` that lies inside the union `cover`."""
    tot = 0.0
    for a, b in iv:
        for c, d in cover:
            lo, hi = max(a, c), min(b, d)
            if hi > lo:
                tot += hi - lo
    return tot


def _subtract(iv, cover):
    """The parts of the intervals `iv` outside the union `cover`."""
    out = []
    for a, b in iv:
        cur = a
        for c, d in cover:
            if d <= cur or c >= b:
                continue
            if c > cur:
                out.append((cur, c))
            cur = max(cur, d)
        if cur < b:
            out.append((cur, b))
    return out


def timeline_summary(tl):
    """Copy/compute overlap and host/GPU concurrency of one profiled step."""
    def ivs(stream):
        return [(r["start_ms"], r["end_ms"]) for r in tl if r["stream"] == stream]
    comp = _union(ivs("compute"))
    host = _union(ivs("host_adam"))
    host_any = _union(ivs("host_adam") + ivs("host_adam_prev"))  # with the previous step's tail
    end = max(r["end_ms"] for r in tl) if tl else 0.0
    out = {"span_ms": end, "gpu_busy_ms": sum(b - a for a, b in comp),
           "host_adam_busy_ms": sum(b - a for a, b in host),
           "host_adam_prev_step_ms": sum(b - a for a, b in _union(ivs("host_adam_prev"))),
           "host_and_gpu_busy_ms": _overlap(host, comp)}
    # a copy costs the device time only where it runs in an idle gap of the
    # compute stream while the host optimizer is not busy
    gaps0 = [(b0, a1) for (a0, b0), (a1, b1) in zip(comp, comp[1:]) if a1 > b0]
    host_any = _union(ivs("host_adam") + ivs("host_adam_prev"))
    exposed_gaps = _subtract(gaps0, host_any)
    for k in ("h2d", "d2h"):
        iv = ivs(k)
        t = sum(b - a for a, b in iv)
        ex = _overlap(_union(iv), exposed_gaps)
        out[k] = {"copies": len(iv), "ms": t, "hidden_under_compute_ms": _overlap(iv, comp),
                  "hidden_frac": _overlap(iv, comp) / t if t else None,
                  "exposed_ms": ex, "not_exposed_frac": 1.0 - ex / t if t else None}
    # Compute-stream idle gaps between the step's first and last launch, by
    # what else was busy: the host optimizer (the device work waits for its
    # updated weights or free slabs), only a copy (waiting on the host link),
    # or neither (launch overhead). Host intervals use the host clock from the
    # start of the call, device ones CUDA events from the first launch.
    gaps = [(b0, a1) for (a0, b0), (a1, b1) in zip(comp, comp[1:]) if a1 > b0]
    copies = _union(ivs("h2d") + ivs("d2h"))
    g_total = sum(b - a for a, b in gaps)
    g_host = _overlap(gaps, host_any)
    g_copy = _overlap(_subtract(gaps, host_any), copies)
    out["gpu_idle"] = {"ms": g_total, "while_host_optimizer_busy_ms": g_host, "copy_only_ms": g_copy,
                       "neither_ms": g_total - g_host - g_copy}
    heads = [r for r in tl if r["stream"] == "compute" and r["cls"] == "ce"]
    if heads:
        out["forward_end_ms"] = min(r["start_ms"] for r in heads)
    return out


def write_trace(tl, path):
    """Chrome / Perfetto trace (one track per stream and one for the host worker)."""
    ev = [{"name": r["cls"], "ph": "X", "ts": r["start_ms"] * 1e3, "dur": max(r["end_ms"] - r["start_ms"], 0.0) * 1e3,
           "pid": 0, "tid": r["stream"]} for r in tl]
    with open(path, "w") as f:
        json.dump({"traceEvents": ev, "displayTimeUnit": "ms"}, f)


def gemm_traffic_record():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current GEMM source (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    src = os.path.join(ROOT, "host_memory_resident_gb300", "csrc", "gemm_tc.cu")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec if rec.get("gemm_source_sha") == h else None


# ----------------------------------------------------------- CPU baseline
def oracle_sample(shape, max_tokens=16384):
    """Time the oracle on a bounded sample of the workload and compose the
    full step. Timed directly on one sequence of ss = min(seq, max_tokens)
    tokens at full width: one layer's forward (oracle.layer_forward) and
    backward (oracle.layer_backward), the attention core inside them
    (oracle.ops.attention_fwd / attention_bwd) on its own, and the head
    (final RMSNorm, logits, cross entropy and their backward). The oracle's
    step runs every layer's forward twice (forward, recompute from the
    checkpoints) and its backward once: t_layer = 2 t_fwd + t_bwd. For a
    longer sequence s the attention part is scaled by (s / ss)^2 and the
    rest of the layer and the head by s / ss. Then
    step = B (L t_layer + t_head) + Adam on the N parameters (a 2^24 slice
    scaled)."""
    import oracle
    from oracle import ops
    s = shape.seq
    ss = min(s, max_tokens)
    d, hd, H, Hkv = shape.d_model, shape.head_dim, shape.n_heads, shape.n_kv_heads
    sh1 = shape.with_(n_layers=1, ckpt_interval=1)
    lay = oracle.build_layout(sh1)
    master = synth.init_master(lay.n_total, lay.segments(), seed=0)
    P = {t.name: master[t.offset:t.offset + t.size].reshape(t.shape) for t in lay.units[1].tensors}
    Ph = {t.name: master[t.offset:t.offset + t.size].reshape(t.shape) for t in lay.units[2].tensors}
    rng = np.random.default_rng(0)
    x = rng.standard_normal((ss, d)).astype(np.float32)
    dy = (rng.standard_normal((ss, d)) * 1e-3).astype(np.float32)
    cos, sin = ops.rope_tables(ss, hd, shape.rope_theta, np.float32)
    t0 = time.perf_counter()
    _, cache = oracle.layer_forward(sh1, P, x, cos, sin, 1, ss)
    t1 = time.perf_counter()
    oracle.layer_backward(sh1, P, dy, cache, cos, sin, 1, ss)
    t2 = time.perf_counter()
    t_layer_ss = 2.0 * (t1 - t0) + (t2 - t1)
    q = rng.standard_normal((1, ss, H, hd)).astype(np.float32)
    k = rng.standard_normal((1, ss, Hkv, hd)).astype(np.float32)
    v = rng.standard_normal((1, ss, Hkv, hd)).astype(np.float32)
    t0 = time.perf_counter()
    ops.attention_fwd(q, k, v)
    t1 = time.perf_counter()
    ops.attention_bwd(q, k, v, q)
    t2 = time.perf_counter()
    t_att_ss = min(2.0 * (t1 - t0) + (t2 - t1), t_layer_ss)
    labels = rng.integers(0, shape.vocab, size=ss)
    t0 = time.perf_counter()
    xh, rf = ops.rmsnorm_fwd(x, Ph["final_norm"], shape.rms_eps)
    _, dlogits = ops.cross_entropy_fwd_bwd(ops.linear_fwd(xh, Ph["head"]), labels)
    dxh, _ = ops.linear_bwd(dlogits, xh, Ph["head"])
    ops.rmsnorm_bwd(dxh, x, Ph["final_norm"], rf)
    t_head_ss = time.perf_counter() - t0
    del master, cache
    r = s / ss
    t_layer = (t_layer_ss - t_att_ss) * r + t_att_ss * r * r
    t_head = t_head_ss * r
    n = 1 << 24
    w = rng.standard_normal(n).astype(np.float32)
    g = rng.standard_normal(n).astype(np.float32) * 1e-3
    t0 = time.perf_counter()
    oracle.adam_update(w, np.zeros(n, np.float32), np.zeros(n, np.float32), g, 1, shape.lr, shape.beta1,
                       shape.beta2, shape.adam_eps, dtype=np.float32)
    t_adam_slice = time.perf_counter() - t0
    lay_full = oracle.build_layout(shape)
    t_adam = t_adam_slice * lay_full.n_total / n
    t_step = shape.batch * (shape.n_layers * t_layer + t_head) + t_adam
    scaled = f"timed at {ss} of {s} tokens, attention scaled by (s/ss)^2, the rest by s/ss; " if ss < s else ""
    return {
        "value": shape.batch * s / t_step, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
        "sample": (f"composed from one full-width layer's forward and backward, its attention core and the head on "
                   f"one sequence (float32 numpy; {scaled}t_layer {t_layer:.2f} s = 2 forwards + 1 backward, of which "
                   f"attention {t_att_ss * r * r:.2f} s; t_head {t_head:.2f} s) + Adam on 2^24 elements scaled to "
                   f"{lay_full.n_total} params; step = {shape.batch} x ({shape.n_layers} t_layer + t_head) + Adam = "
                   f"{t_step:.1f} s"),
    }


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return int(max((i.get("num_threads", 1) for i in info), default=1))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ ranks
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def reduce_over_ranks(pg, x, op):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=op(pg))
    return float(t.item())


def max_over_ranks(pg, x):
    return reduce_over_ranks(pg, x, lambda d: d.ReduceOp.MAX)


def sum_over_ranks(pg, x):
    return reduce_over_ranks(pg, x, lambda d: d.ReduceOp.SUM)


# ------------------------------------------------------------------- arms
def config_dict(args, shape, world, n_total):
    """The workload description both arms print (identical keys and values)."""
    nm = getattr(args, "micro_batches", 1)
    extra = {"micro_batches": nm, "note": f"gradient accumulation over {nm} micro-batches of {shape.batch} x "
                                          f"{shape.seq} tokens, one host Adam per step"} if nm > 1 else {}
    return {"workload": workload_desc(shape), **extra,
            "global_batch_tokens": shape.batch * shape.seq * world * nm,
            "seq_len": shape.seq,
            "parallelism": f"replicas x{world} (no collective)" if world > 1 else "single GPU",
            "overlap_adam": bool(args.overlap),
            "fp32_grad_array": bool(args.keep_grads),
            "fused_epilogues": not args.unfused,
            "keep_attention": bool(args.keep_attention),
            "l2": "inputs larger than L2: each step streams the whole bf16 store "
                  f"({2.0 * n_total / 1e9:.2f} GB) and the activations"}


REFERENCE_MAX_TOKENS = 512   # per-step sample of the reference arm (see run_reference)


def run_reference(args, shape, world, rank, pg):
    """The oracle as it stands, on this host's cores (rank 0 only)."""
    if rank != 0:
        return 0
    import oracle
    vals = []
    base = None
    for i in range(args.warmup + args.steps):
        # each step is a bounded sample (sequences over 512 tokens timed at
        # 256 and 512 and extended) so the whole run takes a few minutes
        b = oracle_sample(shape, max_tokens=REFERENCE_MAX_TOKENS)
        if i >= args.warmup:
            vals.append(b["value"])
            base = b
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": shape.batch * shape.seq / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded uniform token ids, normal(0, 0.02) weights)",
        "config": config_dict(args, shape, world, oracle.build_layout(shape).n_total),
        "cpu_baseline": {k: base[k] for k in ("value", "unit", "cores", "kind", "sample")},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gemm_kernel(args):
    """One GEMM shape through mt_k_gemm (a small case for profiler captures).
    --epilogue swiglu|swiglu_bwd|rope times the fused forms at the same
    M, N, K (N = 2f for SwiGLU forward, f for its backward, the QKV width for
    RoPE with 64-wide heads, 2048-token sequences); wgrad times the weight
    gradient G [M, N] over K tokens (split along K when it has few tiles),
    wgrad_nosplit the same product unsplit."""
    import torch
    import host_memory_resident_gb300 as mt
    M, N, K = (int(x) for x in args.shape.split(","))
    torch.manual_seed(0)
    dev = "cuda"
    mt.k_gemm_tile_policy(args.tile)
    A = torch.randn(M, K, device=dev).to(torch.bfloat16)
    epi = args.epilogue
    if epi in ("wgrad", "wgrad_nosplit"):
        # weight gradient G [M, N] = dY^T X over K tokens, both token-major
        A = torch.randn(K, M, device=dev).to(torch.bfloat16)
        B = (torch.randn(K, N, device=dev) / math.sqrt(K)).to(torch.bfloat16)
        Cm = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        ws = torch.empty(mt.k_gemm_wgrad_ws(M, N), device=dev) if epi == "wgrad" else None
        fn = lambda: mt.k_gemm_wgrad(A, B, Cm, ws)  # noqa: E731
    elif epi == "swiglu_bwd":
        B = (torch.randn(K, N, device=dev) / math.sqrt(K)).to(torch.bfloat16)  # down weight [d, f]
        gu = torch.randn(M, 2 * N, device=dev).to(torch.bfloat16)
        Cm = torch.empty(M, 2 * N, device=dev, dtype=torch.bfloat16)
        fn = lambda: mt.k_gemm_swiglu_bwd(A, B, gu, Cm)  # noqa: E731
    else:
        B = (torch.randn(N, K, device=dev) / math.sqrt(K)).to(torch.bfloat16)
        Cm = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
        if epi == "swiglu":
            a = torch.empty(M, N // 2, device=dev, dtype=torch.bfloat16)
            fn = lambda: mt.k_gemm_swiglu_fwd(A, B, Cm, a)  # noqa: E731
        elif epi == "rope":
            hd, seq = 64, 2048
            pos = torch.arange(seq, device=dev, dtype=torch.float64)[:, None]
            inv = 10000.0 ** (-torch.arange(0, hd, 2, device=dev, dtype=torch.float64) / hd)
            ct, st = torch.cos(pos * inv).float().contiguous(), torch.sin(pos * inv).float().contiguous()
            rot = (N // hd - (N // hd) // 10) * hd  # q and k heads of a 32 + 4 + 4 head layout
            fn = lambda: mt.k_gemm_rope(A, B, Cm, ct, st, rot, hd, seq)  # noqa: E731
        else:
            fn = lambda: mt.k_gemm(A, B, Cm)  # noqa: E731
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(args.iters):
        fn()
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / args.iters
    err = 0.0
    if epi is None:
        ref = A[:256].float() @ B.float().t()
        err = (Cm[:256].float() - ref).abs().max().item() / ref.abs().max().item()
    if epi in ("wgrad", "wgrad_nosplit"):
        ref = A[:, :256].float().t() @ B.float()
        err = (Cm[:256].float() - ref).abs().max().item() / ref.abs().max().item()
    print(json.dumps({"kernel": "gemm_abt" + (f"+{epi}" if epi else ""), "M": M, "N": N, "K": K, "tile": args.tile, "ms": ms,
                      "splits": mt.k_gemm_splitk(M, N, K) if epi == "wgrad" else 1,
                      "tflops": 2.0 * M * N * K / ms / 1e9, "max_rel_err_rows0_255": err}), flush=True)
    return 0 if err < 2e-2 else 1


def run_misc_kernels(args):
    """The memory-bound kernels of one 7B layer step at the workload's sizes
    (M = 8192 tokens, d = 4096, f = 11008, 32 + 32 heads of 128, V = 32000,
    the head's logits for every token), each timed with CUDA events and
    reported as GB/s of algorithmic bytes against the measured HBM copy
    bandwidth. The RMSNorm input is the fp32 residual stream, as in the step.
    Inputs of each kernel exceed L2 (129 MB) except the RoPE tables and norm
    weights."""
    import torch
    import host_memory_resident_gb300 as mt
    torch.manual_seed(0)
    dev = "cuda"
    M, d, f, H, Hkv, hd, V, s = 8192, 4096, 11008, 32, 32, 128, 32000, 4096
    B = M // s
    qn = (H + 2 * Hkv) * hd
    mc = (1 << 28) // V
    bf = torch.bfloat16
    x = torch.randn(M, d, device=dev)                 # fp32 residual stream
    w = (1 + 0.1 * torch.randn(d, device=dev)).to(bf)
    y = torch.empty(M, d, device=dev, dtype=bf)
    rstd = torch.empty(M, device=dev)
    dy = torch.randn(M, d, device=dev)
    dres = torch.randn(M, d, device=dev)
    dx32 = torch.empty(M, d, device=dev)
    dxb = torch.empty(M, d, device=dev, dtype=bf)
    part = torch.empty(mt.k_rmsnorm_bwd_parts(M), d, device=dev)
    dw = torch.empty(d, device=dev, dtype=bf)
    qkv = torch.randn(M, qn, device=dev).to(bf)
    pos = torch.arange(s, device=dev, dtype=torch.float64)[:, None]
    inv = 10000.0 ** (-torch.arange(0, hd, 2, device=dev, dtype=torch.float64) / hd)
    cos_t, sin_t = torch.cos(pos * inv).float().contiguous(), torch.sin(pos * inv).float().contiguous()
    gu = torch.randn(M, 2 * f, device=dev).to(bf)
    a = torch.empty(M, f, device=dev, dtype=bf)
    da = torch.randn(M, f, device=dev).to(bf)
    dgu = torch.empty(M, 2 * f, device=dev, dtype=bf)
    logits = torch.randn(mc, V, device=dev)
    labels = torch.randint(0, V, (mc,), device=dev, dtype=torch.int32)
    dz = torch.empty(mc, V, device=dev, dtype=bf)
    loss_rows = torch.empty(mc, device=dev)
    cases = [
        ("rmsnorm_fwd", lambda: mt.k_rmsnorm_fwd(x, w, y, rstd, 1e-5), 6.0 * M * d + 4.0 * M + 2.0 * d),
        ("rmsnorm_bwd (+ column sums)", lambda: mt.k_rmsnorm_bwd(dy, x, w, rstd, dres, dx32, dxb, part, dw),
         (4.0 + 4.0 + 4.0 + 4.0 + 2.0) * M * d + 4.0 * M),
        ("rope (q and k heads, in place)", lambda: mt.k_rope(qkv, B, s, H + Hkv, hd, cos_t, sin_t),
         4.0 * M * (H + Hkv) * hd),
        ("swiglu_fwd", lambda: mt.k_swiglu_fwd(gu, a), 6.0 * M * f),
        ("swiglu_bwd", lambda: mt.k_swiglu_bwd(da, gu, dgu), 10.0 * M * f),
        ("cross_entropy (one logits chunk)", lambda: mt.k_cross_entropy(logits, labels, dz, loss_rows, 1.0 / M),
         6.0 * mc * V),
    ]
    pk, pk_kind = peaks()
    peak = pk.get("hbm_gbs")
    for name, fn, nbytes in cases:
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.iters):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.iters
        gbs = nbytes / (ms / 1e3) / 1e9
        print(json.dumps({"kernel": name, "ms": ms, "algorithmic_bytes": nbytes, "gbs": gbs, "hbm_peak_gbs": peak,
                          "peak_source": pk_kind, "frac": gbs / peak if peak else None}), flush=True)
    return 0


def run_attn_kernel(args):
    """One attention forward shape through mt_k_attn_fwd (profiler captures)."""
    import torch
    import host_memory_resident_gb300 as mt
    B, s, H, Hkv, hd = (int(x) for x in args.shape.split(","))
    torch.manual_seed(0)
    qkv = torch.randn(B * s, (H + 2 * Hkv) * hd, device="cuda").to(torch.bfloat16)
    o = torch.empty(B * s, H * hd, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(B, H, s, device="cuda")
    fwd = mt.k_attn_fwd_mma if args.legacy else mt.k_attn_fwd
    if args.backward:
        fwd(qkv, o, lse, B, s, H, Hkv, hd)
        dout = torch.randn(B * s, H * hd, device="cuda").to(torch.bfloat16)
        delta = torch.empty(B, H, s, device="cuda")
        dqkv = torch.empty_like(qkv)
        bwd = mt.k_attn_bwd_mma if args.legacy else mt.k_attn_bwd
        if args.rope:
            # RoPE tables [s, hd/2] (base 10000): the backward rotates dq, dk back in its stores
            inv = 10000.0 ** (-torch.arange(0, hd // 2, device="cuda", dtype=torch.float64) * 2.0 / hd)
            ang = torch.arange(s, device="cuda", dtype=torch.float64)[:, None] * inv[None, :]
            cos_t, sin_t = ang.cos().float().contiguous(), ang.sin().float().contiguous()

            def fn(*_):
                mt.k_attn_bwd_rope(qkv, o, dout, lse, delta, dqkv, B, s, H, Hkv, hd, cos_t, sin_t)
        else:
            def fn(*_):
                bwd(qkv, o, dout, lse, delta, dqkv, B, s, H, Hkv, hd)
    else:
        fn = fwd
    for _ in range(2):
        fn(qkv, o, lse, B, s, H, Hkv, hd)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(args.iters):
        fn(qkv, o, lse, B, s, H, Hkv, hd)
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / args.iters
    # causal: two (forward) or five (backward) products over half the score matrix
    flops = (5.0 if args.backward else 2.0) * B * H * s * s * hd
    name = ("attn_bwd" if args.backward else "attn_fwd") + ("_mma" if args.legacy else "") + \
        ("_rope" if args.backward and args.rope else "")
    print(json.dumps({"kernel": name, "shape": [B, s, H, Hkv, hd], "ms": ms,
                      "tflops": flops / ms / 1e9}), flush=True)
    return 0


def host_mem_available():
    """MemAvailable of /proc/meminfo in bytes (None where it is not readable)."""
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        return None
    return None


def host_memory_refusal(mt, cfg, shape, keep_grads, avail, ranks=1):
    """The error line for a workload whose host state and pinned buffers,
    times the `ranks` replicas on this host, exceed 90% of the available
    host memory `avail` (bytes), else None."""
    plan = mt.plan(cfg)
    need = (plan["host_state_bytes"] * (16 if keep_grads else 12) // 16 + plan["pinned_bytes"]) * ranks
    if avail is None or need <= 0.9 * avail:
        return None
    return {"metric": METRIC, "config": {"workload": shape.name}, "value": None,
            "error": f"host memory: {ranks} replica(s) of the workload need {need / 1e9:.1f} GB of host state "
                     f"and pinned buffers, {avail / 1e9:.1f} GB available"}


def run_ours(args, shape, world, rank, local, pg):
    import torch
    import host_memory_resident_gb300 as mt
    cfg = mt.make_config(shape, device=local, host_threads=args.host_threads, overlap_adam=args.overlap,
                         unfused_epilogues=args.unfused, keep_attention=args.keep_attention)
    descs, n_total = mt.layout(cfg)
    # refuse, before touching the GPU or allocating, a workload whose host
    # state and pinned buffers do not fit the host's memory (14B: ~285 GB)
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    refusal = host_memory_refusal(mt, cfg, shape, args.keep_grads, host_mem_available(), ranks=local_ranks)
    if refusal is not None:
        if rank == 0:
            print(json.dumps(refusal), flush=True)
        return 3
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    segs = [(t["offset"], t["rows"] * t["cols"], "normal" if t["kind"] == 0 else "ones") for t in descs]
    master = synth.init_master(n_total, segs, seed=0)
    B, s = shape.batch, shape.seq
    NM = args.micro_batches
    M = B * s * NM             # tokens per step (all micro-batches)
    W, K = args.warmup, args.steps
    batches = [[synth.make_tokens(shape.vocab, B, s, seed=1 + 1000 * rank, step=i * NM + j) for j in range(NM)]
               for i in range(W + 2 * K)]
    dev_batches = [[(torch.from_numpy(t).to(dev), torch.from_numpy(l).to(dev)) for t, l in mb]
                   for mb in batches[:W + K]]
    link = host_link_probe(torch, dev)
    torch.cuda.empty_cache()
    adam_gbs = host_adam_probe(mt, threads=args.host_threads, keep_grads=args.keep_grads)
    # host bytes per parameter per step: one accumulate pass per micro-batch
    # but the last (bf16 slab in, fp32 running sum read and written), then Adam
    hb = host_bytes_per_param(args.keep_grads) + (NM - 1) * 10.0

    tr = mt.Trainer(cfg, master, keep_grads=args.keep_grads)
    comp = torch.cuda.ExternalStream(tr.stream(0), device=dev)

    def step_dev(i):
        """One step from device-resident ids: one mt_train_step_device, or
        NM micro-steps of gradient accumulation (host ids; Adam after the
        last)."""
        if NM == 1:
            tk, lb = dev_batches[i][0]
            return tr.step_device(tk.data_ptr(), lb.data_ptr(), B, s)
        return [tr.step_accum(tk, lb, j, NM) for j, (tk, lb) in enumerate(batches[i])][-1]

    def step_host(i):
        if NM == 1:
            tk, lb = batches[i][0]
            return tr.step(tk, lb)
        return [tr.step_accum(tk, lb, j, NM) for j, (tk, lb) in enumerate(batches[i])][-1]

    for i in range(W):
        step_dev(i)
    tr.sync()  # the warm-up's host Adam (overlap mode) ends before the timed region starts

    # ---- timed region: K steps, token/label arrays resident in device memory,
    # per-launch profiling off (the per-class profile is a separate pass below)
    tr.profile(False)
    st0 = tr.stats()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.5)
    barrier(pg)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    t0 = time.perf_counter()
    losses = []
    for i in range(K):
        losses.append(step_dev(W + i))
    tr.sync()  # the last step's host Adam belongs to the timed work
    e1.record(comp)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    barrier(pg)
    clk = clocks.stop()
    st1 = tr.stats()
    t_max = max_over_ranks(pg, e0.elapsed_time(e1) / 1e3)

    # ---- end to end: host token/label arrays through mt_train_step
    barrier(pg)
    torch.cuda.synchronize(dev)
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(comp)
    for i in range(K):
        losses.append(step_host(W + K + i))
    tr.sync()
    e3.record(comp)
    torch.cuda.synchronize(dev)
    barrier(pg)
    e2e_max = max_over_ranks(pg, e2.elapsed_time(e3) / 1e3)
    stats = tr.stats()
    # ---- per-class profile: the same steps again, back to back, with CUDA
    # events around every launch and copy (on the stream each runs on); the
    # launch / copy / host-worker timeline is that of the last of them (a
    # step in the steady state, overlapping the previous step's host tail)
    KP = min(K, args.profile_steps)
    tr.profile(True)
    tr.read_profile(reset=True)
    for i in range(KP):
        step_dev(W + i)
    tr.sync()
    prof = tr.read_profile(reset=True)
    tl = tr.timeline() if not args.no_timeline else None
    tr.profile(False)
    tl_sum = None
    if tl:
        tl_sum = timeline_summary(tl)
        tl_sum["step"] = f"the last of {KP} profiled steps run back to back"
        if args.timeline and rank == 0:
            write_trace(tl, args.timeline)
            tl_sum["trace"] = args.timeline
    tr.close()

    tokens_all = sum_over_ranks(pg, float(M * K))
    value = tokens_all / t_max
    pk, pk_kind = peaks()
    F = model_flops(shape, B, s) * NM
    t_step = t_max / K
    g = prof["gemm"]
    gemm_tf = g["flops"] / (g["ms"] / 1e3) / 1e12 if g["ms"] > 0 else None
    peak_tf = pk["bf16_tflops_sustained"]
    traffic = gemm_traffic_record()
    w_bytes = 2.0 * n_total
    t_comp = F / (pk["bf16_tflops"] * 1e12)
    t_link = NM * max(2 * w_bytes / (link["bidir_h2d_gbs"] * 1e9), w_bytes / (link["bidir_d2h_gbs"] * 1e9))
    t_roof = max(t_comp, t_link)
    prof_out = {k: {"launches_per_step": v["launches"] / KP, "ms_per_step": v["ms"] / KP,
                    "tflops": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["flops"] and v["ms"] else None,
                    "gbs": (v["bytes"] / (v["ms"] / 1e3) / 1e9) if v["bytes"] and v["ms"] else None}
                for k, v in prof.items() if v["launches"] and k not in ("h2d", "d2h")}
    copies = {k: {"copies_per_step": prof[k]["launches"] / KP, "ms_per_step": prof[k]["ms"] / KP,
                  "gb_per_step": prof[k]["bytes"] / KP / 1e9,
                  "gbs_while_copying": prof[k]["bytes"] / (prof[k]["ms"] / 1e3) / 1e9 if prof[k]["ms"] else None}
              for k in ("h2d", "d2h") if k in prof}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded uniform token ids, normal(0, 0.02) weights, norms 1.0)",
        "config": config_dict(args, shape, world, n_total),
        "model_tflops": F / t_step / 1e12,
        "step_roofline": {"model_flops": F, "t_compute_s": t_comp, "t_link_s": t_link, "t_roof_s": t_roof,
                          "frac": t_roof / t_step, "peak_tflops": pk["bf16_tflops"], "host_link": link,
                          "weight_bytes": w_bytes, "peak_source": pk_kind},
        "roofline": {"bound": "tensor", "kernel": "gemm_abt (tcgen05)", "achieved": gemm_tf, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": (gemm_tf / peak_tf) if gemm_tf else None,
                     "measured_over": f"{KP} profiled steps run after the timed ones (CUDA events around each "
                                      "launch on the compute stream)",
                     "peak_source": f"bf16_tflops_sustained, of {pk_kind}",
                     "traffic": (traffic["traffic_over_algorithmic"] * g["bytes"] / max(g["launches"], 1))
                     if traffic else None,
                     "traffic_note": "ncu DRAM bytes of one captured GEMM launch (profiles/gemm_traffic.json) as a "
                                     "ratio to its algorithmic bytes, times the step's mean algorithmic bytes per "
                                     "GEMM launch" if traffic else "no capture of the current GEMM source"},
        "host_bound": {"adam_probe_gbs": adam_gbs, "t_host_s": hb * n_total / (adam_gbs * 1e9),
                       "frac": hb * n_total / (adam_gbs * 1e9) / t_step, "bytes_per_param": hb,
                       "note": "host Adam + bf16 emit (+ FP32 grad out when kept) over the rate the same pass "
                               "reaches alone on one layer-sized slice; the step roofline (FLOPs vs host link) leaves this "
                               "bound out"},
        "kernels": prof_out,
        "copies": copies,
        "timeline": tl_sum,
        "host": {"adam_s_per_step": (st1["host_adam_s"] - st0["host_adam_s"]) / K,
                 "adam_compute_s_per_step": (st1["host_compute_s"] - st0["host_compute_s"]) / K,
                 "adam_compute_gbs": hb * n_total * K / max(st1["host_compute_s"] - st0["host_compute_s"], 1e-9)
                 / 1e9,
                 "copy_wait_s_per_step": (st1["host_copy_wait_s"] - st0["host_copy_wait_s"]) / K,
                 "slab_wait_s_per_step": (st1["host_wait_s"] - st0["host_wait_s"]) / K,
                 "h2d_gb_per_step": (st1["h2d_bytes"] - st0["h2d_bytes"]) / K / 1e9,
                 "d2h_gb_per_step": (st1["d2h_bytes"] - st0["d2h_bytes"]) / K / 1e9,
                 "threads": args.host_threads or os.cpu_count(),
                 "device_gb": stats["device_bytes"] / 1e9, "pinned_gb": stats["pinned_bytes"] / 1e9},
        "clocks": clk,
        "gpu_launches": int(st1["kernel_launches"] - st0["kernel_launches"]),
        "e2e": {"value": tokens_all / e2e_max, "unit": "tokens/s", "h2d_bytes_per_step": 2 * 4 * M,
                "d2h_bytes_per_step": 4 * NM},
        "loss": {"first": losses[0], "last": losses[-1]},
        "wall_s_timed": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # about 10-30 s of host work: sequences longer than 2048 tokens (1024
        # from d = 4096 up) are timed at half and full budget and extrapolated
        cb = oracle_sample(shape, max_tokens=2048 if shape.d_model < 4096 else 1024)
        line["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="7b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--profile-steps", type=int, default=5,
                    help="steps of the separate per-class profiled pass (at most --steps)")
    ap.add_argument("--kernel", default=None, choices=[None, "gemm", "attn", "misc"])
    ap.add_argument("--legacy", action="store_true", help="with --kernel attn: the mma.sync kernels")
    ap.add_argument("--backward", action="store_true", help="with --kernel attn: time the backward")
    ap.add_argument("--rope", action="store_true",
                    help="with --kernel attn --backward: the form that rotates dq, dk back (the step's)")
    ap.add_argument("--shape", default="8192,8192,2048")
    ap.add_argument("--epilogue", default=None, choices=[None, "swiglu", "swiglu_bwd", "rope", "wgrad", "wgrad_nosplit"],
                    help="with --kernel gemm: a fused-epilogue form")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--tile", type=int, default=0, choices=[0, 1, 2],
                    help="with --kernel gemm: tile shape of plain products (0 library's choice, 1 128x256, 2 256x256)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-threads", type=int, default=0)
    ap.add_argument("--timeline", default=None, help="write the profiled step's Chrome/Perfetto trace here")
    ap.add_argument("--no-timeline", action="store_true", help="leave the copy/compute timeline out of the line")
    ap.add_argument("--keep-attention", action="store_true",
                    help="keep attention outputs from the forward so the recompute skips attention (same results)")
    ap.add_argument("--unfused", action="store_true",
                    help="RoPE and SwiGLU as separate kernels instead of GEMM epilogues (same results)")
    ap.add_argument("--fused-grads", action="store_true",
                    help="no FP32 gradient array: each slab goes straight into Adam (same arithmetic)")
    ap.add_argument("--layers", type=int, default=0,
                    help="run the workload at this depth instead of its own (a reduced-depth variant, named as "
                         "such in the line; for widths whose full-depth host state does not fit the host)")
    ap.add_argument("--micro-batches", type=int, default=1,
                    help="one step = this many micro-batches of gradient accumulation (host ids), Adam after the "
                         "last (global batch grows by this factor)")
    ap.add_argument("--no-overlap", action="store_true",
                    help="overlap_adam = 0: each step returns only after its host Adam has finished")
    args = ap.parse_args()
    args.keep_grads = not args.fused_grads
    args.overlap = not args.no_overlap
    if args.kernel == "gemm":
        return run_gemm_kernel(args)
    if args.kernel == "attn":
        return run_attn_kernel(args)
    if args.kernel == "misc":
        return run_misc_kernels(args)
    shape = synth.workload(args.config)
    if args.layers:
        shape = shape.with_(name=f"{shape.name} ({args.layers} of {shape.n_layers} layers)", n_layers=args.layers)
    world, rank, local, pg = dist_setup()
    if args.impl == "reference":
        return run_reference(args, shape, world, rank, pg)
    return run_ours(args, shape, world, rank, local, pg)


if __name__ == "__main__":
    sys.exit(main())
