"""Resource calculator: memory and time of a streamed-layer training step.

The RAM-centric method's users first size their run from the model and the
machine (the lqnn.cn article, section 七, runs a resource calculator that
picks the batch size; the travelaiplan blog, 核心功能 point 1, estimates host
RAM as parameters x 4 bytes x about 4). This module answers the same
questions for this library exactly where it can: device and pinned bytes
come from the library's own planner (``mt_plan``, the one ``mt_init`` uses);
host state is 16 bytes per parameter (FP32 master, grad, m, v); per-step
traffic and FLOPs are counted from the shapes; time is bounded below by the
measured rates passed in.
"""
from __future__ import annotations

import host_memory_resident_gb300 as mt


def model_flops(shape, batch: int, seq: int) -> float:
    """6 * matmul parameters + 6 * L * s * H * hd per token (causal), per step."""
    d, f, V = shape.d_model, shape.ffn_dim, shape.vocab
    qkv = (shape.n_heads + 2 * shape.n_kv_heads) * shape.head_dim
    hq = shape.n_heads * shape.head_dim
    n_mm = shape.n_layers * (qkv * d + d * hq + 2 * f * d + d * f) + V * d
    return (6.0 * n_mm + 6.0 * shape.n_layers * seq * shape.n_heads * shape.head_dim) * batch * seq


def streamed_units(n_layers: int, ckpt_interval: int) -> list[int]:
    """Units copied host-to-device in one streamed step, in order.

    The step visits units as: embedding, layers 1..L, head (forward); then per
    checkpoint segment, last to first, its layers in order (recompute, except
    for the last segment, whose activations the forward keeps) and in reverse
    (backward). Two device buffers hold the two most recently used units; a
    visit to a unit not held loads it into the least recently used.
    """
    L, C = n_layers, ckpt_interval
    visits = list(range(L + 2))
    starts = list(range(0, L, C))
    for a in reversed(starts):
        seg = list(range(1 + a, 1 + min(L, a + C)))
        visits += (seg if a != starts[-1] else []) + seg[::-1]
    held, loads = [], []
    for u in visits:
        if u in held:
            held.remove(u)
        else:
            loads.append(u)
            if len(held) == 2:
                held.pop(0)
        held.append(u)
    return loads


def estimate(shape, batch: int | None = None, seq: int | None = None, ckpt_interval: int | None = None,
             n_slabs: int | None = None, keep_grads: bool = True, gemm_tflops: float = 1500.0,
             host_gbs: float = 150.0, link_gbs: float = 170.0) -> dict:
    """Memory (exact) and per-step traffic, FLOPs and lower-bound times.

    keep_grads=False is a handle made without the FP32 gradient array: 12
    instead of 16 bytes of host state per parameter, 28 instead of 32 bytes
    of host DRAM traffic per parameter and step."""
    B = batch or shape.batch
    s = seq or shape.seq
    cfg = mt.make_config(shape, batch=B, seq=s, ckpt_interval=ckpt_interval, n_slabs=n_slabs)
    plan = mt.plan(cfg)
    lay, n_total = mt.layout(cfg)
    unit_len = {}
    for t in lay:
        unit_len[t["unit"]] = unit_len.get(t["unit"], 0) + t["rows"] * t["cols"]
    h2d = 2.0 * sum(unit_len[u] for u in streamed_units(shape.n_layers, cfg.ckpt_interval))
    d2h = 2.0 * n_total
    flops = model_flops(shape, B, s)
    hw_flops = flops + flops * (1.0 / 3.0)          # recompute adds one forward (about 1/3 of 6N)
    t_gpu = hw_flops / (gemm_tflops * 1e12)
    state = plan["host_state_bytes"] if keep_grads else plan["host_state_bytes"] * 12 // 16
    t_host = (32.0 if keep_grads else 28.0) * n_total / (host_gbs * 1e9)
    t_link = max(h2d, d2h) / (link_gbs * 1e9)
    return {
        "params": n_total, "tokens_per_step": B * s,
        "device_bytes": plan["device_bytes"], "pinned_bytes": plan["pinned_bytes"],
        "host_state_bytes": state,
        "host_total_bytes": state + plan["pinned_bytes"],
        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
        "model_flops_per_step": flops,
        "t_gpu_s": t_gpu, "t_host_s": t_host, "t_link_s": t_link,
        "t_step_lower_bound_s": max(t_gpu, t_host, t_link),
        "bound": max((("gpu", t_gpu), ("host", t_host), ("link", t_link)), key=lambda x: x[1])[0],
    }


def suggest_batch(shape, seq: int | None = None, device_budget: float = 250e9, host_budget: float | None = None,
                  max_batch: int = 4096) -> int | None:
    """Largest batch whose plan fits the device budget (and, if given, whose
    host state plus pinned memory fits the host budget); None if even 1 does not."""
    s = seq or shape.seq

    def fits(b):
        e = estimate(shape, batch=b, seq=s)
        if e["device_bytes"] > device_budget:
            return False
        return host_budget is None or e["host_total_bytes"] <= host_budget

    if not fits(1):
        return None
    lo, hi = 1, 2
    while hi <= max_batch and fits(hi):
        lo, hi = hi, hi * 2
    hi = min(hi, max_batch + 1)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if fits(mid):
            lo = mid
        else:
            hi = mid
    return lo
