"""The oracle's step with bf16 rounding at the device's storage points.

TEST INFRASTRUCTURE ONLY, used to derive tolerances, never as a reference
for parity. The method computes on bf16 copies of the weights and gradients
with an FP32 optimizer state (zhichai.net article, introduction: mixed
precision with bf16 weights and gradients, FP32 optimizer state); any such
implementation stores bf16 values at fixed points of the layer (weights,
normalised activations, q/k/v, attention output, gate/up pre-activations,
SwiGLU output, the residual stream, gradient operands, softmax and dS
operands of attention, gradient slabs). This module evaluates the plain
definition of the step (the same operators as ``oracle.ops``) and rounds the
value to bf16 at exactly those points, in float64 otherwise. The distance
between its gradients and the exact oracle's is the error floor that bf16
storage alone imposes on the step; it says nothing about any kernel's
arithmetic order and shares no code with the CUDA library.
"""
from __future__ import annotations

import numpy as np

from . import ops
from .layout import build_layout


def to_bf16(x):
    """Round-to-nearest-even to bf16, returned as float64 (plain numpy)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = a.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    out = (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
    out = np.where(np.isnan(a), np.float32(np.nan), out)
    return out.astype(np.float64)


def _attn_fwd(q, k, v, R):
    B, s, H, hd = q.shape
    grp = H // k.shape[2]
    o = np.zeros_like(q)
    lse = np.zeros((B, H, s))
    mask = np.arange(s)[None, :] > np.arange(s)[:, None]
    for b in range(B):
        for h in range(H):
            g = h // grp
            sc = np.where(mask, -np.inf, (q[b, :, h] @ k[b, :, g].T) / np.sqrt(hd))
            mx = sc.max(1, keepdims=True)
            e = np.exp(sc - mx)
            den = e.sum(1, keepdims=True)
            o[b, :, h] = (R(e) @ v[b, :, g]) / den      # unnormalised P is a bf16 operand
            lse[b, h] = (mx + np.log(den))[:, 0]
    return o, lse


def _attn_bwd(q, k, v, o, lse, do, R):
    B, s, H, hd = q.shape
    grp = H // k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    mask = np.arange(s)[None, :] > np.arange(s)[:, None]
    for b in range(B):
        for h in range(H):
            g = h // grp
            sc = (q[b, :, h] @ k[b, :, g].T) / np.sqrt(hd)
            p = np.where(mask, 0.0, np.exp(sc - lse[b, h][:, None]))
            D = np.sum(do[b, :, h] * o[b, :, h], axis=1, keepdims=True)   # rowsum(dO * O)
            ds = p * (do[b, :, h] @ v[b, :, g].T - D)
            pb, dsb = R(p), R(ds)
            dv[b, :, g] += pb.T @ do[b, :, h]
            dq[b, :, h] = (dsb @ k[b, :, g]) / np.sqrt(hd)
            dk[b, :, g] += (dsb.T @ q[b, :, h]) / np.sqrt(hd)
    return dq, dk, dv


def step_grads_bf16_storage(shape, master, tokens, labels):
    """Loss and flat gradient of one step with bf16 storage points (float64)."""
    R = to_bf16
    lay = build_layout(shape)
    W = R(master)
    B, s = tokens.shape
    H, Hkv, hd, f = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim
    cos, sin = ops.rope_tables(s, hd, shape.rope_theta)

    def P(u):
        return {t.name: W[t.offset:t.offset + t.size].reshape(t.shape) for t in lay.units[u].tensors}

    grad = np.zeros(lay.n_total)

    def put(u, name, g):
        t = next(t for t in lay.units[u].tensors if t.name == name)
        grad[t.offset:t.offset + t.size] = R(g).reshape(-1)      # bf16 gradient slab

    x = R(P(0)["embed"][tokens.reshape(-1)])
    caches = []
    for layer in range(shape.n_layers):
        p = P(1 + layer)
        M = x.shape[0]
        u, r1 = ops.rmsnorm_fwd(x, p["attn_norm"], shape.rms_eps)
        u = R(u)
        qkv = R(u @ p["wqkv"].T)
        q = qkv[:, :H * hd].reshape(B, s, H, hd)
        k = qkv[:, H * hd:(H + Hkv) * hd].reshape(B, s, Hkv, hd)
        v = qkv[:, (H + Hkv) * hd:].reshape(B, s, Hkv, hd)
        qr, kr = R(ops.rope_fwd(q, cos, sin)), R(ops.rope_fwd(k, cos, sin))
        o, lse = _attn_fwd(qr, kr, v, R)
        o2 = R(o.reshape(M, -1))
        h = R(x + o2 @ p["wo"].T)
        z, r2 = ops.rmsnorm_fwd(h, p["mlp_norm"], shape.rms_eps)
        z = R(z)
        gu = R(z @ p["wgu"].T)
        g_, up = gu[:, :f], gu[:, f:]
        a = R(ops.swiglu_fwd(g_, up))
        y = R(h + a @ p["wdown"].T)
        caches.append(dict(x=x, u=u, r1=r1, qr=qr, kr=kr, v=v, o2=o2, lse=lse, h=h, z=z, r2=r2, g=g_, up=up,
                           a=a))
        x = y
    ph = P(shape.n_layers + 1)
    xh, rf = ops.rmsnorm_fwd(x, ph["final_norm"], shape.rms_eps)
    xh = R(xh)
    loss, dz = ops.cross_entropy_fwd_bwd(xh @ ph["head"].T, labels.reshape(-1))
    dz = R(dz)
    put(shape.n_layers + 1, "head", dz.T @ xh)
    dx, dfin = ops.rmsnorm_bwd(dz @ ph["head"], x, ph["final_norm"], rf)
    put(shape.n_layers + 1, "final_norm", dfin)
    for layer in reversed(range(shape.n_layers)):
        c, p = caches[layer], P(1 + layer)
        M = dx.shape[0]
        dyb = R(dx)
        put(1 + layer, "wdown", dyb.T @ c["a"])
        da = R(dyb @ p["wdown"])
        dg, dup = ops.swiglu_bwd(da, c["g"], c["up"])
        dgu = R(np.concatenate([dg, dup], 1))
        put(1 + layer, "wgu", dgu.T @ c["z"])
        dhn, dmlp = ops.rmsnorm_bwd(dgu @ p["wgu"], c["h"], p["mlp_norm"], c["r2"])
        put(1 + layer, "mlp_norm", dmlp)
        dh = dx + dhn
        dhb = R(dh)
        put(1 + layer, "wo", dhb.T @ c["o2"])
        do = R(dhb @ p["wo"])
        dq, dk, dv = _attn_bwd(c["qr"], c["kr"], c["v"], c["o2"].reshape(B, s, H, hd), c["lse"],
                               do.reshape(B, s, H, hd), R)
        dq, dk = ops.rope_bwd(dq, cos, sin), ops.rope_bwd(dk, cos, sin)
        dqkv = R(np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), dv.reshape(M, -1)], 1))
        put(1 + layer, "wqkv", dqkv.T @ c["u"])
        dxn, dan = ops.rmsnorm_bwd(dqkv @ p["wqkv"], c["x"], p["attn_norm"], c["r1"])
        put(1 + layer, "attn_norm", dan)
        dx = dh + dxn
    put(0, "embed", ops.embedding_bwd(dx, tokens, shape.vocab))
    return float(loss), grad
