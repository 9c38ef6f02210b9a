"""One training step of the decoder, restated plainly (forward, backward).

The step follows the zhichai.net article ("以内存为中心的训练新范式",
points 2-4) and the lqnn.cn article (section 三.1-三.4): units are used one at
a time in forward order (embedding, layers, final norm + head); the input of
every ``ckpt_interval``-th layer is checkpointed; backward walks the segments
from last to first, recomputes each segment's forward from its checkpoint and
then runs the layers' backward in reverse. With ``streamed`` the weights of a
unit are copied into one of two scratch slots before each use, standing in for
the two device flat buffers. Neither knob changes the arithmetic, which is what
the invariance tests check.
"""
from __future__ import annotations

import numpy as np

from . import ops
from .layout import build_layout


class _Weights:
    """Hands out a unit's tensors, either as views of the master or from a
    two-slot scratch copy (the double buffer of the streamed engine)."""

    def __init__(self, layout, master, dtype, streamed):
        self.layout = layout
        self.master = master
        self.dtype = dtype
        self.streamed = streamed
        self.slots = [None, None]
        self.uses = 0
        self.resident = None if streamed else master.astype(dtype, copy=False)

    def unit(self, index):
        u = self.layout.units[index]
        if self.streamed:
            slot = self.uses % 2
            self.uses += 1
            self.slots[slot] = np.array(
                self.master[u.offset:u.offset + u.length], dtype=self.dtype)
            base, off0 = self.slots[slot], u.offset
        else:
            base, off0 = self.resident, 0
        out = {}
        for t in u.tensors:
            a = t.offset - off0
            out[t.name] = base[a:a + t.size].reshape(t.shape)
        return out


def layer_forward(shape, P, x, cos, sin, B, s):
    """Forward of one decoder layer; returns the output and what backward needs."""
    H, Hkv, hd, f = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim
    M = x.shape[0]
    u, r1 = ops.rmsnorm_fwd(x, P["attn_norm"], shape.rms_eps)
    qkv = ops.linear_fwd(u, P["wqkv"])
    q = qkv[:, :H * hd].reshape(B, s, H, hd)
    k = qkv[:, H * hd:(H + Hkv) * hd].reshape(B, s, Hkv, hd)
    v = qkv[:, (H + Hkv) * hd:].reshape(B, s, Hkv, hd)
    qr = ops.rope_fwd(q, cos, sin)
    kr = ops.rope_fwd(k, cos, sin)
    o, lse = ops.attention_fwd(qr, kr, v)
    o2 = o.reshape(M, H * hd)
    h = x + ops.linear_fwd(o2, P["wo"])
    z, r2 = ops.rmsnorm_fwd(h, P["mlp_norm"], shape.rms_eps)
    gu = ops.linear_fwd(z, P["wgu"])
    g, up = gu[:, :f], gu[:, f:]
    a = ops.swiglu_fwd(g, up)
    y = h + ops.linear_fwd(a, P["wdown"])
    cache = dict(x=x, u=u, r1=r1, qr=qr, kr=kr, v=v, o2=o2, lse=lse, h=h, z=z,
                 r2=r2, g=g, up=up, a=a)
    return y, cache


def layer_backward(shape, P, dy, c, cos, sin, B, s):
    """Backward of one decoder layer given dL/dy; returns dL/dx and weight grads."""
    H, hd = shape.n_heads, shape.head_dim
    M = dy.shape[0]
    da, dwdown = ops.linear_bwd(dy, c["a"], P["wdown"])
    dg, dup = ops.swiglu_bwd(da, c["g"], c["up"])
    dgu = np.concatenate([dg, dup], axis=1)
    dz, dwgu = ops.linear_bwd(dgu, c["z"], P["wgu"])
    dhn, dmlp = ops.rmsnorm_bwd(dz, c["h"], P["mlp_norm"], c["r2"])
    dh = dy + dhn
    do2, dwo = ops.linear_bwd(dh, c["o2"], P["wo"])
    dq, dk, dv = ops.attention_bwd(c["qr"], c["kr"], c["v"], do2.reshape(B, s, H, hd))
    dq = ops.rope_bwd(dq, cos, sin)
    dk = ops.rope_bwd(dk, cos, sin)
    dqkv = np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), dv.reshape(M, -1)], axis=1)
    du, dwqkv = ops.linear_bwd(dqkv, c["u"], P["wqkv"])
    dxn, dattn = ops.rmsnorm_bwd(du, c["x"], P["attn_norm"], c["r1"])
    dx = dh + dxn
    grads = dict(attn_norm=dattn, wqkv=dwqkv, wo=dwo, mlp_norm=dmlp, wgu=dwgu, wdown=dwdown)
    return dx, grads


def step_grads(shape, master, tokens, labels, ckpt_interval=None, streamed=False,
               dtype=np.float64, out_dtype=None):
    """Loss (mean cross entropy) and flat gradient of one step at ``master``.

    ``tokens``/``labels`` are int [B, s]. Returns ``(loss, grad)`` with ``grad``
    a flat array of the layout's n_total elements (padding stays 0).
    """
    lay = build_layout(shape)
    C = int(ckpt_interval or shape.ckpt_interval)
    if C < 1:
        raise ValueError("ckpt_interval must be >= 1")
    B, s = tokens.shape
    L = shape.n_layers
    W = _Weights(lay, master, dtype, streamed)
    cos, sin = ops.rope_tables(s, shape.head_dim, shape.rope_theta, dtype)
    grad = np.zeros(lay.n_total, dtype=out_dtype or dtype)

    def put(unit_index, name, g):
        t = next(t for t in lay.units[unit_index].tensors if t.name == name)
        grad[t.offset:t.offset + t.size] = g.reshape(-1)

    # forward: embedding, then layers with a checkpoint every C layers
    x = ops.embedding_fwd(W.unit(0)["embed"], tokens)
    ckpt = {}
    for layer in range(L):
        if layer % C == 0:
            ckpt[layer] = x
        x, _ = layer_forward(shape, W.unit(1 + layer), x, cos, sin, B, s)

    # head: final norm, logits, cross entropy and its gradient
    Ph = W.unit(L + 1)
    xh, rf = ops.rmsnorm_fwd(x, Ph["final_norm"], shape.rms_eps)
    logits = ops.linear_fwd(xh, Ph["head"])
    loss, dlogits = ops.cross_entropy_fwd_bwd(logits, labels.reshape(-1))
    del logits
    dxh, dhead = ops.linear_bwd(dlogits, xh, Ph["head"])
    del dlogits
    dx, dfinal = ops.rmsnorm_bwd(dxh, x, Ph["final_norm"], rf)
    put(L + 1, "head", dhead)
    put(L + 1, "final_norm", dfinal)

    # backward: segments from last to first, recomputing each from its checkpoint
    for start in reversed(range(0, L, C)):
        stop = min(start + C, L)
        caches = []
        xs = ckpt[start]
        for layer in range(start, stop):
            xs, cache = layer_forward(shape, W.unit(1 + layer), xs, cos, sin, B, s)
            caches.append(cache)
        for layer in reversed(range(start, stop)):
            dx, gl = layer_backward(shape, W.unit(1 + layer), dx, caches[layer - start],
                                    cos, sin, B, s)
            caches[layer - start] = None
            for name, g in gl.items():
                put(1 + layer, name, g)

    put(0, "embed", ops.embedding_bwd(dx, tokens, shape.vocab))
    return float(loss), grad
