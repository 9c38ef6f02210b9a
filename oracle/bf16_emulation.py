"""The oracle's step with bf16 rounding at chosen storage points.

TEST INFRASTRUCTURE ONLY, used to study tolerances, never as a reference
for parity. The method computes on bf16 copies of the weights and gradients
with an FP32 optimizer state (zhichai.net article, introduction: mixed
precision with bf16 weights and gradients, FP32 optimizer state), and its
products take bf16 operands with FP32 accumulation. A bf16 implementation
of the step stores bf16 values at some fixed points of the layer; this
module evaluates the plain definition of the step (the same operators as
``oracle.ops``, in float64) and rounds the value to bf16 at the points named
in ``points`` only. Each point can be switched on or off on its own, so the
error that each storage point adds to every gradient tensor can be measured
against the exact oracle. With no point switched on the step is the exact
one (equal to ``oracle.step_grads`` up to float64 rounding order). It says
nothing about any kernel's arithmetic order and shares no code with the
CUDA library.

Storage points (``POINTS``). The first group are operands of the step's
products, which a bf16 product needs in bf16 (``OPERAND_POINTS``):

* ``norm_out``      outputs of the three RMSNorms (u, z, final x-hat):
                    operands of the projections after them;
* ``qkv``           the rotated q, k and v: operands of the attention products;
* ``attn_p``        the softmax weights as an operand of P V (forward: the
                    unnormalised exponentials) and of P^T dO (backward);
* ``attn_ds``       dS as an operand of dS K and dS^T Q;
* ``attn_out``      the attention output O: operand of the output projection
                    and of the backward's rowsum(dO * O);
* ``swiglu_out``    a = silu(gate) * up: operand of the down projection;
* ``grad_operands`` the output-side gradients of the products (dz of the
                    head, dy, d(gate|up), dh, dO, dqkv);
* ``grad_slab``     every weight gradient as written (the bf16 gradient slab).

The second group are storage points an implementation may or may not have:

* ``residual``       the residual stream h = x + O Wo^T, y = h + a Wdown^T
                     (and so the layer inputs and checkpoints);
* ``qk_pre_rope``    q and k rounded once more before the rotation;
* ``gate_up``        the gate/up projection's output rounded before the
                     forward's SwiGLU;
* ``gate_up_saved``  the copy of gate/up the backward's SwiGLU reads;
* ``swiglu_da``      da = dy Wdown rounded before the SwiGLU backward;
* ``dqk_pre_rope``   dq and dk rounded before the inverse rotation.
"""
from __future__ import annotations

import numpy as np

from . import ops
from .layout import build_layout

OPERAND_POINTS = ("norm_out", "qkv", "attn_p", "attn_ds", "attn_out", "swiglu_out", "grad_operands",
                  "grad_slab")
OTHER_POINTS = ("residual", "qk_pre_rope", "gate_up", "gate_up_saved", "swiglu_da", "dqk_pre_rope")
POINTS = OPERAND_POINTS + OTHER_POINTS


def to_bf16(x):
    """Round-to-nearest-even to bf16, returned as float64 (plain numpy; done
    in slices of 2^24 elements so the integer temporaries stay small)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(a.shape, dtype=np.float64)
    flat_a, flat_o = a.reshape(-1), out.reshape(-1)
    step = 1 << 24
    for i in range(0, flat_a.size, step):
        c = flat_a[i:i + step]
        u = c.view(np.uint32).astype(np.uint64)
        r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
        b = (r & 0xFFFFFFFF).astype(np.uint32).view(np.float32)
        flat_o[i:i + step] = np.where(np.isnan(c), np.float32(np.nan), b)
    return out


def _identity(x):
    return np.asarray(x, dtype=np.float64)


def _attn_fwd(q, k, v, Rp):
    """Causal softmax attention; the unnormalised weights pass through Rp
    before the P V product and the row sum divides afterwards (a bf16
    implementation cannot store P/den without a second pass)."""
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
            o[b, :, h] = (Rp(e) @ v[b, :, g]) / den
            lse[b, h] = (mx + np.log(den))[:, 0]
    return o, lse


def _attn_bwd(q, k, v, o, lse, do, Rp, Rds):
    """Gradients of _attn_fwd from the saved log-sum-exp; delta = rowsum(dO * O)."""
    B, s, H, hd = q.shape
    grp = H // k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    mask = np.arange(s)[None, :] > np.arange(s)[:, None]
    for b in range(B):
        for h in range(H):
            g = h // grp
            sc = (q[b, :, h] @ k[b, :, g].T) / np.sqrt(hd)
            p = np.where(mask, 0.0, np.exp(sc - lse[b, h][:, None]))
            D = np.sum(do[b, :, h] * o[b, :, h], axis=1, keepdims=True)
            ds = p * (do[b, :, h] @ v[b, :, g].T - D)
            pb, dsb = Rp(p), Rds(ds)
            dv[b, :, g] += pb.T @ do[b, :, h]
            dq[b, :, h] = (dsb @ k[b, :, g]) / np.sqrt(hd)
            dk[b, :, g] += (dsb.T @ q[b, :, h]) / np.sqrt(hd)
    return dq, dk, dv


def step_grads_bf16_storage(shape, master, tokens, labels, points=POINTS, out_dtype=np.float64):
    """Loss and flat gradient of one step at the bf16 values of ``master``,
    rounding to bf16 at the storage points in ``points`` (arithmetic in
    float64; the gradient is returned in ``out_dtype``)."""
    points = frozenset(points)
    unknown = points - frozenset(POINTS)
    if unknown:
        raise ValueError(f"unknown storage points {sorted(unknown)}")

    def rnd(name):
        return to_bf16 if name in points else _identity

    Rn, Rq, Rp, Rds, Ro = rnd("norm_out"), rnd("qkv"), rnd("attn_p"), rnd("attn_ds"), rnd("attn_out")
    Ra, Rg, Rs = rnd("swiglu_out"), rnd("grad_operands"), rnd("grad_slab")
    Rh, Rq0, Rgu, Rgus = rnd("residual"), rnd("qk_pre_rope"), rnd("gate_up"), rnd("gate_up_saved")
    Rda, Rdq0 = rnd("swiglu_da"), rnd("dqk_pre_rope")

    lay = build_layout(shape)
    B, s = tokens.shape
    H, Hkv, hd, f = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim
    cos, sin = ops.rope_tables(s, hd, shape.rope_theta)

    def P(u):
        """The unit's tensors at their bf16 values (float64)."""
        un = lay.units[u]
        base = to_bf16(master[un.offset:un.offset + un.length])
        return {t.name: base[t.offset - un.offset:t.offset - un.offset + t.size].reshape(t.shape)
                for t in un.tensors}

    grad = np.zeros(lay.n_total, dtype=out_dtype)

    def put(u, name, g):
        t = next(t for t in lay.units[u].tensors if t.name == name)
        grad[t.offset:t.offset + t.size] = Rs(g).reshape(-1)

    x = P(0)["embed"][tokens.reshape(-1)]          # bf16 weights: exact either way
    caches = []
    for layer in range(shape.n_layers):
        p = P(1 + layer)
        M = x.shape[0]
        u, r1 = ops.rmsnorm_fwd(x, p["attn_norm"], shape.rms_eps)
        u = Rn(u)
        qkv = u @ p["wqkv"].T
        q = Rq0(qkv[:, :H * hd]).reshape(B, s, H, hd)
        k = Rq0(qkv[:, H * hd:(H + Hkv) * hd]).reshape(B, s, Hkv, hd)
        v = Rq(qkv[:, (H + Hkv) * hd:]).reshape(B, s, Hkv, hd)
        qr, kr = Rq(ops.rope_fwd(q, cos, sin)), Rq(ops.rope_fwd(k, cos, sin))
        o, lse = _attn_fwd(qr, kr, v, Rp)
        o2 = Ro(o.reshape(M, -1))
        h = Rh(x + o2 @ p["wo"].T)
        z, r2 = ops.rmsnorm_fwd(h, p["mlp_norm"], shape.rms_eps)
        z = Rn(z)
        gu = Rgu(z @ p["wgu"].T)
        a = Ra(ops.swiglu_fwd(gu[:, :f], gu[:, f:]))
        gus = Rgus(gu)
        y = Rh(h + a @ p["wdown"].T)
        caches.append(dict(x=x, u=u, r1=r1, qr=qr, kr=kr, v=v, o2=o2, lse=lse, h=h, z=z, r2=r2, g=gus[:, :f],
                           up=gus[:, f:], a=a))
        x = y
    ph = P(shape.n_layers + 1)
    xh, rf = ops.rmsnorm_fwd(x, ph["final_norm"], shape.rms_eps)
    xh = Rn(xh)
    loss, dz = ops.cross_entropy_fwd_bwd(xh @ ph["head"].T, labels.reshape(-1))
    dz = Rg(dz)
    put(shape.n_layers + 1, "head", dz.T @ xh)
    dx, dfin = ops.rmsnorm_bwd(dz @ ph["head"], x, ph["final_norm"], rf)
    del dz
    put(shape.n_layers + 1, "final_norm", dfin)
    for layer in reversed(range(shape.n_layers)):
        c, p = caches[layer], P(1 + layer)
        caches[layer] = None
        M = dx.shape[0]
        dyb = Rg(dx)
        put(1 + layer, "wdown", dyb.T @ c["a"])
        da = Rda(dyb @ p["wdown"])
        dg, dup = ops.swiglu_bwd(da, c["g"], c["up"])
        dgu = Rg(np.concatenate([dg, dup], 1))
        put(1 + layer, "wgu", dgu.T @ c["z"])
        dhn, dmlp = ops.rmsnorm_bwd(dgu @ p["wgu"], c["h"], p["mlp_norm"], c["r2"])
        put(1 + layer, "mlp_norm", dmlp)
        dh = dx + dhn
        dhb = Rg(dh)
        put(1 + layer, "wo", dhb.T @ c["o2"])
        do = Rg(dhb @ p["wo"])
        dq, dk, dv = _attn_bwd(c["qr"], c["kr"], c["v"], c["o2"].reshape(B, s, H, hd), c["lse"],
                               do.reshape(B, s, H, hd), Rp, Rds)
        dq, dk = ops.rope_bwd(Rdq0(dq), cos, sin), ops.rope_bwd(Rdq0(dk), cos, sin)
        dqkv = Rg(np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), dv.reshape(M, -1)], 1))
        put(1 + layer, "wqkv", dqkv.T @ c["u"])
        dxn, dan = ops.rmsnorm_bwd(dqkv @ p["wqkv"], c["x"], p["attn_norm"], c["r1"])
        put(1 + layer, "attn_norm", dan)
        dx = dh + dxn
    put(0, "embed", ops.embedding_bwd(dx, tokens, shape.vocab))
    return float(loss), grad
