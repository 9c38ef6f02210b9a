"""Per-operator forward and hand-written backward, plain numpy.

Each function is the textbook definition of one operator of a Llama-style
decoder layer (the "stateless layer template" of the zhichai.net article,
section "以内存为中心的训练新范式" point 4, and of the travelaiplan blog,
"核心功能" point 3). No blocking, fusion or reordering beyond the definition.
All inputs and outputs are numpy arrays in the caller's dtype; tokens are laid
out row-major (batch, position).
"""
from __future__ import annotations

import numpy as np


# ----------------------------------------------------------------- RMSNorm
def rmsnorm_fwd(x, w, eps):
    """y = x * rstd * w with rstd = 1 / sqrt(mean(x^2) + eps) per row."""
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)
    return x * rstd[:, None] * w[None, :], rstd


def rmsnorm_bwd(dy, x, w, rstd):
    """Gradients of rmsnorm_fwd.

    dx_j = rstd * w_j dy_j - x_j * rstd^3 / d * sum_i dy_i w_i x_i
    dw_i = sum_rows dy_i * x_i * rstd
    """
    d = x.shape[-1]
    wdy = dy * w[None, :]
    dot = np.sum(wdy * x, axis=-1)
    dx = wdy * rstd[:, None] - x * (rstd ** 3 * dot / d)[:, None]
    dw = np.sum(dy * x * rstd[:, None], axis=0)
    return dx, dw


# -------------------------------------------------------------------- RoPE
def rope_tables(seq, head_dim, theta, dtype=np.float64):
    """cos/sin of angle pos * theta^(-2i/hd) for i < hd/2, shape [seq, hd/2]."""
    half = head_dim // 2
    inv = theta ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    ang = np.arange(seq, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(dtype), np.sin(ang).astype(dtype)


def rope_fwd(x, cos, sin):
    """Rotate-half RoPE on x [B, s, nh, hd]; pair (i, i + hd/2) is rotated by
    the angle of its position: (a, b) -> (a cos - b sin, b cos + a sin)."""
    half = x.shape[-1] // 2
    a, b = x[..., :half], x[..., half:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rope_bwd(dy, cos, sin):
    """Transpose of the rotation: rotate by the negative angle."""
    half = dy.shape[-1] // 2
    a, b = dy[..., :half], dy[..., half:]
    c = cos[None, :, None, :]
    s = sin[None, :, None, :]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


# --------------------------------------------------------------- attention
def _group(n_heads, n_kv_heads):
    return n_heads // n_kv_heads


def attention_fwd(q, k, v, rows=None):
    """Causal softmax attention with grouped KV heads.

    q [B, s, H, hd], k and v [B, s, Hkv, hd]; query head h reads KV head
    h // (H / Hkv); key j is visible to query i iff j <= i; scale 1/sqrt(hd).
    Returns o [B, s, H, hd] and lse [B, H, s] (natural log of the softmax
    denominator of the scaled scores). With ``rows`` (an array of query
    positions) only those query rows are computed: o [B, len(rows), H, hd],
    lse [B, H, len(rows)].
    """
    B, s, H, hd = q.shape
    Hkv = k.shape[2]
    grp = _group(H, Hkv)
    scale = 1.0 / np.sqrt(hd)
    qi = np.arange(s) if rows is None else np.asarray(rows)
    o = np.zeros((B, len(qi), H, hd), dtype=q.dtype)
    lse = np.zeros((B, H, len(qi)), dtype=q.dtype)
    kj = np.arange(s)
    mask = kj[None, :] > qi[:, None]
    for b in range(B):
        for h in range(H):
            g = h // grp
            sc = (q[b, qi, h, :] @ k[b, :, g, :].T) * scale
            sc = np.where(mask, -np.inf, sc)
            mx = np.max(sc, axis=1, keepdims=True)
            e = np.exp(sc - mx)
            den = np.sum(e, axis=1, keepdims=True)
            p = e / den
            o[b, :, h, :] = p @ v[b, :, g, :]
            lse[b, h, :] = (mx + np.log(den))[:, 0]
    return o, lse


def attention_bwd(q, k, v, do):
    """Gradients of attention_fwd (full rows), plain definition.

    P = softmax(mask(q k^T * scale)); dV = P^T dO; dP = dO V^T;
    dS = P * (dP - rowsum(P * dP)); dQ = dS K * scale; dK = dS^T Q * scale.
    Query heads sharing a KV head add their dK, dV.
    """
    B, s, H, hd = q.shape
    Hkv = k.shape[2]
    grp = _group(H, Hkv)
    scale = 1.0 / np.sqrt(hd)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    mask = np.arange(s)[None, :] > np.arange(s)[:, None]
    for b in range(B):
        for h in range(H):
            g = h // grp
            sc = (q[b, :, h, :] @ k[b, :, g, :].T) * scale
            sc = np.where(mask, -np.inf, sc)
            mx = np.max(sc, axis=1, keepdims=True)
            e = np.exp(sc - mx)
            p = e / np.sum(e, axis=1, keepdims=True)
            dov = do[b, :, h, :]
            dv[b, :, g, :] += p.T @ dov
            dp = dov @ v[b, :, g, :].T
            ds = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
            dq[b, :, h, :] = (ds @ k[b, :, g, :]) * scale
            dk[b, :, g, :] += (ds.T @ q[b, :, h, :]) * scale
    return dq, dk, dv


# ------------------------------------------------------------------ SwiGLU
def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def swiglu_fwd(g, u):
    """a = silu(g) * u with silu(g) = g * sigmoid(g)."""
    return g * _sigmoid(g) * u


def swiglu_bwd(da, g, u):
    """dg = da * u * sigmoid(g) * (1 + g (1 - sigmoid(g))); du = da * silu(g)."""
    sg = _sigmoid(g)
    dg = da * u * sg * (1.0 + g * (1.0 - sg))
    du = da * g * sg
    return dg, du


# ------------------------------------------------------------ cross entropy
def cross_entropy_fwd_bwd(logits, labels):
    """Mean over rows of logsumexp(z) - z[label]; gradient (softmax - onehot)/M."""
    M = logits.shape[0]
    mx = np.max(logits, axis=1, keepdims=True)
    e = np.exp(logits - mx)
    den = np.sum(e, axis=1, keepdims=True)
    lse = (mx + np.log(den))[:, 0]
    rows = np.arange(M)
    loss = np.sum(lse - logits[rows, labels]) / M
    dz = e / den
    dz[rows, labels] -= 1.0
    dz /= M
    return loss, dz


# --------------------------------------------------------------- embedding
def embedding_fwd(E, tokens):
    return E[tokens.reshape(-1)]


def embedding_bwd(dx, tokens, vocab):
    """dE[v] = sum over tokens t with id v of dx[t]."""
    dE = np.zeros((vocab, dx.shape[1]), dtype=dx.dtype)
    np.add.at(dE, tokens.reshape(-1), dx)
    return dE


# ------------------------------------------------------------------ linear
def linear_fwd(x, W):
    """y = x W^T with W [out, in]."""
    return x @ W.T


def linear_bwd(dy, x, W):
    """dx = dy W; dW = dy^T x."""
    return dy @ W, dy.T @ x
