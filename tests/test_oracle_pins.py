"""Pins of the oracle against facts other than itself (CPU only).

* finite differences of the whole step (backward against forward);
* torch autograd of the same decoder built from torch library operators
  (F.rms_norm, complex-number RoPE, F.scaled_dot_product_attention,
  F.silu, F.cross_entropy), which pins the forward and the backward;
* closed forms: CE with a zero head is ln V; RMSNorm of a constant row;
  RoPE identity at position 0, norm preservation, inverse rotation;
  attention with zero queries is the running mean of v; s = 1 gives v;
* torch.optim.Adam on hand-set tensors and Adam's closed forms;
* the flat layout against the published parameter counts of the
  TinyLlama-1.1B, Llama-2-7B and (bias-free) Qwen2.5-14B shapes;
* invariance of the gradient under the checkpoint interval and streaming.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth
from oracle import ops


def _inputs(shape, seed=0, tok_seed=1):
    lay = oracle.build_layout(shape)
    master = synth.init_master(lay.n_total, lay.segments(), seed=seed)
    tokens, labels = synth.make_tokens(shape.vocab, shape.batch, shape.seq, seed=tok_seed)
    return lay, master, tokens, labels


# ------------------------------------------------------------------ layout
@pytest.mark.parametrize("name,expected", [
    ("tiny", 196_928),
    ("1.1b", 1_100_048_384),   # TinyLlama-1.1B published parameter count
    ("7b", 6_738_415_616),     # Llama-2-7B published parameter count
    ("14b", 14_770_033_664 - 48 * (5120 + 2 * 1024)),  # Qwen2.5-14B minus its QKV biases
])
def test_layout_totals(name, expected):
    lay = oracle.build_layout(synth.workload(name))
    n_params = sum(t.size for t in lay.tensors())
    assert n_params == expected
    # every width in these shapes is a multiple of 64, so no padding
    assert lay.n_total == expected


def test_layout_offsets_aligned_and_disjoint(tiny):
    shape = tiny.with_(d_model=72, ffn_dim=200, head_dim=18)  # forces padding
    lay = oracle.build_layout(shape)
    prev_end = 0
    for u in lay.units:
        assert u.offset == prev_end and u.offset % oracle.ALIGN == 0
        for t in u.tensors:
            assert t.offset % oracle.ALIGN == 0
            assert t.offset >= prev_end
            prev_end = t.offset + t.size
        prev_end = u.offset + u.length
        assert u.length % oracle.ALIGN == 0
    assert lay.n_total == prev_end


# ------------------------------------------------------------ closed forms
def test_ce_zero_head_is_ln_v():
    for V in (512, 32000):
        M = 6
        logits = np.zeros((M, V))
        labels = np.arange(M) % V
        loss, dz = ops.cross_entropy_fwd_bwd(logits, labels)
        assert loss == pytest.approx(math.log(V), rel=1e-15)
        expect = np.full((M, V), 1.0 / V)
        expect[np.arange(M), labels] -= 1.0
        np.testing.assert_allclose(dz, expect / M, rtol=1e-14, atol=0)


def test_rmsnorm_constant_row():
    d, c, eps = 64, 0.37, 1e-5
    w = np.linspace(0.5, 1.5, d)
    x = np.full((3, d), c)
    y, r = ops.rmsnorm_fwd(x, w, eps)
    np.testing.assert_allclose(y, np.tile(w * c / math.sqrt(c * c + eps), (3, 1)), rtol=1e-14)
    np.testing.assert_allclose(r, 1.0 / math.sqrt(c * c + eps), rtol=1e-14)


def test_rope_identity_norm_inverse():
    rng = np.random.default_rng(3)
    B, s, nh, hd = 2, 9, 3, 16
    x = rng.standard_normal((B, s, nh, hd))
    cos, sin = ops.rope_tables(s, hd, 10000.0)
    y = ops.rope_fwd(x, cos, sin)
    np.testing.assert_array_equal(y[:, 0], x[:, 0])            # position 0
    half = hd // 2
    n_in = x[..., :half] ** 2 + x[..., half:] ** 2
    n_out = y[..., :half] ** 2 + y[..., half:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-13)         # pairwise norm
    np.testing.assert_allclose(ops.rope_bwd(y, cos, sin), x, rtol=1e-13, atol=1e-14)
    # position 1, pair 0 rotates by exactly 1 radian
    assert y[0, 1, 0, 0] == pytest.approx(x[0, 1, 0, 0] * math.cos(1) - x[0, 1, 0, half] * math.sin(1))


def test_attention_closed_forms():
    rng = np.random.default_rng(4)
    B, s, H, Hkv, hd = 2, 7, 4, 2, 8
    k = rng.standard_normal((B, s, Hkv, hd))
    v = rng.standard_normal((B, s, Hkv, hd))
    q = np.zeros((B, s, H, hd))
    o, lse = ops.attention_fwd(q, k, v)
    grp = H // Hkv
    for h in range(H):
        running_mean = np.cumsum(v[:, :, h // grp], axis=1) / np.arange(1, s + 1)[None, :, None]
        np.testing.assert_allclose(o[:, :, h], running_mean, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse[:, h], np.tile(np.log(np.arange(1, s + 1)), (B, 1)), rtol=1e-13, atol=1e-15)
    q1 = rng.standard_normal((B, 1, H, hd))
    o1, _ = ops.attention_fwd(q1, k[:, :1], v[:, :1])
    for h in range(H):
        np.testing.assert_allclose(o1[:, 0, h], v[:, 0, h // grp], rtol=1e-14)


def test_attention_rows_match_full():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 11, 2, 8))
    k = rng.standard_normal((1, 11, 1, 8))
    v = rng.standard_normal((1, 11, 1, 8))
    o, lse = ops.attention_fwd(q, k, v)
    rows = np.array([0, 4, 10])
    o_r, lse_r = ops.attention_fwd(q, k, v, rows=rows)
    np.testing.assert_allclose(o_r, o[:, rows], rtol=1e-13)
    np.testing.assert_allclose(lse_r, lse[:, :, rows], rtol=1e-13)


def test_embedding_bwd_is_onehot_transpose():
    rng = np.random.default_rng(6)
    V, d = 13, 5
    tokens = rng.integers(0, V, size=(3, 8))
    dx = rng.standard_normal((24, d))
    onehot = np.zeros((24, V))
    onehot[np.arange(24), tokens.reshape(-1)] = 1.0
    np.testing.assert_allclose(ops.embedding_bwd(dx, tokens, V), onehot.T @ dx, rtol=1e-14, atol=1e-15)


# ------------------------------------------------------------------- Adam
def test_adam_closed_forms():
    w = np.array([0.5, -1.0, 2.0, 0.0])
    g = np.array([0.3, -2.0, 0.0, 1e-3])
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    w1, m1, v1 = oracle.adam_update(w, np.zeros(4), np.zeros(4), g, 1, lr, b1, b2, eps)
    np.testing.assert_allclose(w1, w - lr * g / (np.abs(g) + eps), rtol=0, atol=1e-16)
    assert w1[2] == w[2]                               # zero gradient: unchanged
    # constant gradient: m_hat = g and v_hat = g^2 at every t
    m, v, ww = np.zeros(4), np.zeros(4), w.copy()
    for t in range(1, 6):
        prev = ww
        ww, m, v = oracle.adam_update(ww, m, v, g, t, lr, b1, b2, eps)
        np.testing.assert_allclose(prev - ww, lr * g / (np.abs(g) + eps), rtol=1e-9, atol=1e-18)


def test_adam_matches_torch_optim():
    rng = np.random.default_rng(7)
    n = 1000
    w0 = rng.standard_normal(n)
    p = torch.nn.Parameter(torch.tensor(w0, dtype=torch.float64))
    opt = torch.optim.Adam([p], lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0)
    w, m, v = w0.copy(), np.zeros(n), np.zeros(n)
    for t in range(1, 8):
        g = rng.standard_normal(n) * (10.0 ** rng.integers(-6, 1, size=n))
        p.grad = torch.tensor(g)
        opt.step()
        w, m, v = oracle.adam_update(w, m, v, g, t, 1e-3, 0.9, 0.999, 1e-8)
        np.testing.assert_allclose(w, p.detach().numpy(), rtol=0, atol=1e-15)


# ------------------------------------------------- whole step vs torch ops
def _torch_step(shape, master, tokens, labels):
    lay = oracle.build_layout(shape)
    flat = torch.tensor(master, dtype=torch.float64)
    leaves = {}

    def param(unit, name):
        t = lay.find(unit, name)
        p = flat[t.offset:t.offset + t.size].reshape(t.shape).clone().requires_grad_(True)
        leaves[(unit, name)] = (t, p)
        return p

    B, s = tokens.shape
    H, Hkv, hd, f, d = shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim, shape.d_model
    pos = torch.arange(s, dtype=torch.float64)
    inv = shape.rope_theta ** (-torch.arange(0, hd // 2, dtype=torch.float64) * 2.0 / hd)
    rot = torch.polar(torch.ones(s, hd // 2, dtype=torch.float64), pos[:, None] * inv[None, :])

    def rope(x):  # x [B, s, n, hd]; complex pair (x_i, x_{i+hd/2})
        z = torch.complex(x[..., :hd // 2], x[..., hd // 2:]) * rot[None, :, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    tok = torch.tensor(tokens, dtype=torch.long)
    x = F.embedding(tok, param("embed", "embed")).reshape(B * s, d)
    for layer in range(shape.n_layers):
        un = f"layer{layer}"
        u = F.rms_norm(x, (d,), param(un, "attn_norm"), eps=shape.rms_eps)
        qkv = F.linear(u, param(un, "wqkv"))
        q = rope(qkv[:, :H * hd].reshape(B, s, H, hd))
        k = rope(qkv[:, H * hd:(H + Hkv) * hd].reshape(B, s, Hkv, hd))
        v = qkv[:, (H + Hkv) * hd:].reshape(B, s, Hkv, hd)
        rep = H // Hkv
        k = k.repeat_interleave(rep, dim=2)
        v = v.repeat_interleave(rep, dim=2)
        o = F.scaled_dot_product_attention(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2),
                                           is_causal=True)
        o = o.transpose(1, 2).reshape(B * s, H * hd)
        h = x + F.linear(o, param(un, "wo"))
        z = F.rms_norm(h, (d,), param(un, "mlp_norm"), eps=shape.rms_eps)
        gu = F.linear(z, param(un, "wgu"))
        x = h + F.linear(F.silu(gu[:, :f]) * gu[:, f:], param(un, "wdown"))
    xh = F.rms_norm(x, (d,), param("head", "final_norm"), eps=shape.rms_eps)
    loss = F.cross_entropy(F.linear(xh, param("head", "head")), torch.tensor(labels, dtype=torch.long).reshape(-1))
    loss.backward()
    grad = np.zeros(lay.n_total)
    for (t, p) in leaves.values():
        grad[t.offset:t.offset + t.size] = p.grad.reshape(-1).numpy()
    return float(loss.detach()), grad


@pytest.mark.parametrize("variant", ["tiny", "gqa"])
def test_step_matches_torch_autograd(tiny, variant):
    shape = tiny if variant == "tiny" else tiny.with_(n_heads=4, n_kv_heads=2, n_layers=3, ckpt_interval=2)
    lay, master, tokens, labels = _inputs(shape)
    master = master * 20.0  # larger weights so every term matters
    for t in lay.tensors():
        if t.kind == "ones":
            master[t.offset:t.offset + t.size] = 1.0 + 0.1 * np.sin(np.arange(t.size))
    loss, grad = oracle.step_grads(shape, master, tokens, labels)
    tl, tg = _torch_step(shape, master, tokens, labels)
    assert loss == pytest.approx(tl, rel=1e-12)
    for t in lay.tensors():
        a = grad[t.offset:t.offset + t.size]
        b = tg[t.offset:t.offset + t.size]
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-12 * np.abs(b).max(), err_msg=t.name)


# ---------------------------------------------------- finite differences
def test_step_finite_differences(tiny):
    shape = tiny.with_(n_heads=4, n_kv_heads=2)
    lay, master, tokens, labels = _inputs(shape, seed=11)
    master = master.astype(np.float64) * 5.0
    loss, grad = oracle.step_grads(shape, master, tokens, labels)
    f = lambda w: oracle.step_grads(shape, w, tokens, labels)[0]  # noqa: E731
    rng = np.random.default_rng(0)
    # directional derivatives over all parameters at once
    for _ in range(3):
        dirn = rng.standard_normal(lay.n_total)
        dirn /= np.linalg.norm(dirn)
        h = 1e-6
        fd = (f(master + h * dirn) - f(master - h * dirn)) / (2 * h)
        assert fd == pytest.approx(float(grad @ dirn), rel=1e-6)
    # coordinates: the largest-gradient entry of every tensor plus random ones
    gmax = np.abs(grad).max()
    for t in lay.tensors():
        seg = grad[t.offset:t.offset + t.size]
        idx = [int(np.argmax(np.abs(seg)))] + list(rng.integers(0, t.size, size=2))
        for i in idx:
            j = t.offset + i
            h = 1e-6
            wp, wm = master.copy(), master.copy()
            wp[j] += h
            wm[j] -= h
            fd = (f(wp) - f(wm)) / (2 * h)
            assert abs(fd - grad[j]) <= 1e-6 * gmax, (t.name, i, fd, grad[j])


# ------------------------------------------------------------- invariants
@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_grads_invariant_to_ckpt_interval_and_streaming(tiny, dtype):
    shape = tiny.with_(n_layers=4)
    _, master, tokens, labels = _inputs(shape)
    ref_loss, ref = oracle.step_grads(shape, master, tokens, labels, ckpt_interval=1, dtype=dtype)
    for C in (1, 2, 3, 4):
        for streamed in (False, True):
            loss, g = oracle.step_grads(shape, master, tokens, labels, ckpt_interval=C,
                                        streamed=streamed, dtype=dtype)
            assert loss == ref_loss
            np.testing.assert_array_equal(g, ref)


def test_loss_at_init_near_ln_v(tiny):
    _, master, tokens, labels = _inputs(tiny)
    loss, _ = oracle.step_grads(tiny, master, tokens, labels)
    assert abs(loss - math.log(tiny.vocab)) < 0.05


# ------------------------------------------- planted mistakes are caught
def _mut_rmsnorm_bwd(dy, x, w, rstd):
    dx, dw = _ORIG["rmsnorm_bwd"](dy, x, w, rstd)
    return dy * w[None, :] * rstd[:, None], dw          # dropped projection term


def _mut_rope_bwd(dy, cos, sin):
    return _ORIG["rope_fwd"](dy, cos, sin)                # wrong rotation sign


def _mut_swiglu_bwd(da, g, u):
    dg, du = _ORIG["swiglu_bwd"](da, g, u)
    sg = 1.0 / (1.0 + np.exp(-g))
    return da * u * sg, du                                # dropped silu' term


def _mut_attention_bwd(q, k, v, do):
    dq, dk, dv = _ORIG["attention_bwd"](q, k, v, do)
    return dq, dk, dv * 0.5 + dv * 0.5 * (1 + 1e-3)       # perturbed dV


def _mut_linear_bwd(dy, x, W):
    dx, dW = _ORIG["linear_bwd"](dy, x, W)
    return dx, (dW.T if dW.shape[0] == dW.shape[1] else dW * (1 + 1e-6))  # transposed operand


def _mut_ce(logits, labels):
    loss, dz = _ORIG["cross_entropy_fwd_bwd"](logits, labels)
    return loss, dz * logits.shape[0]                     # missing 1/M


_ORIG = {n: getattr(ops, n) for n in
         ("rmsnorm_bwd", "rope_fwd", "rope_bwd", "swiglu_bwd", "attention_bwd", "linear_bwd",
          "cross_entropy_fwd_bwd")}


@pytest.mark.parametrize("name,fn", [
    ("rmsnorm_bwd", _mut_rmsnorm_bwd), ("rope_bwd", _mut_rope_bwd),
    ("swiglu_bwd", _mut_swiglu_bwd), ("attention_bwd", _mut_attention_bwd),
    ("linear_bwd", _mut_linear_bwd), ("cross_entropy_fwd_bwd", _mut_ce),
])
def test_planted_mistake_is_caught(tiny, monkeypatch, name, fn):
    lay, master, tokens, labels = _inputs(tiny)
    master = master * 20.0
    _, tg = _torch_step(tiny, master, tokens, labels)
    monkeypatch.setattr(ops, name, fn)
    _, grad = oracle.step_grads(tiny, master, tokens, labels)
    caught = False
    for t in lay.tensors():
        a = grad[t.offset:t.offset + t.size]
        b = tg[t.offset:t.offset + t.size]
        if not np.allclose(a, b, rtol=1e-9, atol=1e-12 * np.abs(b).max()):
            caught = True
    assert caught


def test_bf16_emulation_rounding_matches_torch():
    """The rounding used to derive tolerance floors is torch's bf16 rounding."""
    from oracle.bf16_emulation import to_bf16
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-38, 38, 200000),
                        [np.inf, -np.inf, np.nan, 0.0, -0.0, 1.00390625, 1.01171875, 3.4e38]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = to_bf16(x)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(got[~nan], ref[~nan].astype(np.float64))
    assert np.isnan(got[nan]).all()


def test_bf16_emulation_is_close_to_exact_step(tiny):
    """With bf16 storage the tiny step moves by well under 1%: the emulation
    is the exact step plus rounding, not a different computation."""
    from oracle.bf16_emulation import step_grads_bf16_storage
    lay, master, tokens, labels = _inputs(tiny)
    loss, g = step_grads_bf16_storage(tiny, master, tokens, labels)
    rl, rg = oracle.step_grads(tiny, master, tokens, labels)
    assert abs(loss - rl) / rl < 1e-3
    assert np.linalg.norm(g - rg) / np.linalg.norm(rg) < 1e-2
