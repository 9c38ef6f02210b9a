"""Pins of oracle.bf16_emulation, the exact step with bf16 rounding at chosen
storage points, which derives the per-tensor error floors of bf16 operands.

It must reduce to the exact oracle with no point switched on, round exactly
like torch, and each switch must act only where it says: a point of the
backward leaves the loss unchanged, the gradient-slab point is the exact
gradient rounded once, and every point alone moves each gradient tensor by
no more than a few bf16 roundings.
"""
import numpy as np
import pytest

import oracle
import synth
from oracle.bf16_emulation import OPERAND_POINTS, OTHER_POINTS, POINTS, step_grads_bf16_storage, to_bf16

BACKWARD_POINTS = ("attn_ds", "grad_operands", "grad_slab", "gate_up_saved", "swiglu_da", "dqk_pre_rope")


def _case(n_layers=2, **kw):
    shape = synth.workload("tiny").with_(n_layers=n_layers, ckpt_interval=1, **kw)
    lay = oracle.build_layout(shape)
    master = synth.init_master(lay.n_total, lay.segments(), seed=0)
    tokens, labels = synth.make_tokens(shape.vocab, shape.batch, shape.seq, seed=1)
    return shape, lay, master, tokens, labels


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def test_points_partition():
    assert set(OPERAND_POINTS) | set(OTHER_POINTS) == set(POINTS)
    assert not set(OPERAND_POINTS) & set(OTHER_POINTS)
    shape, lay, master, tokens, labels = _case()
    with pytest.raises(ValueError):
        step_grads_bf16_storage(shape, master, tokens, labels, points=("bogus",))


def test_to_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        [0.0, -0.0, 1e-40, -1e-40, 3.4e38, np.inf, -np.inf]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(to_bf16(x), ref)


@pytest.mark.parametrize("kw", [{}, {"n_heads": 4, "n_kv_heads": 2, "n_layers": 3}])
def test_no_point_is_the_exact_step(kw):
    """With every switch off the emulation is the plain step: equal to the
    oracle (float64, at the bf16 weight values) up to float64 rounding order."""
    shape, lay, master, tokens, labels = _case(**kw)
    loss, g = step_grads_bf16_storage(shape, master, tokens, labels, points=())
    ref_loss, ref = oracle.step_grads(shape, to_bf16(master), tokens, labels, dtype=np.float64)
    assert abs(loss - ref_loss) <= 1e-12 * abs(ref_loss)
    for t in lay.tensors():
        sl = slice(t.offset, t.offset + t.size)
        assert _rel(g[sl], ref[sl]) <= 1e-10, t.name


def test_backward_points_leave_the_loss_unchanged():
    shape, lay, master, tokens, labels = _case()
    loss0, _ = step_grads_bf16_storage(shape, master, tokens, labels, points=())
    for p in BACKWARD_POINTS:
        loss, _ = step_grads_bf16_storage(shape, master, tokens, labels, points=(p,))
        assert loss == loss0, p
    for p in set(POINTS) - set(BACKWARD_POINTS):
        loss, _ = step_grads_bf16_storage(shape, master, tokens, labels, points=(p,))
        assert loss != loss0, p      # every forward point rounds something the loss sees


def test_gradient_slab_point_rounds_the_exact_gradient_once():
    shape, lay, master, tokens, labels = _case()
    _, g0 = step_grads_bf16_storage(shape, master, tokens, labels, points=())
    _, g1 = step_grads_bf16_storage(shape, master, tokens, labels, points=("grad_slab",))
    assert np.array_equal(g1, to_bf16(g0))


def test_each_point_alone_stays_within_a_few_roundings():
    """One rounding of relative size 2^-9 at one storage point moves every
    gradient tensor of the tiny step by well under 1%; each point moves at
    least one tensor (so no switch is dead)."""
    shape, lay, master, tokens, labels = _case()
    _, g0 = step_grads_bf16_storage(shape, master, tokens, labels, points=())
    for p in POINTS:
        _, g = step_grads_bf16_storage(shape, master, tokens, labels, points=(p,))
        errs = [_rel(g[t.offset:t.offset + t.size], g0[t.offset:t.offset + t.size]) for t in lay.tensors()]
        assert max(errs) < 1e-2, (p, max(errs))
        assert max(errs) > 0.0, p


def test_operand_points_bound_the_full_set():
    """Rounding at the operand points only is no farther from the exact step
    than rounding at every point (the other points only add error)."""
    shape, lay, master, tokens, labels = _case(n_layers=3)
    _, g0 = step_grads_bf16_storage(shape, master, tokens, labels, points=())
    _, go = step_grads_bf16_storage(shape, master, tokens, labels, points=OPERAND_POINTS)
    _, ga = step_grads_bf16_storage(shape, master, tokens, labels, points=POINTS)
    assert _rel(go, g0) < _rel(ga, g0)
