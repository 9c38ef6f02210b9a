"""Host-side checks of libmt.so that need no GPU.

* the library loads and exports every function declared in include/*.h;
* its flat layout equals the oracle's, independently written, bit for bit;
* its fp32 -> bf16 rounding equals torch's on all 2^32 bit patterns;
* its host Adam, fed the same FP32 gradients, matches the oracle's Adam
  within 1e-6 * (lr / 1e-3) (the post-Adam master tolerance);
* argument validation and host-side fault injection fail cleanly.
"""
import ctypes as C
import glob
import os
import re

import numpy as np
import pytest
import torch

import host_memory_resident_gb300 as mt
import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(mt.LIB_PATH):
        import host_memory_resident_gb300.build as b
        b.build()
    return mt.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(mt_\w+)\s*\(", text):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert len(names) >= 30
    missing = [n for n in sorted(names) if not hasattr(L, n)]
    assert not missing, missing
    assert set(mt.EXPORTS) <= names


def test_binding_structs_match_the_header():
    """The ctypes mirrors of mt_kernel_profile and mt_config have the header's
    sizes (a mismatch would let the library write past the Python buffer)."""
    text = open(os.path.join(ROOT, "include", "mt.h")).read()
    classes = {int(v): n.lower() for n, v in re.findall(r"#define MT_PROF_(\w+) (\d+)", text) if n != "N"}
    n_prof = int(re.search(r"#define MT_PROF_N (\d+)", text).group(1))
    assert len(mt.PROF_CLASSES) == n_prof == len(classes)
    assert [classes[i] for i in range(n_prof)] == mt.PROF_CLASSES
    assert C.sizeof(mt.KernelProfile) == n_prof * 8 * 4
    body = re.search(r"typedef struct mt_config \{(.*?)\} mt_config;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    n_fields = sum(len(decl.split(",")) for decl in re.findall(r"(?:int32_t|float)\s+([^;]+);", body))
    assert C.sizeof(mt.Config) == 4 * n_fields


@pytest.mark.parametrize("name", ["tiny", "1.1b", "7b", "14b", "7b-256k", "padded", "gqa"])
def test_layout_matches_oracle(L, name):
    if name == "padded":
        shape = synth.workload("tiny").with_(d_model=128, ffn_dim=192, vocab=520)
    elif name == "gqa":
        shape = synth.workload("tiny").with_(n_heads=8, n_kv_heads=2, head_dim=16, n_layers=3)
    else:
        shape = synth.workload(name)
    cfg = mt.make_config(shape)
    descs, n_total = mt.layout(cfg)
    lay = oracle.build_layout(shape)
    assert n_total == lay.n_total
    ts = list(lay.tensors())
    assert len(ts) == len(descs)
    unit_index = {u.name: i for i, u in enumerate(lay.units)}
    for t, dsc in zip(ts, descs):
        u = next(u for u in lay.units if t in u.tensors)
        assert dsc["name"] == t.name
        assert dsc["offset"] == t.offset
        assert dsc["unit"] == unit_index[u.name]
        rows, cols = (t.shape[0], t.shape[1]) if len(t.shape) == 2 else (t.shape[0], 1)
        assert (dsc["rows"], dsc["cols"]) == (rows, cols)
        assert dsc["kind"] == (0 if t.kind == "normal" else 1)
    for i, u in enumerate(lay.units):
        assert mt.unit_range(cfg, i) == (u.offset, u.length)


def test_layout_rejects_bad_shapes(L):
    base = synth.workload("tiny")
    for bad in (dict(head_dim=32), dict(n_kv_heads=3), dict(d_model=100), dict(vocab=511), dict(n_slabs=1),
                dict(ckpt_interval=0)):
        cfg = mt.make_config(base.with_(**{k: v for k, v in bad.items() if k not in ("n_slabs", "ckpt_interval")}))
        if "n_slabs" in bad:
            cfg.n_slabs = bad["n_slabs"]
        if "ckpt_interval" in bad:
            cfg.ckpt_interval = bad["ckpt_interval"]
        n = C.c_int()
        tot = C.c_int64()
        assert L.mt_layout(C.byref(cfg), None, 0, C.byref(n), C.byref(tot)) == mt.MT_EINVAL


def test_bf16_rounding_all_patterns(L):
    step = 1 << 26
    for lo in range(0, 1 << 32, step):
        bits = np.arange(lo, lo + step, dtype=np.uint64).astype(np.uint32)
        f = bits.view(np.float32)
        ours = mt.host_to_bf16(f)
        ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        nan = np.isnan(f)
        assert np.array_equal(ours[~nan], ref[~nan]), hex(lo)
        # every NaN stays a NaN (canonical quiet NaN)
        assert np.all((ours[nan] & 0x7f80) == 0x7f80) and np.all((ours[nan] & 0x7f) != 0)


def test_host_adam_matches_oracle_with_identical_grads(L):
    rng = np.random.default_rng(0)
    n = 100_003
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    wo, mo, vo = w.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    store = np.empty(n, np.uint16)
    for t in range(1, 6):
        g = (rng.standard_normal(n) * 10.0 ** rng.integers(-7, -1, size=n)).astype(np.float32)
        g[::97] = 0.0
        mt.host_adam(w, m, v, g, t, lr, b1, b2, eps, store=store)
        wo, mo, vo = oracle.adam_update(wo, mo, vo, g.astype(np.float64), t, lr, b1, b2, eps)
        assert np.max(np.abs(w - wo)) <= 1e-6 * (lr / 1e-3)
        # beta1 / beta2 reach the library as float32 (0.999f differs from 0.999
        # by 1.3e-8, i.e. 1.3e-5 relative on 1 - beta2)
        np.testing.assert_allclose(m, mo, rtol=5e-5, atol=1e-6 * np.abs(mo).max())
        np.testing.assert_allclose(v, vo, rtol=5e-5, atol=1e-18)
        assert np.array_equal(store, mt.host_to_bf16(w))


def test_host_adam_closed_form_first_step(L):
    g = np.array([0.3, -2.0, 0.0, 1e-3, 5e-9], np.float32)
    w = np.array([0.5, -1.0, 2.0, 0.0, 1.0], np.float32)
    w0 = w.copy()
    m = np.zeros(5, np.float32)
    v = np.zeros(5, np.float32)
    mt.host_adam(w, m, v, g, 1, 1e-3, 0.9, 0.999, 1e-8)
    expect = w0.astype(np.float64) - 1e-3 * g / (np.abs(g.astype(np.float64)) + 1e-8)
    np.testing.assert_allclose(w, expect, rtol=0, atol=2e-7)
    assert w[2] == w0[2]


def test_init_rejects_bad_arguments_without_gpu(L):
    cfg = mt.make_config(synth.workload("tiny"))
    h = C.c_void_p()
    a = np.zeros(10, np.float32)
    p = a.ctypes.data_as(C.c_void_p)
    assert L.mt_init(C.byref(cfg), p, p, p, p, 10, C.byref(h)) == mt.MT_EINVAL  # wrong n_total
    assert "n_total" in L.mt_last_error(None).decode()
    assert L.mt_init(C.byref(cfg), None, p, p, p, 10, C.byref(h)) == mt.MT_EINVAL
    assert h.value is None


def test_injected_allocation_failure_is_clean(L):
    shape = synth.workload("tiny")
    cfg = mt.make_config(shape)
    _, n_total = mt.layout(cfg)
    arrs = [np.zeros(n_total, np.float32) for _ in range(4)]
    ptrs = [a.ctypes.data_as(C.c_void_p) for a in arrs]
    assert L.mt_debug_inject_global(4, 1) == mt.MT_OK
    h = C.c_void_p()
    assert L.mt_init(C.byref(cfg), *ptrs, n_total, C.byref(h)) == mt.MT_ENOMEM
    assert h.value is None
    assert "injected" in L.mt_last_error(None).decode()


def test_null_handle_calls_fail_cleanly(L):
    loss = C.c_float()
    assert L.mt_train_step(None, None, None, 1, 1, C.byref(loss)) == mt.MT_EINVAL
    assert L.mt_read_grads(None, None, 0) == mt.MT_EINVAL
    assert L.mt_destroy(None) == mt.MT_EINVAL


def test_gemm_splitk_factor_choices(L):
    # 160 tiles of the 1.1B QKV gradient over 16384 tokens: split; 2000 tiles
    # of the head gradient, or a short K: not split
    assert mt.k_gemm_splitk(2560, 2048, 16384) > 1
    assert mt.k_gemm_splitk(32000, 2048, 16384) == 1
    assert mt.k_gemm_splitk(2560, 2048, 512) == 1
    assert mt.k_gemm_wgrad_ws(32000, 2048) == 0
