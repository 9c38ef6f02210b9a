"""Resource calculator (no GPU): the pages' sizing rules and the planner."""
import pytest

import host_memory_resident_gb300 as mt
import synth
from host_memory_resident_gb300 import resources


def test_host_state_matches_the_pages_sizing_rules():
    e7 = resources.estimate(synth.workload("7b"))
    n = e7["params"]
    # FP32 master + m + v: 12 bytes per parameter, about 12 GB per billion
    # parameters (lqnn.cn article, section 一), so about 81 GB at 7B
    master_m_v = resources.estimate(synth.workload("7b"), keep_grads=False)["host_state_bytes"]
    assert master_m_v == 12 * n
    assert 80e9 < master_m_v < 84e9
    # full precision with the gradient: parameters x 4 bytes x about 4, so a
    # 70B model needs about 1.1 TB (travelaiplan blog, 核心功能 point 1); a
    # Llama-2-70B-shaped decoder here
    s70 = synth.workload("7b").with_(n_layers=80, d_model=8192, n_heads=64, n_kv_heads=8, ffn_dim=28672)
    e70 = resources.estimate(s70, batch=1, seq=4096)
    assert 68e9 < e70["params"] < 70e9
    assert e70["host_state_bytes"] == 16 * e70["params"]
    assert 1.05e12 < e70["host_state_bytes"] < 1.15e12
    assert e7["host_state_bytes"] == 16 * n
    # the bf16 store is 2 bytes per parameter (lqnn.cn section 一: 120B -> ~240 GB)
    assert e7["pinned_bytes"] >= 2 * n


def test_plan_grows_with_tokens_and_not_with_depth_beyond_checkpoints():
    base = synth.workload("1.1b")
    a = resources.estimate(base, batch=4)["device_bytes"]
    b = resources.estimate(base, batch=8)["device_bytes"]
    assert b > a
    # deeper model with the same checkpoint interval: only checkpoints grow
    d1 = resources.estimate(base.with_(n_layers=8), batch=4)["device_bytes"]
    d2 = resources.estimate(base.with_(n_layers=16), batch=4)["device_bytes"]
    ckpt = 4 * 2048 * 2048 * 4  # one [M, d] fp32 checkpoint (the residual stream is fp32)
    assert d2 - d1 == pytest.approx(2 * ckpt, rel=0.01)


def test_suggest_batch_is_the_largest_that_fits():
    shape = synth.workload("1.1b")
    budget = resources.estimate(shape, batch=8)["device_bytes"]
    b = resources.suggest_batch(shape, device_budget=budget)
    assert b == 8
    assert resources.suggest_batch(shape, device_budget=1e6) is None


def test_streamed_units_follow_the_two_buffer_cache():
    # 4 layers, 2-layer segments: the last segment is not recomputed (its
    # last layer is still held, the other one is loaded again); the first
    # segment's layers stay resident from recompute into backward
    assert resources.streamed_units(4, 2) == [0, 1, 2, 3, 4, 5, 3, 1, 2]
    # 1-layer segments: the last layer is still held when backward begins
    assert resources.streamed_units(3, 1) == [0, 1, 2, 3, 4, 2, 1]
    # one 4-layer segment: no recompute; backward re-loads all but the last layer
    assert resources.streamed_units(4, 4) == [0, 1, 2, 3, 4, 5, 3, 2, 1]
    # two 4-layer segments: the first segment's backward re-streams all but
    # the last two of its layers
    assert resources.streamed_units(8, 4) == list(range(10)) + [7, 6, 5, 1, 2, 3, 4, 2, 1]


def test_traffic_matches_the_unit_model():
    shape = synth.workload("tiny").with_(n_layers=4, ckpt_interval=2)
    e = resources.estimate(shape)
    cfg = mt.make_config(shape)
    lay, n = mt.layout(cfg)
    units = [0] * 6
    for t in lay:
        units[t["unit"]] += t["rows"] * t["cols"]
    assert e["h2d_bytes_per_step"] == 2 * (sum(units) + units[3] + units[1] + units[2])
    assert e["d2h_bytes_per_step"] == 2 * n
    e7 = resources.estimate(synth.workload("7b"))
    # 4-layer segments: layer weights cross the link about 2.4 times, the rest once
    assert 4.5 * e7["params"] < e7["h2d_bytes_per_step"] < 5.0 * e7["params"]
