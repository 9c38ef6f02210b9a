"""bench.py's multi-rank plumbing on CPU: two gloo ranks (replicas only, no
data-path collective) agree on the max step time and the summed tokens."""
import os
import socket

import pytest
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local, pg = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(pg)
    t = bench.max_over_ranks(pg, 1.0 + rank)
    tok = bench.sum_over_ranks(pg, 100.0 * (rank + 1))
    out.put((rank, t, tok))
    pg.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_tokens():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2.0, 300.0), (1, 2.0, 300.0)]


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench

    class A:
        gpus, steps, warmup = 2, 1, 0
    assert bench.run_reference(A, None, 2, 1, None) == 0


def test_bench_refuses_workloads_beyond_host_memory():
    """The bench's guard: the 14B workload's host state and pinned buffers
    (about 285 GB) do not fit 199 GB of host memory; the 1.1B workload's do."""
    import bench
    import host_memory_resident_gb300 as mt
    import synth
    big, small = synth.workload("14b"), synth.workload("1.1b")
    avail = 199 * 2**30
    r = bench.host_memory_refusal(mt, mt.make_config(big), big, True, avail)
    assert r is not None and r["value"] is None and "host memory" in r["error"]
    assert bench.host_memory_refusal(mt, mt.make_config(small), small, True, avail) is None
    # unknown available memory: no refusal
    assert bench.host_memory_refusal(mt, mt.make_config(big), big, True, None) is None


def test_default_workload_fits_the_host():
    """The bench's default workload (7B: about 126 GB of host state and
    pinned buffers) fits 199 GB of host memory once, not twice: replicas on
    one host are refused before anything is allocated."""
    import bench
    import host_memory_resident_gb300 as mt
    import synth
    sh = synth.workload("7b")
    assert bench.host_memory_refusal(mt, mt.make_config(sh), sh, True, 199 * 2**30) is None
    r = bench.host_memory_refusal(mt, mt.make_config(sh), sh, True, 199 * 2**30, ranks=2)
    assert r is not None and "2 replica(s)" in r["error"]


def test_reference_arm_line_carries_the_repo_arms_config(capsys):
    """Both arms describe the workload with the same config dict, so their
    lines compare like for like; run here on the tiny workload."""
    import json

    import bench
    import oracle
    import synth

    class A:
        gpus, steps, warmup = 1, 1, 0
        overlap, keep_grads, unfused, keep_attention = True, True, False, False
    sh = synth.workload("tiny")
    assert bench.run_reference(A, sh, 1, 0, None) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.config_dict(A, sh, 1, oracle.build_layout(sh).n_total)
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"


def test_timeline_gap_classification():
    """Idle gaps of the compute stream are split into time the host
    optimizer was busy, time only a copy was, and the rest."""
    import bench
    tl = [{"stream": "compute", "cls": "gemm", "start_ms": 0, "end_ms": 10},
          {"stream": "compute", "cls": "gemm", "start_ms": 20, "end_ms": 30},
          {"stream": "compute", "cls": "ce", "start_ms": 40, "end_ms": 50},
          {"stream": "h2d", "cls": "unit 1", "start_ms": 12, "end_ms": 18},
          {"stream": "host_adam", "cls": "unit 1", "start_ms": 31, "end_ms": 35},
          {"stream": "d2h", "cls": "unit 2", "start_ms": 33, "end_ms": 38}]
    s = bench.timeline_summary(tl)
    assert s["gpu_idle"] == {"ms": 20, "while_host_optimizer_busy_ms": 4.0, "copy_only_ms": 9.0, "neither_ms": 7.0}
    assert s["h2d"]["hidden_frac"] == 0.0 and s["d2h"]["hidden_frac"] == 0.0
    # the d2h copy runs 2 ms of its 5 under the host optimizer: not exposed
    assert s["h2d"]["exposed_ms"] == 6.0 and s["d2h"]["exposed_ms"] == 3.0
    assert abs(s["d2h"]["not_exposed_frac"] - 0.4) < 1e-12
    assert bench._subtract([(0, 10)], [(2, 3), (5, 12)]) == [(0, 2), (3, 5)]
