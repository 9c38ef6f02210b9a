"""Seeded synthetic workloads: model shapes and the random inputs of a step.

This module holds no arithmetic of the training method. It names the model
shapes of the five decoder workloads and draws the seeded random numbers that
both the CUDA path and the oracle consume: the initial FP32 master weights
(normal(0, 0.02) for matrices, 1.0 for norm weights) and the uniform token /
label ids. Which flat ranges are matrices and which are norm weights is
passed in by the caller as a list of segments, so this module does not know
the flat layout either.

The shapes follow the RAM-centric training articles' running examples
(MegaTrain articles: "单卡训百亿大模型的突破与实践", section on performance,
and "單卡也能練 100B+", section 3 on long context); the exact widths are the
common Llama-family shapes at 1.1B / 7B / 14B parameters.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

__all__ = [
    "ModelShape", "WORKLOADS", "workload", "init_master", "make_tokens",
]


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Shape and run settings of one synthetic decoder workload."""
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    batch: int
    seq: int
    ckpt_interval: int
    n_slabs: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    adam_eps: float = 1e-8

    def with_(self, **kw) -> "ModelShape":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": ModelShape("tiny", 2, 64, 4, 4, 16, 256, 512, 2, 32, 1, 2),
    "1.1b": ModelShape("1.1b", 22, 2048, 32, 4, 64, 5632, 32000, 8, 2048, 4, 12),
    "7b": ModelShape("7b", 32, 4096, 32, 32, 128, 11008, 32000, 2, 4096, 4, 12),
    "14b": ModelShape("14b", 48, 5120, 40, 8, 128, 13824, 152064, 1, 4096, 4, 12),
    "7b-256k": ModelShape("7b-256k", 32, 4096, 32, 32, 128, 11008, 32000, 1, 262144, 1, 12),
}


def workload(name: str) -> ModelShape:
    return WORKLOADS[name]


_CHUNK = 1 << 24  # elements per independently seeded chunk


def _fill_normal(out: np.ndarray, seed: int, chunk_index: int, std: float) -> None:
    rng = np.random.Generator(np.random.Philox(key=seed, counter=[0, 0, 0, chunk_index]))
    rng.standard_normal(out=out, dtype=np.float32)
    out *= np.float32(std)


def init_master(n_total: int, segments, seed: int = 0, std: float = 0.02,
                threads: int | None = None) -> np.ndarray:
    """Initial FP32 master weights of length ``n_total``.

    ``segments`` is an iterable of ``(offset, length, kind)`` with kind
    ``"normal"`` (normal(0, std)) or ``"ones"`` (norm weights). Elements not
    covered (alignment padding) are 0. The normal draw of an element is a fixed
    function of (seed, element index): the flat array is cut into fixed chunks
    of 2**24 elements, each drawn from its own Philox stream, so the result does
    not depend on the thread count or on how the segments are split.
    """
    out = np.zeros(n_total, dtype=np.float32)
    segs = [(int(o), int(n), k) for o, n, k in segments]
    for o, n, k in segs:
        if k not in ("normal", "ones"):
            raise ValueError(f"unknown segment kind {k!r}")
        if o < 0 or n < 0 or o + n > n_total:
            raise ValueError("segment out of range")
    normal = [(o, n) for o, n, k in segs if k == "normal" and n > 0]
    chunks = sorted({c for o, n in normal
                     for c in range(o // _CHUNK, (o + n - 1) // _CHUNK + 1)})

    def work(c):
        lo = c * _CHUNK
        hi = min(n_total, lo + _CHUNK)
        tmp = np.empty(hi - lo, dtype=np.float32)
        _fill_normal(tmp, seed, c, std)
        for o, n in normal:
            a, b = max(o, lo), min(o + n, hi)
            if a < b:
                out[a:b] = tmp[a - lo:b - lo]

    nthr = threads or min(32, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(nthr) as ex:
        list(ex.map(work, chunks))
    for o, n, k in segs:
        if k == "ones":
            out[o:o + n] = 1.0
    return out


def make_tokens(vocab: int, batch: int, seq: int, seed: int = 1, step: int = 0):
    """Uniform token ids: ``seq + 1`` ids per row; tokens are the first ``seq``,
    labels the last ``seq`` (next-token targets). int32, row-major [batch, seq]."""
    rng = np.random.Generator(np.random.Philox(key=seed + step))
    ids = rng.integers(0, vocab, size=(batch, seq + 1), dtype=np.int64).astype(np.int32)
    return np.ascontiguousarray(ids[:, :seq]), np.ascontiguousarray(ids[:, 1:])
