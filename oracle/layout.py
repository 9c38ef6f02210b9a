"""Flat parameter layout, restated independently of the CUDA library.

The articles say only that each layer's weights are kept pre-flattened and
page-locked ("layer_pinned_flats", lqnn.cn article section 三.1) and that a
flat tensor layout keeps host memory linear in the parameter count
(zhichai.net article, section "MegaTrain 的性能与能力"). The order is a
reading:

    unit 0          : embed            [V, d]
    unit 1 + l      : layer l: attn_norm [d], Wqkv [(H + 2 Hkv) hd, d]
                      (q rows, then k rows, then v rows), Wo [d, H hd],
                      mlp_norm [d], Wgu [2 f, d] (gate rows, then up rows),
                      Wdown [d, f]
    unit L + 1      : final_norm [d], head [V, d] (untied)

Matrices are row-major [out, in]. Every tensor starts at a multiple of
ALIGN elements; padding elements are zero and are counted in n_total. FP32
host arrays and the bf16 store share these element indices.
"""
from __future__ import annotations

import dataclasses

ALIGN = 64


@dataclasses.dataclass(frozen=True)
class Tensor:
    name: str
    offset: int          # absolute element offset in the flat arrays
    shape: tuple
    kind: str            # "normal" (matrix) or "ones" (norm weight)

    @property
    def size(self) -> int:
        n = 1
        for s in self.shape:
            n *= s
        return n


@dataclasses.dataclass(frozen=True)
class Unit:
    name: str
    offset: int
    length: int          # elements including trailing padding
    tensors: tuple


@dataclasses.dataclass(frozen=True)
class Layout:
    units: tuple
    n_total: int

    def tensors(self):
        for u in self.units:
            yield from u.tensors

    def segments(self):
        return [(t.offset, t.size, t.kind) for t in self.tensors()]

    def find(self, unit: str, name: str) -> Tensor:
        for u in self.units:
            if u.name == unit:
                for t in u.tensors:
                    if t.name == name:
                        return t
        raise KeyError((unit, name))


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def build_layout(shape) -> Layout:
    d, V = shape.d_model, shape.vocab
    qkv = (shape.n_heads + 2 * shape.n_kv_heads) * shape.head_dim
    hq = shape.n_heads * shape.head_dim
    f = shape.ffn_dim

    units = []
    cursor = 0

    def unit(name, specs):
        nonlocal cursor
        start = cursor
        ts = []
        for tname, tshape, kind in specs:
            cursor = _round_up(cursor, ALIGN)
            t = Tensor(tname, cursor, tuple(tshape), kind)
            ts.append(t)
            cursor += t.size
        cursor = _round_up(cursor, ALIGN)
        units.append(Unit(name, start, cursor - start, tuple(ts)))

    unit("embed", [("embed", (V, d), "normal")])
    for layer in range(shape.n_layers):
        unit(f"layer{layer}", [
            ("attn_norm", (d,), "ones"),
            ("wqkv", (qkv, d), "normal"),
            ("wo", (d, hq), "normal"),
            ("mlp_norm", (d,), "ones"),
            ("wgu", (2 * f, d), "normal"),
            ("wdown", (d, f), "normal"),
        ])
    unit("head", [("final_norm", (d,), "ones"), ("head", (V, d), "normal")])
    return Layout(tuple(units), cursor)
