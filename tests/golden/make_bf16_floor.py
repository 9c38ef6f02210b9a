"""Writes bf16_floor.json: the gradient error that bf16 operands alone impose.

The method's products take bf16 operands with FP32 accumulation and its
weights and gradients are bf16 (zhichai.net article, introduction: mixed
precision with bf16 weights and gradients, FP32 optimizer state). For each
parity case of test_step_gpu.py this writes, per gradient tensor, the
relative L2 distance between oracle.bf16_emulation with rounding at exactly
those points (OPERAND_POINTS: the operands of every product and the gradient
slab) and the exact oracle evaluated at the same bf16 weight values. Calls
only oracle/ and synth/. Run from the repository root:
``python tests/golden/make_bf16_floor.py [case ...]``. The 14B cases need
about 60 GB of host memory and the full-depth 1.1B case about 30 minutes on
16 cores.
"""
import gc
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402
from oracle.bf16_emulation import OPERAND_POINTS, step_grads_bf16_storage, to_bf16  # noqa: E402


def cases():
    """name -> (shape, batch, seq, weight scale); batch/seq None = the shape's."""
    tiny = synth.workload("tiny")
    out = {
        "tiny": (tiny, None, None, 1.0),
        "tiny-gqa-ragged": (tiny.with_(n_heads=4, n_kv_heads=2, n_layers=3, ckpt_interval=2), 3, 21, 1.0),
        "tiny-x10": (tiny, None, None, 10.0),
    }
    for name, B, s in (("1.1b", 1, 512), ("7b", 1, 256), ("14b", 1, 128), ("7b-s4096", 1, 4096),
                       ("14b-s4096", 1, 4096)):
        out[name] = (synth.workload(name.split("-")[0]).with_(n_layers=2, ckpt_interval=1), B, s, 1.0)
    out["1.1b-full"] = (synth.workload("1.1b"), 1, 2048, 1.0)
    return out


def master_for(shape, scale):
    lay = oracle.build_layout(shape)
    master = synth.init_master(lay.n_total, lay.segments(), seed=0)
    if scale != 1.0:
        master = master * scale
        for t in lay.tensors():
            if t.kind == "ones":
                master[t.offset:t.offset + t.size] = 1.0
    return lay, master


def floor_for(shape, B, s, scale):
    lay, master = master_for(shape, scale)
    tokens, labels = synth.make_tokens(shape.vocab, B or shape.batch, s or shape.seq, seed=1)
    wb = np.empty(master.shape, dtype=np.float32)  # the bf16 weight values both sides use
    for i in range(0, master.size, 1 << 26):
        wb[i:i + (1 << 26)] = to_bf16(master[i:i + (1 << 26)])
    del master
    gc.collect()
    _, ref = oracle.step_grads(shape, wb, tokens, labels, dtype=np.float64, streamed=True, out_dtype=np.float32)
    gc.collect()
    _, emu = step_grads_bf16_storage(shape, wb, tokens, labels, points=OPERAND_POINTS, out_dtype=np.float32)
    res = {}
    for t in lay.tensors():
        a = emu[t.offset:t.offset + t.size].astype(np.float64)
        b = ref[t.offset:t.offset + t.size].astype(np.float64)
        res[f"{t.name}@{t.offset}"] = float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
    return res


def main(names):
    path = os.path.join(HERE, "bf16_floor.json")
    data = json.load(open(path)) if os.path.exists(path) else {}
    data["points"] = list(OPERAND_POINTS)
    allc = cases()
    for name in names or list(allc):
        shape, B, s, scale = allc[name]
        data[name] = floor_for(shape, B, s, scale)
        print(name, max(data[name].values()), flush=True)
        with open(path, "w") as f:
            json.dump(data, f, indent=1, sort_keys=True)
        gc.collect()


if __name__ == "__main__":
    main(sys.argv[1:])
