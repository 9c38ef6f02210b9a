"""Oracle: a plain, slow CPU restatement of one streamed-layer training step.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
package; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it. It shares no code with the CUDA library: the flat
layout, every operator and its hand-written backward, and Adam are restated
here from their definitions in numpy (float64 by default, float32 on request).

What it computes follows the RAM-centric training articles:

* "MegaTrain：单卡训百亿大模型的突破与实践" (zhichai.net), section
  "以内存为中心的训练新范式", points 1-4: parameters, gradients and Adam state
  live in host memory; layers are streamed in, run through a stateless layer
  template and released; activations are checkpointed every few layers and
  recomputed in backward.
* lqnn.cn MegaTrain article, section 二 (ParameterState: FP32 master, grad,
  m, v per parameter; the optimizer step updates the host master) and
  section 三 (double-buffered flat layer buffers, a K-slab gradient pool, a
  CPU worker adding slabs into FP32 master gradients, checkpoint_interval).

Streaming, recompute and host placement change where numbers live, not what
they are, so the step's result is the plain training step of a Llama-style
decoder followed by one Adam update. The oracle is that definition written
out, with two structural knobs kept so their invariance can be tested:
``ckpt_interval`` (segment recompute) and ``streamed`` (weights copied into a
two-slot scratch before use). Readings of points the articles leave open
(flat order, RoPE convention, loss normalisation, init, Adam constants) are
stated in the docstring of the function that takes them (``layout``,
``ops``, ``adam``).

Pins (tests marked ``not gpu``): central finite differences of the whole
step, comparison with torch autograd built from torch library ops, closed
forms for CE / RMSNorm / RoPE / attention special cases, torch.optim.Adam on
hand-set tensors, and the published parameter counts of the 1.1B and 7B
Llama-family shapes for the layout.
"""
from .layout import Tensor, Unit, Layout, build_layout, ALIGN  # noqa: F401
from .ops import (  # noqa: F401
    rmsnorm_fwd, rmsnorm_bwd, rope_tables, rope_fwd, rope_bwd,
    attention_fwd, attention_bwd, swiglu_fwd, swiglu_bwd,
    cross_entropy_fwd_bwd, embedding_fwd, embedding_bwd, linear_fwd,
    linear_bwd,
)
from .model import step_grads, layer_forward, layer_backward  # noqa: F401
from .adam import adam_update  # noqa: F401
