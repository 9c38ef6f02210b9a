"""Readings taken where the articles are silent, garbled or disagree.

This module holds no code; it records each reading the oracle (and, written
independently, the CUDA library) follows, with the passage it answers.

R1  Flat order and alignment (lqnn.cn article, 三.1 "layer_pinned_flats";
    zhichai.net article, "性能与能力", flat tensor layout). Order
    [embed][layer 0..L-1][final_norm, head]; within a layer attn_norm, Wqkv
    (q, k, v rows), Wo, mlp_norm, Wgu (gate rows, then up rows), Wdown;
    matrices row-major [out, in]; every tensor offset a multiple of 64
    elements; untied head; no biases.
R2  RMSNorm epsilon 1e-5 (articles silent; Llama-family default).
R3  RoPE: rotate-half pairs (i, i + hd/2), base 10000, positions restart at
    0 in every sequence (articles silent; HF models are implied by the
    lqnn.cn article's section 四, AutoModelForCausalLM introspection).
R4  Attention: scale 1/sqrt(hd), causal (key j visible to query i iff
    j <= i), no dropout.
R5  Grouped KV: query head h reads KV head h // (H / Hkv).
R6  Loss: mean cross entropy over all B*s tokens; every label in [0, V).
R7  Labels are caller supplied; the synthetic recipe draws s + 1 ids per row
    and shifts by one.
R8  Init: normal(0, 0.02) for embedding, every linear weight and the head;
    norm weights 1.0; m = v = grad = 0.
R9  Adam: beta1 0.9, beta2 0.999, eps 1e-8 added outside the square root,
    bias correction, t starts at 1, no weight decay, lr 1e-3 (lqnn.cn article
    section 二: FP32 master, grad, m, v per parameter).
R10 Rounding to bf16 is round-to-nearest-even; the device computes on bf16
    copies of the FP32 master, the oracle on the FP32 master itself.
R11 Gradient slabs hold bf16 gradients that the host adds into FP32 master
    gradients (lqnn.cn article 三.3: "flat gradient slab" + FP32 master grad).
R12 Segments are [jC, (j+1)C); the input of the first layer of each segment is
    checkpointed; the last segment is recomputed too (zhichai.net article,
    point 3 "every K layers"; lqnn.cn article 三.4, checkpoint_interval: 4).
R13 Three streams (compute, host-to-device, device-to-host) as the lqnn.cn
    article 三.2 names; its table of their roles was lost in extraction; the
    travelaiplan blog, 核心功能 point 2, describes a two-stream variant.
"""
