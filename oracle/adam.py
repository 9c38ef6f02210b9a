"""Host Adam on the FP32 master, restated from its definition.

The articles place the optimizer step on the CPU over host-resident FP32
master, m and v (zhichai.net article, "以内存为中心的训练新范式" point 1;
lqnn.cn article, section 二, ParameterState and CPU Adam). The update is the
standard Adam with bias correction and no weight decay:

    m <- b1 m + (1 - b1) g ;  v <- b2 v + (1 - b2) g^2
    m_hat = m / (1 - b1^t) ;  v_hat = v / (1 - b2^t)
    w <- w - lr * m_hat / (sqrt(v_hat) + eps)
"""
from __future__ import annotations

import numpy as np


def adam_update(w, m, v, g, t, lr, beta1, beta2, eps, dtype=np.float64):
    """Returns (w, m, v) after step ``t`` (t >= 1), computed in ``dtype``."""
    if t < 1:
        raise ValueError("Adam step count starts at 1")
    w = np.asarray(w, dtype=dtype)
    m = np.asarray(m, dtype=dtype)
    v = np.asarray(v, dtype=dtype)
    g = np.asarray(g, dtype=dtype)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    w = w - lr * m_hat / (np.sqrt(v_hat) + eps)
    return w, m, v
