"""Python binding of libmt.so: the streamed-layer training step and its kernels.

Argument marshalling only: every step of the path runs in the library's
CUDA kernels and host C++. If libmt.so is missing the import of ``lib()``
raises; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmt.so")

MT_OK = 0
ERRORS = {
    -1: "MT_EINVAL", -2: "MT_ENOMEM", -3: "MT_ECUDA", -4: "MT_ETIMEOUT",
    -5: "MT_EWORKER", -6: "MT_ENONFINITE", -7: "MT_ESTATE", -8: "MT_EDEVICE",
}
_NAMES = {v: k for k, v in ERRORS.items()}
globals().update(_NAMES)


class MtError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class Config(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
        ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
        ("vocab", C.c_int32), ("max_batch", C.c_int32), ("max_seq", C.c_int32),
        ("ckpt_interval", C.c_int32), ("n_slabs", C.c_int32), ("streamed", C.c_int32),
        ("rms_eps", C.c_float), ("rope_theta", C.c_float), ("lr", C.c_float),
        ("beta1", C.c_float), ("beta2", C.c_float), ("adam_eps", C.c_float),
        ("device", C.c_int32), ("host_threads", C.c_int32), ("overlap_adam", C.c_int32),
        ("unfused_epilogues", C.c_int32), ("keep_attention", C.c_int32), ("head_chunk_rows", C.c_int32),
    ]


class TimelineRec(C.Structure):
    _fields_ = [("cls", C.c_int32), ("stream", C.c_int32), ("start_ms", C.c_double), ("end_ms", C.c_double)]


class TensorDesc(C.Structure):
    _fields_ = [("unit", C.c_int32), ("kind", C.c_int32), ("offset", C.c_int64),
                ("rows", C.c_int64), ("cols", C.c_int64), ("name", C.c_char * 24)]


class Stats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("h2d_bytes", C.c_int64), ("d2h_bytes", C.c_int64),
                ("h2d_units", C.c_int64), ("host_adam_s", C.c_double), ("host_wait_s", C.c_double),
                ("last_step_s", C.c_double), ("device_bytes", C.c_int64), ("pinned_bytes", C.c_int64),
                ("kernel_launches", C.c_int64), ("host_compute_s", C.c_double), ("host_copy_wait_s", C.c_double)]


PROF_CLASSES = ["gemm", "attn_fwd", "attn_bwd", "norm", "rope", "swiglu", "reserved", "ce", "embed", "other",
                "h2d", "d2h"]


class KernelProfile(C.Structure):
    _fields_ = [("launches", C.c_int64 * len(PROF_CLASSES)), ("ms", C.c_double * len(PROF_CLASSES)),
                ("flops", C.c_double * len(PROF_CLASSES)), ("bytes", C.c_double * len(PROF_CLASSES))]


EXPORTS = [
    "mt_layout", "mt_unit_range", "mt_plan", "mt_init", "mt_train_step", "mt_train_step_device", "mt_train_step_accum",
    "mt_read_grads", "mt_sync", "mt_get_step", "mt_set_step", "mt_sync_store", "mt_get_stats",
    "mt_get_stream", "mt_profile_enable", "mt_profile_read", "mt_profile_timeline", "mt_destroy", "mt_last_error", "mt_debug_inject", "mt_debug_inject_global",
    "mt_host_adam", "mt_host_adam_slab", "mt_host_to_bf16",
    "mt_k_gemm", "mt_k_gemm_ex", "mt_k_gemm_rope", "mt_k_gemm_swiglu_fwd", "mt_k_gemm_swiglu_bwd", "mt_k_gemm_wgrad", "mt_k_gemm_splitk", "mt_k_gemm_tile_policy", "mt_k_gemm_wgrad_ws", "mt_k_rmsnorm_fwd", "mt_k_rmsnorm_bwd", "mt_k_rmsnorm_bwd_parts",
    "mt_k_rope", "mt_k_swiglu_fwd", "mt_k_swiglu_bwd", "mt_k_attn_fwd", "mt_k_attn_fwd_mma", "mt_k_attn_bwd", "mt_k_attn_bwd_rope", "mt_k_attn_bwd_mma",
    "mt_k_cross_entropy", "mt_k_sum", "mt_k_embedding_fwd", "mt_k_embedding_bwd",
    "mt_k_embedding_bwd_work", "mt_k_check_ids", "mt_k_device_error",
]

_lib = None
P = C.c_void_p
I = C.c_int
I64 = C.c_int64
F = C.c_float


def lib():
    """The loaded libmt.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m host_memory_resident_gb300.build`")
    L = C.CDLL(LIB_PATH)
    sig = {
        "mt_layout": ([C.POINTER(Config), C.POINTER(TensorDesc), I, C.POINTER(I), C.POINTER(I64)], I),
        "mt_unit_range": ([C.POINTER(Config), I, C.POINTER(I64), C.POINTER(I64)], I),
        "mt_plan": ([C.POINTER(Config), C.POINTER(I64), C.POINTER(I64), C.POINTER(I64)], I),
        "mt_init": ([C.POINTER(Config), P, P, P, P, I64, C.POINTER(P)], I),
        "mt_train_step": ([P, P, P, C.c_int32, C.c_int32, C.POINTER(F)], I),
        "mt_train_step_device": ([P, P, P, C.c_int32, C.c_int32, C.POINTER(F)], I),
        "mt_train_step_accum": ([P, P, P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.POINTER(F)], I),
        "mt_read_grads": ([P, P, I64], I),
        "mt_sync": ([P], I),
        "mt_get_step": ([P, C.POINTER(I64)], I),
        "mt_set_step": ([P, I64], I),
        "mt_sync_store": ([P], I),
        "mt_get_stats": ([P, C.POINTER(Stats)], I),
        "mt_get_stream": ([P, I, C.POINTER(P)], I),
        "mt_profile_enable": ([P, I], I),
        "mt_profile_read": ([P, C.POINTER(KernelProfile), I], I),
        "mt_profile_timeline": ([P, C.POINTER(TimelineRec), I, C.POINTER(I)], I),
        "mt_destroy": ([P], I),
        "mt_last_error": ([P], C.c_char_p),
        "mt_debug_inject": ([P, I, I64], I),
        "mt_debug_inject_global": ([I, I64], I),
        "mt_host_adam": ([P, P, P, P, P, I64, I64, F, F, F, F, I], I),
        "mt_host_adam_slab": ([P, P, P, P, P, P, I64, I64, F, F, F, F, I], I),
        "mt_host_to_bf16": ([P, P, I64], I),
        "mt_k_gemm": ([P, I64, P, I64, P, I64, I, P, I64, I, I, I, P], I),
        "mt_k_gemm_ex": ([P, I64, I, P, I64, I, P, I64, I, P, I64, I, I, I, P], I),
        "mt_k_gemm_rope": ([P, I64, P, I64, P, I64, I, I, I, P, P, I, I, I, P], I),
        "mt_k_gemm_swiglu_fwd": ([P, I64, P, I64, P, I64, P, I64, I, I, I, P], I),
        "mt_k_gemm_swiglu_bwd": ([P, I64, P, I64, P, I64, P, I64, I, I, I, P], I),
        "mt_k_gemm_wgrad": ([P, I64, P, I64, P, I64, I, I, I, P, I64, P], I),
        "mt_k_gemm_splitk": ([I, I, I], I),
        "mt_k_gemm_tile_policy": ([I], I),
        "mt_k_gemm_wgrad_ws": ([I, I], I64),
        "mt_k_rmsnorm_fwd": ([P, I, P, P, P, I, I, F, P], I),
        "mt_k_rmsnorm_bwd": ([P, P, I, P, P, P, P, P, P, P, I, I, P], I),
        "mt_k_rmsnorm_bwd_parts": ([I], I),
        "mt_k_rope": ([P, I64, I, I, I, I, P, P, I, P], I),
        "mt_k_swiglu_fwd": ([P, P, I, I, P], I),
        "mt_k_swiglu_bwd": ([P, P, P, I, I, P], I),
        "mt_k_attn_fwd": ([P, I64, P, I64, P, I, I, I, I, I, P], I),
        "mt_k_attn_fwd_mma": ([P, I64, P, I64, P, I, I, I, I, I, P], I),
        "mt_k_attn_bwd": ([P, I64, P, I64, P, I64, P, P, P, I64, I, I, I, I, I, P], I),
        "mt_k_attn_bwd_rope": ([P, I64, P, I64, P, I64, P, P, P, I64, I, I, I, I, I, P, P, P], I),
        "mt_k_attn_bwd_mma": ([P, I64, P, I64, P, I64, P, P, P, I64, I, I, I, I, I, P], I),
        "mt_k_cross_entropy": ([P, I64, P, P, I64, P, I, I, F, P], I),
        "mt_k_sum": ([P, I, P, P], I),
        "mt_k_embedding_fwd": ([P, P, P, I, I, I, I, P], I),
        "mt_k_embedding_bwd": ([P, P, P, I, I, I, P, P], I),
        "mt_k_embedding_bwd_work": ([I, I], I64),
        "mt_k_check_ids": ([P, I, I, P, P], I),
        "mt_k_device_error": ([C.POINTER(I), I], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def check(code, handle=None):
    if code != MT_OK:
        msg = lib().mt_last_error(handle)
        raise MtError(code, msg.decode() if msg else "")
    return code


def make_config(shape, batch=None, seq=None, streamed=True, device=0, host_threads=0, ckpt_interval=None,
                n_slabs=None, overlap_adam=False, unfused_epilogues=False, keep_attention=False,
                head_chunk_rows=0) -> Config:
    """mt_config from a synth.ModelShape-like object."""
    c = Config()
    c.n_layers = shape.n_layers
    c.d_model = shape.d_model
    c.n_heads = shape.n_heads
    c.n_kv_heads = shape.n_kv_heads
    c.head_dim = shape.head_dim
    c.ffn_dim = shape.ffn_dim
    c.vocab = shape.vocab
    c.max_batch = batch or shape.batch
    c.max_seq = seq or shape.seq
    c.ckpt_interval = ckpt_interval or shape.ckpt_interval
    c.n_slabs = n_slabs or shape.n_slabs
    c.streamed = 1 if streamed else 0
    c.rms_eps = shape.rms_eps
    c.rope_theta = shape.rope_theta
    c.lr = shape.lr
    c.beta1 = shape.beta1
    c.beta2 = shape.beta2
    c.adam_eps = shape.adam_eps
    c.device = device
    c.host_threads = host_threads
    c.overlap_adam = 1 if overlap_adam else 0
    c.unfused_epilogues = 1 if unfused_epilogues else 0
    c.keep_attention = 1 if keep_attention else 0
    c.head_chunk_rows = int(head_chunk_rows)
    return c


def layout(cfg: Config):
    """List of dicts (unit, kind, offset, rows, cols, name) and n_total."""
    L = lib()
    n = C.c_int()
    total = C.c_int64()
    check(L.mt_layout(C.byref(cfg), None, 0, C.byref(n), C.byref(total)))
    arr = (TensorDesc * n.value)()
    check(L.mt_layout(C.byref(cfg), arr, n.value, C.byref(n), C.byref(total)))
    out = [dict(unit=t.unit, kind=t.kind, offset=t.offset, rows=t.rows, cols=t.cols, name=t.name.decode())
           for t in arr]
    return out, total.value


def unit_range(cfg: Config, unit: int):
    off, ln = C.c_int64(), C.c_int64()
    check(lib().mt_unit_range(C.byref(cfg), unit, C.byref(off), C.byref(ln)))
    return off.value, ln.value


def plan(cfg: Config) -> dict:
    """Exact memory plan of a handle for `cfg` (no GPU, nothing allocated)."""
    dev, pin, state = C.c_int64(), C.c_int64(), C.c_int64()
    check(lib().mt_plan(C.byref(cfg), C.byref(dev), C.byref(pin), C.byref(state)))
    return {"device_bytes": dev.value, "pinned_bytes": pin.value, "host_state_bytes": state.value}


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


class Trainer:
    """Owns an mt_handle over caller numpy FP32 arrays (master, m, v, grad).

    keep_grads=False passes no gradient array: gradients go straight from the
    staging slabs into Adam (read_grads and accumulation are then refused)."""

    def __init__(self, cfg: Config, master: np.ndarray, m=None, v=None, grad=None, keep_grads: bool = True):
        _, n_total = layout(cfg)
        for a in (master, m, v, grad):
            if a is not None and (a.dtype != np.float32 or a.shape != (n_total,) or not a.flags.c_contiguous):
                raise ValueError("host state arrays must be contiguous float32 of n_total elements")
        self.cfg = cfg
        self.n_total = n_total
        self.master = master
        self.m = m if m is not None else np.zeros(n_total, np.float32)
        self.v = v if v is not None else np.zeros(n_total, np.float32)
        if not keep_grads and grad is not None:
            raise ValueError("keep_grads=False takes no gradient array")
        self.grad = None if not keep_grads else (grad if grad is not None else np.zeros(n_total, np.float32))
        h = C.c_void_p()
        check(lib().mt_init(C.byref(cfg), _ptr(self.master), _ptr(self.m), _ptr(self.v),
                            _ptr(self.grad) if self.grad is not None else None,
                            n_total, C.byref(h)))
        self.h = h

    def step(self, tokens: np.ndarray, labels: np.ndarray) -> float:
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        labels = np.ascontiguousarray(labels, dtype=np.int32)
        B, s = tokens.shape
        loss = C.c_float()
        check(lib().mt_train_step(self.h, _ptr(tokens), _ptr(labels), B, s, C.byref(loss)), self.h)
        return loss.value

    def step_accum(self, tokens, labels, micro_index: int, n_micro: int) -> float:
        """One micro-step of gradient accumulation (Adam after the last)."""
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        labels = np.ascontiguousarray(labels, dtype=np.int32)
        B, s = tokens.shape
        loss = C.c_float()
        check(lib().mt_train_step_accum(self.h, _ptr(tokens), _ptr(labels), B, s, micro_index, n_micro,
                                        C.byref(loss)), self.h)
        return loss.value

    def step_device(self, tok_ptr: int, lab_ptr: int, B: int, s: int) -> float:
        loss = C.c_float()
        check(lib().mt_train_step_device(self.h, C.c_void_p(tok_ptr), C.c_void_p(lab_ptr), B, s, C.byref(loss)),
              self.h)
        return loss.value

    def step_code(self, tokens, labels):
        """Like step() but returns (code, loss) instead of raising."""
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        labels = np.ascontiguousarray(labels, dtype=np.int32)
        B, s = tokens.shape
        loss = C.c_float()
        code = lib().mt_train_step(self.h, _ptr(tokens), _ptr(labels), B, s, C.byref(loss))
        return code, loss.value

    def read_grads(self) -> np.ndarray:
        out = np.empty(self.n_total, np.float32)
        check(lib().mt_read_grads(self.h, _ptr(out), self.n_total), self.h)
        return out

    def sync(self):
        """Wait for the host worker (needed with overlap_adam before reading master/m/v)."""
        check(lib().mt_sync(self.h), self.h)

    def stats(self) -> dict:
        s = Stats()
        check(lib().mt_get_stats(self.h, C.byref(s)), self.h)
        return {k: getattr(s, k) for k, _ in Stats._fields_}

    def profile(self, on: bool = True):
        check(lib().mt_profile_enable(self.h, 1 if on else 0))

    def read_profile(self, reset: bool = False) -> dict:
        p = KernelProfile()
        check(lib().mt_profile_read(self.h, C.byref(p), 1 if reset else 0))
        return {name: dict(launches=p.launches[i], ms=p.ms[i], flops=p.flops[i], bytes=p.bytes[i])
                for i, name in enumerate(PROF_CLASSES)}

    def timeline(self) -> list:
        """Launches and copies of the last profiled step: dicts with the class
        name, stream (compute / h2d / d2h) and start / end in ms."""
        n = C.c_int()
        check(lib().mt_profile_timeline(self.h, None, 0, C.byref(n)), self.h)
        buf = (TimelineRec * max(n.value, 1))()
        check(lib().mt_profile_timeline(self.h, buf, n.value, C.byref(n)), self.h)
        names = ("compute", "h2d", "d2h", "host_adam", "host_wait", "host_adam_prev", "host_wait_prev")
        return [dict(cls=PROF_CLASSES[r.cls] if r.stream < 3 else f"unit {r.cls}", stream=names[r.stream],
                     start_ms=r.start_ms, end_ms=r.end_ms) for r in buf[:n.value]]

    def get_step(self) -> int:
        t = C.c_int64()
        check(lib().mt_get_step(self.h, C.byref(t)))
        return t.value

    def stream(self, which: int = 0) -> int:
        p = C.c_void_p()
        check(lib().mt_get_stream(self.h, which, C.byref(p)))
        return p.value or 0

    def inject(self, what: int, value: int):
        check(lib().mt_debug_inject(self.h, what, value))

    def last_error(self) -> str:
        m = lib().mt_last_error(self.h)
        return m.decode() if m else ""

    def close(self):
        if getattr(self, "h", None):
            lib().mt_destroy(self.h)
            self.h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def host_adam(w, m, v, g, t, lr, beta1, beta2, eps, store=None, threads=0):
    """The library's host Adam on numpy float32 arrays (in place)."""
    n = w.shape[0]
    sp = _ptr(store) if store is not None else None
    check(lib().mt_host_adam(_ptr(w), _ptr(m), _ptr(v), _ptr(g), sp, n, t, lr, beta1, beta2, eps, threads))


def host_adam_slab(w, m, v, slab, t, lr, beta1, beta2, eps, grad_out=None, store=None, threads=0):
    """The worker's pass: bf16 slab -> FP32 grad_out, Adam, bf16 store (numpy arrays)."""
    n = w.shape[0]
    check(lib().mt_host_adam_slab(_ptr(w), _ptr(m), _ptr(v), _ptr(slab),
                                  _ptr(grad_out) if grad_out is not None else None,
                                  _ptr(store) if store is not None else None, n, t, lr, beta1, beta2, eps, threads))


def host_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    check(lib().mt_host_to_bf16(_ptr(x), _ptr(out), x.size))
    return out


# ---------------------------------------------------------------- kernels
def _dp(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _st(stream):
    if stream is None:
        return None
    return C.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)


def k_gemm(A, B, Cout, R=None, stream=None):
    """Cout = A @ B.T (+ R). A [M,K], B [N,K] bf16; Cout bf16 or fp32 [M,N];
    R (optional) of Cout's dtype."""
    import torch
    M, K = A.shape
    N = B.shape[0]
    f32 = 1 if Cout.dtype == torch.float32 else 0
    check(lib().mt_k_gemm(_dp(A), A.stride(0), _dp(B), B.stride(0), _dp(Cout), Cout.stride(0), f32, _dp(R),
                          R.stride(0) if R is not None else 0, M, N, K, _st(stream)))


def k_gemm_ex(A, a_mn, B, b_mn, Cout, R=None, stream=None):
    """Cout = op(A) op(B)^T (+ R): A is [M,K] (a_mn False) or stored [K,M] (a_mn True);
    B is [N,K] (b_mn False) or stored [K,N] (b_mn True)."""
    import torch
    M, N = Cout.shape
    K = A.shape[0] if a_mn else A.shape[1]
    f32 = 1 if Cout.dtype == torch.float32 else 0
    check(lib().mt_k_gemm_ex(_dp(A), A.stride(0), 1 if a_mn else 0, _dp(B), B.stride(0), 1 if b_mn else 0, _dp(Cout),
                             Cout.stride(0), f32, _dp(R), R.stride(0) if R is not None else 0, M, N, K, _st(stream)))


def _is_f32(t):
    import torch
    return 1 if t.dtype == torch.float32 else 0


def k_rmsnorm_fwd(x, w, y, rstd, eps, stream=None):
    """x bf16 or fp32 [M, d]; y bf16."""
    M, d = x.shape
    check(lib().mt_k_rmsnorm_fwd(_dp(x), _is_f32(x), _dp(w), _dp(y), _dp(rstd), M, d, eps, _st(stream)))


def k_rmsnorm_bwd_parts(M):
    return lib().mt_k_rmsnorm_bwd_parts(M)


def k_rmsnorm_bwd(dy, x, w, rstd, dres, dx32, dxb, partial, dw, stream=None):
    M, d = x.shape
    check(lib().mt_k_rmsnorm_bwd(_dp(dy), _dp(x), _is_f32(x), _dp(w), _dp(rstd), _dp(dres), _dp(dx32), _dp(dxb),
                                 _dp(partial), _dp(dw), M, d, _st(stream)))


def k_gemm_rope(A, B, Cout, cos_t, sin_t, rot_cols, hd, seq, stream=None):
    """Cout = A B^T with RoPE on columns [0, rot_cols) (position = row mod seq)."""
    M, N = Cout.shape
    check(lib().mt_k_gemm_rope(_dp(A), A.stride(0), _dp(B), B.stride(0), _dp(Cout), Cout.stride(0), M, N, A.shape[1],
                               _dp(cos_t), _dp(sin_t), rot_cols, hd, seq, _st(stream)))


def k_gemm_swiglu_fwd(A, W, gu, a, stream=None):
    """gu = A W^T (W = [gate rows; up rows]) and a = silu(gate) * up."""
    M, f = a.shape
    check(lib().mt_k_gemm_swiglu_fwd(_dp(A), A.stride(0), _dp(W), W.stride(0), _dp(gu), gu.stride(0), _dp(a),
                                     a.stride(0), M, f, A.shape[1], _st(stream)))


def k_gemm_swiglu_bwd(dy, W, gu, dgu, stream=None):
    """dgu = SwiGLU backward of da = dy W (W [K, f] read in place) at gate | up = gu."""
    M, f = dy.shape[0], W.shape[1]
    check(lib().mt_k_gemm_swiglu_bwd(_dp(dy), dy.stride(0), _dp(W), W.stride(0), _dp(gu), gu.stride(0), _dp(dgu),
                                     dgu.stride(0), M, f, dy.shape[1], _st(stream)))


def k_gemm_wgrad(dY, X, G, ws=None, stream=None):
    """G = dY^T X (dY [K, M], X [K, N], G bf16 [M, N]), split along K into the
    fp32 workspace ws when the output has few tiles."""
    K, M = dY.shape
    N = X.shape[1]
    check(lib().mt_k_gemm_wgrad(_dp(dY), dY.stride(0), _dp(X), X.stride(0), _dp(G), G.stride(0), M, N, K, _dp(ws),
                                ws.numel() if ws is not None else 0, _st(stream)))


def k_gemm_tile_policy(policy):
    """0: library's tile choice; 1: 128 x 256 tiles; 2: 256 x 256 (plain products)."""
    check(lib().mt_k_gemm_tile_policy(policy))


def k_gemm_splitk(M, N, K):
    return lib().mt_k_gemm_splitk(M, N, K)


def k_gemm_wgrad_ws(M, N):
    return lib().mt_k_gemm_wgrad_ws(M, N)


def k_rope(x, B, s, n_rot_heads, hd, cos_t, sin_t, inverse=False, stream=None):
    check(lib().mt_k_rope(_dp(x), x.stride(0), B, s, n_rot_heads, hd, _dp(cos_t), _dp(sin_t), 1 if inverse else 0,
                          _st(stream)))


def k_swiglu_fwd(gu, a, stream=None):
    M, f = a.shape
    check(lib().mt_k_swiglu_fwd(_dp(gu), _dp(a), M, f, _st(stream)))


def k_swiglu_bwd(da, gu, dgu, stream=None):
    M, f = da.shape
    check(lib().mt_k_swiglu_bwd(_dp(da), _dp(gu), _dp(dgu), M, f, _st(stream)))


def k_attn_fwd(qkv, o, lse, B, s, H, Hkv, hd, stream=None):
    check(lib().mt_k_attn_fwd(_dp(qkv), qkv.stride(0), _dp(o), o.stride(0), _dp(lse), B, s, H, Hkv, hd,
                              _st(stream)))


def k_attn_fwd_mma(qkv, o, lse, B, s, H, Hkv, hd, stream=None):
    check(lib().mt_k_attn_fwd_mma(_dp(qkv), qkv.stride(0), _dp(o), o.stride(0), _dp(lse), B, s, H, Hkv, hd,
                                  _st(stream)))


def k_attn_bwd(qkv, o, dout, lse, delta, dqkv, B, s, H, Hkv, hd, stream=None):
    check(lib().mt_k_attn_bwd(_dp(qkv), qkv.stride(0), _dp(o), o.stride(0), _dp(dout), dout.stride(0), _dp(lse),
                              _dp(delta), _dp(dqkv), dqkv.stride(0), B, s, H, Hkv, hd, _st(stream)))


def k_attn_bwd_rope(qkv, o, dout, lse, delta, dqkv, B, s, H, Hkv, hd, cos_t, sin_t, stream=None):
    """Attention backward with dq, dk rotated back by RoPE's inverse."""
    check(lib().mt_k_attn_bwd_rope(_dp(qkv), qkv.stride(0), _dp(o), o.stride(0), _dp(dout), dout.stride(0),
                                   _dp(lse), _dp(delta), _dp(dqkv), dqkv.stride(0), B, s, H, Hkv, hd, _dp(cos_t),
                                   _dp(sin_t), _st(stream)))


def k_attn_bwd_mma(qkv, o, dout, lse, delta, dqkv, B, s, H, Hkv, hd, stream=None):
    check(lib().mt_k_attn_bwd_mma(_dp(qkv), qkv.stride(0), _dp(o), o.stride(0), _dp(dout), dout.stride(0),
                                  _dp(lse), _dp(delta), _dp(dqkv), dqkv.stride(0), B, s, H, Hkv, hd, _st(stream)))


def k_cross_entropy(logits, labels, dz, loss_rows, scale, stream=None):
    M, V = logits.shape
    check(lib().mt_k_cross_entropy(_dp(logits), logits.stride(0), _dp(labels), _dp(dz), dz.stride(0),
                                   _dp(loss_rows), M, V, scale, _st(stream)))


def k_sum(x, out, stream=None):
    check(lib().mt_k_sum(_dp(x), x.numel(), _dp(out), _st(stream)))


def k_embedding_fwd(E, tok, x, stream=None):
    """x bf16 or fp32 [M, d]."""
    V, d = E.shape
    check(lib().mt_k_embedding_fwd(_dp(E), _dp(tok), _dp(x), _is_f32(x), tok.numel(), d, V, _st(stream)))


def k_embedding_bwd_work(M, V):
    return lib().mt_k_embedding_bwd_work(M, V)


def k_embedding_bwd(dx, tok, dE, work, stream=None):
    V, d = dE.shape
    check(lib().mt_k_embedding_bwd(_dp(dx), _dp(tok), _dp(dE), tok.numel(), d, V, _dp(work), _st(stream)))


def device_error(reset=True) -> int:
    c = C.c_int()
    check(lib().mt_k_device_error(C.byref(c), 1 if reset else 0))
    return c.value
