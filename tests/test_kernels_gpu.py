"""Per-kernel parity of libmt.so's sm_103a kernels against the oracle.

Every kernel is called through the C ABI on seeded inputs and compared
element by element with the oracle's function evaluated in float64 on the
same (bf16-rounded) inputs. Sizes span several tiles with ragged tails and
include one full-width layer shape of each large workload.

Tolerances follow from the arithmetic: inputs and outputs are bf16 (relative
rounding 2^-9), accumulation is fp32. A bf16 output is within ~2^-8 of the
exact value relative to the row/column scale, so element checks use
|err| <= 2e-2 * scale and relative L2 error <= 1e-2 (5e-3 for a single
rounding); integer / byte work (the gather) is bit-exact.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import host_memory_resident_gb300 as mt  # noqa: E402
from oracle import ops  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda"


def bf(a):
    """numpy -> (device bf16 tensor, float64 numpy of its exact values)."""
    t = torch.from_numpy(np.asarray(a, dtype=np.float32)).to(DEV).to(torch.bfloat16)
    return t, t.float().cpu().numpy().astype(np.float64)


def f32(a):
    t = torch.from_numpy(np.asarray(a, dtype=np.float32)).to(DEV)
    return t, t.cpu().numpy().astype(np.float64)


def host(t):
    return t.float().cpu().numpy().astype(np.float64)


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def assert_close(got, ref, l2=1e-2, elem=2e-2, what="", floor=0.0):
    """floor: a magnitude below which the reference counts as zero (for
    outputs that vanish exactly, e.g. dq with a single visible key)."""
    scale = max(np.abs(ref).max(), floor, 1e-30)
    e = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), floor * np.sqrt(ref.size), 1e-30))
    assert e <= l2, f"{what}: rel L2 {e:.3e}"
    m = np.abs(got - ref).max() / scale
    assert m <= elem, f"{what}: max err / scale {m:.3e}"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mt.lib()
    mt.device_error(reset=True)
    yield
    torch.cuda.synchronize()
    assert mt.device_error(reset=True) == 0


# --------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K,out,res", [
    (64, 192, 64, "bf16", False),      # tiny QKV
    (200, 296, 136, "bf16", True),     # ragged M, N, K
    (200, 300, 72, "f32", False),      # ragged N with fp32 output
    (130, 8, 8, "bf16", False),        # smallest N and K
    (2048, 2048, 512, "f32", True),
    (4096, 4096, 1024, "bf16", False),  # several tiles per CTA (TMEM ping-pong)
    (512, 12288, 4096, "bf16", False),  # 7B QKV, 512 tokens
    (384, 5120, 13824, "f32", False),   # 14B down projection K
])
def test_gemm(M, N, K, out, res):
    """The residual R has C's type: fp32 with fp32 output (the residual
    stream), bf16 with bf16 output."""
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A, Ah = bf(rng.standard_normal((M, K)))
    B, Bh = bf(rng.standard_normal((N, K)) / np.sqrt(K))
    R, Rh = ((f32 if out == "f32" else bf)(rng.standard_normal((M, N)))) if res else (None, 0.0)
    Cout = torch.empty((M, N), device=DEV, dtype=torch.float32 if out == "f32" else torch.bfloat16)
    mt.k_gemm(A, B, Cout, R)
    torch.cuda.synchronize()
    ref = ops.linear_fwd(Ah, Bh) + Rh
    assert_close(host(Cout), ref, l2=5e-3 if out == "bf16" else 1e-4, elem=1e-2 if out == "bf16" else 1e-3,
                 what=f"gemm {M}x{N}x{K}")


def test_gemm_strided_operands_and_rejects_misaligned():
    rng = np.random.default_rng(1)
    big, bigh = bf(rng.standard_normal((256, 200)))
    A = big[:, 8:136]            # row pitch 200, K = 128
    B, Bh = bf(rng.standard_normal((64, 128)))
    Cout = torch.empty((256, 64), device=DEV, dtype=torch.float32)
    mt.k_gemm(A, B, Cout)
    torch.cuda.synchronize()
    assert_close(host(Cout), bigh[:, 8:136] @ Bh.T, l2=1e-4, elem=1e-3, what="strided")
    bad = big[:, 1:129]          # not 16-byte aligned
    with pytest.raises(mt.MtError):
        mt.k_gemm(bad, B, Cout)


def test_gemm_deterministic():
    rng = np.random.default_rng(2)
    A, _ = bf(rng.standard_normal((1000, 777 // 8 * 8)))
    B, _ = bf(rng.standard_normal((600, 777 // 8 * 8)))
    c1 = torch.empty((1000, 600), device=DEV)
    c2 = torch.empty((1000, 600), device=DEV)
    mt.k_gemm(A, B, c1)
    mt.k_gemm(A, B, c2)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2)


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, False), (True, True)])
def test_gemm_wide_tiles_bitwise(a_mn, b_mn):
    """256 x 256 tiles give the same bits as 128 x 256 tiles (both sum K in
    the same order), for either operand layout, with a residual and with
    fp32 output, on ragged M, N and K; and match the fp64 product."""
    rng = np.random.default_rng(7 + 2 * a_mn + b_mn)
    M, N, K = 600, 520, 1000
    A, Ah = bf(rng.standard_normal((K, M) if a_mn else (M, K)))
    B, Bh = bf(rng.standard_normal((K, N) if b_mn else (N, K)) / np.sqrt(K))
    R, Rh = bf(rng.standard_normal((M, N)))
    outs = {}
    try:
        for pol in (1, 2):
            mt.k_gemm_tile_policy(pol)
            c16 = torch.full((M, N), float("nan"), device=DEV, dtype=torch.bfloat16)
            c32 = torch.full((M, N), float("nan"), device=DEV, dtype=torch.float32)
            mt.k_gemm_ex(A, a_mn, B, b_mn, c16, R)
            mt.k_gemm_ex(A, a_mn, B, b_mn, c32)
            torch.cuda.synchronize()
            outs[pol] = (c16, c32)
    finally:
        mt.k_gemm_tile_policy(0)
    assert torch.equal(outs[1][0], outs[2][0])
    assert torch.equal(outs[1][1], outs[2][1])
    a64 = Ah.T if a_mn else Ah
    b64 = Bh.T if b_mn else Bh
    ref = a64 @ b64.T
    assert_close(host(outs[2][1]), ref, l2=1e-4, elem=1e-3, what="wide tiles fp32")
    assert_close(host(outs[2][0]), ref + Rh, l2=5e-3, elem=1e-2, what="wide tiles bf16 + residual")


def test_gemm_tile_policy_rejects_bad_values():
    with pytest.raises(mt.MtError):
        mt.k_gemm_tile_policy(3)
    mt.k_gemm_tile_policy(0)


@pytest.mark.parametrize("M,N,K", [(384, 512, 8192), (296, 520, 5000), (2560, 2048, 16384)])
def test_gemm_wgrad_split_k(M, N, K):
    """Split-K weight gradient: near the fp64 product, deterministic, and the
    unsplit product (bit for bit) when the workspace is missing or short."""
    sp = mt.k_gemm_splitk(M, N, K)
    assert sp > 1
    rng = np.random.default_rng(M + N + K)
    dY, dYh = bf(rng.standard_normal((K, M)) / np.sqrt(K))
    X, Xh = bf(rng.standard_normal((K, N)))
    ws = torch.empty(mt.k_gemm_wgrad_ws(M, N), device=DEV, dtype=torch.float32)
    assert ws.numel() >= sp * M * N
    g1 = torch.full((M, N), float("nan"), device=DEV, dtype=torch.bfloat16)
    g2 = torch.full((M, N), float("nan"), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_wgrad(dY, X, g1, ws)
    ws.fill_(float("nan"))
    mt.k_gemm_wgrad(dY, X, g2, ws)
    plain = torch.empty((M, N), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_ex(dY, True, X, True, plain)
    g3 = torch.empty((M, N), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_wgrad(dY, X, g3, ws[: sp * M * N - 1])
    torch.cuda.synchronize()
    assert torch.equal(g1, g2)
    assert torch.equal(g3, plain)
    if M * N * K <= 8192 * 512 * 384:
        ref = dYh.T @ Xh
    else:   # rows sampled from the full product
        rows = np.arange(0, M, 37)
        ref, g1 = dYh[:, rows].T @ Xh, g1[torch.as_tensor(rows, device=DEV)]
    assert_close(host(g1), ref, l2=5e-3, elem=1e-2, what=f"wgrad {M}x{N}x{K} split {sp}")


# ------------------------------------------------------------------ RMSNorm
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
@pytest.mark.parametrize("M,d", [(64, 64), (333, 2048), (257, 5120)])
def test_rmsnorm_fwd_bwd(M, d, xdt):
    """x bf16, or fp32 (the residual stream, read without rounding)."""
    rng = np.random.default_rng(M + d)
    x, xh = (bf if xdt == "bf16" else f32)(rng.standard_normal((M, d)) * 3.0)
    w, wh = bf(1.0 + 0.1 * rng.standard_normal(d))
    y = torch.empty((M, d), device=DEV, dtype=torch.bfloat16)
    rstd = torch.empty(M, device=DEV)
    mt.k_rmsnorm_fwd(x, w, y, rstd, 1e-5)
    yr, rr = ops.rmsnorm_fwd(xh, wh, 1e-5)
    torch.cuda.synchronize()
    assert_close(host(y), yr, l2=5e-3, elem=1e-2, what="rmsnorm y")
    np.testing.assert_allclose(host(rstd), rr, rtol=1e-5)
    dy, dyh = f32(rng.standard_normal((M, d)))
    dres, dresh = f32(rng.standard_normal((M, d)))
    dx32 = torch.empty((M, d), device=DEV)
    dxb = torch.empty((M, d), device=DEV, dtype=torch.bfloat16)
    part = torch.empty((mt.k_rmsnorm_bwd_parts(M), d), device=DEV)
    dw = torch.empty(d, device=DEV, dtype=torch.bfloat16)
    mt.k_rmsnorm_bwd(dy, x, w, rstd, dres, dx32, dxb, part, dw)
    dxr, dwr = ops.rmsnorm_bwd(dyh, xh, wh, host(rstd))
    torch.cuda.synchronize()
    assert_close(host(dx32), dxr + dresh, l2=1e-5, elem=1e-4, what="rmsnorm dx")
    assert_close(host(dxb), dxr + dresh, l2=5e-3, elem=1e-2, what="rmsnorm dx bf16")
    assert_close(host(dw), dwr, l2=5e-3, elem=1e-2, what="rmsnorm dw")


# --------------------------------------------------------------------- RoPE
@pytest.mark.parametrize("B,s,H,Hkv,hd", [(2, 32, 4, 4, 16), (1, 300, 4, 2, 64), (2, 129, 2, 2, 128)])
def test_rope_fwd_inverse(B, s, H, Hkv, hd):
    rng = np.random.default_rng(s + hd)
    qn = (H + 2 * Hkv) * hd
    x, xh = bf(rng.standard_normal((B * s, qn)))
    cos, sin = ops.rope_tables(s, hd, 10000.0)
    ct, _ = f32(cos)
    st, _ = f32(sin)
    y = x.clone()
    mt.k_rope(y, B, s, H + Hkv, hd, ct, st)
    torch.cuda.synchronize()
    rot = (H + Hkv) * hd
    ref = xh.copy()
    ref[:, :rot] = ops.rope_fwd(xh[:, :rot].reshape(B, s, H + Hkv, hd), cos, sin).reshape(B * s, rot)
    assert_close(host(y), ref, l2=5e-3, elem=1e-2, what="rope")
    assert torch.equal(y[:, rot:], x[:, rot:])                 # v untouched
    z = y.clone()
    mt.k_rope(z, B, s, H + Hkv, hd, ct, st, inverse=True)
    torch.cuda.synchronize()
    back = ops.rope_bwd(host(y)[:, :rot].reshape(B, s, H + Hkv, hd), cos, sin).reshape(B * s, rot)
    assert_close(host(z)[:, :rot], back, l2=5e-3, elem=1e-2, what="rope inverse")


def test_rope_unaligned_pitch_matches_aligned():
    """A row pitch that is not a multiple of 8 elements takes the scalar
    kernel; it must give the bits of the 16-byte-vector kernel."""
    rng = np.random.default_rng(7)
    B, s, H, Hkv, hd = 2, 70, 4, 2, 64
    qn = (H + 2 * Hkv) * hd
    x, _ = bf(rng.standard_normal((B * s, qn)))
    cos, sin = ops.rope_tables(s, hd, 10000.0)
    ct, _ = f32(cos)
    st, _ = f32(sin)
    wide = torch.zeros((B * s, qn + 2), device=DEV, dtype=torch.bfloat16)
    wide[:, :qn] = x
    y = x.clone()
    mt.k_rope(y, B, s, H + Hkv, hd, ct, st)
    z = wide[:, :qn]
    mt.k_rope(z, B, s, H + Hkv, hd, ct, st)
    torch.cuda.synchronize()
    assert torch.equal(z, y)


# ------------------------------------------------------------------- SwiGLU
@pytest.mark.parametrize("M,f", [(64, 256), (199, 5632)])
def test_swiglu(M, f):
    rng = np.random.default_rng(M + f)
    gu, guh = bf(rng.standard_normal((M, 2 * f)) * 2)
    a = torch.empty((M, f), device=DEV, dtype=torch.bfloat16)
    mt.k_swiglu_fwd(gu, a)
    da, dah = bf(rng.standard_normal((M, f)))
    dgu = torch.empty((M, 2 * f), device=DEV, dtype=torch.bfloat16)
    mt.k_swiglu_bwd(da, gu, dgu)
    torch.cuda.synchronize()
    assert_close(host(a), ops.swiglu_fwd(guh[:, :f], guh[:, f:]), l2=5e-3, elem=1e-2, what="swiglu")
    dg, du = ops.swiglu_bwd(dah, guh[:, :f], guh[:, f:])
    assert_close(host(dgu), np.concatenate([dg, du], 1), l2=5e-3, elem=1e-2, what="swiglu bwd")


# ------------------------------------------------------- fused GEMM epilogues
# Each fused epilogue works on the fp32 accumulator and rounds to bf16 only
# what it stores: its output equals the element-wise function (float64, the
# oracle's) of the fp32 product, rounded once, to within one bf16 rounding,
# and it is closer to the exact result than the unfused sequence (GEMM to
# bf16, then the separate kernel), which rounds twice.
def within_one_rounding(got, ref, what):
    """|got - ref| <= 2^-8 |ref| elementwise (one bf16 rounding of a value
    within 1e-5 of ref), with an absolute floor of 1e-6 of the scale."""
    scale = max(np.abs(ref).max(), 1e-30)
    bad = np.abs(got - ref) > 2.0 ** -8 * np.abs(ref) + 1e-6 * scale
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond one rounding"


@pytest.mark.parametrize("Bt,seq,H,Hkv,hd,K", [(3, 100, 8, 2, 64, 192), (1, 257, 4, 2, 128, 128),
                                               (2, 260, 32, 4, 64, 2048)])
def test_gemm_rope_rounds_once(Bt, seq, H, Hkv, hd, K):
    rng = np.random.default_rng(seq + hd + K)
    M, N = Bt * seq, (H + 2 * Hkv) * hd
    A, Ah = bf(rng.standard_normal((M, K)))
    W, Wh = bf(rng.standard_normal((N, K)) / np.sqrt(K))
    cos, sin = ops.rope_tables(seq, hd, 10000.0)
    ct, _ = f32(cos)
    st, _ = f32(sin)
    y32 = torch.empty((M, N), device=DEV)
    mt.k_gemm(A, W, y32)
    twice = torch.empty((M, N), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm(A, W, twice)
    mt.k_rope(twice, Bt, seq, H + Hkv, hd, ct, st)
    got = torch.full((M, N), float("nan"), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_rope(A, W, got, ct, st, (H + Hkv) * hd, hd, seq)
    torch.cuda.synchronize()
    rot = (H + Hkv) * hd

    def rotate(y):
        y = y.copy()
        y[:, :rot] = ops.rope_fwd(y[:, :rot].reshape(Bt, seq, H + Hkv, hd), cos, sin).reshape(M, rot)
        return y
    within_one_rounding(host(got), rotate(host(y32)), "gemm+rope")
    exact = rotate(ops.linear_fwd(Ah, Wh))
    assert_close(host(got), exact, l2=5e-3, elem=2e-2, what="gemm+rope")
    assert rel_l2(host(got), exact) < rel_l2(host(twice), exact)


@pytest.mark.parametrize("M,f,K", [(64, 256, 64), (300, 5632, 2048), (130, 11008, 512)])
def test_gemm_swiglu_fwd_from_fp32(M, f, K):
    rng = np.random.default_rng(M + f + K)
    A, Ah = bf(rng.standard_normal((M, K)))
    W, Wh = bf(rng.standard_normal((2 * f, K)) * (2.0 / np.sqrt(K)))
    gu_ref = torch.empty((M, 2 * f), device=DEV, dtype=torch.bfloat16)
    y32 = torch.empty((M, 2 * f), device=DEV)
    mt.k_gemm(A, W, gu_ref)
    mt.k_gemm(A, W, y32)
    a_twice = torch.empty((M, f), device=DEV, dtype=torch.bfloat16)
    mt.k_swiglu_fwd(gu_ref, a_twice)
    gu = torch.full((M, 2 * f), float("nan"), device=DEV, dtype=torch.bfloat16)
    a = torch.full((M, f), float("nan"), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_swiglu_fwd(A, W, gu, a)
    torch.cuda.synchronize()
    assert torch.equal(gu, gu_ref)      # the stored gate | up: the product rounded once
    yh = host(y32)
    within_one_rounding(host(a), ops.swiglu_fwd(yh[:, :f], yh[:, f:]), "gemm+swiglu")
    y = ops.linear_fwd(Ah, Wh)
    exact = ops.swiglu_fwd(y[:, :f], y[:, f:])
    assert_close(host(a), exact, l2=1e-2, elem=2e-2, what="gemm+swiglu")
    assert rel_l2(host(a), exact) < rel_l2(host(a_twice), exact)


@pytest.mark.parametrize("M,f,K", [(64, 256, 64), (300, 5632, 2048), (130, 11008, 512)])
def test_gemm_swiglu_bwd_from_fp32(M, f, K):
    rng = np.random.default_rng(M + f + K + 1)
    dy, dyh = bf(rng.standard_normal((M, K)))
    Wd, Wdh = bf(rng.standard_normal((K, f)) / np.sqrt(K))  # the down weight [d, f]
    gu, guh = bf(rng.standard_normal((M, 2 * f)) * 2)
    da32 = torch.empty((M, f), device=DEV)
    mt.k_gemm_ex(dy, False, Wd, True, da32)
    da = torch.empty((M, f), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_ex(dy, False, Wd, True, da)
    dgu_twice = torch.empty((M, 2 * f), device=DEV, dtype=torch.bfloat16)
    mt.k_swiglu_bwd(da, gu, dgu_twice)
    dgu = torch.full((M, 2 * f), float("nan"), device=DEV, dtype=torch.bfloat16)
    mt.k_gemm_swiglu_bwd(dy, Wd, gu, dgu)
    torch.cuda.synchronize()
    dg, du = ops.swiglu_bwd(host(da32), guh[:, :f], guh[:, f:])
    within_one_rounding(host(dgu), np.concatenate([dg, du], 1), "gemm+swiglu bwd")
    dg, du = ops.swiglu_bwd(dyh @ Wdh, guh[:, :f], guh[:, f:])
    exact = np.concatenate([dg, du], 1)
    assert_close(host(dgu), exact, l2=1e-2, elem=2e-2, what="gemm+swiglu bwd")
    assert rel_l2(host(dgu), exact) < rel_l2(host(dgu_twice), exact)


# ---------------------------------------------------------------- attention
ATTN_CASES = [
    (2, 32, 4, 4, 16),     # tiny
    (1, 100, 4, 2, 16),    # ragged s, GQA
    (2, 130, 4, 1, 64),    # ragged, 4 query heads per KV head
    (1, 257, 2, 2, 128),   # ragged, hd 128
    (1, 1, 2, 1, 64),      # single token: output = v
    (1, 1024, 2, 2, 128),
    (1, 1, 2, 1, 128),     # single token at hd 128
    (2, 300, 8, 2, 128),   # GQA, several 128-query sub-tiles per key tile, ragged
    (1, 640, 5, 1, 128),   # 5 query heads per KV head (the 14B grouping), 5 tiles
]


def _attn_inputs(B, s, H, Hkv, hd, seed):
    rng = np.random.default_rng(seed)
    qn = (H + 2 * Hkv) * hd
    qkv, qkvh = bf(rng.standard_normal((B * s, qn)))
    q = qkvh[:, :H * hd].reshape(B, s, H, hd)
    k = qkvh[:, H * hd:(H + Hkv) * hd].reshape(B, s, Hkv, hd)
    v = qkvh[:, (H + Hkv) * hd:].reshape(B, s, Hkv, hd)
    return qkv, q, k, v


@pytest.mark.parametrize("B,s,H,Hkv,hd", ATTN_CASES)
def test_attention_fwd(B, s, H, Hkv, hd):
    qkv, q, k, v = _attn_inputs(B, s, H, Hkv, hd, s * hd)
    o = torch.empty((B * s, H * hd), device=DEV, dtype=torch.bfloat16)
    lse = torch.empty((B, H, s), device=DEV)
    mt.k_attn_fwd(qkv, o, lse, B, s, H, Hkv, hd)
    torch.cuda.synchronize()
    orf, lr = ops.attention_fwd(q, k, v)
    assert_close(host(o), orf.reshape(B * s, H * hd), l2=1e-2, elem=2e-2, what="attn o")
    np.testing.assert_allclose(host(lse), lr, rtol=0, atol=2e-2)


@pytest.mark.parametrize("B,s,H,Hkv,hd", ATTN_CASES)
def test_attention_bwd(B, s, H, Hkv, hd):
    qkv, q, k, v = _attn_inputs(B, s, H, Hkv, hd, s * hd + 1)
    o = torch.empty((B * s, H * hd), device=DEV, dtype=torch.bfloat16)
    lse = torch.empty((B, H, s), device=DEV)
    mt.k_attn_fwd(qkv, o, lse, B, s, H, Hkv, hd)
    rng = np.random.default_rng(s)
    do, doh = bf(rng.standard_normal((B * s, H * hd)))
    delta = torch.empty((B, H, s), device=DEV)
    dqkv = torch.zeros_like(qkv)
    mt.k_attn_bwd(qkv, o, do, lse, delta, dqkv, B, s, H, Hkv, hd)
    dqkv2 = torch.zeros_like(qkv)
    mt.k_attn_bwd(qkv, o, do, lse, delta, dqkv2, B, s, H, Hkv, hd)
    torch.cuda.synchronize()
    assert torch.equal(dqkv, dqkv2)                    # deterministic
    dq, dk, dv = ops.attention_bwd(q, k, v, doh.reshape(B, s, H, hd))
    g = host(dqkv)
    fl = 1e-3 * np.abs(dv).max()  # dq, dk vanish exactly when s = 1
    assert_close(g[:, :H * hd], dq.reshape(B * s, -1), l2=2e-2, elem=3e-2, what="dq", floor=fl)
    assert_close(g[:, H * hd:(H + Hkv) * hd], dk.reshape(B * s, -1), l2=2e-2, elem=3e-2, what="dk", floor=fl)
    assert_close(g[:, (H + Hkv) * hd:], dv.reshape(B * s, -1), l2=2e-2, elem=3e-2, what="dv")


@pytest.mark.parametrize("B,s,H,Hkv,hd", [(2, 32, 4, 4, 16), (2, 130, 4, 1, 64), (1, 257, 2, 2, 128),
                                          (2, 300, 8, 2, 128)])
def test_attention_bwd_with_rope_inverse(B, s, H, Hkv, hd):
    """dq and dk rotated back by RoPE's inverse in the backward's stores: the
    oracle's attention backward followed by its RoPE backward; at hd 64 / 128
    within one bf16 rounding of the rotation of the unfused kernel's fp32
    result (so rounded once), and closer to the exact values than the
    unfused sequence (backward to bf16, then the separate rotation)."""
    qkv, q, k, v = _attn_inputs(B, s, H, Hkv, hd, s * hd + 5)
    o = torch.empty((B * s, H * hd), device=DEV, dtype=torch.bfloat16)
    lse = torch.empty((B, H, s), device=DEV)
    mt.k_attn_fwd(qkv, o, lse, B, s, H, Hkv, hd)
    rng = np.random.default_rng(s + 1)
    do, doh = bf(rng.standard_normal((B * s, H * hd)))
    cos, sin = ops.rope_tables(s, hd, 10000.0)
    ct, _ = f32(cos)
    st, _ = f32(sin)
    delta = torch.empty((B, H, s), device=DEV)
    got = torch.zeros_like(qkv)
    mt.k_attn_bwd_rope(qkv, o, do, lse, delta, got, B, s, H, Hkv, hd, ct, st)
    twice = torch.zeros_like(qkv)
    mt.k_attn_bwd(qkv, o, do, lse, delta, twice, B, s, H, Hkv, hd)
    mt.k_rope(twice, B, s, H + Hkv, hd, ct, st, inverse=True)
    torch.cuda.synchronize()
    dq, dk, dv = ops.attention_bwd(q, k, v, doh.reshape(B, s, H, hd))
    dq, dk = ops.rope_bwd(dq, cos, sin), ops.rope_bwd(dk, cos, sin)
    g, g2 = host(got), host(twice)
    exact_qk = np.concatenate([dq.reshape(B * s, -1), dk.reshape(B * s, -1)], 1)
    assert_close(g[:, :(H + Hkv) * hd], exact_qk, l2=2e-2, elem=3e-2, what="dq, dk rotated back")
    assert torch.equal(got[:, (H + Hkv) * hd:], twice[:, (H + Hkv) * hd:])   # dv untouched
    if hd != 16:
        assert rel_l2(g[:, :(H + Hkv) * hd], exact_qk) < rel_l2(g2[:, :(H + Hkv) * hd], exact_qk)


# ------------------------------------------------------------ cross entropy
@pytest.mark.parametrize("M,V", [(64, 512), (37, 32000), (5, 152064), (2000, 512), (400, 152064)])
def test_cross_entropy(M, V):
    """Rows are spread over a fixed grid of a few blocks per SM, so the
    larger cases give each block several rows."""
    rng = np.random.default_rng(M + V)
    z, zh = f32(rng.standard_normal((M, V)) * 3)
    lab_np = rng.integers(0, V, size=M).astype(np.int32)
    lab = torch.from_numpy(lab_np).to(DEV)
    dz = torch.empty((M, V), device=DEV, dtype=torch.bfloat16)
    rows = torch.empty(M, device=DEV)
    total = torch.empty(1, device=DEV)
    mt.k_cross_entropy(z, lab, dz, rows, 1.0 / M)
    mt.k_sum(rows, total)
    torch.cuda.synchronize()
    loss, dref = ops.cross_entropy_fwd_bwd(zh, lab_np)
    assert float(total.item()) / M == pytest.approx(loss, rel=1e-5)
    assert_close(host(dz), dref, l2=5e-3, elem=1e-2, what="dz")


def test_cross_entropy_zero_logits_is_ln_v():
    M, V = 8, 32000
    z = torch.zeros((M, V), device=DEV)
    lab = torch.arange(M, device=DEV, dtype=torch.int32)
    dz = torch.empty((M, V), device=DEV, dtype=torch.bfloat16)
    rows = torch.empty(M, device=DEV)
    mt.k_cross_entropy(z, lab, dz, rows, 1.0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(host(rows), np.log(V), rtol=1e-6)


# ---------------------------------------------------------------- embedding
@pytest.mark.parametrize("M,V,d,dup", [(64, 512, 64, False), (1000, 97, 128, True), (4096, 152064, 512, False),
                                       (3000, 5, 64, True)])
def test_embedding_fwd_bwd(M, V, d, dup):
    rng = np.random.default_rng(M + V)
    E, Eh = bf(rng.standard_normal((V, d)))
    tok_np = (rng.integers(0, min(V, 3), size=M) if dup else rng.integers(0, V, size=M)).astype(np.int32)
    tok = torch.from_numpy(tok_np).to(DEV)
    x = torch.empty((M, d), device=DEV, dtype=torch.bfloat16)
    mt.k_embedding_fwd(E, tok, x)
    x32 = torch.empty((M, d), device=DEV)
    mt.k_embedding_fwd(E, tok, x32)     # the fp32 residual stream: exact
    torch.cuda.synchronize()
    assert torch.equal(x, E[tok.long()])
    assert torch.equal(x32, E[tok.long()].float())
    dx, dxh = f32(rng.standard_normal((M, d)))
    work = torch.empty(mt.k_embedding_bwd_work(M, V), device=DEV, dtype=torch.int32)
    dE = torch.empty((V, d), device=DEV, dtype=torch.bfloat16)
    dE2 = torch.empty_like(dE)
    mt.k_embedding_bwd(dx, tok, dE, work)
    mt.k_embedding_bwd(dx, tok, dE2, work)
    torch.cuda.synchronize()
    assert torch.equal(dE, dE2)
    ref = ops.embedding_bwd(dxh, tok_np, V)
    assert_close(host(dE), ref, l2=5e-3, elem=1e-2, what="dE")
    untouched = np.setdiff1d(np.arange(V), tok_np)
    assert np.all(host(dE)[untouched] == 0)


# ------------------------------------------------- GEMM with MN-major operands
@pytest.mark.parametrize("a_mn,b_mn", [(False, True), (True, False), (True, True)])
@pytest.mark.parametrize("M,N,K,out", [
    (64, 192, 64, "f32"),          # tiny
    (200, 296, 136, "bf16"),       # ragged M, N, K
    (2048, 5632, 2048, "bf16"),    # 1.1B down-projection dgrad / wgrad shapes
    (4096, 4096, 1000, "f32"),     # ragged K (tokens) for a weight gradient
])
def test_gemm_mn_major(M, N, K, out, a_mn, b_mn):
    rng = np.random.default_rng(M + N + K + 7 * a_mn + 3 * b_mn)
    Ah = rng.standard_normal((M, K))
    Bh = rng.standard_normal((N, K)) / np.sqrt(K)
    # store MN-major operands as [K, M] / [K, N] arrays (the product uses their transposes)
    A, Ab = bf(Ah.T.copy() if a_mn else Ah)
    B, Bb = bf(Bh.T.copy() if b_mn else Bh)
    Aop = Ab.T if a_mn else Ab
    Bop = Bb.T if b_mn else Bb
    Cout = torch.empty((M, N), device=DEV, dtype=torch.float32 if out == "f32" else torch.bfloat16)
    mt.k_gemm_ex(A, a_mn, B, b_mn, Cout)
    torch.cuda.synchronize()
    ref = Aop @ Bop.T
    assert_close(host(Cout), ref, l2=5e-3 if out == "bf16" else 1e-4, elem=1e-2 if out == "bf16" else 1e-3,
                 what=f"gemm_ex a_mn={a_mn} b_mn={b_mn} {M}x{N}x{K}")


@pytest.mark.parametrize("B,s,H,Hkv,hd", [(3, 200, 4, 2, 128), (2, 129, 8, 2, 64), (1, 2048, 4, 4, 64),
                                          (2, 640, 2, 1, 128)])
def test_attention_fwd_tcgen05_matches_mma_and_oracle(B, s, H, Hkv, hd):
    """The tcgen05/TMEM forward against the oracle and against the mma.sync
    kernel (several sequences per batch with ragged length: rows past each
    sequence's end must read as zeros)."""
    qkv, q, k, v = _attn_inputs(B, s, H, Hkv, hd, 11 * s + hd)
    o = torch.empty((B * s, H * hd), device=DEV, dtype=torch.bfloat16)
    lse = torch.empty((B, H, s), device=DEV)
    o2 = torch.empty_like(o)
    lse2 = torch.empty_like(lse)
    mt.k_attn_fwd(qkv, o, lse, B, s, H, Hkv, hd)
    mt.k_attn_fwd_mma(qkv, o2, lse2, B, s, H, Hkv, hd)
    torch.cuda.synchronize()
    orf, lr = ops.attention_fwd(q, k, v)
    assert_close(host(o), orf.reshape(B * s, H * hd), l2=1e-2, elem=2e-2, what="tc o")
    np.testing.assert_allclose(host(lse), lr, rtol=0, atol=2e-2)
    assert_close(host(o), host(o2), l2=1e-2, elem=2e-2, what="tc vs mma")


@pytest.mark.parametrize("B,s,H,Hkv,hd", [(3, 200, 4, 2, 128), (2, 129, 8, 2, 64), (1, 1024, 4, 4, 64),
                                          (2, 384, 2, 1, 128)])
def test_attention_bwd_tcgen05_matches_mma_and_oracle(B, s, H, Hkv, hd):
    """The tcgen05 backward (dK/dV and dQ kernels) against the oracle and the
    mma.sync backward, several ragged sequences per batch; deterministic."""
    qkv, q, k, v = _attn_inputs(B, s, H, Hkv, hd, 13 * s + hd)
    o = torch.empty((B * s, H * hd), device=DEV, dtype=torch.bfloat16)
    lse = torch.empty((B, H, s), device=DEV)
    mt.k_attn_fwd(qkv, o, lse, B, s, H, Hkv, hd)
    rng = np.random.default_rng(s + 1)
    do, doh = bf(rng.standard_normal((B * s, H * hd)))
    delta = torch.empty((B, H, s), device=DEV)
    g1, g2, g3 = (torch.zeros_like(qkv) for _ in range(3))
    mt.k_attn_bwd(qkv, o, do, lse, delta, g1, B, s, H, Hkv, hd)
    mt.k_attn_bwd(qkv, o, do, lse, delta, g2, B, s, H, Hkv, hd)
    mt.k_attn_bwd_mma(qkv, o, do, lse, delta, g3, B, s, H, Hkv, hd)
    torch.cuda.synchronize()
    assert torch.equal(g1, g2)
    dq, dk, dv = ops.attention_bwd(q, k, v, doh.reshape(B, s, H, hd))
    g = host(g1)
    fl = 1e-3 * np.abs(dv).max()
    assert_close(g[:, :H * hd], dq.reshape(B * s, -1), l2=2e-2, elem=3e-2, what="dq", floor=fl)
    assert_close(g[:, H * hd:(H + Hkv) * hd], dk.reshape(B * s, -1), l2=2e-2, elem=3e-2, what="dk", floor=fl)
    assert_close(g[:, (H + Hkv) * hd:], dv.reshape(B * s, -1), l2=2e-2, elem=3e-2, what="dv")
    assert_close(g, host(g3), l2=2e-2, elem=3e-2, what="tc vs mma", floor=fl)
