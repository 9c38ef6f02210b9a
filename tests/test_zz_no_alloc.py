"""The embedding backward that allocates nothing, checked against the regular one.

mt_k_embedding_bwd_noalloc serves callers that cannot allocate device memory
themselves (code running inside another framework's memory pool, or in a
process whose allocator belongs to someone else), so they cannot hand the
regular entry point its `work` buffer. Its workspace is a fixed device array
inside the library. Both entry points run the same kernels, so their outputs
must agree; the test uses the embedding tolerance of the kernel tests
(relative L2 <= 5e-3 against the oracle) and, since the arithmetic is the
same, also requires bit equality with the regular entry point. Two calls in a
row with different token ids make sure nothing left in the shared array by
the first call leaks into the second. This file is collected last.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import host_memory_resident_gb300 as mt  # noqa: E402
from oracle import ops  # noqa: E402

pytestmark = pytest.mark.gpu


def _noalloc():
    fn = mt.lib().mt_k_embedding_bwd_noalloc
    fn.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p]
    fn.restype = C.c_int
    return fn


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mt.lib()


@pytest.mark.parametrize("M,V,d", [(64, 512, 64), (4096, 152064, 512)])
def test_noalloc_matches_regular_entry_point_twice(M, V, d):
    fn = _noalloc()
    rng = np.random.default_rng(M + V)
    for call in range(2):
        # the second call uses fewer distinct ids, so stale buckets would show
        hi = V if call == 0 else max(2, V // 64)
        tok_np = rng.integers(0, hi, size=M).astype(np.int32)
        dx_np = rng.standard_normal((M, d)).astype(np.float32)
        tok = torch.from_numpy(tok_np).cuda()
        dx = torch.from_numpy(dx_np).cuda()
        ref = torch.empty((V, d), device="cuda", dtype=torch.bfloat16)
        work = torch.empty(mt.k_embedding_bwd_work(M, V), device="cuda", dtype=torch.int32)
        mt.k_embedding_bwd(dx, tok, ref, work)
        out = torch.full((V, d), 7.0, device="cuda", dtype=torch.bfloat16)
        code = fn(C.c_void_p(dx.data_ptr()), C.c_void_p(tok.data_ptr()), C.c_void_p(out.data_ptr()), M, d, V, None)
        assert code == mt.MT_OK, mt.lib().mt_last_error(None)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}"
        got = out.float().cpu().numpy().astype(np.float64)
        exact = ops.embedding_bwd(dx_np.astype(np.float64), tok_np, V)
        assert np.linalg.norm(got - exact) / np.linalg.norm(exact) <= 5e-3


def test_noalloc_at_its_largest_accepted_sizes():
    """M and V at the limits fill the fixed array exactly (start[V + 1],
    cursor[V], perm[M]); the result must still be the regular entry point's,
    bit for bit, twice in a row."""
    fn = _noalloc()
    M, V, d = 524288, 262144, 8
    rng = np.random.default_rng(5)
    for call in range(2):
        tok = torch.from_numpy(rng.integers(0, V if call == 0 else 1000, size=M).astype(np.int32)).cuda()
        dx = torch.from_numpy(rng.standard_normal((M, d)).astype(np.float32)).cuda()
        ref = torch.empty((V, d), device="cuda", dtype=torch.bfloat16)
        work = torch.empty(mt.k_embedding_bwd_work(M, V), device="cuda", dtype=torch.int32)
        mt.k_embedding_bwd(dx, tok, ref, work)
        out = torch.full((V, d), 7.0, device="cuda", dtype=torch.bfloat16)
        code = fn(C.c_void_p(dx.data_ptr()), C.c_void_p(tok.data_ptr()), C.c_void_p(out.data_ptr()), M, d, V, None)
        assert code == mt.MT_OK, mt.lib().mt_last_error(None)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"call {call}"


def test_noalloc_rejects_sizes_above_its_limits():
    fn = _noalloc()
    dx = torch.zeros((8, 64), device="cuda")
    tok = torch.zeros(8, device="cuda", dtype=torch.int32)
    out = torch.empty((8, 64), device="cuda", dtype=torch.bfloat16)
    code = fn(C.c_void_p(dx.data_ptr()), C.c_void_p(tok.data_ptr()), C.c_void_p(out.data_ptr()),
              524288 + 1, 64, 8, None)
    assert code == mt.MT_EINVAL
    assert b"limits" in mt.lib().mt_last_error(None)
    code = fn(C.c_void_p(dx.data_ptr()), C.c_void_p(tok.data_ptr()), C.c_void_p(out.data_ptr()),
              8, 64, 262144 + 1, None)
    assert code == mt.MT_EINVAL
