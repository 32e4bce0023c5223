"""The allocation-free GEMM entry point, for callers that cannot allocate
device memory (their allocator belongs to another runtime, or they may not
call cudaMalloc while a captured graph or a latency-critical loop is live).

Called twice in a row through the C ABI (the shared scratch array keeps the
previous call's contents, so the second call checks that the kernels leave it
reusable), both results are compared with the oracle within the tolerance the
other GEMM tests use.  The shapes reach both kernels that read the scratch:
the decode kernel (activation images, stream-K pieces, flags) and the general
kernel (tile counters, pieces).  This file sorts last so that a run stopping at the
first failure has run every other test; it also passes on its own."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    from dense_sparse_int4_gb300 import mq
    L = mq.lib()
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn = L.mq_w4a4_residual_gemm_noalloc
    fn.restype = i32
    fn.argtypes = [P, P, i64, P, i64, i64, P, P, i64, P, P, i32, P]
    return L


def _noalloc(L, xq, xs, M, pl, out):
    from dense_sparse_int4_gb300 import mq
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    nz = pl.nnzb > 0
    return L.mq_w4a4_residual_gemm_noalloc(p(xq), p(xs), M, p(pl.wpk), pl.N, pl.K, p(pl.row_ptr),
                                           p(pl.col_idx) if nz else None, pl.nnzb, p(pl.rpk) if nz else None,
                                           p(out), mq._dtype_code(out.dtype),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("M,N,K,budget", [(4, 512, 512, 0.10), (32, 4096, 4096, 0.10), (17, 1024, 2048, 0.30),
                                          (40, 512, 1024, 0.20), (64, 1024, 512, 0.10), (160, 512, 640, 0.20)])
def test_noalloc_matches_oracle_twice(lib, M, N, K, budget):
    from dense_sparse_int4_gb300 import mq, synth
    from tests.gpu_helpers import check_close, dev_half
    import oracle as O
    x = synth.activations(M, K, seed=M + K, count=synth.n_outliers(K))
    w = synth.weights(N, K, seed=N + 1)
    xcal = synth.calibration(K, seed=3, count=synth.n_outliers(K))
    pl = mq.prepare_linear(dev_half(w), dev_half(xcal), budget)
    xq, xs = mq.quantize_act(dev_half(x))
    qx, sx = O.quantize_act(x, False)
    y, a = O.linear(qx, sx, O.prepare(w, xcal, False, budget))
    assert mq.gemm_plan(M, N, K)["decode"] == (M <= 32)
    # 160 tokens: the image form, whose operand images fit the fixed scratch at this size
    assert (mq.gemm_plan(M, N, K)["variant"] == "image") == (M >= 128)
    assert int(lib.mq_gemm_workspace_bytes(M, N, K)) > 0
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        st = _noalloc(lib, xq, xs, M, pl, out)
        assert st == mq.MQ_OK, lib.mq_last_error()
        mq.check_device_error()
        check_close(out.cpu().numpy(), y, a)


def test_noalloc_rejects_oversized(lib):
    from dense_sparse_int4_gb300 import mq
    M, N, K = 128, 4096, 4096  # 128-token tiles need more than the fixed scratch
    xq = torch.zeros((K // 128, M, 64), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((K // 128, M), dtype=torch.float16, device="cuda")
    w = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    pl = mq.pack_weights(w, torch.zeros(N // 64 + 1, dtype=torch.int32, device="cuda"),
                         torch.zeros(0, dtype=torch.int32, device="cuda"))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, xq, xs, M, pl, out) == mq.MQ_ERR_WORKSPACE
    assert b"scratch" in lib.mq_last_error()
