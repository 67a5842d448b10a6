"""w8a8_gemm_noalloc: the W8A8 GEMM on the library's built-in scratch array.

The GPU test compares it with w8a8_gemm (caller workspace) on two calls in a
row with different inputs and shapes, under the tests' floating-point bar
(|y - y_ref| <= 1e-3 * sum_k |x_k w_kn| + 1e-5 + 2^-8 |y_ref|, the magnitude
sum from the oracle); the row quantization and the int32 product are compared
bit for bit.  The host test checks the size limit and the argument checks,
which return before any CUDA call.  The file name sorts last, so the GPU test
also runs after every other test of the suite.
"""
import numpy as np
import pytest

# fake, never-dereferenced device addresses (aligned / misaligned)
A = 0x7f0000000000
MIS = A + 4


@pytest.fixture(scope="module")
def wq():
    import gemm_dequant_gemv_gb300 as m
    return m


def test_noalloc_rejects_before_any_cuda_call(wq):
    f = wq.library().w8a8_gemm_noalloc
    cap = wq.w8a8_gemm_noalloc_max_scratch_bytes()
    assert cap == 8 << 20
    base = [A, A, A, A, 64, 128, 64, None, None, None, 0, 0]
    assert f(*([0] + base[1:])) == wq.WQ_ERR_NULL
    b = list(base); b[5] = 100
    assert f(*b) == wq.WQ_ERR_SHAPE                 # K % 64
    b = list(base); b[6] = 40
    assert f(*b) == wq.WQ_ERR_SHAPE                 # N % 16
    b = list(base); b[7] = MIS
    assert f(*b) == wq.WQ_ERR_ALIGN
    # the largest M that fits at K = 8192 is 511 (the 256-byte padding of Sx
    # takes the rest); one more row needs more than the built-in scratch
    assert wq.w8a8_gemm_workspace_bytes(511, 8192, 64) <= cap < wq.w8a8_gemm_workspace_bytes(512, 8192, 64)
    b = list(base); b[4], b[5] = 512, 8192
    assert f(*b) == wq.WQ_ERR_WORKSPACE
    b = list(base); b[4], b[5] = 2048, 8192
    assert f(*b) == wq.WQ_ERR_WORKSPACE


def _run(wq, G, d, noalloc):
    import torch
    M, K = d["X"].shape
    N = d["W"].shape[1]
    X, W, Sw = G.dev(d["X"]), G.dev(d["W"]), G.dev(d["Sw"])
    buf, Y = G.guarded((M, N), torch.bfloat16)
    Xq = torch.empty((M, K), dtype=torch.int8, device=G.DEV)
    Sx = torch.empty((M,), dtype=torch.float32, device=G.DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=G.DEV)
    if noalloc:
        wq.w8a8_gemm_noalloc(X, W, Sw, Y, M, K, N, Xq, Sx, acc)
    else:
        nbytes = wq.w8a8_gemm_workspace_bytes(M, K, N)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=G.DEV)
        wq.w8a8_gemm(X, W, Sw, Y, M, K, N, Xq, Sx, acc, ws, nbytes)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    return G.to_f64(Y), Xq.cpu().numpy(), Sx.cpu().numpy(), acc.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_w8a8_gemm_two_calls_in_a_row(wq):
    import gpu_util as G
    import oracle
    import synthetic as syn
    from tolerance import U_BF16, within
    cases = [syn.make_w8a8(seed=5, M=200, K=4096, N=272), syn.make_w8a8(seed=6, M=511, K=8192, N=384)]
    # both no-alloc calls first, back to back on the same scratch, then the references
    got = [_run(wq, G, d, noalloc=True) for d in cases]
    for d, (y, xq, sx, acc) in zip(cases, got):
        y_ref, xq_ref, sx_ref, acc_ref = _run(wq, G, d, noalloc=False)
        assert np.array_equal(sx.view(np.uint32), sx_ref.view(np.uint32)), "Sx differs"
        assert np.array_equal(xq, xq_ref), "Xq differs"
        assert np.array_equal(acc, acc_ref), "int32 product differs"
        _, _, a, ovf = oracle.w8a8_gemm_rows(xq_ref, sx_ref, d["W"], d["Sw"], None)
        assert not ovf
        ok, worst = within(y, y_ref, a, U_BF16)
        assert ok, f"max |err|/bound = {worst:.3g}"
