"""w8a8_gemm_noalloc: the W8A8 GEMM on the library's built-in scratch array.

Some callers cannot allocate device memory for a workspace (their memory is
reserved up front by a host framework, they run under a fixed budget, or they
cannot afford cudaMalloc / cudaFree, which may block or synchronize the
device).  This entry point serves them from a fixed array compiled into the
library, so these tests check that it computes exactly what the caller-
workspace entry point w8a8_gemm computes, and what the oracle computes:

* two calls in a row with different inputs and shapes on the one shared
  scratch array: the row scales, the int8 codes and the int32 product bit for
  bit against the oracle and against w8a8_gemm, and Y against the oracle
  under the tests' floating-point bar (|y - y_ref| <= 1e-3 * sum_k |x_k w_kn|
  + 1e-5 + 2^-8 |y_ref|: bf16 output) and against w8a8_gemm's Y bit for bit;
* two calls back to back on one stream with programmatic dependent launch
  and no synchronization between them, so the second call's quantization
  kernel may start while the first call's GEMM still reads the scratch: the
  quantization kernel waits for the preceding grid before its first write,
  and both calls' results must still match the oracle;
* on the host, the size limit and the argument checks, which return before
  any CUDA call.

The file name sorts last, so the GPU tests also run after every other test of
the suite (and pass alone in a fresh process as well).
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


def _outputs(G, M, K, N):
    import torch
    buf, Y = G.guarded((M, N), torch.bfloat16)
    Xq = torch.empty((M, K), dtype=torch.int8, device=G.DEV)
    Sx = torch.empty((M,), dtype=torch.float32, device=G.DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=G.DEV)
    return buf, Y, Xq, Sx, acc


def _host(G, o, M, N):
    buf, Y, Xq, Sx, acc = o
    G.check_canary(buf, M * N)
    return G.bits_u16(Y), Xq.cpu().numpy(), Sx.cpu().numpy(), acc.cpu().numpy()


def _run(wq, G, d, noalloc, flags=0, sync=True):
    """One call; returns the device outputs (the inputs stay alive in the tuple)."""
    import torch
    M, K = d["X"].shape
    N = d["W"].shape[1]
    X, W, Sw = G.dev(d["X"]), G.dev(d["W"]), G.dev(d["Sw"])
    o = _outputs(G, M, K, N)
    _, Y, Xq, Sx, acc = o
    if noalloc:
        wq.w8a8_gemm_noalloc(X, W, Sw, Y, M, K, N, Xq, Sx, acc, flags=flags)
    else:
        nbytes = wq.w8a8_gemm_workspace_bytes(M, K, N)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=G.DEV)
        wq.w8a8_gemm(X, W, Sw, Y, M, K, N, Xq, Sx, acc, ws, nbytes, flags=flags)
    if sync:
        torch.cuda.synchronize()
    return o, (X, W, Sw)


def _check_against_oracle(d, y_bits, xq, sx, acc):
    """Sx, Xq and the int32 product bit for bit, Y under the bar, all from the oracle."""
    import oracle
    from tolerance import U_BF16, within
    xq_ref, sx_ref = oracle.w8a8_quant_rows(d["X"])
    assert np.array_equal(sx.view(np.uint32), sx_ref.view(np.uint32)), "Sx differs from the oracle"
    assert np.array_equal(xq, xq_ref), "Xq differs from the oracle"
    acc_ref, y_ref, a, ovf = oracle.w8a8_gemm_rows(xq_ref, sx_ref, d["W"], d["Sw"], None)
    assert not ovf
    assert np.array_equal(acc.astype(np.int64), acc_ref), "int32 product differs from the oracle"
    y = oracle.decode_bf16(y_bits)
    ok, worst = within(y, y_ref, a, U_BF16)
    assert ok, f"Y: max |err|/bound = {worst:.3g}"


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_w8a8_gemm_two_calls_in_a_row(wq):
    import gpu_util as G
    import synthetic as syn
    cases = [syn.make_w8a8(seed=5, M=200, K=4096, N=272), syn.make_w8a8(seed=6, M=511, K=8192, N=384)]
    # both no-alloc calls first, one after the other on the same scratch, then the checks
    got = []
    for d in cases:
        o, _ = _run(wq, G, d, noalloc=True)
        got.append(_host(G, o, d["X"].shape[0], d["W"].shape[1]))
    for d, (y, xq, sx, acc) in zip(cases, got):
        _check_against_oracle(d, y, xq, sx, acc)
        o, _ = _run(wq, G, d, noalloc=False)
        y_ws, xq_ws, sx_ws, acc_ws = _host(G, o, d["X"].shape[0], d["W"].shape[1])
        assert np.array_equal(sx.view(np.uint32), sx_ws.view(np.uint32)), "Sx differs from w8a8_gemm"
        assert np.array_equal(xq, xq_ws), "Xq differs from w8a8_gemm"
        assert np.array_equal(acc, acc_ws), "int32 product differs from w8a8_gemm"
        assert np.array_equal(y, y_ws), "Y differs from w8a8_gemm"


@pytest.mark.gpu
def test_noalloc_back_to_back_pdl_on_one_stream(wq):
    import torch

    import gpu_util as G
    import synthetic as syn
    cases = [syn.make_w8a8(seed=11, M=384, K=8192, N=256), syn.make_w8a8(seed=12, M=256, K=8192, N=512)]
    stream = torch.cuda.Stream(device=G.DEV)
    torch.cuda.synchronize()
    keep = []
    with torch.cuda.stream(stream):
        for d in cases:  # no synchronization between the two calls
            o, inputs = _run(wq, G, d, noalloc=True, flags=wq.WQ_FLAG_PDL, sync=False)
            keep.append((o, inputs))
    torch.cuda.synchronize()
    for d, (o, _) in zip(cases, keep):
        _check_against_oracle(d, *_host(G, o, d["X"].shape[0], d["W"].shape[1]))
    assert wq.read_timeout_flag(clear=True) == 0
