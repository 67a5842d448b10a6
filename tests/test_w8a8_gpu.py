"""GPU parity of the W8A8 dynamic-quantization GEMM against the oracle.

The row quantization (Sx, Xq) and the int32 product are compared bit for bit;
Y is compared under |y - y_ref| <= 1e-3 * sum_k |x_k w_kn| + 1e-5 + 2^-8 |y_ref|
with x = Sx Xq and w = Sw Wq (the last term is the bf16 rounding of the stored
output).  Shapes cover one and several 128 x 128 tiles, ragged M and N,
a K that is not a multiple of the 256-value exact chunk, adversarial
full-magnitude codes, an all-zero row, and the full 2048 x 8192 x 8192
workload (every row's quantization, sampled rows of the product).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import gpu_util
    return gpu_util


def run_w8a8(G, X_bits, W, Sw, want_acc=True):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    M, K = X_bits.shape
    N = W.shape[1]
    X, Wd, Swd = G.dev(X_bits), G.dev(W), G.dev(Sw)
    buf, Y = G.guarded((M, N), torch.bfloat16)
    Xq = torch.empty((M, K), dtype=torch.int8, device=G.DEV)
    Sx = torch.empty((M,), dtype=torch.float32, device=G.DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=G.DEV) if want_acc else None
    ws_bytes = wq.w8a8_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=G.DEV)
    wq.w8a8_gemm(X, Wd, Swd, Y, M, K, N, Xq, Sx, acc, ws, ws_bytes)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    return (Y, Xq.cpu().numpy(), Sx.cpu().numpy(),
            None if acc is None else acc.cpu().numpy().astype(np.int64))


def _check(G, X_bits, W, Sw, rows=None):
    import oracle
    from tolerance import U_BF16, within
    Y, Xq, Sx, acc = run_w8a8(G, X_bits, W, Sw)
    Xq_ref, Sx_ref = oracle.w8a8_quant_rows(X_bits)
    assert np.array_equal(Sx.view(np.uint32), Sx_ref.view(np.uint32)), "Sx differs"
    assert np.array_equal(Xq, Xq_ref), "Xq differs"
    acc_ref, y_ref, a, ovf = oracle.w8a8_gemm_rows(Xq_ref, Sx_ref, W, Sw, rows)
    assert not ovf
    r = np.arange(X_bits.shape[0]) if rows is None else np.asarray(rows)
    assert np.array_equal(acc[r], acc_ref), "int32 accumulator differs"
    ok, worst = within(G.to_f64(Y)[r], y_ref, a, U_BF16)
    assert ok, f"max |err|/bound = {worst:.3g}"


@pytest.mark.parametrize("M,K,N", [(64, 256, 128), (200, 512, 272), (128, 320, 128), (300, 1024, 512)])
def test_w8a8_parity_small(G, M, K, N):
    import synthetic as syn
    d = syn.make_w8a8(seed=5, M=M, K=K, N=N)
    _check(G, d["X"], d["W"], d["Sw"])


def test_w8a8_more_tiles_than_sms_ragged_odd_stages(G):
    """187 output tiles (11 x 17, ragged in both M and N): more CTAs than SMs,
    so later CTAs run on SMs whose previous CTA has just released its tensor
    memory; K = 320 gives three 128-value stages (an odd count) and two exact
    chunks, the second of one stage."""
    import synthetic as syn
    d = syn.make_w8a8(seed=11, M=1300, K=320, N=2064)
    _check(G, d["X"], d["W"], d["Sw"])


def test_w8a8_adversarial_full_magnitude(G):
    """Every code of X +-127 with aligned signs: |acc| up to K * 127 * 128 (133 M at
    K = 8192) with W = -128 in some columns, the edge of the exact 256-value chunk
    (256 * 127 * 128 < 2^22)."""
    import synthetic as syn
    M, K, N = 128, 8192, 256
    Xf = np.full((M, K), 2.0, np.float32)
    Xf[1::2] = -2.0                      # rows of alternating sign
    Xf[5] = 0.0                          # an all-zero row
    W = np.full((K, N), 127, np.int8)
    W[:, 1::3] = -127
    W[:, 2::5] = -128
    Sw = np.full((N,), 0.01, np.float32)
    _check(G, syn.f32_to_bf16_bits(Xf), W, Sw)


def full_workload_rows(M=2048, tile=128, n=256, seed=0):
    """Both sides of every 128-row tile edge, the first and last rows, and seeded
    random rows up to n in all."""
    edges = {0, M - 1}
    for e in range(tile, M, tile):
        edges.update((e - 1, e))
    r = np.random.default_rng(seed)
    rest = r.permutation(np.setdiff1d(np.arange(M), sorted(edges)))[: n - len(edges)]
    return np.sort(np.concatenate([np.array(sorted(edges)), rest])).astype(np.int64)


def test_w8a8_full_workload_sampled_rows(G):
    """The benchmarked 2048 x 8192 x 8192 shape: every row's Sx and Xq, and the
    int32 product and Y of 256 rows (every tile edge and seeded random rows)."""
    import synthetic as syn
    d = syn.make_w8a8(seed=5)
    rows = full_workload_rows()
    assert len(rows) == 256 and {127, 128, 1919, 1920, 2047} <= set(rows.tolist())
    _check(G, d["X"], d["W"], d["Sw"], rows)


def test_w8a8_repeat_bit_identical(G):
    import synthetic as syn
    d = syn.make_w8a8(seed=6, M=256, K=1024, N=384)
    y1 = G.bits_u16(run_w8a8(G, d["X"], d["W"], d["Sw"], want_acc=False)[0])
    y2 = G.bits_u16(run_w8a8(G, d["X"], d["W"], d["Sw"], want_acc=False)[0])
    assert np.array_equal(y1, y2)


def test_w8a8_smooth_parity(G):
    """Smoothquant: X / s per channel before the row quantization; the weights are the
    int8 codes of diag(s) W.  Sx, Xq and the int32 product bit-exact, Y under the bar."""
    import torch
    import gemm_dequant_gemv_gb300 as wq
    import oracle
    import synthetic as syn
    from tolerance import U_BF16, within
    M, K, N = 200, 512, 272
    r = np.random.default_rng(31)
    Xf = r.normal(0, 1, (M, K)).astype(np.float32)
    Xf[:, [5, 77, 300]] *= 30.0                              # outlier channels
    X_bits = syn.f32_to_bf16_bits(Xf)
    amax_c = np.abs(syn.bf16_bits_to_f32(X_bits)).max(axis=0)
    smooth = np.sqrt(np.maximum(amax_c, 1e-3)).astype(np.float32)   # s = sqrt(max|X[:, k]|)
    Wf = r.normal(0, 0.02, (K, N)).astype(np.float32) * smooth[:, None]   # diag(s) W
    Sw = (np.abs(Wf).max(axis=0) / np.float32(127.0)).astype(np.float32)
    Wq = np.clip(np.rint(Wf / Sw[None, :]), -127, 127).astype(np.int8)
    X, Wd, Swd, sd = G.dev(X_bits), G.dev(Wq), G.dev(Sw), G.dev(smooth)
    buf, Y = G.guarded((M, N), torch.bfloat16)
    Xq = torch.empty((M, K), dtype=torch.int8, device=G.DEV)
    Sx = torch.empty((M,), dtype=torch.float32, device=G.DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=G.DEV)
    nb = wq.w8a8_gemm_workspace_bytes(M, K, N)
    ws = torch.empty(nb, dtype=torch.uint8, device=G.DEV)
    wq.w8a8_gemm_smooth(X, sd, Wd, Swd, Y, M, K, N, Xq, Sx, acc, ws, nb)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    Xq_ref, Sx_ref = oracle.w8a8_quant_rows_smooth(X_bits, smooth)
    assert np.array_equal(Sx.cpu().numpy().view(np.uint32), Sx_ref.view(np.uint32)), "Sx differs"
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref), "Xq differs"
    acc_ref, y_ref, a, ovf = oracle.w8a8_gemm_rows(Xq_ref, Sx_ref, Wq, Sw)
    assert not ovf
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref), "int32 accumulator differs"
    ok, worst = within(G.to_f64(Y), y_ref, a, U_BF16)
    assert ok, f"max |err|/bound = {worst:.3g}"
    # smoothing lowers the row scales that the outlier channels set
    _, Sx_plain = oracle.w8a8_quant_rows(X_bits)
    assert np.all(Sx_ref <= Sx_plain) and np.mean(Sx_ref) < 0.5 * np.mean(Sx_plain)


@pytest.mark.parametrize("M,K,N,threshold", [(200, 512, 272, 6.0), (128, 8192, 256, 6.0), (64, 256, 128, -1.0),
                                             (96, 320, 144, float("inf"))])
def test_w8a8_outlier_parity(G, M, K, N, threshold):
    """LLM.int8(): outlier columns flagged as the oracle flags them, Sx / Xq / the int8
    part's int32 product bit-exact, Y (int8 part + 16-bit outlier part) under the bar."""
    import torch
    import gemm_dequant_gemv_gb300 as wq
    import oracle
    import synthetic as syn
    from tolerance import U_BF16, within
    r = np.random.default_rng(41 + K)
    Xf = r.normal(0, 1, (M, K)).astype(np.float32)
    cols = r.choice(K, size=min(40, K // 8), replace=False)   # more than one staging round of 32
    for i, c in enumerate(cols):
        Xf[r.integers(0, M), c] = (8.0 + i) * (1 if i % 2 else -1)
    Xf[0, (cols[0] + 1) % K] = 6.0                               # equal to the threshold
    X_bits = syn.f32_to_bf16_bits(Xf)
    W = r.integers(-127, 128, (K, N), dtype=np.int8)
    Sw = r.uniform(0.001, 0.01, N).astype(np.float32)
    Xd, Wd, Swd = G.dev(X_bits), G.dev(W), G.dev(Sw)
    buf, Y = G.guarded((M, N), torch.bfloat16)
    Xq = torch.empty((M, K), dtype=torch.int8, device=G.DEV)
    Sx = torch.empty((M,), dtype=torch.float32, device=G.DEV)
    acc = torch.empty((M, N), dtype=torch.int32, device=G.DEV)
    nout = torch.zeros((4,), dtype=torch.int32, device=G.DEV)
    nb = wq.w8a8_gemm_outlier_workspace_bytes(M, K, N)
    ws = torch.empty(nb, dtype=torch.uint8, device=G.DEV)
    wq.w8a8_gemm_outlier(Xd, Wd, Swd, Y, M, K, N, threshold, Xq, Sx, acc, nout, ws, nb)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    flags, Xq_ref, Sx_ref, acc_ref, y_ref, a, ovf = oracle.w8a8_outlier(X_bits, W, Sw, threshold)
    assert int(nout[0]) == int(flags.sum())
    assert np.array_equal(Sx.cpu().numpy().view(np.uint32), Sx_ref.view(np.uint32)), "Sx differs"
    assert np.array_equal(Xq.cpu().numpy(), Xq_ref), "Xq differs"
    assert not ovf
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref), "int32 accumulator differs"
    ok, worst = within(G.to_f64(Y), y_ref, a, U_BF16)
    assert ok, f"max |err|/bound = {worst:.3g}"
