"""GPU parity of the standalone dequantization kernels (the unfused baseline).

Each dense matrix is compared bit for bit with the oracle's exact weights
rounded once to the output format: fp32 for W8 (numpy's IEEE float32 cast of
the exact double), fp16 for W3 and W4 (numpy's IEEE half cast), bf16 (the
round-to-nearest-even of the exact fp32 value's top 16 bits).  A sample of each
matrix is also rounded by the oracle's own format routines, which ties the
numpy casts to the oracle.  W8 and W4 are exact in fp32 before that one
rounding; W3 (s*q - zero, fp32 fma then fp16) is too at the configuration's
scales and zeros.  The unfused product (dense weights, then a dense fp32
matrix product) is checked against the oracle's GEMV under the project's
numerical bar.  Shapes: the three 4096-wide configurations in full, a bf16
W4A16 slice, and small ragged cases.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import gpu_util
    return gpu_util


def _u16(a):
    """fp16 / bf16 data as bit patterns (the oracle takes bits, never converted values)."""
    return a if a.dtype == np.uint16 else a.view(np.uint16)


def _bf16_rne(v):
    """bf16 bit patterns of float64 values that are exact in fp32 (RNE on the fp32 bits)."""
    u = np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _sample_matches(got_bits, exact, rounder, n=2000, seed=0):
    r = np.random.default_rng(seed)
    idx = r.integers(0, exact.size, n)
    want = rounder(exact.ravel()[idx])
    assert np.array_equal(got_bits.ravel()[idx], want)


def run_dq8(G, d):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    K, N = d["w"].shape
    buf, out = G.guarded((K, N), torch.float32)
    wq.wq8_dequant(G.dev(d["w"]), G.dev(d["scales"]), out, K, N, d["group"])
    torch.cuda.synchronize()
    G.check_canary(buf, K * N)
    return out


def run_dq3(G, d):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    K, N = d["K"], d["N"]
    buf, out = G.guarded((K, N), torch.float16)
    wq.wq3_dequant(G.dev(d["mat"]), G.dev(d["scales"]), G.dev(d["zeros"]), out, K, N)
    torch.cuda.synchronize()
    G.check_canary(buf, K * N)
    return out


def run_dq4(G, d):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    K, N, g = d["K"], d["N"], d["group"]
    act = wq.WQ_BF16 if d["act_bf16"] else wq.WQ_F16
    qz = None if d["qzeros"] is None else G.dev(d["qzeros"])
    gi = None if d["g_idx"] is None else G.dev(d["g_idx"])
    buf, out = G.guarded((K, N), torch.bfloat16 if d["act_bf16"] else torch.float16)
    wq.wq4_dequant(G.dev(d["qweight"]), G.dev(d["scales"]), qz, gi, out, K, N, g, act)
    torch.cuda.synchronize()
    G.check_canary(buf, K * N)
    return out


@pytest.mark.parametrize("K,N,group", [(4096, 4096, 128), (32, 16, 16), (384, 48, 64)])
def test_wq8_dequant_bit_exact(G, K, N, group):
    import oracle
    import synthetic as syn
    d = syn.make_wq8(seed=1, K=K, N=N, group=group)
    got = run_dq8(G, d).cpu().numpy()
    exact = oracle.wq8_dequant(d["w"], d["scales"], group)
    assert np.array_equal(got.view(np.uint32), exact.astype(np.float32).view(np.uint32))
    _sample_matches(got.view(np.uint32), exact, lambda v: oracle.round_f32(v).view(np.uint32))


@pytest.mark.parametrize("K,N", [(4096, 4096), (32, 8), (96, 40)])
def test_wq3_dequant_bit_exact(G, K, N):
    import oracle
    import synthetic as syn
    d = syn.make_wq3(seed=2, K=K, N=N)
    got = G.bits_u16(run_dq3(G, d))
    exact = oracle.wq3_dequant(d["mat"], _u16(d["scales"]), _u16(d["zeros"]), K)
    assert np.array_equal(got, exact.astype(np.float16).view(np.uint16))
    _sample_matches(got, exact, oracle.round_f16)


@pytest.mark.parametrize("case", ["actorder_f16", "sym_bf16", "asym_f16_ragged", "actorder_bf16_small"])
def test_wq4_dequant_bit_exact(G, case):
    import oracle
    import synthetic as syn
    if case == "actorder_f16":
        d = syn.make_wq4_actorder(seed=3)
        d.update(act_bf16=False)
    elif case == "sym_bf16":
        d = syn.make_wq4_sym(seed=4, K=1024, N=2048)
        d.update(act_bf16=True, qzeros=None, g_idx=None)
    elif case == "asym_f16_ragged":
        r = np.random.default_rng(7)
        K, N, g = 96, 24, 32
        d = dict(qweight=syn.pack4(r.integers(0, 16, (K, N), dtype=np.uint8)),
                 scales=r.uniform(0.002, 0.03, (K // g, N)).astype(np.float16),
                 qzeros=syn.pack_zeros4(r.integers(0, 16, (K // g, N), dtype=np.uint8)),
                 g_idx=None, K=K, N=N, group=g, act_bf16=False)
    else:
        d = syn.make_wq4_actorder(seed=8, K=512, N=264, group=128)
        d.update(act_bf16=True, scales=syn.f32_to_bf16_bits(d["scales"].astype(np.float32)))
    K, N = d["K"], d["N"]
    got = G.bits_u16(run_dq4(G, d))
    exact = oracle.wq4_dequant(int(d["act_bf16"]), d["qweight"], _u16(d["scales"]), d["qzeros"], d["g_idx"],
                               d["group"])
    want = _bf16_rne(exact) if d["act_bf16"] else exact.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    _sample_matches(got, exact, oracle.round_bf16 if d["act_bf16"] else oracle.round_f16)


def test_unfused_products_match_the_oracle(G):
    """dequantize, then a dense fp32 product: y within the numerical bar of the fused kernels."""
    import torch
    import oracle
    import synthetic as syn
    from tolerance import U_F16, within
    d8 = syn.make_wq8(seed=1)
    w8 = run_dq8(G, d8)
    y8 = torch.from_numpy(d8["x"]).to(G.DEV) @ w8
    ref, a = oracle.wq8_gemv(d8["x"], d8["w"], d8["scales"], d8["group"])
    ok, worst = within(G.to_f64(y8), ref, a)
    assert ok, worst
    d3 = syn.make_wq3(seed=2)
    w3 = run_dq3(G, d3).float()
    x3 = torch.from_numpy(d3["x"].view(np.float16).astype(np.float32)).to(G.DEV)
    y3 = (x3 @ w3).half()
    ref, a = oracle.wq3_gemv(_u16(d3["x"]), d3["mat"], _u16(d3["scales"]), _u16(d3["zeros"]))
    ok, worst = within(G.to_f64(y3), ref, a, U_F16)
    assert ok, worst
    d4 = syn.make_wq4_actorder(seed=3)
    d4.update(act_bf16=False)
    w4 = run_dq4(G, d4).float()
    x4 = torch.from_numpy(d4["x"].view(np.float16).astype(np.float32)).to(G.DEV)
    y4 = (x4 @ w4).half()
    ref, a = oracle.wq4_gemm(_u16(d4["x"]), 0, d4["qweight"], _u16(d4["scales"]), d4["qzeros"], d4["g_idx"],
                             d4["group"])
    ok, worst = within(G.to_f64(y4), ref, a, U_F16)
    assert ok, worst
