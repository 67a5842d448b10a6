"""GPU parity of the CUDA-core GEMV kernels against the oracle.

Every case compares each output element with the oracle's exact value under
|y - y_ref| <= 1e-3 * sum_k |x_k w_kn| + 1e-5, with outputs poisoned with NaN
beforehand (an unwritten element fails) and a canary tail after each output
(an out-of-bounds write fails).  Shapes cover several tiles and K-slices,
ragged column tiles, one-group K, M from 1 to 8, and the full workload sizes
in the launch configuration the benchmark times.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    import gpu_util  # imports the library: fails loudly when it is missing
    return gpu_util


def _tol(y, y_ref, a, out="f32", stated=False):
    """The tests' bar (tolerance.within); stated=True holds the output to the
    stated bound alone, with no allowance for rounding it to a bf16 output
    (random inputs with K large enough that |y| stays far below the magnitude sum)."""
    from tolerance import unit_roundoff, within, within_stated
    ok, worst = (within_stated(y, y_ref, a) if stated else within(y, y_ref, a, unit_roundoff(out)))
    assert ok, f"max |err|/bound = {worst:.3g}"
    return worst


# ------------------------------------------------------------------- int8 ----
WQ8_CASES = [(1, 128, 16, 128), (1, 512, 272, 128), (3, 1024, 512, 64), (8, 256, 48, 16),
             (2, 2048, 1040, 128), (1, 4096, 4096, 128), (5, 4096, 4096, 128)]


@pytest.mark.parametrize("M,K,N,g", WQ8_CASES)
def test_wq8_parity(G, M, K, N, g):
    import oracle
    import synthetic as syn
    d = syn.make_wq8(seed=1, M=M, K=K, N=N, group=g)
    y = G.run_wq8(d)
    y_ref, a = oracle.wq8_gemv(d["x"], d["w"], d["scales"], g)
    _tol(G.to_f64(y), y_ref, a)


def test_wq8_onehot_exact(G):
    """x = e_k returns fp32(s * q) exactly (one rounding of an exact product)."""
    import oracle
    import synthetic as syn
    d = syn.make_wq8(seed=7, M=1, K=1024, N=512, group=128)
    for k in (0, 127, 128, 513, 1023):
        d["x"] = np.zeros((1, 1024), np.float32)
        d["x"][0, k] = 1.0
        y = G.to_f64(G.run_wq8(d))
        y_ref, _ = oracle.wq8_gemv(d["x"], d["w"], d["scales"], 128)
        assert np.array_equal(y, y_ref.astype(np.float32).astype(np.float64)), k


# ------------------------------------------------------------------- 3-bit ----
WQ3_CASES = [(1, 32, 8), (1, 96, 136), (2, 1024, 1000), (8, 512, 256), (1, 4096, 4096), (3, 4096, 4096)]


@pytest.mark.parametrize("M,K,N", WQ3_CASES)
def test_wq3_parity(G, M, K, N):
    import oracle
    import synthetic as syn
    d = syn.make_wq3(seed=2, M=M, K=K, N=N)
    y = G.run_wq3(d)
    y_ref, a = oracle.wq3_gemv(d["x"].view(np.uint16), d["mat"], d["scales"].view(np.uint16),
                               d["zeros"].view(np.uint16))
    _tol(G.to_f64(y), y_ref, a, "f16")


# shapes that steer the 3-bit tensor-core kernel (M >= 3) and its plan: K not
# a multiple of the 128-value unit, N not a multiple of the 32-column slab, M
# between the MMA rows; K-slices over a cluster (small N, long K); column tiles
# in several waves (N beyond what one wave holds); and a pair-ordered x too
# large for shared memory (M = 8 at very long K), which goes to the CUDA-core
# kernel like every M <= 2
WQ3T_CASES = [(5, 96, 264), (7, 1056, 1000), (3, 4128, 520), (4, 16384, 256), (8, 16384, 256),
              (3, 64, 40960), (8, 131072, 64), (2, 4128, 520)]


@pytest.mark.parametrize("M,K,N", WQ3T_CASES)
def test_wq3_plan_shapes(G, M, K, N):
    import oracle
    import synthetic as syn
    d = syn.make_wq3(seed=4, M=M, K=K, N=N)
    y = G.to_f64(G.run_wq3(d))
    cols = None
    if N > 4096:
        r = np.random.default_rng(6)
        cols = np.unique(np.concatenate([np.arange(0, 256), np.arange(N - 256, N), r.integers(0, N, 512)]))
    y_ref, a = oracle.wq3_gemv(d["x"].view(np.uint16), d["mat"], d["scales"].view(np.uint16),
                               d["zeros"].view(np.uint16), cols=cols)
    _tol(y if cols is None else y[:, cols], y_ref, a, "f16")


W3_ADV_CASES = [(1, 4096, 4096, "same"), (8, 4096, 512, "same"), (1, 16384, 20480, "same"),
                (8, 16384, 1024, "same"), (1, 4096, 4096, "halves"), (1, 16384, 20480, "halves")]


@pytest.mark.parametrize("M,K,N,signs", W3_ADV_CASES)
def test_wq3_same_sign_large_x(G, M, K, N, signs):
    """Every activation of one sign and large (or +a / -a in alternating halves of
    each 32-value block) with random codes: no cancellation between terms, so any
    bias or offset the kernel adds and later removes shows up in full against the
    bar.  a = 60 at K = 4096 and 12 at K = 16384 (|y| stays inside the fp16
    range); N = 20480 gives enough column tiles that one CTA runs over all of K."""
    import oracle
    import synthetic as syn
    d = syn.make_wq3(seed=21, M=M, K=K, N=N)
    amp = 60.0 if K <= 4096 else 12.0
    x = np.full((M, K), amp, np.float16)
    if signs == "halves":
        x.reshape(M, K // 16, 16)[:, 1::2, :] = -amp
    d["x"] = x
    y = G.run_wq3(d)
    cols = None
    if N > 4096:
        r = np.random.default_rng(2)
        cols = np.unique(np.concatenate([np.arange(0, 128), np.arange(N - 128, N), r.integers(0, N, 256)]))
    y_ref, a = oracle.wq3_gemv(x.view(np.uint16), d["mat"], d["scales"].view(np.uint16), d["zeros"].view(np.uint16),
                               cols=cols)
    yv = G.to_f64(y)
    _tol(yv if cols is None else yv[:, cols], y_ref, a, "f16")


def test_wq3_onehot_exact(G):
    """Every code position of a block, including the straddling codes 10 and 21."""
    import oracle
    import synthetic as syn
    d = syn.make_wq3(seed=5, M=1, K=256, N=136)
    for k in list(range(32)) + [32 * 5 + 10, 32 * 7 + 21, 255]:
        x = np.zeros((1, 256), np.float16)
        x[0, k] = 1.0
        d["x"] = x
        y = G.bits_u16(G.run_wq3(d))
        y_ref, _ = oracle.wq3_gemv(x.view(np.uint16), d["mat"], d["scales"].view(np.uint16),
                                   d["zeros"].view(np.uint16))
        assert np.array_equal(y, oracle.round_f16(y_ref)), k


def test_wq3_tensor_core_onehot_exact(G):
    """The 3-bit tensor-core path (M >= 3) reads every code of a block through
    its pair cover (16 pairs from seven 32-bit windows): one-hot rows of x at
    all 32 positions of a block -- the straddling codes 10 and 21 included --
    and at a few other blocks return the dequantized weight rows rounded once."""
    import oracle
    import synthetic as syn
    d = syn.make_wq3(seed=7, M=8, K=512, N=264)
    positions = list(range(32)) + [32 * 3 + 10, 32 * 6 + 21, 32 * 9 + 31, 32 * 15 + 0, 511, 300, 129, 64]
    for c0 in range(0, len(positions), 8):
        x = np.zeros((8, 512), np.float16)
        for m, k in enumerate(positions[c0:c0 + 8]):
            x[m, k] = 1.0
        d["x"] = x
        y = G.bits_u16(G.run_wq3(d))
        y_ref, _ = oracle.wq3_gemv(x.view(np.uint16), d["mat"], d["scales"].view(np.uint16),
                                   d["zeros"].view(np.uint16))
        assert np.array_equal(y, oracle.round_f16(y_ref)), positions[c0:c0 + 8]


def test_tensor_core_paths_repeat_bit_identical_and_pdl(G):
    """The 3-bit tensor-core GEMM (M = 5) and the 4-bit n-tile GEMMs (M = 16,
    24): two runs and a run with programmatic dependent launch give identical
    bits (fixed summation order, no dependence on timing)."""
    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    d3 = syn.make_wq3(seed=8, M=5, K=4096, N=4096)
    a = G.bits_u16(G.run_wq3(d3))
    assert np.array_equal(a, G.bits_u16(G.run_wq3(d3)))
    assert np.array_equal(a, G.bits_u16(G.run_wq3(d3, flags=wq.WQ_FLAG_PDL)))
    for M in (16, 24):
        d4 = _make_wq4(M, 2048, 4096, 128, True, True, seed=9)
        b = G.bits_u16(G.run_wq4(d4))
        assert np.array_equal(b, G.bits_u16(G.run_wq4(d4)))
        assert np.array_equal(b, G.bits_u16(G.run_wq4(d4, flags=wq.WQ_FLAG_PDL)))


# ------------------------------------------------------------------- 4-bit ----
WQ4_CASES = [  # M, K, N, group, bf16, asym zeros
    (1, 256, 128, 32, False, True), (3, 512, 264, 128, True, False), (8, 1024, 520, 64, False, True),
    (2, 2048, 1032, 128, True, True), (1, 8192, 28672, 128, True, False), (8, 8192, 28672, 128, True, False),
    # K not a multiple of the 256-value stage, M between the tile sizes
    (1, 320, 136, 64, False, True), (5, 576, 200, 64, True, True), (7, 1088, 264, 64, False, False)]


def _make_wq4(M, K, N, g, bf16, asym, seed=4):
    import synthetic as syn
    if bf16 and not asym:
        return syn.make_wq4_sym(seed=seed, M=M, K=K, N=N, group=g)
    r = np.random.default_rng(seed)
    codes = r.integers(0, 16, (K, N), dtype=np.uint8)
    G_ = K // g
    s = r.uniform(0.002, 0.03, (G_, N)).astype(np.float32)
    x = syn.normal(seed, 1, (M, K), 1.0, np.float32)
    if bf16:
        xb, sb = syn.f32_to_bf16_bits(x), syn.f32_to_bf16_bits(s)
    else:
        xb, sb = x.astype(np.float16), s.astype(np.float16)
    z = r.integers(0, 16, (G_, N), dtype=np.uint8)
    return dict(x=xb, qweight=syn.pack4(codes), scales=sb, qzeros=syn.pack_zeros4(z) if asym else None,
                g_idx=None, M=M, K=K, N=N, group=g, act_bf16=int(bf16))


@pytest.mark.parametrize("M,K,N,g,bf16,asym", WQ4_CASES)
def test_wq4_parity(G, M, K, N, g, bf16, asym):
    d = _make_wq4(M, K, N, g, bf16, asym)
    y = G.run_wq4(d)
    cols = None
    if N > 4096:  # sampled columns: both ends of every tile edge region plus a random sample
        r = np.random.default_rng(0)
        cols = np.unique(np.concatenate([np.arange(0, 256), np.arange(N - 256, N), r.integers(0, N, 1024)]))
    y_ref, a = G.oracle_wq4(d, cols)
    yv = G.to_f64(y)
    _tol(yv if cols is None else yv[:, cols], y_ref, a, "bf16" if bf16 else "f16", stated=K >= 1024)


WQ4G_CASES = [(1, 256, 128, 32), (1, 1024, 392, 128), (4, 2048, 1024, 64), (1, 4096, 11008, 128),
              (2, 4096, 11008, 128), (8, 4096, 1024, 128)]


@pytest.mark.parametrize("M,K,N,g", WQ4G_CASES)
def test_wq4_actorder_parity(G, M, K, N, g):
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=3, M=M, K=K, N=N, group=g)
    y = G.run_wq4(d)
    y_ref, a = G.oracle_wq4(d)
    _tol(G.to_f64(y), y_ref, a, "f16")


@pytest.mark.parametrize("act_order", [False, True])
def test_wq4_onehot_exact(G, act_order):
    import oracle
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=9, M=1, K=512, N=264, group=128)
    if not act_order:
        d["g_idx"] = None
    for k in (0, 7, 8, 129, 300, 511):
        x = np.zeros((1, 512), np.float16)
        x[0, k] = 1.0
        d["x"] = x
        y = G.bits_u16(G.run_wq4(d))
        y_ref, _ = G.oracle_wq4(d)
        assert np.array_equal(y, oracle.round_f16(y_ref)), k


def test_wq4_onehot_exact_multirow(G):
    """M = 3 (tensor-core path): each row of x a different one-hot vector; y rows
    are the dequantized weight rows, rounded once (bit for bit)."""
    import oracle
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=9, M=3, K=512, N=264, group=128)
    d["g_idx"] = None
    x = np.zeros((3, 512), np.float16)
    for m, k in enumerate((5, 130, 511)):
        x[m, k] = 1.0
    d["x"] = x
    y = G.bits_u16(G.run_wq4(d))
    y_ref, _ = G.oracle_wq4(d)
    assert np.array_equal(y, oracle.round_f16(y_ref))


# ------------------------------------------------------------ invariants ----

def test_repeat_bit_identical_and_pdl(G):
    """Two runs, and a run with programmatic dependent launch, give identical bits."""
    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=3, M=1, K=4096, N=11008, group=128)
    y1 = G.bits_u16(G.run_wq4(d))
    y2 = G.bits_u16(G.run_wq4(d))
    y3 = G.bits_u16(G.run_wq4(d, flags=wq.WQ_FLAG_PDL))
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)
    d3 = syn.make_wq3(seed=2, M=1, K=4096, N=4096)
    assert np.array_equal(G.bits_u16(G.run_wq3(d3)), G.bits_u16(G.run_wq3(d3, flags=wq.WQ_FLAG_PDL)))


def test_decode_step_chain_matches_oracle(G):
    """The benchmark's launch configuration: two layers of [W4 act-order on
    sorted rows, W8, W3] at full size, chained with programmatic dependent
    launch in one CUDA graph and replayed twice; every output matches the oracle."""
    import torch
    import gemm_dequant_gemv_gb300 as wq
    import oracle
    import synthetic as syn
    layers = []
    for l in range(2):
        d8 = syn.make_wq8(seed=1000 * l + 1)
        d3 = syn.make_wq3(seed=1000 * l + 2)
        d4 = syn.make_wq4_actorder(seed=1000 * l + 3)
        t8 = {k: G.dev(d8[k]) for k in ("x", "w", "scales")}
        t3 = {k: G.dev(d3[k]) for k in ("x", "mat", "scales", "zeros")}
        t4 = {k: G.dev(d4[k]) for k in ("x", "qweight", "scales", "qzeros", "g_idx")}
        qs, perm = torch.empty_like(t4["qweight"]), torch.empty_like(t4["g_idx"])
        wq.wq4_actorder_prepare(t4["qweight"], t4["g_idx"], 4096, 11008, 128, qs, perm)
        y8 = torch.empty((1, 4096), dtype=torch.float32, device=G.DEV)
        y3 = torch.empty((1, 4096), dtype=torch.float16, device=G.DEV)
        y4 = torch.empty((1, 11008), dtype=torch.float16, device=G.DEV)
        layers.append((d8, d3, d4, t8, t3, t4, qs, perm, y8, y3, y4))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    P = wq.WQ_FLAG_PDL

    def step():
        for d8, d3, d4, t8, t3, t4, qs, perm, y8, y3, y4 in layers:
            wq.wq4_gemm_sorted(t4["x"], qs, t4["scales"], t4["qzeros"], perm, y4, 1, 4096, 11008, 128, wq.WQ_F16,
                               flags=P, stream=stream)
            wq.wq8_gemv(t8["x"], t8["w"], t8["scales"], y8, 1, 4096, 4096, 128, flags=P, stream=stream)
            wq.wq3_gemv(t3["x"], t3["mat"], t3["scales"], t3["zeros"], y3, 1, 4096, 4096, flags=P, stream=stream)

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        step()
    for _ in range(2):
        for L in layers:  # poison the outputs: the replay must rewrite every element
            for y in L[8:]:
                y.fill_(float("nan"))
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        for d8, d3, d4, t8, t3, t4, qs, perm, y8, y3, y4 in layers:
            r8, a8 = oracle.wq8_gemv(d8["x"], d8["w"], d8["scales"], 128)
            _tol(G.to_f64(y8), r8, a8, "f32")
            r3, a3 = oracle.wq3_gemv(d3["x"].view(np.uint16), d3["mat"], d3["scales"].view(np.uint16),
                                     d3["zeros"].view(np.uint16))
            _tol(G.to_f64(y3), r3, a3, "f16")
            r4, a4 = G.oracle_wq4(d4)
            _tol(G.to_f64(y4), r4, a4, "f16")
    assert wq.read_timeout_flag(clear=True) == 0


def test_no_timeouts(G):
    import gemm_dequant_gemv_gb300 as wq
    assert wq.read_timeout_flag(clear=True) == 0


# ------------------------------------------------------------------ M > 8 ----
# 9 .. 32 rows take the warp-level MMA kernel with two or four n-tiles (rows
# past M inside an n-tile read TMA zero fill); more rows the tcgen05 kernel in
# 64-row chunks, whose last chunk picks the 16-, 32- or 64-row instance
WQ4_MMA_CASES = [  # M, K, N, group, bf16, asym zeros
    (16, 8192, 28672, 128, True, False), (32, 8192, 28672, 128, True, False),
    (16, 256, 128, 64, True, False), (17, 512, 264, 128, False, True), (33, 1024, 392, 256, True, True),
    (9, 2048, 1024, 128, False, False), (50, 1024, 520, 64, True, False), (100, 512, 256, 128, False, True),
    # one K slice per CTA with 16 / 32 scale groups and stored zeros: the scales and
    # zeros fetched eight groups ahead cross several chunks (128-k and 64-k stages)
    (17, 2048, 20480, 128, False, True), (24, 2048, 20480, 64, True, True),
    (80, 512, 264, 128, True, False), (96, 1024, 136, 64, False, True), (31, 4096, 1056, 128, True, True)]


@pytest.mark.parametrize("M,K,N,g,bf16,asym", WQ4_MMA_CASES)
def test_wq4_mma_parity(G, M, K, N, g, bf16, asym):
    d = _make_wq4(M, K, N, g, bf16, asym, seed=11)
    y = G.run_wq4(d)
    cols = None
    if N > 4096:
        r = np.random.default_rng(1)
        cols = np.unique(np.concatenate([np.arange(0, 256), np.arange(N - 256, N), r.integers(0, N, 768)]))
    y_ref, a = G.oracle_wq4(d, cols)
    yv = G.to_f64(y)
    _tol(yv if cols is None else yv[:, cols], y_ref, a, "bf16" if bf16 else "f16", stated=K >= 1024)


def test_wq4_mma_onehot_exact(G):
    """One-hot rows of x through the tensor-core path return the dequantized weight rows
    exactly (integer A operand, scale applied once in fp32)."""
    import oracle
    d = _make_wq4(16, 512, 264, 128, True, True, seed=12)
    x = np.zeros((16, 512), np.float32)
    for m, k in enumerate((0, 7, 8, 63, 64, 127, 128, 200, 255, 256, 300, 383, 384, 450, 510, 511)):
        x[m, k] = 1.0
    import synthetic as syn
    d["x"] = syn.f32_to_bf16_bits(x)
    y = G.bits_u16(G.run_wq4(d))
    y_ref, _ = G.oracle_wq4(d)
    assert np.array_equal(y, oracle.round_bf16(y_ref))


# ------------------------------------------- act-order on group-sorted rows ----
WQ4S_CASES = [(1, 256, 128, 32), (1, 4096, 11008, 128), (3, 2048, 1032, 64), (8, 1024, 256, 128),
              (5, 704, 136, 64), (2, 4096, 11008, 128)]


@pytest.mark.parametrize("M,K,N,g", WQ4S_CASES)
def test_wq4_sorted_matches_actorder_oracle(G, M, K, N, g):
    """Prepared (row-sorted) weights + perm reproduce the act-order product of the
    original weights and g_idx; the repack itself is checked bit for bit."""
    import torch
    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=13, M=M, K=K, N=N, group=g)
    qw, gi = G.dev(d["qweight"]), G.dev(d["g_idx"])
    qs = torch.empty_like(qw)
    perm = torch.empty_like(gi)
    wq.wq4_actorder_prepare(qw, gi, K, N, g, qs, perm)
    p = perm.cpu().numpy()
    assert np.array_equal(np.sort(p), np.arange(K))
    assert np.array_equal(d["g_idx"][p], np.arange(K) // g)
    assert np.array_equal(qs.cpu().numpy(), syn.pack4(d["codes"][p]))
    x, sc, qz = G.dev(d["x"]), G.dev(d["scales"]), G.dev(d["qzeros"])
    buf, y = G.guarded((M, N), torch.float16)
    wq.wq4_gemm_sorted(x, qs, sc, qz, perm, y, M, K, N, g, wq.WQ_F16)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    y_ref, a = G.oracle_wq4(d)
    _tol(G.to_f64(y), y_ref, a, "f16")


@pytest.mark.parametrize("M", [1, 4])
def test_wq4_sorted_bf16(G, M):
    """The sorted act-order path with bf16 activations and scales (CUDA-core
    kernel at M = 1, tensor-core kernel at M = 4) against the act-order oracle."""
    import torch
    import gemm_dequant_gemv_gb300 as wq
    import synthetic as syn
    K, N, g = 1024, 392, 128
    d = syn.make_wq4_actorder(seed=17, M=M, K=K, N=N, group=g)
    xb = syn.f32_to_bf16_bits(d["x"].astype(np.float32))
    sb = syn.f32_to_bf16_bits(d["scales"].astype(np.float32))
    qw, gi = G.dev(d["qweight"]), G.dev(d["g_idx"])
    qs, perm = torch.empty_like(qw), torch.empty_like(gi)
    wq.wq4_actorder_prepare(qw, gi, K, N, g, qs, perm)
    buf, y = G.guarded((M, N), torch.bfloat16)
    wq.wq4_gemm_sorted(G.dev(xb), qs, G.dev(sb), G.dev(d["qzeros"]), perm, y, M, K, N, g, wq.WQ_BF16)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    import oracle
    y_ref, a = oracle.wq4_gemm(xb, 1, d["qweight"], sb, d["qzeros"], d["g_idx"], g)
    _tol(G.to_f64(y), y_ref, a, "bf16")


def test_wq4_prepare_rejects_unequal_groups(G):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    K, N, g = 256, 128, 64
    gi = np.repeat(np.arange(K // g), g).astype(np.int32)
    gi[0], gi[-1] = 1, 1   # group 0 loses a row, group 1 gains one
    qw = torch.zeros((K // 8, N), dtype=torch.int32, device=G.DEV)
    qs, perm = torch.empty_like(qw), torch.empty(K, dtype=torch.int32, device=G.DEV)
    with pytest.raises(wq.WQError) as e:
        wq.wq4_actorder_prepare(qw, G.dev(gi), K, N, g, qs, perm)
    assert e.value.status == wq.WQ_ERR_SHAPE
