"""Pins that tie the oracle to facts outside itself.

Each pin_* function raises AssertionError when the oracle disagrees with:
  * a hand-worked value (tests/golden/*, each with its derivation and source),
  * a library routine the definition reduces to in a special case
    (numpy float64 / int64 matmul, numpy's IEEE half conversion),
  * an invariant of the mathematics (linearity, permutation of the summation
    index, homogeneity in the scales, group/column equivalences).

They are plain functions so that the mutation test can run them against
oracle builds with a planted mistake and check that at least one pin fails.
"""
import numpy as np

import oracle
import synthetic as syn
from conftest import read_golden


def _golden_map(name):
    return {r[0]: r[1:] for r in read_golden(name)}


def _rng(seed):
    return np.random.default_rng(seed)


def _f16_bits(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16)


# ---------------------------------------------------------------- formats ----

def pin_pack3_words():
    for label, codes, words in read_golden("pack3_words.txt"):
        c = np.array([int(v) for v in codes.split()], dtype=np.uint8).reshape(32, 1)
        want = np.array([int(w, 16) for w in words.split()], dtype=np.uint64).astype(np.uint32).view(np.int32)
        got = syn.pack3(c).reshape(3)
        assert np.array_equal(got, want), (label, got, want)
        dec = oracle.unpack3(want.reshape(3, 1), 32, 1).reshape(32)
        assert np.array_equal(dec, c.reshape(32)), (label, dec)


def pin_pack4_words():
    for kind, codes, word in read_golden("pack4_words.txt"):
        c = np.array([int(v) for v in codes.split()], dtype=np.uint8)
        want = np.array([int(word, 16)], dtype=np.uint64).astype(np.uint32).view(np.int32)
        if kind == "weight":
            got = syn.pack4(c.reshape(8, 1)).reshape(1)
            dec = oracle.unpack4(want.reshape(1, 1), 8, 1).reshape(8)
        else:
            got = syn.pack_zeros4(c.reshape(1, 8)).reshape(1)
            dec = oracle.unpack_zeros4(want.reshape(1, 1), 1, 8).reshape(8)
        assert np.array_equal(got, want), (kind, codes, got, want)
        assert np.array_equal(dec, c), (kind, codes, dec)


def pin_pack_roundtrip():
    r = _rng(11)
    for K, N in ((32, 8), (64, 24), (256, 40)):
        c3 = r.integers(0, 8, (K, N), dtype=np.uint8)
        assert np.array_equal(oracle.unpack3(syn.pack3(c3), K, N), c3)
        c4 = r.integers(0, 16, (K, N), dtype=np.uint8)
        assert np.array_equal(oracle.unpack4(syn.pack4(c4), K, N), c4)
        z = r.integers(0, 16, (K // 8, N), dtype=np.uint8)
        assert np.array_equal(oracle.unpack_zeros4(syn.pack_zeros4(z), K // 8, N), z)


def pin_code3_exhaustive():
    """Every value at every one of the 32 positions of a block, alone."""
    for j in range(32):
        for v in range(8):
            c = np.zeros((32, 1), dtype=np.uint8)
            c[j, 0] = v
            mat = syn.pack3(c)
            # the bit-stream value of the block must be v << 3j
            stream = sum(int(np.uint32(mat[i, 0])) << (32 * i) for i in range(3))
            assert stream == v << (3 * j), (j, v)
            assert np.array_equal(oracle.unpack3(mat, 32, 1), c), (j, v)


def pin_scalar_formats():
    # hand-checked binary16 / bfloat16 patterns
    cases16 = {0x3C00: 1.0, 0xC000: -2.0, 0x7BFF: 65504.0, 0x0001: 2.0 ** -24,
               0x0400: 2.0 ** -14, 0x3555: 0.333251953125, 0x0000: 0.0}
    for b, v in cases16.items():
        assert oracle.f16_to_double(b) == v, hex(b)
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0x4049) == 3.140625
    assert oracle.bf16_to_double(0xC2F7) == -123.5
    # rounding: ties to even, overflow, subnormal
    r16 = {1 + 2.0 ** -11: 0x3C00, 1 + 3 * 2.0 ** -11: 0x3C02, 65520.0: 0x7C00,
           65519.99: 0x7BFF, 2.0 ** -25: 0x0000, 3 * 2.0 ** -25: 0x0002, -1.5: 0xBE00}
    for v, b in r16.items():
        assert oracle.double_to_f16(v) == b, (v, hex(oracle.double_to_f16(v)))
    rb = {1 + 2.0 ** -8: 0x3F80, 1 + 3 * 2.0 ** -8: 0x3F82, -3.140625: 0xC049}
    for v, b in rb.items():
        assert oracle.double_to_bf16(v) == b, (v, hex(oracle.double_to_bf16(v)))
    # library pin: numpy's IEEE double -> half conversion on many values
    r = _rng(12)
    vals = np.concatenate([r.normal(0, 1, 3000), r.normal(0, 1e-5, 500), r.normal(0, 2e4, 500)])
    vals = vals[np.abs(vals) < 65504]
    ours = oracle.round_f16(vals)
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    back = oracle.decode_f16(ref)
    assert np.array_equal(back, ref.view(np.float16).astype(np.float64))
    # bf16 of float32-representable values: the round-to-nearest-even bit trick
    f = r.normal(0, 10, 4000).astype(np.float32)
    assert np.array_equal(oracle.round_bf16(f.astype(np.float64)), syn.f32_to_bf16_bits(f))


# ------------------------------------------------------------------- wq8 ----

def pin_wq8_hand():
    want = [float(v) for v in _golden_map("products_small.txt")["wq8"][0].split()]
    q = np.array([[1, -2], [3, 4], [-5, 6], [7, -8]], dtype=np.int8)
    s = np.array([[0.5, 0.25], [2, 1]], dtype=np.float32)
    x = np.array([[1, 2, 3, 4]], dtype=np.float32)
    y, _ = oracle.wq8_gemv(x, q, s, 2)
    assert y.tolist() == [want], (y, want)


def pin_wq8_library():
    """Unit scales reduce to an integer-matrix product (numpy float64 matmul)."""
    r = _rng(13)
    M, K, N, g = 3, 256, 40, 64
    x = r.normal(0, 1, (M, K)).astype(np.float32)
    q = r.integers(-127, 128, (K, N), dtype=np.int8)
    y, a = oracle.wq8_gemv(x, q, np.ones((K // g, N), np.float32), g)
    ref = x.astype(np.float64) @ q.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9)
    assert np.allclose(a, np.abs(x.astype(np.float64)) @ np.abs(q.astype(np.float64)), rtol=1e-12)
    # one scale per group: multiplying group 1's scales by 4 adds 3x its partial product
    s = np.ones((K // g, N), np.float32)
    s[1] = 4.0
    y2, _ = oracle.wq8_gemv(x, q, s, g)
    part = x[:, g:2 * g].astype(np.float64) @ q[g:2 * g].astype(np.float64)
    assert np.allclose(y2, ref + 3 * part, rtol=1e-12, atol=1e-9)


def pin_wq8_invariants():
    r = _rng(14)
    M, K, N, g = 2, 256, 24, 128
    d = syn.make_wq8(seed=3, M=M, K=K, N=N, group=g)
    y, _ = oracle.wq8_gemv(d["x"], d["w"], d["scales"], g)
    # homogeneity in the scales and linearity in x (dyadic x: every sum is exact)
    y2, _ = oracle.wq8_gemv(d["x"], d["w"], d["scales"] * np.float32(2), g)
    assert np.allclose(y2, 2 * y, rtol=1e-12, atol=1e-12)
    x1 = (r.integers(-64, 64, (M, K)) / 16).astype(np.float32)
    x2 = (r.integers(-64, 64, (M, K)) / 16).astype(np.float32)
    y1, _ = oracle.wq8_gemv(x1, d["w"], d["scales"], g)
    ya, _ = oracle.wq8_gemv(x2, d["w"], d["scales"], g)
    yb, _ = oracle.wq8_gemv(x1 + x2, d["w"], d["scales"], g)
    assert np.allclose(yb, y1 + ya, rtol=1e-12, atol=1e-12)
    # group = K equals one scale per column
    s_col = r.uniform(0.01, 0.02, (1, N)).astype(np.float32)
    yk, _ = oracle.wq8_gemv(d["x"], d["w"], s_col, K)
    ref = (d["x"].astype(np.float64) @ d["w"].astype(np.float64)) * s_col.astype(np.float64)
    assert np.allclose(yk, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- wq3 ----

def pin_wq3_hand():
    gm = _golden_map("products_small.txt")
    j = np.arange(32)
    codes = np.stack([j % 8, 7 - (j % 8)], axis=1).astype(np.uint8)
    mat = syn.pack3(codes)
    s = _f16_bits([0.5, 0.25]); z = _f16_bits([0.25, 1.0])
    y, _ = oracle.wq3_gemv(_f16_bits(np.ones((1, 32))), mat, s, z)
    assert y.tolist() == [[float(v) for v in gm["wq3_ones"][0].split()]], y
    e = np.zeros((1, 32)); e[0, 10] = 1
    y, _ = oracle.wq3_gemv(_f16_bits(e), mat, s, z)
    assert y.tolist() == [[float(v) for v in gm["wq3_e10"][0].split()]], y


def pin_wq3_library():
    """scale 1, zero 0: y = x . codes (numpy float64 matmul)."""
    r = _rng(15)
    M, K, N = 3, 256, 24
    codes = r.integers(0, 8, (K, N), dtype=np.uint8)
    x = r.normal(0, 1, (M, K)).astype(np.float16)
    y, a = oracle.wq3_gemv(x.view(np.uint16), syn.pack3(codes), _f16_bits(np.ones(N)), _f16_bits(np.zeros(N)))
    ref = x.astype(np.float64) @ codes.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9)
    # the stored zero enters once per row with a minus sign: y(zero=c) = y - c * sum_k x_k
    y2, _ = oracle.wq3_gemv(x.view(np.uint16), syn.pack3(codes), _f16_bits(np.ones(N)), _f16_bits(np.full(N, 0.5)))
    assert np.allclose(y2, ref - 0.5 * x.astype(np.float64).sum(axis=1, keepdims=True), rtol=1e-12, atol=1e-9)
    # per-column scales multiply columns
    s = r.uniform(0.005, 0.02, N).astype(np.float16)
    y3, _ = oracle.wq3_gemv(x.view(np.uint16), syn.pack3(codes), s.view(np.uint16), _f16_bits(np.zeros(N)))
    assert np.allclose(y3, ref * s.astype(np.float64)[None, :], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------- wq4 ----

def _wq4_hand_inputs(act_order):
    K, N, g = 16, 8, 8
    codes = np.zeros((K, N), dtype=np.uint8)
    codes[:8, 0] = 3; codes[8:, 0] = 12
    codes[:, 7] = np.arange(16)
    s = np.ones((2, N)); s[0, 0] = 0.5; s[0, 7] = 2; s[1, 0] = 0.25; s[1, 7] = 1
    z = np.zeros((2, N), dtype=np.uint8); z[0, 0] = 1; z[1, 0] = 8; z[1, 7] = 15
    x = np.ones((1, K)); x[0, 8:] = 2
    g_idx = (np.arange(K) // g).astype(np.int32)
    if act_order:
        g_idx[0], g_idx[8] = 1, 0
    return (_f16_bits(x), syn.pack4(codes), _f16_bits(s), syn.pack_zeros4(z), g_idx, g)


def pin_wq4_hand():
    gm = _golden_map("products_small.txt")
    for key, ao in (("wq4_plain", False), ("wq4_actorder", True)):
        x, qw, s, qz, gi, g = _wq4_hand_inputs(ao)
        y, _ = oracle.wq4_gemm(x, 0, qw, s, qz, gi if ao else None, g)
        want = [float(v) for v in gm[key][0].split()]
        assert [y[0, 0], y[0, 7]] == want, (key, y)
        assert np.all(y[0, 1:7] == 0), (key, y)


def pin_wq4_library():
    """unit scales, zero 0: y = x . codes; zero 8 (symmetric) subtracts 8 * sum_k x."""
    r = _rng(16)
    M, K, N, g = 2, 256, 16, 64
    codes = r.integers(0, 16, (K, N), dtype=np.uint8)
    x = r.normal(0, 1, (M, K)).astype(np.float16)
    xd = x.astype(np.float64)
    ones = _f16_bits(np.ones((K // g, N)))
    y, _ = oracle.wq4_gemm(x.view(np.uint16), 0, syn.pack4(codes), ones,
                           syn.pack_zeros4(np.zeros((K // g, N), np.uint8)), None, g)
    ref = xd @ codes.astype(np.float64)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9)
    ysym, _ = oracle.wq4_gemm(x.view(np.uint16), 0, syn.pack4(codes), ones, None, None, g)
    assert np.allclose(ysym, ref - 8 * xd.sum(axis=1, keepdims=True), rtol=1e-12, atol=1e-9)
    # qzeros all 8 is the same as the symmetric (NULL) form, bit for bit
    y8, _ = oracle.wq4_gemm(x.view(np.uint16), 0, syn.pack4(codes), ones,
                            syn.pack_zeros4(np.full((K // g, N), 8, np.uint8)), None, g)
    assert np.array_equal(y8, ysym)


def pin_wq4_invariants():
    r = _rng(17)
    M, K, N, g = 2, 512, 16, 128
    G = K // g
    codes = r.integers(0, 16, (K, N), dtype=np.uint8)
    z = r.integers(0, 16, (G, N), dtype=np.uint8)
    s = r.uniform(0.005, 0.05, (G, N)).astype(np.float16)
    x = r.normal(0, 1, (M, K)).astype(np.float16)
    xb, qw, sb, qz = x.view(np.uint16), syn.pack4(codes), s.view(np.uint16), syn.pack_zeros4(z)
    y, _ = oracle.wq4_gemm(xb, 0, qw, sb, qz, None, g)
    # identity act-order equals no act-order, bit for bit
    yid, _ = oracle.wq4_gemm(xb, 0, qw, sb, qz, (np.arange(K) // g).astype(np.int32), g)
    assert np.array_equal(y, yid)
    # permuting the summation index (x columns, weight rows, g_idx together)
    perm = syn.permutation(7, 1, K)
    gi = syn.gidx_from_permutation(perm, g)
    ya, _ = oracle.wq4_gemm(xb, 0, qw, sb, qz, gi, g)
    p2 = r.permutation(K)
    yb, _ = oracle.wq4_gemm(np.ascontiguousarray(xb[:, p2]), 0, syn.pack4(codes[p2]), sb, qz,
                            np.ascontiguousarray(gi[p2]), g)
    assert np.allclose(ya, yb, rtol=1e-12, atol=1e-12)
    # group = K equals per-column scale and zero
    s1 = s[:1]; z1 = z[:1]
    yk, _ = oracle.wq4_gemm(xb, 0, qw, s1.view(np.uint16), syn.pack_zeros4(z1), None, K)
    ref = (x.astype(np.float64) @ (codes.astype(np.float64) - z1.astype(np.float64))) * s1.astype(np.float64)
    assert np.allclose(yk, ref, rtol=1e-12, atol=1e-12)
    # bf16 activations and scales decode through their own format
    xb16 = syn.f32_to_bf16_bits(x.astype(np.float32))
    sb16 = syn.f32_to_bf16_bits(np.full((G, N), 0.5, np.float32))
    yb16, _ = oracle.wq4_gemm(xb16, 1, qw, sb16, None, None, g)
    xv16 = syn.bf16_bits_to_f32(xb16).astype(np.float64)
    ref = 0.5 * (xv16 @ (codes.astype(np.float64) - 8))
    assert np.allclose(yb16, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- smoothquant ----

def pin_w8a8_smooth():
    """Smoothquant's activation division: s = 1 is the plain quantizer bit for bit;
    powers of two scale X exactly, so the result is the plain quantizer applied to
    X * 2^-e (numpy, exact in bf16); an outlier channel divided by a large s no
    longer sets the row scale."""
    r = _rng(23)
    M, K = 6, 256
    Xf = r.normal(0, 1, (M, K)).astype(np.float32)
    Xf[:, 17] = np.where(np.arange(M) % 2 == 0, 100.0, -100.0)  # an outlier channel
    X = syn.f32_to_bf16_bits(Xf)
    Xq0, Sx0 = oracle.w8a8_quant_rows(X)
    Xq1, Sx1 = oracle.w8a8_quant_rows_smooth(X, np.ones(K, np.float32))
    assert np.array_equal(Xq0, Xq1) and np.array_equal(Sx0.view(np.uint32), Sx1.view(np.uint32))
    e = r.integers(-3, 4, K)
    s = (2.0 ** e).astype(np.float32)
    Xs = syn.f32_to_bf16_bits(syn.bf16_bits_to_f32(X) / s)   # exact: a power-of-two rescale
    Xq2, Sx2 = oracle.w8a8_quant_rows(Xs)
    Xq3, Sx3 = oracle.w8a8_quant_rows_smooth(X, s)
    assert np.array_equal(Xq2, Xq3) and np.array_equal(Sx2.view(np.uint32), Sx3.view(np.uint32))
    s_out = np.ones(K, np.float32)
    s_out[17] = 64.0
    _, Sx4 = oracle.w8a8_quant_rows_smooth(X, s_out)
    assert np.all(Sx4 < Sx0), (Sx4, Sx0)


# ------------------------------------------------------------------ LLM.int8() ----

def pin_w8a8_outlier():
    """LLM.int8(): no column above the threshold is the plain W8A8 path bit for bit;
    every column above it is the 16-bit product X . (Sw W) (numpy float64); a value
    equal to the threshold is not an outlier (strictly greater); in general the
    result is the plain path on X with the outlier columns zeroed plus the
    16-bit product over those columns (numpy)."""
    r = _rng(29)
    M, K, N = 5, 128, 24
    Xf = r.normal(0, 1, (M, K)).astype(np.float32)
    Xf[2, 9] = 6.0                         # equal to the threshold: regular
    Xf[1, 40] = -7.5                       # above it: column 40 is an outlier
    Xf[3, 100] = 12.0                      # column 100 too
    X = syn.f32_to_bf16_bits(Xf)
    W = r.integers(-127, 128, (K, N), dtype=np.int8)
    Sw = r.uniform(0.001, 0.01, N).astype(np.float32)
    xv = syn.bf16_bits_to_f32(X).astype(np.float64)
    wv = W.astype(np.float64) * Sw.astype(np.float64)[None, :]
    flags, Xq, Sx, acc, y, a, ovf = oracle.w8a8_outlier(X, W, Sw, np.inf)
    Xq0, Sx0, acc0, y0, a0, _ = oracle.w8a8_gemm(X, W, Sw)
    assert not flags.any() and np.array_equal(Xq, Xq0) and np.array_equal(acc, acc0) and np.array_equal(y, y0)
    flags, Xq, Sx, acc, y, a, ovf = oracle.w8a8_outlier(X, W, Sw, -1.0)
    assert flags.all() and not Xq.any() and not acc.any()
    assert np.allclose(y, xv @ wv, rtol=1e-12, atol=1e-15)
    flags, Xq, Sx, acc, y, a, ovf = oracle.w8a8_outlier(X, W, Sw, 6.0)
    assert sorted(np.nonzero(flags)[0].tolist()) == [40, 100], np.nonzero(flags)
    Xm = X.copy()
    Xm[:, [40, 100]] = 0
    _, _, acc_m, y_m, _, _ = oracle.w8a8_gemm(Xm, W, Sw)
    assert np.array_equal(acc, acc_m)
    assert np.allclose(y, y_m + xv[:, [40, 100]] @ wv[[40, 100]], rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------- dequantization ----

def pin_dequant_hand():
    """The hand-worked products, recomputed as x . (dense dequantized W) with numpy."""
    gm = _golden_map("products_small.txt")
    q = np.array([[1, -2], [3, 4], [-5, 6], [7, -8]], dtype=np.int8)
    s = np.array([[0.5, 0.25], [2, 1]], dtype=np.float32)
    x = np.array([[1, 2, 3, 4]], dtype=np.float64)
    assert (x @ oracle.wq8_dequant(q, s, 2)).tolist() == [[float(v) for v in gm["wq8"][0].split()]]
    j = np.arange(32)
    codes3 = np.stack([j % 8, 7 - (j % 8)], axis=1).astype(np.uint8)
    w3 = oracle.wq3_dequant(syn.pack3(codes3), _f16_bits([0.5, 0.25]), _f16_bits([0.25, 1.0]), 32)
    assert w3.sum(axis=0).tolist() == [float(v) for v in gm["wq3_ones"][0].split()]
    assert w3[10].tolist() == [float(v) for v in gm["wq3_e10"][0].split()]
    for key, ao in (("wq4_plain", False), ("wq4_actorder", True)):
        xb, qw, sb, qz, gi, g = _wq4_hand_inputs(ao)
        w4 = oracle.wq4_dequant(0, qw, sb, qz, gi if ao else None, g)
        y = np.asarray(xb, np.uint16).view(np.float16).astype(np.float64) @ w4
        assert [y[0, 0], y[0, 7]] == [float(v) for v in gm[key][0].split()], (key, y)


def pin_dequant_closed_forms():
    """Against the hand-worked packed words and the generator's own codes:
    w = s * (q - z) (4-bit), s * q - zero (3-bit), s[g_idx[k]] rows (act-order)."""
    zrow = [r for r in read_golden("pack4_words.txt") if r[0] == "zeros"][0]
    zeros = np.array([int(v) for v in zrow[1].split()], dtype=np.float64)  # columns 0..7
    zword = np.array([int(zrow[2], 16)], dtype=np.uint64).astype(np.uint32).view(np.int32).reshape(1, 1)
    for kind, codes, word in read_golden("pack4_words.txt"):
        if kind != "weight":
            continue
        c = np.array([int(v) for v in codes.split()], dtype=np.float64)
        wd = np.array([int(word, 16)], dtype=np.uint64).astype(np.uint32).view(np.int32)
        qw = np.repeat(wd.reshape(1, 1), 8, axis=1)
        got = oracle.wq4_dequant(0, qw, _f16_bits(np.full((1, 8), 0.5)), zword, None, 8)
        assert np.array_equal(got, 0.5 * (c[:, None] - zeros[None, :])), (codes, got)
    for label, codes, words in read_golden("pack3_words.txt"):
        c = np.array([int(v) for v in codes.split()], dtype=np.float64)
        wd = np.array([int(w, 16) for w in words.split()], dtype=np.uint64).astype(np.uint32).view(np.int32)
        got = oracle.wq3_dequant(wd.reshape(3, 1), _f16_bits([0.25]), _f16_bits([0.125]), 32)
        assert np.array_equal(got[:, 0], 0.25 * c - 0.125), label
    r = _rng(21)
    K, N, g = 64, 16, 16
    G = K // g
    codes = r.integers(0, 16, (K, N), dtype=np.uint8)
    z = r.integers(0, 16, (G, N), dtype=np.uint8)
    s = r.uniform(0.005, 0.05, (G, N)).astype(np.float16)
    gi = syn.gidx_from_permutation(syn.permutation(5, 1, K), g)
    got = oracle.wq4_dequant(0, syn.pack4(codes), s.view(np.uint16), syn.pack_zeros4(z), gi, g)
    want = s.astype(np.float64)[gi] * (codes.astype(np.float64) - z.astype(np.float64)[gi])
    assert np.array_equal(got, want)
    q8 = r.integers(-128, 128, (K, N), dtype=np.int8)
    s8 = r.uniform(0.01, 0.02, (G, N)).astype(np.float32)
    got8 = oracle.wq8_dequant(q8, s8, g)
    assert np.array_equal(got8, np.repeat(s8.astype(np.float64), g, axis=0) * q8.astype(np.float64))


# ------------------------------------------------------------------ w8a8 ----

def pin_w8a8_hand():
    gm = _golden_map("products_small.txt")
    X = syn.f32_to_bf16_bits(np.array([[15.875, -1.0625, 0.1875, -0.0625, 3.0]], np.float32))
    Xq, Sx = oracle.w8a8_quant_rows(X)
    assert Sx.tolist() == [0.125]
    assert Xq.ravel().tolist() == [int(v) for v in gm["w8a8_xq"][0].split()], Xq
    W = np.array([[2], [-1], [3], [5], [-4]], np.int8)
    acc, y, a, ovf = oracle.w8a8_gemm_rows(Xq, Sx, W, np.array([0.5], np.float32))
    assert acc.ravel().tolist() == [int(gm["w8a8_acc"][0])]
    assert y.ravel().tolist() == [float(gm["w8a8_y"][0])]
    assert not ovf


def pin_w8a8_quant_properties():
    r = _rng(18)
    M, K = 16, 300
    Xf = r.normal(0, 1, (M, K)).astype(np.float32)
    Xf[3] = 0.0                          # an all-zero row
    Xf[5, 17] = -40.0                    # a negative extreme
    X = syn.f32_to_bf16_bits(Xf)
    Xv = syn.bf16_bits_to_f32(X).astype(np.float64)
    Xq, Sx = oracle.w8a8_quant_rows(X)
    assert Sx[3] == 0 and np.all(Xq[3] == 0)
    assert np.all(np.abs(Xq.astype(np.int32)) <= 127)
    amax = np.abs(Xv).max(axis=1)
    assert np.array_equal(Sx, (amax.astype(np.float32) / np.float32(127)).astype(np.float32))
    for m in range(M):
        if Sx[m] == 0:
            continue
        i = int(np.argmax(np.abs(Xv[m])))
        assert abs(int(Xq[m, i])) == 127 and np.sign(Xq[m, i]) == np.sign(Xv[m, i])
        # half a code step, plus the fp32 rounding of X / Sx (at most 127 * 2^-24)
        err = np.abs(Sx[m] * Xq[m].astype(np.float64) - Xv[m])
        assert np.all(err <= Sx[m] * (0.5 + 2.0 ** -16)), m
    assert Xq[5, 17] == -127


def pin_w8a8_library():
    """The integer product equals numpy's int64 matmul; y = Sx * acc * Sw."""
    r = _rng(19)
    M, K, N = 6, 512, 48
    Xq = r.integers(-127, 128, (M, K), dtype=np.int8)
    W = r.integers(-127, 128, (K, N), dtype=np.int8)
    Sx = r.uniform(0.001, 0.1, M).astype(np.float32)
    Sw = r.uniform(0.001, 0.1, N).astype(np.float32)
    acc, y, a, ovf = oracle.w8a8_gemm_rows(Xq, Sx, W, Sw)
    ref = Xq.astype(np.int64) @ W.astype(np.int64)
    assert np.array_equal(acc, ref) and not ovf
    assert np.allclose(y, Sx[:, None].astype(np.float64) * ref * Sw[None, :].astype(np.float64), rtol=1e-15)
    # row subset returns the same rows
    acc2, _, _, _ = oracle.w8a8_gemm_rows(Xq, Sx, W, Sw, rows=[5, 0])
    assert np.array_equal(acc2, ref[[5, 0]])
    # adversarial magnitudes: all +-127 still fit int32 at K = 8192
    Xq = np.full((1, 8192), -127, np.int8); W = np.full((8192, 2), -127, np.int8)
    acc3, _, _, ovf3 = oracle.w8a8_gemm_rows(Xq, np.ones(1, np.float32), W, np.ones(2, np.float32))
    assert acc3[0, 0] == 8192 * 127 * 127 and not ovf3


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
