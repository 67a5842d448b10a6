"""The tiled 4-bit layout of wq4_repack_tiled / wq4_gemm_tiled.

CPU: the layout formula (written out in synthetic.tile4_index from the
header's definition) is a bijection, hand-worked word positions land where
the formula says, and the oracle's own unpacker reads the original codes back
from untiled words bit for bit; the argument checks of both entry points
return before any CUDA call.

GPU: the repack kernel writes exactly the formula's layout (plain, and with
the rows sorted by act-order group), and wq4_gemm_tiled matches the oracle
under the tests' bar (|y - y_ref| <= 1e-3 * sum_k |x_k w_kn| + 1e-5, plus the
bf16 output rounding only where it alone exceeds half of that) for several
tiles, K-slices and a ragged last stage, M = 1 .. 8, fp16 and bf16, symmetric
and stored zeros, and at the full workload sizes.
"""
import numpy as np
import pytest

A = 0x7f0000000000
MIS = A + 4


def test_tile_index_is_a_bijection_with_hand_worked_positions():
    import synthetic as syn
    K, N = 128, 96
    idx = syn.tile4_index(K, N)
    assert idx.shape == (K // 8, N)
    assert np.array_equal(np.sort(idx.ravel()), np.arange(K // 8 * N))
    # worked by hand from the header's formula (K = 128: two 64-value units; N = 96: three slabs)
    assert idx[0, 0] == 0
    assert idx[9, 37] == (1 * 3 + 1) * 256 + 1 * 128 + (4 * 1 + 0) * 4 + 1 == 1169
    assert idx[15, 31] == (1 * 3 + 0) * 256 + 1 * 128 + (4 * 7 + 3) * 4 + 3 == 1023
    assert idx[6, 95] == (0 * 3 + 2) * 256 + 0 * 128 + (4 * 7 + 3) * 4 + 3 == 639
    # one 1 KB block = one unit of one slab: rows 8u .. 8u+7, columns 32s .. 32s+31
    blk = idx[8:16, 32:64]
    assert blk.min() == (1 * 3 + 1) * 256 and blk.max() == (1 * 3 + 1) * 256 + 255


def test_untiled_words_unpack_to_the_original_codes():
    import oracle
    import synthetic as syn
    r = np.random.default_rng(3)
    K, N = 256, 96
    codes = r.integers(0, 16, (K, N), dtype=np.uint8)
    qw = syn.pack4(codes)
    tiled = syn.tile4(qw)
    assert tiled.size == qw.size and not np.array_equal(tiled, qw.ravel())
    back = syn.untile4(tiled, K, N)
    assert np.array_equal(back, qw)
    assert np.array_equal(oracle.unpack4(back, K, N), codes)


def test_tiled_entry_points_reject_before_any_cuda_call():
    import gemm_dequant_gemv_gb300 as wq
    lib = wq.library()
    rp = lib.wq4_repack_tiled
    assert rp(0, None, 128, 64, 64, A, None, None) == wq.WQ_ERR_NULL
    assert rp(A, A, 128, 64, 64, A, None, None) == wq.WQ_ERR_NULL        # g_idx without perm
    assert rp(A, None, 96, 64, 64, A, None, None) == wq.WQ_ERR_SHAPE     # K % 64
    assert rp(A, None, 128, 48, 64, A, None, None) == wq.WQ_ERR_SHAPE    # N % 32
    assert rp(A, None, 128, 64, 32, A, None, None) == wq.WQ_ERR_SHAPE    # group % 64
    assert rp(MIS, None, 128, 64, 64, A, None, None) == wq.WQ_ERR_ALIGN
    g = lib.wq4_gemm_tiled
    args = [A, A, A, None, None, A, 1, 128, 64, 64, wq.WQ_F16, 0, None]
    assert g(*([0] + args[1:])) == wq.WQ_ERR_NULL
    b = list(args); b[6] = 9
    assert g(*b) == wq.WQ_ERR_SHAPE                                      # M <= 8
    b = list(args); b[8] = 40
    assert g(*b) == wq.WQ_ERR_SHAPE                                      # N % 32
    b = list(args); b[9] = 32
    assert g(*b) == wq.WQ_ERR_SHAPE                                      # group % 64
    b = list(args); b[10] = 7
    assert g(*b) == wq.WQ_ERR_UNSUPPORTED
    b = list(args); b[1] = MIS
    assert g(*b) == wq.WQ_ERR_ALIGN


# ---------------------------------------------------------------------- GPU --

def _repack(G, d, act_order):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    K, N, g = d["K"], d["N"], d["group"]
    qw = G.dev(d["qweight"])
    tiled = torch.empty(K // 8 * N, dtype=torch.int32, device=G.DEV)
    perm = None
    if act_order:
        perm = torch.empty(K, dtype=torch.int32, device=G.DEV)
        wq.wq4_repack_tiled(qw, G.dev(d["g_idx"]), K, N, g, tiled, perm)
    else:
        wq.wq4_repack_tiled(qw, None, K, N, g, tiled, None)
    torch.cuda.synchronize()
    return tiled, perm


@pytest.mark.gpu
@pytest.mark.parametrize("act_order", [False, True])
def test_repack_writes_the_documented_layout(act_order):
    import gpu_util as G
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=23, M=1, K=1024, N=352, group=128)
    tiled, perm = _repack(G, d, act_order)
    got = tiled.cpu().numpy()
    if act_order:
        p = perm.cpu().numpy()
        assert np.array_equal(np.sort(p), np.arange(d["K"]))
        assert np.array_equal(d["g_idx"][p], np.arange(d["K"]) // d["group"])
        want = syn.tile4(syn.pack4(d["codes"][p]))
    else:
        want = syn.tile4(d["qweight"])
    assert np.array_equal(got, want)


def _run_tiled(G, d, tiled, perm, flags=0):
    import torch
    import gemm_dequant_gemv_gb300 as wq
    M, K, N, g = d["M"], d["K"], d["N"], d["group"]
    act = wq.WQ_BF16 if d["act_bf16"] else wq.WQ_F16
    qz = None if d["qzeros"] is None else G.dev(d["qzeros"])
    buf, y = G.guarded((M, N), torch.bfloat16 if d["act_bf16"] else torch.float16)
    wq.wq4_gemm_tiled(G.dev(d["x"]), tiled, G.dev(d["scales"]), qz, perm, y, M, K, N, g, act, flags=flags)
    torch.cuda.synchronize()
    G.check_canary(buf, M * N)
    return y


TILED_CASES = [  # M, K, N, group, act_order, bf16
    (1, 64, 32, 64, False, False), (1, 320, 160, 64, False, True), (3, 1088, 288, 64, False, False),
    (8, 2048, 1056, 128, False, True), (1, 4096, 11008, 128, True, False), (2, 4096, 11008, 128, True, False),
    (5, 704, 160, 64, True, False), (8, 1024, 256, 128, True, True), (1, 8192, 28672, 128, False, True),
    (8, 8192, 28672, 128, False, True)]


@pytest.mark.gpu
@pytest.mark.parametrize("M,K,N,g,act_order,bf16", TILED_CASES)
def test_wq4_gemm_tiled_parity(M, K, N, g, act_order, bf16):
    import gpu_util as G
    import synthetic as syn
    from tolerance import unit_roundoff, within
    if act_order:
        d = syn.make_wq4_actorder(seed=29, M=M, K=K, N=N, group=g)
        if bf16:
            d["x"] = syn.f32_to_bf16_bits(d["x"].astype(np.float32))
            d["scales"] = syn.f32_to_bf16_bits(d["scales"].astype(np.float32))
            d["act_bf16"] = 1
    else:
        d = syn.make_wq4_sym(seed=31, M=M, K=K, N=N, group=g) if bf16 else None
        if d is None:
            d = syn.make_wq4_actorder(seed=31, M=M, K=K, N=N, group=g)
            d["g_idx"] = None  # the same codes, scales and zeros read as contiguous groups
    tiled, perm = _repack(G, d, act_order)
    y = G.to_f64(_run_tiled(G, d, tiled, perm))
    cols = None
    if N > 4096:
        r = np.random.default_rng(5)
        cols = np.unique(np.concatenate([np.arange(0, 256), np.arange(N - 256, N), r.integers(0, N, 768)]))
    y_ref, a = G.oracle_wq4(d, cols)
    ok, worst = within(y if cols is None else y[:, cols], y_ref, a, unit_roundoff("bf16" if bf16 else "f16"))
    assert ok, f"max |err|/bound = {worst:.3g}"


@pytest.mark.gpu
def test_wq4_gemm_tiled_onehot_exact_and_pdl_repeat():
    """One-hot x returns the dequantized rows rounded once; a PDL launch gives the same bits."""
    import gemm_dequant_gemv_gb300 as wq
    import gpu_util as G
    import oracle
    import synthetic as syn
    d = syn.make_wq4_actorder(seed=9, M=3, K=512, N=288, group=128)
    tiled, perm = _repack(G, d, True)
    x = np.zeros((3, 512), np.float16)
    for m, k in enumerate((0, 130, 511)):
        x[m, k] = 1.0
    d["x"] = x
    y1 = G.bits_u16(_run_tiled(G, d, tiled, perm))
    y2 = G.bits_u16(_run_tiled(G, d, tiled, perm, flags=wq.WQ_FLAG_PDL))
    y_ref, _ = G.oracle_wq4(d)
    assert np.array_equal(y1, oracle.round_f16(y_ref))
    assert np.array_equal(y1, y2)
    assert wq.read_timeout_flag(clear=True) == 0
