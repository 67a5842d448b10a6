"""Seeded synthetic inputs for the quantized GEMV/GEMM workloads.

This module is the one piece the tests, the benchmark, the oracle side and the
CUDA side all use.  It holds no arithmetic of the hot path (no dequantization,
no products, no activation quantization): only

  * a counter-based splitmix64 stream and Box-Muller normals,
  * the offline weight preparation that produces the stored inputs
    (round-to-nearest quantizers and the bit packers of the storage formats),
  * builders for the five workloads (shapes, distributions, seeds).

splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): output i of a stream with key c is
mix(c + (i+1) * 0x9E3779B97F4A7C15) with the published mix constants.
Box-Muller: z0 = sqrt(-2 ln(1-u1)) cos(2 pi u2), z1 = ... sin(2 pi u2).

Storage formats (the same conventions the library documents):
  * int8 weights [K, N] row-major;
  * 4-bit: int32 [K/8, N], nibble j of word [r, n] holds row 8r + j;
  * 3-bit: int32 [3K/32, N]; the 32 codes of rows 32b..32b+31 of a column
    form a 96-bit little-endian bit stream over word rows 3b..3b+2, code j at
    bits [3j, 3j+3);
  * 4-bit zeros: int32 [G, N/8], nibble j of word [g, c] is column 8c + j.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = np.array([(seed * 0x100000001B3 + stream * 0x2545F4914F6CDD1D) & 0xFFFFFFFFFFFFFFFF],
                     dtype=np.uint64)
        return _mix(a)[0]


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive 64-bit outputs of splitmix64 stream (seed, stream)."""
    key = _key(seed, stream)
    out = np.empty(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            i = np.arange(offset + s + 1, offset + e + 1, dtype=np.uint64)
            out[s:e] = _mix(key + i * _GOLDEN)
    return out


def uniform(seed: int, stream: int, shape) -> np.ndarray:
    """float64 uniforms in [0, 1): top 53 bits of each output."""
    n = int(np.prod(shape))
    return ((u64(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)).reshape(shape)


def normal(seed: int, stream: int, shape, sigma: float = 1.0, dtype=np.float32) -> np.ndarray:
    """Box-Muller normals N(0, sigma^2), generated in float64 and rounded to dtype."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=dtype)
    half = (n + 1) // 2
    for s in range(0, half, _CHUNK):
        e = min(half, s + _CHUNK)
        u = (u64(seed, stream, 2 * (e - s), offset=2 * s) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * np.pi * u2
        z = np.empty(2 * (e - s))
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        z *= sigma
        lo, hi = 2 * s, min(n, 2 * e)
        out[lo:hi] = z[: hi - lo].astype(dtype)
    return out.reshape(shape)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded random permutation of 0..n-1 (argsort of distinct 64-bit keys)."""
    keys = u64(seed, stream, n)
    return np.argsort(keys, kind="stable").astype(np.int32)


# ---- bf16 helpers (numpy has no bf16 dtype: bit patterns in uint16) ---------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); finite inputs."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---- bit packers of the storage formats ---------------------------------------

def pack4(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [K, N] in 0..15 -> int32 [K/8, N], nibble j = row 8r + j."""
    codes = np.asarray(codes)
    K, N = codes.shape
    assert K % 8 == 0 and codes.min(initial=0) >= 0 and codes.max(initial=0) <= 15
    c = codes.astype(np.uint32).reshape(K // 8, 8, N)
    w = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        w |= c[:, j, :] << np.uint32(4 * j)
    return w.view(np.int32)


def tile4_index(K: int, N: int) -> np.ndarray:
    """Destination of every word of a [K/8, N] 4-bit matrix in the library's
    tiled layout (wq4_repack_tiled): word (r, n) goes to
    ((r//8) * (N//32) + n//32) * 256 + ((r%8) % 2) * 128 + (4 * ((n%32)//4) + (r%8)//2) * 4 + n%4."""
    assert K % 64 == 0 and N % 32 == 0
    r = np.arange(K // 8, dtype=np.int64)[:, None]
    n = np.arange(N, dtype=np.int64)[None, :]
    rr = r % 8
    return (((r // 8) * (N // 32) + n // 32) * 256 + (rr % 2) * 128 + (4 * ((n % 32) // 4) + rr // 2) * 4 + n % 4)


def tile4(qweight: np.ndarray) -> np.ndarray:
    """The tiled layout of a packed [K/8, N] 4-bit matrix (a flat int32 array)."""
    R, N = qweight.shape
    out = np.empty(R * N, dtype=qweight.dtype)
    out[tile4_index(8 * R, N).ravel()] = qweight.ravel()
    return out


def untile4(tiled: np.ndarray, K: int, N: int) -> np.ndarray:
    """Inverse of tile4: the [K/8, N] matrix back from the tiled words."""
    return np.asarray(tiled).ravel()[tile4_index(K, N)]


def pack3(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [K, N] in 0..7 -> int32 [3K/32, N] (96-bit little-endian blocks)."""
    codes = np.asarray(codes)
    K, N = codes.shape
    assert K % 32 == 0 and codes.min(initial=0) >= 0 and codes.max(initial=0) <= 7
    c = codes.astype(np.uint64).reshape(K // 32, 32, N)
    words = np.zeros((K // 32, 3, N), dtype=np.uint64)
    for j in range(32):
        bit = 3 * j
        wi, off = divmod(bit, 32)
        words[:, wi, :] |= (c[:, j, :] << np.uint64(off)) & np.uint64(0xFFFFFFFF)
        if off > 29:
            words[:, wi + 1, :] |= c[:, j, :] >> np.uint64(32 - off)
    return words.reshape(3 * K // 32, N).astype(np.uint32).view(np.int32)


def pack_zeros4(zeros: np.ndarray) -> np.ndarray:
    """uint8 zero points [G, N] in 0..15 -> int32 [G, N/8], nibble j = column 8c + j."""
    zeros = np.asarray(zeros)
    G, N = zeros.shape
    assert N % 8 == 0
    z = zeros.astype(np.uint32).reshape(G, N // 8, 8)
    w = np.zeros((G, N // 8), dtype=np.uint32)
    for j in range(8):
        w |= z[:, :, j] << np.uint32(4 * j)
    return w.view(np.int32)


# ---- offline round-to-nearest weight quantizers (input preparation) ------------

def rtn_int8_groups(wf: np.ndarray, group: int):
    """Symmetric int8, one fp32 scale per (group of `group` rows, column):
    s = max|w| / 127 (fp32), q = clamp(rint(w / s), -127, 127); all-zero group: s = 1."""
    K, N = wf.shape
    g = wf.astype(np.float32).reshape(K // group, group, N)
    s = (np.abs(g).max(axis=1) / np.float32(127.0)).astype(np.float32)
    s[s == 0] = 1.0
    q = np.clip(np.rint(g / s[:, None, :]), -127, 127).astype(np.int8)
    return q.reshape(K, N), s


def rtn_uint4_sym(wf: np.ndarray, group: int):
    """Symmetric uint4 with zero 8, bf16 scale per (group, column):
    s = bf16(max|w| / 7), q = clamp(rint(w / s) + 8, 0, 15).  Returns (codes, scale bits)."""
    K, N = wf.shape
    g = wf.astype(np.float32).reshape(K // group, group, N)
    s_bits = f32_to_bf16_bits(np.abs(g).max(axis=1) / np.float32(7.0))
    s = bf16_bits_to_f32(s_bits)
    zero = s == 0
    s_bits[zero] = f32_to_bf16_bits(np.ones(1, np.float32))[0]
    s[zero] = 1.0
    q = np.clip(np.rint(g / s[:, None, :]) + 8, 0, 15).astype(np.uint8)
    return q.reshape(K, N), s_bits


def rtn_uint4_asym_gidx(wf: np.ndarray, g_idx: np.ndarray, group: int):
    """Asymmetric uint4 over the row groups named by g_idx, fp16 scales:
    s = fp16((max - min) / 15), z = clamp(rint(-min / s), 0, 15),
    q = clamp(rint(w / s) + z, 0, 15).  Returns (codes [K,N], scales fp16 [G,N], zeros [G,N])."""
    K, N = wf.shape
    G = K // group
    wf = wf.astype(np.float32)
    s = np.empty((G, N), dtype=np.float16)
    z = np.empty((G, N), dtype=np.uint8)
    q = np.empty((K, N), dtype=np.uint8)
    for g in range(G):
        rows = np.nonzero(g_idx == g)[0]
        blk = wf[rows]
        lo, hi = blk.min(axis=0), blk.max(axis=0)
        sg = ((hi - lo) / np.float32(15.0)).astype(np.float16)
        sg[sg == 0] = 1.0
        sf = sg.astype(np.float32)
        zg = np.clip(np.rint(-lo / sf), 0, 15)
        s[g] = sg
        z[g] = zg.astype(np.uint8)
        q[rows] = np.clip(np.rint(blk / sf) + zg, 0, 15).astype(np.uint8)
    return q, s, z


def gidx_from_permutation(perm: np.ndarray, group: int) -> np.ndarray:
    """Act-order group index: g_idx[perm[i]] = i // group (every group has `group` rows)."""
    g_idx = np.empty(perm.size, dtype=np.int32)
    g_idx[perm] = np.arange(perm.size, dtype=np.int32) // group
    return g_idx


# ---- the workloads --------------------------------------------------------------
# Stream tags keep the tensors of one workload independent of each other.
_X, _W, _S, _Z, _P = 1, 2, 3, 4, 5


def make_wq8(seed=1, M=1, K=4096, N=4096, group=128):
    """INT8 weight-only GEMV: x fp32 ~N(0,1); W ~N(0, 0.02) -> symmetric int8,
    group-wise fp32 scales."""
    x = normal(seed, _X, (M, K), 1.0, np.float32)
    wf = normal(seed, _W, (K, N), 0.02, np.float32)
    q, s = rtn_int8_groups(wf, group)
    return dict(x=x, w=q, scales=s, M=M, K=K, N=N, group=group)


def make_wq3(seed=2, M=1, K=4096, N=4096):
    """3-bit GEMV: x fp16 ~N(0,1); codes U{0..7}; per-column fp16 scale
    ~U(0.005, 0.02); zero stored as fp16(scale * z), z U{0..7}."""
    x = normal(seed, _X, (M, K), 1.0, np.float32).astype(np.float16)
    codes = np.floor(uniform(seed, _W, (K, N)) * 8).astype(np.uint8)
    s = (0.005 + 0.015 * uniform(seed, _S, (N,))).astype(np.float16)
    z = np.floor(uniform(seed, _Z, (N,)) * 8)
    zeros = (s.astype(np.float64) * z).astype(np.float16)
    return dict(x=x, mat=pack3(codes), scales=s, zeros=zeros, codes=codes, z=z.astype(np.uint8),
                M=M, K=K, N=N)


def make_wq4_actorder(seed=3, M=1, K=4096, N=11008, group=128):
    """4-bit group-wise GEMV with act-order: x fp16 ~N(0,1); W ~N(0, 0.02) ->
    asymmetric uint4 over g_idx groups, fp16 scales, 4-bit zeros."""
    x = normal(seed, _X, (M, K), 1.0, np.float32).astype(np.float16)
    wf = normal(seed, _W, (K, N), 0.02, np.float32)
    perm = permutation(seed, _P, K)
    g_idx = gidx_from_permutation(perm, group)
    q, s, z = rtn_uint4_asym_gidx(wf, g_idx, group)
    return dict(x=x, qweight=pack4(q), scales=s, qzeros=pack_zeros4(z), g_idx=g_idx,
                codes=q, zeros=z, perm=perm, M=M, K=K, N=N, group=group, act_bf16=0)


def make_wq4_sym(seed=4, M=1, K=8192, N=28672, group=128, x_seed=None):
    """W4A16: x bf16 ~N(0,1) [M, K]; W ~N(0, 0.02) -> symmetric uint4 (zero 8),
    bf16 scales.  The weights come from `seed`, x from `x_seed` (default seed + M)."""
    xs = seed + M if x_seed is None else x_seed
    x = f32_to_bf16_bits(normal(xs, _X, (M, K), 1.0, np.float32))
    wf = normal(seed, _W, (K, N), 0.02, np.float32)
    q, s_bits = rtn_uint4_sym(wf, group)
    return dict(x=x, qweight=pack4(q), scales=s_bits, qzeros=None, g_idx=None, codes=q,
                M=M, K=K, N=N, group=group, act_bf16=1)


def make_w8a8(seed=5, M=2048, K=8192, N=8192):
    """W8A8: X bf16 ~N(0,1) [M, K]; W ~N(0, 0.02) -> int8 with per-column fp32
    scale Sw = max|W[:, n]| / 127."""
    X = f32_to_bf16_bits(normal(seed, _X, (M, K), 1.0, np.float32))
    wf = normal(seed, _W, (K, N), 0.02, np.float32)
    Sw = (np.abs(wf).max(axis=0) / np.float32(127.0)).astype(np.float32)
    Sw[Sw == 0] = 1.0
    Wq = np.clip(np.rint(wf / Sw[None, :]), -127, 127).astype(np.int8)
    return dict(X=X, W=Wq, Sw=Sw, M=M, K=K, N=N)


# The five workloads, by what they are.
WORKLOADS = {
    "wq8_gemv_4096x4096_g128": dict(builder="make_wq8", seed=1, M=1, K=4096, N=4096, group=128),
    "wq3_gemv_4096x4096": dict(builder="make_wq3", seed=2, M=1, K=4096, N=4096),
    "wq4_actorder_gemv_4096x11008_g128": dict(builder="make_wq4_actorder", seed=3, M=1, K=4096, N=11008, group=128),
    "wq4_sym_gemm_8192x28672_g128": dict(builder="make_wq4_sym", seed=4, K=8192, N=28672, group=128,
                                         M_sweep=(1, 2, 4, 8, 16, 32)),
    "w8a8_gemm_2048x8192x8192": dict(builder="make_w8a8", seed=5, M=2048, K=8192, N=8192),
}
