"""The C ABI on the host: the library loads, exports every entry point the
header declares, and rejects invalid arguments before touching the GPU (every
case here returns before its first CUDA call, so no GPU is needed)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")

# fake, never-dereferenced device addresses: aligned and misaligned
A = 0x7f0000000000
MIS = A + 4


@pytest.fixture(scope="module")
def wq():
    import gemm_dequant_gemv_gb300 as m
    return m


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"WQ_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_symbols()
    for n in ("wq8_gemv", "wq3_gemv", "wq4_gemm", "w8a8_gemm", "w8a8_gemm_workspace_bytes",
              "wq_status_string", "wq_abi_version", "wq_read_timeout_flag"):
        assert n in names


def test_library_exports_every_declared_symbol(wq):
    lib = wq.library()
    for n in declared_symbols():
        assert hasattr(lib, n), n
    assert set(declared_symbols()) <= set(wq.SIGNATURES)


def test_only_the_abi_is_exported(wq):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", wq.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared_symbols()) <= exported
    stray = {s for s in exported if s.startswith("wq") and s not in declared_symbols()}
    assert not stray, stray


def test_status_strings(wq):
    assert wq.abi_version() == 1
    for s in range(8):
        assert wq.status_string(s) and wq.status_string(s) != "unknown status"
    assert wq.status_string(99) == "unknown status"


def _st(fn, *args):
    return fn(*args)


def test_wq8_validation(wq):
    f = wq.library().wq8_gemv
    ok = (A, A, A, A, 1, 256, 256, 128, 0, 0)
    bad = [((0, A, A, A, 1, 256, 256, 128, 0, 0), wq.WQ_ERR_NULL),
           ((A, A, A, 0, 1, 256, 256, 128, 0, 0), wq.WQ_ERR_NULL),
           ((A, A, A, A, 0, 256, 256, 128, 0, 0), wq.WQ_ERR_SHAPE),
           ((A, A, A, A, 9, 256, 256, 128, 0, 0), wq.WQ_ERR_SHAPE),
           ((A, A, A, A, 1, 200, 256, 128, 0, 0), wq.WQ_ERR_SHAPE),   # K % group
           ((A, A, A, A, 1, 256, 264, 128, 0, 0), wq.WQ_ERR_SHAPE),   # N % 16
           ((A, A, A, A, 1, 256, 256, 24, 0, 0), wq.WQ_ERR_SHAPE),    # group % 16
           ((MIS, A, A, A, 1, 256, 256, 128, 0, 0), wq.WQ_ERR_ALIGN),
           ((A, MIS, A, A, 1, 256, 256, 128, 0, 0), wq.WQ_ERR_ALIGN),
           ((A, A, A, MIS, 1, 256, 256, 128, 0, 0), wq.WQ_ERR_ALIGN)]
    for args, want in bad:
        assert f(*args) == want, args
    assert len(ok) == 10


def test_wq3_validation(wq):
    f = wq.library().wq3_gemv
    cases = [((A, A, A, 0, A, 1, 64, 64, 0, 0), wq.WQ_ERR_NULL),
             ((A, A, A, A, A, 1, 48, 64, 0, 0), wq.WQ_ERR_SHAPE),      # K % 32
             ((A, A, A, A, A, 1, 64, 60, 0, 0), wq.WQ_ERR_SHAPE),      # N % 8
             ((A, A, A, A, A, 9, 64, 64, 0, 0), wq.WQ_ERR_SHAPE),
             ((A, A, A, A, MIS, 1, 64, 64, 0, 0), wq.WQ_ERR_ALIGN)]
    for args, want in cases:
        assert f(*args) == want, args


def test_wq4_validation(wq):
    f = wq.library().wq4_gemm
    base = [A, A, A, None, None, A, 1, 256, 256, 128, wq.WQ_F16, None, 0, 0, 0]

    def call(**kw):
        a = list(base)
        names = ["x", "qw", "s", "qz", "gi", "y", "M", "K", "N", "g", "act", "ws", "wsb", "flags", "stream"]
        for k, v in kw.items():
            a[names.index(k)] = v
        return f(*a)

    assert call(x=0) == wq.WQ_ERR_NULL
    assert call(s=0) == wq.WQ_ERR_NULL
    assert call(M=0) == wq.WQ_ERR_SHAPE
    assert call(g=48) == wq.WQ_ERR_SHAPE          # group % 32
    assert call(K=320) == wq.WQ_ERR_SHAPE         # K % group
    assert call(N=260) == wq.WQ_ERR_SHAPE         # N % 8
    assert call(act=0) == wq.WQ_ERR_UNSUPPORTED   # not fp16 / bf16
    assert call(qz=MIS) == wq.WQ_ERR_ALIGN
    assert call(gi=MIS) == wq.WQ_ERR_ALIGN
    assert call(M=12, gi=A) == wq.WQ_ERR_UNSUPPORTED  # act-order is a CUDA-core path only (M <= 8)
    assert call(M=32, g=32, K=256) == wq.WQ_ERR_UNSUPPORTED  # the tensor-core path needs group % 64


def test_dequant_validation(wq):
    lib = wq.library()
    f8, f3, f4 = lib.wq8_dequant, lib.wq3_dequant, lib.wq4_dequant
    cases8 = [((0, A, A, 256, 256, 128, 0, 0), wq.WQ_ERR_NULL),
              ((A, A, 0, 256, 256, 128, 0, 0), wq.WQ_ERR_NULL),
              ((A, A, A, 200, 256, 128, 0, 0), wq.WQ_ERR_SHAPE),   # K % group
              ((A, A, A, 256, 264, 128, 0, 0), wq.WQ_ERR_SHAPE),   # N % 16
              ((A, A, A, 256, 256, 24, 0, 0), wq.WQ_ERR_SHAPE),    # group % 16
              ((A, A, MIS, 256, 256, 128, 0, 0), wq.WQ_ERR_ALIGN)]
    for args, want in cases8:
        assert f8(*args) == want, args
    cases3 = [((A, A, 0, A, 64, 64, 0, 0), wq.WQ_ERR_NULL),
              ((A, A, A, A, 48, 64, 0, 0), wq.WQ_ERR_SHAPE),       # K % 32
              ((A, A, A, A, 64, 60, 0, 0), wq.WQ_ERR_SHAPE),       # N % 8
              ((A, A, A, MIS, 64, 64, 0, 0), wq.WQ_ERR_ALIGN)]
    for args, want in cases3:
        assert f3(*args) == want, args
    ok4 = [A, A, None, None, A, 256, 256, 128, wq.WQ_F16, 0, 0]
    cases4 = [({0: 0}, wq.WQ_ERR_NULL), ({4: 0}, wq.WQ_ERR_NULL),
              ({7: 48}, wq.WQ_ERR_SHAPE),                            # group % 32
              ({5: 320}, wq.WQ_ERR_SHAPE),                           # K % group
              ({6: 260}, wq.WQ_ERR_SHAPE),                           # N % 8
              ({8: 0}, wq.WQ_ERR_UNSUPPORTED),                       # not fp16 / bf16
              ({2: MIS}, wq.WQ_ERR_ALIGN), ({3: MIS}, wq.WQ_ERR_ALIGN), ({4: MIS}, wq.WQ_ERR_ALIGN)]
    for edits, want in cases4:
        a = list(ok4)
        for i, v in edits.items():
            a[i] = v
        assert f4(*a) == want, edits


def test_w8a8_smooth_validation(wq):
    f = wq.library().w8a8_gemm_smooth
    ok = [A, A, A, A, A, 128, 256, 256, None, None, None, A, 1 << 20, 0, 0]
    for edits, want in (({1: 0}, wq.WQ_ERR_NULL), ({1: MIS}, wq.WQ_ERR_ALIGN), ({0: 0}, wq.WQ_ERR_NULL),
                        ({6: 96}, wq.WQ_ERR_SHAPE), ({7: 40}, wq.WQ_ERR_SHAPE), ({12: 16}, wq.WQ_ERR_WORKSPACE)):
        a = list(ok)
        for i, v in edits.items():
            a[i] = v
        assert f(*a) == want, edits


def test_w8a8_outlier_validation(wq):
    lib = wq.library()
    f = lib.w8a8_gemm_outlier
    need = lib.w8a8_gemm_outlier_workspace_bytes(128, 256, 256)
    assert need > lib.w8a8_gemm_workspace_bytes(128, 256, 256)
    ok = [A, A, A, A, 128, 256, 256, 6.0, None, None, None, None, A, need, 0, 0]
    for edits, want in (({0: 0}, wq.WQ_ERR_NULL), ({5: 96}, wq.WQ_ERR_SHAPE), ({6: 40}, wq.WQ_ERR_SHAPE),
                        ({11: A + 2}, wq.WQ_ERR_ALIGN), ({12: A + 16}, wq.WQ_ERR_ALIGN),
                        ({13: need - 1}, wq.WQ_ERR_WORKSPACE)):
        a = list(ok)
        for i, v in edits.items():
            a[i] = v
        assert f(*a) == want, edits


def test_w8a8_validation(wq):
    f = wq.library().w8a8_gemm
    need = wq.w8a8_gemm_workspace_bytes(64, 128, 64)
    assert need > 0 and wq.w8a8_gemm_workspace_bytes(0, 128, 64) == 0
    base = [A, A, A, A, 64, 128, 64, None, None, None, A, need, 0, 0]
    assert f(*([0] + base[1:])) == wq.WQ_ERR_NULL
    b = list(base); b[10] = None
    assert f(*b) == wq.WQ_ERR_WORKSPACE
    b = list(base); b[11] = need - 1
    assert f(*b) == wq.WQ_ERR_WORKSPACE
    b = list(base); b[5] = 100
    assert f(*b) == wq.WQ_ERR_SHAPE                # K % 64
    b = list(base); b[6] = 40
    assert f(*b) == wq.WQ_ERR_SHAPE                # N % 16
    b = list(base); b[10] = A + 16
    assert f(*b) == wq.WQ_ERR_ALIGN                # workspace 256-byte aligned
    b = list(base); b[7] = MIS
    assert f(*b) == wq.WQ_ERR_ALIGN
