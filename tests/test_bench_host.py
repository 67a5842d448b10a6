"""Host-side logic of bench.py that needs no GPU: the packed step buffers
(every layer's x and y become 256-byte-aligned views into one buffer each, so
that a step's inputs and results move with one copy each way), the algorithmic
byte counts, and the job-throughput arithmetic."""
import os
import sys
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _fake_layer(torch, seed):
    g = torch.Generator().manual_seed(seed)
    return types.SimpleNamespace(
        w8={"x": torch.randn(1, 4096, generator=g)},
        w3={"x": torch.randn(1, 4096, generator=g).half()},
        w4={"x": torch.randn(1, 4096, generator=g).half()},
        y8=torch.randn(1, 4096, generator=g),
        y3=torch.randn(1, 4096, generator=g).half(),
        y4=torch.randn(1, 11008, generator=g).half())


def test_pack_io_views_share_one_buffer_each():
    torch = pytest.importorskip("torch")
    import bench
    layers = [_fake_layer(torch, s) for s in range(3)]
    before = [(L.w8["x"].clone(), L.w3["x"].clone(), L.w4["x"].clone(), L.y8.clone(), L.y3.clone(), L.y4.clone())
              for L in layers]
    xbuf, ybuf = bench.pack_io(layers, torch.device("cpu"))
    xs = [t for L in layers for t in (L.w8["x"], L.w3["x"], L.w4["x"])]
    ys = [t for L in layers for t in (L.y8, L.y3, L.y4)]
    for t, base in [(t, xbuf) for t in xs] + [(t, ybuf) for t in ys]:
        off = t.data_ptr() - base.data_ptr()
        assert 0 <= off and off + t.numel() * t.element_size() <= base.numel()
        assert off % 256 == 0                       # tensor maps want 16-byte starts
    for L, b in zip(layers, before):                # contents carried over
        for t, ref in zip((L.w8["x"], L.w3["x"], L.w4["x"], L.y8, L.y3, L.y4), b):
            assert torch.equal(t, ref)
    # a write through the packed buffer lands in the layer's tensor (one copy per step suffices)
    xbuf.zero_()
    assert all(float(t.abs().sum()) == 0.0 for t in xs)
    # sizes: 3 layers x (16 KB + 8 KB + 8 KB) of x, 3 x (16 KB + 8 KB + 21.5 KB) of y
    assert xbuf.numel() == 3 * (4096 * 4 + 4096 * 2 + 4096 * 2)
    assert ybuf.numel() == 3 * (4096 * 4 + 4096 * 2 + 11008 * 2)


def test_algorithmic_bytes():
    import bench
    # W8: codes + fp32 group scales + fp32 x + fp32 y
    assert bench.alg_bytes_w8() == 4096 * 4096 + 32 * 4096 * 4 + 4096 * 4 + 4096 * 4
    # W3: 3-bit codes + fp16 scale and zero per column + fp16 x + fp16 y
    assert bench.alg_bytes_w3() == 4096 * 4096 * 3 // 8 + 4096 * 2 * 2 + 4096 * 2 + 4096 * 2
    assert bench.alg_bytes_w4g() == 23471616


def test_job_throughput_is_total_bytes_over_the_slowest_rank():
    import bench
    assert bench.job_throughput(1_000_000, 10, 2, 5.0) == pytest.approx(2 * 10 * 1_000_000 / 5e-3 / 1e9)
    assert np.isclose(bench.job_throughput(2_000_000, 4, 1, 1.0), 2_000_000 * 4 / 1e-3 / 1e9)
