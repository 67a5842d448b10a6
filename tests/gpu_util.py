"""Helpers for the GPU parity tests: move seeded numpy inputs to the device,
call the library through its binding, and guard outputs (NaN poisoning and a
canary tail after every output buffer)."""
import numpy as np
import torch

import gemm_dequant_gemv_gb300 as wq

DEV = torch.device("cuda:0")
CANARY = 64        # elements of guard tail after each output
SENTINEL = 1024.0  # exact in fp32, fp16 and bf16


def dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:  # bf16 bit patterns
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def guarded(shape, dtype):
    """Output tensor poisoned with NaN, followed by a canary tail of NaN-free sentinels."""
    n = int(np.prod(shape))
    buf = torch.full((n + CANARY,), float("nan"), dtype=dtype, device=DEV)
    buf[n:] = SENTINEL
    return buf, buf[:n].view(*shape)


def check_canary(buf, n):
    tail = buf[n:].float().cpu().numpy()
    assert np.all(tail == SENTINEL), "an output was written past its end"


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def bits_u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_wq8(d, flags=0):
    M, K, N, g = d["M"], d["K"], d["N"], d["group"]
    x, w, s = dev(d["x"]), dev(d["w"]), dev(d["scales"])
    buf, y = guarded((M, N), torch.float32)
    wq.wq8_gemv(x, w, s, y, M, K, N, g, flags=flags)
    torch.cuda.synchronize()
    check_canary(buf, M * N)
    return y


def run_wq3(d, flags=0):
    M, K, N = d["M"], d["K"], d["N"]
    x, mat, s, z = dev(d["x"]), dev(d["mat"]), dev(d["scales"]), dev(d["zeros"])
    buf, y = guarded((M, N), torch.float16)
    wq.wq3_gemv(x, mat, s, z, y, M, K, N, flags=flags)
    torch.cuda.synchronize()
    check_canary(buf, M * N)
    return y


def run_wq4(d, flags=0):
    M, K, N, g = d["M"], d["K"], d["N"], d["group"]
    act = wq.WQ_BF16 if d["act_bf16"] else wq.WQ_F16
    x, qw, s = dev(d["x"]), dev(d["qweight"]), dev(d["scales"])
    qz = None if d["qzeros"] is None else dev(d["qzeros"])
    gi = None if d["g_idx"] is None else dev(d["g_idx"])
    buf, y = guarded((M, N), torch.bfloat16 if d["act_bf16"] else torch.float16)
    wq.wq4_gemm(x, qw, s, qz, gi, y, M, K, N, g, act, flags=flags)
    torch.cuda.synchronize()
    check_canary(buf, M * N)
    return y


def oracle_wq4(d, cols=None):
    import oracle
    x = d["x"] if d["x"].dtype == np.uint16 else d["x"].view(np.uint16)
    s = d["scales"] if d["scales"].dtype == np.uint16 else d["scales"].view(np.uint16)
    return oracle.wq4_gemm(x, d["act_bf16"], d["qweight"], s, d["qzeros"], d["g_idx"], d["group"], cols=cols)
