"""Helpers for the GPU parity tests: run the library through its binding with
canary-guarded output buffers, and run the oracle on the same inputs."""
import numpy as np
import torch

import bitlinear_w1_a8_gb300 as bl
import oracle

CANARY = 64  # guard elements on each side of every output buffer


def guarded(n, dtype, fill):
    """A CUDA buffer of n elements with `fill` canaries on each side; returns (inner, full)."""
    full = torch.full((n + 2 * CANARY,), fill, dtype=dtype, device="cuda")
    return full[CANARY:CANARY + n], full


def check_canary(full, fill):
    head = full[:CANARY].cpu()
    tail = full[-CANARY:].cpu()
    assert torch.all(head == fill) and torch.all(tail == fill), "output buffer overrun"


def gpu_quantize_weights(W):
    """W: torch CPU fp32 [N, K] -> (packed uint8 numpy, sw float, mean float)."""
    N, K = W.shape
    Wd = W.cuda()
    nbytes = bl.bitlinear_packed_bytes(N, K)
    packed, pfull = guarded(nbytes, torch.uint8, 0xA5)
    scale, sfull = guarded(1, torch.float32, -7.0)
    ws = torch.full((bl.bitlinear_quantize_weights_workspace(N, K),), 0x5A, dtype=torch.uint8,
                    device="cuda")
    bl.bitlinear_quantize_weights(Wd, packed, scale, ws)
    assert bl.bitlinear_device_status() == 0
    check_canary(pfull, 0xA5)
    check_canary(sfull, -7.0)
    mean = ws[2048:2052].view(torch.float32).item()  # the kernel leaves mean|W| there
    return packed.cpu().numpy(), float(scale.item()), mean, (packed, scale)


def gpu_act_quant(x, mul=None, gamma=None, eps=1e-6):
    M, K = x.shape
    xq, xfull = guarded(M * K, torch.int8, 77)
    sx, sfull = guarded(M, torch.float32, -3.0)
    xq2 = xq.view(M, K)
    bl.bitlinear_quant_act(x.cuda(), xq2, sx,
                           mul=None if mul is None else mul.cuda(),
                           rms_weight=None if gamma is None else gamma.cuda(), rms_eps=eps)
    assert bl.bitlinear_device_status() == 0
    check_canary(xfull, 77)
    check_canary(sfull, -3.0)
    return xq2.cpu().numpy(), sx.cpu().numpy(), (xq2, sx)


def gpu_forward(xq_d, sx_d, packed_d, sw_d, N, algo=bl.ALGO_AUTO, flags=0, workspace=False):
    """bitlinear_forward_ex, or with workspace=True (always for ALGO_WIDE)
    bitlinear_forward_ws with a canary-guarded workspace."""
    M, K = xq_d.shape
    y, yfull = guarded(M * N, torch.float32, 1234.5)
    acc, afull = guarded(M * N, torch.int32, -99)
    y2, acc2 = y.view(M, N), acc.view(M, N)
    if workspace or algo == bl.ALGO_WIDE:
        ws, wfull = guarded(bl.bitlinear_forward_workspace(M, K), torch.uint8, 0x3C)
        bl.bitlinear_forward_ws(xq_d, sx_d, packed_d, sw_d, N, y2, acc2, workspace=ws, algo=algo, flags=flags)
        assert bl.bitlinear_device_status() == 0
        check_canary(wfull, 0x3C)
    else:
        bl.bitlinear_forward_ex(xq_d, sx_d, packed_d, sw_d, N, y2, acc2, algo=algo, flags=flags)
        assert bl.bitlinear_device_status() == 0
    check_canary(yfull, 1234.5)
    check_canary(afull, -99)
    return acc2.cpu().numpy(), y2.cpu().numpy()


def max_rel_err(y_gpu, y_ref):
    y_gpu = np.asarray(y_gpu, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    denom = np.maximum(np.abs(y_ref), np.finfo(np.float64).tiny)
    err = np.where(y_ref == 0, np.abs(y_gpu), np.abs(y_gpu - y_ref) / denom)
    return float(err.max()) if err.size else 0.0


# Output tolerance: the outputs are one fp32 product and one fp32 division of
# exact operands (|error| <= ~1.2e-7 relative); the bar is 1e-5.
Y_RTOL = 1e-5


# Rows of one repeated value c (signs varied), K = 2560: the RMSNorm sum is
# exactly K*c^2, so the scale's fp64 chain is 1/sqrt(c^2 + eps) rounded at
# each step, and these c put that fp64 value within ~32 fp64 ulps of an fp32
# rounding boundary (the midpoint between two fp32 values), where a faster
# estimate of the scale would round the other way if it were trusted.  Each
# entry: eps, the fp32 bit pattern of c, the signed distance of the chain's
# low 29 fraction bits from 2^28 (in fp64 ulps).  With gamma drawn by
# ``RMS_BOUNDARY_GAMMA`` a one-ulp change of the fp32 scale changes sx for
# every entry.
RMS_BOUNDARY_K = 2560
RMS_BOUNDARY_ROWS = [
    (0.0, 0x3DFC3237, 16), (0.0, 0x3DD0AC19, 20), (0.0, 0x3D869913, 30), (0.0, 0x3D87CC45, 30),
    (1e-6, 0x3DD4EE44, 14), (1e-6, 0x3E814329, 1), (1e-6, 0x4138A38E, 4), (1e-6, 0x40978642, -37),
]


def rms_boundary_gamma():
    return np.random.default_rng(91).uniform(0.5, 1.5, RMS_BOUNDARY_K).astype(np.float32)


def rms_boundary_rows(eps):
    """The rows of ``RMS_BOUNDARY_ROWS`` for one eps: (M, K) float32."""
    cs = [np.array([b], dtype=np.uint32).view(np.float32)[0] for e, b, _ in RMS_BOUNDARY_ROWS if e == eps]
    sign = np.where(np.random.default_rng(93).random((len(cs), RMS_BOUNDARY_K)) < 0.5, -1.0, 1.0)
    return (np.array(cs, dtype=np.float32)[:, None] * sign).astype(np.float32)


def full_parity(W, x, mul=None, gamma=None, eps=1e-6, algo=bl.ALGO_AUTO, flags=0, workspace=False):
    """Every stage of the library against the oracle on the same inputs."""
    N, K = W.shape
    Wn, xn = W.numpy(), x.numpy()
    Wq_o, sw_o, mean_o = oracle.weight_quant(Wn)
    packed_o = oracle.pack(Wq_o)
    packed_g, sw_g, mean_g, (packed_d, sw_d) = gpu_quantize_weights(W)
    assert mean_g == mean_o
    assert sw_g == sw_o
    np.testing.assert_array_equal(packed_g, packed_o)
    xq_o, sx_o = oracle.act_quant(xn, mul=None if mul is None else mul.numpy(),
                                  gamma=None if gamma is None else gamma.numpy(), eps=eps)
    xq_g, sx_g, (xq_d, sx_d) = gpu_act_quant(x, mul, gamma, eps)
    np.testing.assert_array_equal(sx_g, sx_o)
    np.testing.assert_array_equal(xq_g, xq_o)
    acc_o, y_o = oracle.forward(xq_o, sx_o, packed_o, sw_o, N, K)
    acc_g, y_g = gpu_forward(xq_d, sx_d, packed_d, sw_d, N, algo=algo, flags=flags, workspace=workspace)
    np.testing.assert_array_equal(acc_g, acc_o)
    assert max_rel_err(y_g, y_o) <= Y_RTOL
    return dict(acc=acc_g, y=y_g, y_ref=y_o)
