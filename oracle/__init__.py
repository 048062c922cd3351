"""CPU oracle for the BitLinear W1.58A8 layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never does, and shares no code with it.

The arithmetic lives in ``bitlinear_oracle.c`` (plain C, built with
``-ffp-contract=off`` and no fast-math); this module builds it with gcc and
marshals numpy arrays into it.  Every function states which part of the
method it follows; the header of the C file lists the readings taken where
the pages leave a step open.

Pins: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` against something other than itself (a
hand-worked example, the pages' printed sizes, exactly rounded sums from the
Python standard library, closed forms, or brute force in exact rational
arithmetic).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitlinear_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libbitlinear_oracle.so")

CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build`` (gcc, no GPU needed)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, f32p, f64p = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
        vp = ctypes.c_void_p
        lib.oracle_exact_abs_sum.argtypes = [vp, i64]
        lib.oracle_exact_abs_sum.restype = ctypes.c_double
        lib.oracle_exact_sq_sum.argtypes = [vp, i64]
        lib.oracle_exact_sq_sum.restype = ctypes.c_double
        lib.oracle_weight_quant.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.oracle_weight_quant.restype = ctypes.c_int
        lib.oracle_packed_bytes.argtypes = [i64, i64]
        lib.oracle_packed_bytes.restype = i64
        lib.oracle_pack.argtypes = [vp, i64, i64, vp]
        lib.oracle_pack.restype = ctypes.c_int
        lib.oracle_unpack.argtypes = [vp, i64, i64, vp]
        lib.oracle_unpack.restype = ctypes.c_int
        lib.oracle_act_quant.argtypes = [vp, vp, i64, i64, vp, ctypes.c_double, vp, vp, vp]
        lib.oracle_act_quant.restype = ctypes.c_int
        lib.oracle_forward.argtypes = [vp, vp, i64, vp, ctypes.c_float, i64, i64, vp, vp]
        lib.oracle_forward.restype = ctypes.c_int
        lib.oracle_forward_unpacked.argtypes = [vp, vp, i64, vp, ctypes.c_float, i64, i64, vp, vp]
        lib.oracle_forward_unpacked.restype = ctypes.c_int
        lib.oracle_argmax.argtypes = [vp, i64, i64, vp]
        lib.oracle_argmax.restype = ctypes.c_int
        del f32p, f64p
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(f"{what} failed with code {rc}")


def exact_abs_sum(v) -> float:
    """Exact sum of |v| over fp32 values, rounded once to fp64 (mean|W| numerator)."""
    v = _c(v, np.float32).ravel()
    return _load().oracle_exact_abs_sum(_ptr(v), v.size)


def exact_sq_sum(v) -> float:
    """Exact sum of v^2 over fp32 values, rounded once to fp64 (RMSNorm numerator)."""
    v = _c(v, np.float32).ravel()
    return _load().oracle_exact_sq_sum(_ptr(v), v.size)


def weight_quant(W):
    """absmean weight_quant (Candle BitNet PR, the changes list): returns (Wq int8 [N,K], sw, mean)."""
    W = _c(W, np.float32)
    N, K = W.shape
    Wq = np.empty((N, K), np.int8)
    sw = np.zeros(1, np.float32)
    mean = np.zeros(1, np.float32)
    _check(_load().oracle_weight_quant(_ptr(W), N, K, _ptr(Wq), _ptr(sw), _ptr(mean)), "weight_quant")
    return Wq, float(sw[0]), float(mean[0])


def packed_bytes(N: int, K: int) -> int:
    """Bytes of the 2-bit packed layout: N * ceil(K/64) * 16 (0.25 B per weight)."""
    return int(_load().oracle_packed_bytes(N, K))


def pack(Wq) -> np.ndarray:
    """Pack ternary codes (Wq+1) into the 16-byte-chunk layout."""
    Wq = _c(Wq, np.int8)
    N, K = Wq.shape
    out = np.empty(packed_bytes(N, K), np.uint8)
    _check(_load().oracle_pack(_ptr(Wq), N, K, _ptr(out)), "pack")
    return out


def unpack(packed, N: int, K: int) -> np.ndarray:
    """Inverse of pack; raises on an invalid code 3."""
    packed = _c(packed, np.uint8).ravel()
    if packed.size != packed_bytes(N, K):
        raise OracleError("packed buffer has the wrong size")
    Wq = np.empty((N, K), np.int8)
    _check(_load().oracle_unpack(_ptr(packed), N, K, _ptr(Wq)), "unpack")
    return Wq


def act_quant(x, mul=None, gamma=None, eps: float = 1e-6, return_h: bool = False):
    """Per-token absmax activation_quant with the optional ReLU^2*mul and RMSNorm prologues.

    Returns (xq int8 [M,K], sx fp32 [M]) and, if asked, the fp32 rows h fed to
    the quantiser.
    """
    x = _c(x, np.float32)
    M, K = x.shape
    mul = None if mul is None else _c(mul, np.float32)
    gamma = None if gamma is None else _c(gamma, np.float32).ravel()
    if mul is not None and mul.shape != x.shape:
        raise OracleError("mul must match x")
    if gamma is not None and gamma.size != K:
        raise OracleError("gamma must have K entries")
    xq = np.empty((M, K), np.int8)
    sx = np.empty(M, np.float32)
    h = np.empty((M, K), np.float32) if return_h else None
    _check(_load().oracle_act_quant(_ptr(x), _ptr(mul), M, K, _ptr(gamma), float(eps),
                                    _ptr(xq), _ptr(sx), _ptr(h)), "act_quant")
    return (xq, sx, h) if return_h else (xq, sx)


def forward(xq, sx, packed, sw: float, N: int, K: int):
    """Contraction on packed weights: returns (acc int32 [M,N], y fp64 [M,N])."""
    xq = _c(xq, np.int8)
    sx = _c(sx, np.float32).ravel()
    packed = _c(packed, np.uint8).ravel()
    M = xq.shape[0]
    if xq.shape[1] != K or sx.size != M or packed.size != packed_bytes(N, K):
        raise OracleError("shape mismatch")
    acc = np.empty((M, N), np.int32)
    y = np.empty((M, N), np.float64)
    _check(_load().oracle_forward(_ptr(xq), _ptr(sx), M, _ptr(packed), float(sw), N, K,
                                  _ptr(acc), _ptr(y)), "forward")
    return acc, y


def forward_unpacked(xq, sx, Wq, sw: float):
    """Contraction on unpacked ternary weights Wq [N,K]: returns (acc, y fp64)."""
    xq = _c(xq, np.int8)
    sx = _c(sx, np.float32).ravel()
    Wq = _c(Wq, np.int8)
    M, K = xq.shape
    N = Wq.shape[0]
    acc = np.empty((M, N), np.int32)
    y = np.empty((M, N), np.float64)
    _check(_load().oracle_forward_unpacked(_ptr(xq), _ptr(sx), M, _ptr(Wq), float(sw), N, K,
                                           _ptr(acc), _ptr(y)), "forward_unpacked")
    return acc, y


def argmax(y):
    """First index of each row's largest value: y [M, N] (fp32 or fp64) -> int32 [M]."""
    y = _c(y, np.float64)
    M, N = y.shape
    out = np.empty(M, np.int32)
    _check(_load().oracle_argmax(_ptr(y), M, N, _ptr(out)), "argmax")
    return out


def bitlinear(x, W, mul=None, gamma=None, eps: float = 1e-6):
    """The whole layer: weight_quant, pack, act_quant, contraction, rescale.

    Returns a dict with every intermediate (Wq, sw, packed, xq, sx, acc, y).
    """
    Wq, sw, _ = weight_quant(W)
    packed = pack(Wq)
    xq, sx = act_quant(x, mul=mul, gamma=gamma, eps=eps)
    N, K = Wq.shape
    acc, y = forward(xq, sx, packed, sw, N, K)
    return dict(Wq=Wq, sw=sw, packed=packed, xq=xq, sx=sx, acc=acc, y=y)
