"""Python binding of the GB300 BitLinear W1.58A8 C-ABI library (libbitlinear.so).

Argument marshalling only: every function below forwards torch CUDA tensors
(as raw device pointers, sizes and the current CUDA stream) to the
``extern "C"`` entry point of the same name declared in ``include/bitlinear.h``.
All arithmetic runs in the library's CUDA kernels; there is no CPU fallback.
If the library has not been built, importing works but every call raises.
"""
from __future__ import annotations

import ctypes
import functools
import os

__all__ = [
    "BitLinearError", "load_library", "library_path",
    "bitlinear_abi_version", "bitlinear_status_string", "bitlinear_packed_bytes",
    "bitlinear_quantize_weights_workspace", "bitlinear_quantize_weights",
    "bitlinear_quant_act", "bitlinear_forward", "bitlinear_forward_ex",
    "bitlinear_forward_workspace", "bitlinear_forward_ws",
    "bitlinear_device_status", "bitlinear_quantize_weights_noalloc",
    "bitlinear_selftest_wait_timeout", "bitlinear_linear", "bitlinear_linear_ws", "bitlinear_argmax",
    "BitLinearWeight",
    "EXPORTED_SYMBOLS",
    "ALGO_AUTO", "ALGO_DECODE", "ALGO_PREFILL", "ALGO_BATCHED", "ALGO_WIDE", "FLAG_PDL",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libbitlinear.so")

ALGO_AUTO, ALGO_DECODE, ALGO_PREFILL, ALGO_BATCHED, ALGO_WIDE = 0, 1, 2, 3, 4
FLAG_PDL = 1
FLAG_GATED = 2  # bitlinear_linear: gate, up pair; the first output receives (r * r) * up, r = max(gate, 0)

STATUS = {0: "OK", -1: "ERR_NULL", -2: "ERR_SHAPE", -3: "ERR_ALIGN", -4: "ERR_UNSUPPORTED",
          -5: "ERR_CUDA", -6: "ERR_TIMEOUT", -7: "ERR_WORKSPACE"}

# Every entry point include/bitlinear.h declares.
EXPORTED_SYMBOLS = (
    "bitlinear_abi_version", "bitlinear_status_string", "bitlinear_packed_bytes",
    "bitlinear_quantize_weights_workspace", "bitlinear_quantize_weights",
    "bitlinear_quant_act", "bitlinear_forward", "bitlinear_forward_ex",
    "bitlinear_forward_workspace", "bitlinear_forward_ws",
    "bitlinear_device_status", "bitlinear_quantize_weights_noalloc",
    "bitlinear_selftest_wait_timeout", "bitlinear_linear", "bitlinear_linear_ws", "bitlinear_argmax",
)

_lib = None


class BitLinearWeight(ctypes.Structure):
    """ctypes mirror of the C struct bitlinear_weight."""
    _fields_ = [("packed", ctypes.c_void_p), ("w_scale", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("y", ctypes.c_void_p), ("acc", ctypes.c_void_p)]


class BitLinearError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {bitlinear_status_string(status)} ({status})")


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load libbitlinear.so (raises if it was not built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libbitlinear.so not found at {p}: build it with "
                           "bitlinear_w1_a8_gb300.build.build() (needs nvcc)")
    lib = ctypes.CDLL(p)
    i64, vp, sz, st = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    lib.bitlinear_abi_version.argtypes = []
    lib.bitlinear_abi_version.restype = ctypes.c_int
    lib.bitlinear_status_string.argtypes = [st]
    lib.bitlinear_status_string.restype = ctypes.c_char_p
    lib.bitlinear_packed_bytes.argtypes = [i64, i64]
    lib.bitlinear_packed_bytes.restype = sz
    lib.bitlinear_quantize_weights_workspace.argtypes = [i64, i64]
    lib.bitlinear_quantize_weights_workspace.restype = sz
    lib.bitlinear_quantize_weights.argtypes = [vp, i64, i64, vp, vp, vp, sz, vp]
    lib.bitlinear_quantize_weights.restype = st
    lib.bitlinear_quant_act.argtypes = [vp, vp, i64, i64, vp, ctypes.c_double, vp, vp, vp]
    lib.bitlinear_quant_act.restype = st
    lib.bitlinear_forward.argtypes = [vp, vp, i64, vp, vp, i64, i64, vp, vp, vp]
    lib.bitlinear_forward.restype = st
    lib.bitlinear_forward_ex.argtypes = [vp, vp, i64, vp, vp, i64, i64, vp, vp, ctypes.c_int,
                                         ctypes.c_int, vp]
    lib.bitlinear_forward_ex.restype = st
    lib.bitlinear_forward_workspace.argtypes = [i64, i64]
    lib.bitlinear_forward_workspace.restype = sz
    lib.bitlinear_forward_ws.argtypes = [vp, vp, i64, vp, vp, i64, i64, vp, vp, ctypes.c_int,
                                         ctypes.c_int, vp, sz, vp]
    lib.bitlinear_forward_ws.restype = st
    lib.bitlinear_quantize_weights_noalloc.argtypes = [vp, i64, i64, vp, vp, vp]
    lib.bitlinear_quantize_weights_noalloc.restype = st
    lib.bitlinear_selftest_wait_timeout.argtypes = [i64, vp]
    lib.bitlinear_selftest_wait_timeout.restype = st
    lib.bitlinear_linear.argtypes = [vp, vp, i64, i64, vp, ctypes.c_double, ctypes.POINTER(BitLinearWeight),
                                     ctypes.c_int, vp, vp, ctypes.c_int, vp]
    lib.bitlinear_linear.restype = st
    lib.bitlinear_linear_ws.argtypes = [vp, vp, i64, i64, vp, ctypes.c_double, ctypes.POINTER(BitLinearWeight),
                                        ctypes.c_int, vp, vp, ctypes.c_int, vp, sz, vp]
    lib.bitlinear_linear_ws.restype = st
    lib.bitlinear_argmax.argtypes = [vp, i64, i64, vp, vp]
    lib.bitlinear_argmax.restype = st
    lib.bitlinear_device_status.argtypes = [vp, ctypes.c_int]
    lib.bitlinear_device_status.restype = st
    if path is None:
        _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise BitLinearError(status, what)


# Addresses go to ctypes as plain ints (the argtypes are c_void_p; None is NULL).
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _need(t, dtype, name, shape=None):
    try:  # the common case in one expression; the detailed checks only on failure
        if t.is_cuda and t.dtype == dtype and t.is_contiguous() and (shape is None or t.shape == shape):
            return
    except AttributeError:
        pass
    if not getattr(t, "is_cuda", False):
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def bitlinear_abi_version() -> int:
    return load_library().bitlinear_abi_version()


def bitlinear_status_string(status: int) -> str:
    try:
        return load_library().bitlinear_status_string(status).decode()
    except RuntimeError:
        return STATUS.get(status, "unknown status")


@functools.lru_cache(maxsize=256)
def bitlinear_packed_bytes(N: int, K: int) -> int:
    """Bytes of the packed layout of an [N, K] matrix (asked of the library)."""
    return int(load_library().bitlinear_packed_bytes(int(N), int(K)))


def bitlinear_quantize_weights_workspace(N: int, K: int) -> int:
    return int(load_library().bitlinear_quantize_weights_workspace(N, K))


def bitlinear_quantize_weights(W, packed, w_scale, workspace, stream=None):
    """weight_quant + pack of W [N, K] fp32 into `packed` (uint8) and `w_scale` (fp32 [1])."""
    import torch
    _need(W, torch.float32, "W")
    N, K = W.shape
    _need(packed, torch.uint8, "packed", (bitlinear_packed_bytes(N, K),))
    _need(w_scale, torch.float32, "w_scale")
    _need(workspace, torch.uint8, "workspace")
    _check(load_library().bitlinear_quantize_weights(
        _ptr(W), N, K, _ptr(packed), _ptr(w_scale), _ptr(workspace), workspace.numel(),
        _stream(stream)), "bitlinear_quantize_weights")


def bitlinear_quantize_weights_noalloc(W, packed, w_scale, stream=None):
    """weight_quant + pack like bitlinear_quantize_weights, for callers that cannot
    allocate device memory: the scratch is a fixed array inside the library
    (calls on one device must not overlap on the GPU; see include/bitlinear.h)."""
    import torch
    _need(W, torch.float32, "W")
    N, K = W.shape
    _need(packed, torch.uint8, "packed", (bitlinear_packed_bytes(N, K),))
    _need(w_scale, torch.float32, "w_scale")
    _check(load_library().bitlinear_quantize_weights_noalloc(
        _ptr(W), N, K, _ptr(packed), _ptr(w_scale), _stream(stream)),
        "bitlinear_quantize_weights_noalloc")


def bitlinear_quant_act(x, xq, x_scale, mul=None, rms_weight=None, rms_eps: float = 1e-6,
                        stream=None):
    """activation_quant of x [M, K] fp32 (optional ReLU^2*mul gating, optional RMSNorm)."""
    import torch
    _need(x, torch.float32, "x")
    M, K = x.shape
    _need(xq, torch.int8, "xq", (M, K))
    _need(x_scale, torch.float32, "x_scale", (M,))
    if mul is not None:
        _need(mul, torch.float32, "mul", (M, K))
    if rms_weight is not None:
        _need(rms_weight, torch.float32, "rms_weight", (K,))
    _check(load_library().bitlinear_quant_act(
        _ptr(x), _ptr(mul), M, K, _ptr(rms_weight), float(rms_eps), _ptr(xq), _ptr(x_scale),
        _stream(stream)), "bitlinear_quant_act")


def bitlinear_forward_ex(xq, x_scale, packed, w_scale, N: int, y, acc=None,
                         algo: int = ALGO_AUTO, flags: int = 0, stream=None):
    """y [M, N] = (xq . Wq^T) / (sx * sw) with an explicit algorithm and flags."""
    import torch
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    _need(x_scale, torch.float32, "x_scale", (M,))
    _need(packed, torch.uint8, "packed", (bitlinear_packed_bytes(N, K),))
    _need(w_scale, torch.float32, "w_scale")
    _need(y, torch.float32, "y", (M, N))
    if acc is not None:
        _need(acc, torch.int32, "acc", (M, N))
    _check(load_library().bitlinear_forward_ex(
        _ptr(xq), _ptr(x_scale), M, _ptr(packed), _ptr(w_scale), N, K, _ptr(y), _ptr(acc),
        int(algo), int(flags), _stream(stream)), "bitlinear_forward_ex")


@functools.lru_cache(maxsize=256)
def bitlinear_forward_workspace(M: int, K: int) -> int:
    """Bytes of device workspace bitlinear_forward_ws needs for M tokens of K."""
    return int(load_library().bitlinear_forward_workspace(int(M), int(K)))


def bitlinear_forward_ws(xq, x_scale, packed, w_scale, N: int, y, acc=None, workspace=None,
                         algo: int = ALGO_AUTO, flags: int = 0, stream=None):
    """bitlinear_forward_ex with a device workspace (a uint8 CUDA tensor of at
    least bitlinear_forward_workspace(M, K) bytes, or None: then no algorithm
    that needs one is chosen, and asking for ALGO_WIDE raises)."""
    import torch
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    _need(x_scale, torch.float32, "x_scale", (M,))
    _need(packed, torch.uint8, "packed", (bitlinear_packed_bytes(N, K),))
    _need(w_scale, torch.float32, "w_scale")
    _need(y, torch.float32, "y", (M, N))
    if acc is not None:
        _need(acc, torch.int32, "acc", (M, N))
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
    _check(load_library().bitlinear_forward_ws(
        _ptr(xq), _ptr(x_scale), M, _ptr(packed), _ptr(w_scale), N, K, _ptr(y), _ptr(acc),
        int(algo), int(flags), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream)), "bitlinear_forward_ws")


def bitlinear_forward(xq, x_scale, packed, w_scale, N: int, y, acc=None, stream=None):
    """y [M, N] = (xq . Wq^T) / (sx * sw); the kernel is chosen from M."""
    import torch
    _need(xq, torch.int8, "xq")
    M, K = xq.shape
    _need(x_scale, torch.float32, "x_scale", (M,))
    _need(packed, torch.uint8, "packed", (bitlinear_packed_bytes(N, K),))
    _need(w_scale, torch.float32, "w_scale")
    _need(y, torch.float32, "y", (M, N))
    if acc is not None:
        _need(acc, torch.int32, "acc", (M, N))
    _check(load_library().bitlinear_forward(
        _ptr(xq), _ptr(x_scale), M, _ptr(packed), _ptr(w_scale), N, K, _ptr(y), _ptr(acc),
        _stream(stream)), "bitlinear_forward")


def bitlinear_device_status(stream=None, clear: bool = True) -> int:
    """Synchronise the stream and return the library's device status (0 = OK)."""
    return int(load_library().bitlinear_device_status(_stream(stream), 1 if clear else 0))


def bitlinear_argmax(y, index, stream=None):
    """index[m] = first n of the largest y[m, n] (y [M, N] fp32, index [M] int32)."""
    import torch
    _need(y, torch.float32, "y")
    if y.dim() != 2:
        raise ValueError("y must be [M, N]")
    M, N = y.shape
    _need(index, torch.int32, "index", (M,))
    _check(load_library().bitlinear_argmax(_ptr(y), M, N, _ptr(index), _stream(stream)), "bitlinear_argmax")


def bitlinear_selftest_wait_timeout(limit_ns: int, stream=None):
    """Launch the bounded-wait self-test kernel (a wait nothing satisfies)."""
    _check(load_library().bitlinear_selftest_wait_timeout(int(limit_ns), _stream(stream)),
           "bitlinear_selftest_wait_timeout")


def _packed_size(N: int, K: int) -> int:
    """bitlinear_packed_bytes(N, K) without a call into the library (N * ceil(K/64) * 16,
    the layout the header documents); a CPU test holds the two equal."""
    return N * ((K + 63) // 64) * 16


def _weight_array(weights, M, K):
    import torch
    arr = (BitLinearWeight * len(weights))()
    for i, w in enumerate(weights):
        packed, w_scale, y = w[0], w[1], w[2]
        acc = w[3] if len(w) > 3 else None
        N = y.shape[1]
        _need(packed, torch.uint8, "packed", (_packed_size(N, K),))
        _need(w_scale, torch.float32, "w_scale")
        _need(y, torch.float32, "y", (M, N))
        if acc is not None:
            _need(acc, torch.int32, "acc", (M, N))
        arr[i] = BitLinearWeight(packed.data_ptr(), w_scale.data_ptr(), N, y.data_ptr(),
                                 acc.data_ptr() if acc is not None else None)
    return arr


def _linear_inputs(x, xq, x_scale, mul, rms_weight):
    import torch
    _need(x, torch.float32, "x")
    M, K = x.shape
    _need(xq, torch.int8, "xq", (M, K))
    _need(x_scale, torch.float32, "x_scale", (M,))
    if mul is not None:
        _need(mul, torch.float32, "mul", (M, K))
    if rms_weight is not None:
        _need(rms_weight, torch.float32, "rms_weight", (K,))
    return M, K


def bitlinear_linear(x, weights, xq, x_scale, mul=None, rms_weight=None, rms_eps: float = 1e-6,
                     flags: int = 0, stream=None):
    """act_quant + forward for 1..4 matrices sharing the input x [M, K].

    weights: sequence of (packed, w_scale, y) or (packed, w_scale, y, acc) tuples of
    CUDA tensors (y [M, N] fp32, acc [M, N] int32 or None).
    """
    M, K = _linear_inputs(x, xq, x_scale, mul, rms_weight)
    arr = _weight_array(weights, M, K)
    _check(load_library().bitlinear_linear(
        _ptr(x), _ptr(mul), M, K, _ptr(rms_weight), float(rms_eps), arr, len(weights), _ptr(xq),
        _ptr(x_scale), int(flags), _stream(stream)), "bitlinear_linear")


def bitlinear_linear_ws(x, weights, xq, x_scale, workspace, mul=None, rms_weight=None, rms_eps: float = 1e-6,
                        flags: int = 0, stream=None):
    """bitlinear_linear with a device workspace (uint8 CUDA tensor of at least
    bitlinear_forward_workspace(M, K) bytes, or None)."""
    import torch
    M, K = _linear_inputs(x, xq, x_scale, mul, rms_weight)
    arr = _weight_array(weights, M, K)
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
    _check(load_library().bitlinear_linear_ws(
        _ptr(x), _ptr(mul), M, K, _ptr(rms_weight), float(rms_eps), arr, len(weights), _ptr(xq),
        _ptr(x_scale), int(flags), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream)), "bitlinear_linear_ws")
