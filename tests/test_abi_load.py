"""The C-ABI library loads, exports every symbol include/bitlinear.h declares,
and rejects bad arguments on the host before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import bitlinear_w1_a8_gb300 as bl
from bitlinear_w1_a8_gb300 import build as blbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "bitlinear.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bitlinear_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    blbuild.build()
    return bl.load_library()


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert len(declared) >= 9
    assert sorted(bl.EXPORTED_SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_host_only_calls(lib):
    assert bl.bitlinear_abi_version() == 1
    assert bl.bitlinear_packed_bytes(10240, 2560) == 6553600
    assert bl.bitlinear_packed_bytes(2560, 10240) == 6553600
    assert bl.bitlinear_packed_bytes(50000, 2560) == 32000000
    assert bl.bitlinear_packed_bytes(3, 65) == 96
    assert bl.bitlinear_packed_bytes(0, 64) == 0
    assert bl.bitlinear_quantize_weights_workspace(10240, 2560) >= 256 * 8
    for N, K in ((1, 64), (3, 65), (10240, 2560), (2560, 10240), (50000, 2560), (7, 32768), (0, 64)):
        assert bl._packed_size(N, K) == bl.bitlinear_packed_bytes(N, K)
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert bl.bitlinear_status_string(code).startswith("BITLINEAR_")


# Fake, never dereferenced device addresses: every call below must fail (or
# return OK for an empty batch) during argument checking, before any CUDA call.
A = 0x10000   # 16-byte aligned
U = 0x10004   # misaligned


def test_forward_argument_errors(lib):
    f = lib.bitlinear_forward_ex
    assert f(None, A, 1, A, A, 64, 64, A, None, 0, 0, None) == -1          # NULL xq
    assert f(A, A, 1, A, A, 64, 100, A, None, 0, 0, None) == -2            # K % 64
    assert f(A, A, 1, A, A, 0, 64, A, None, 0, 0, None) == -2              # N == 0
    assert f(A, A, -1, A, A, 64, 64, A, None, 0, 0, None) == -2            # M < 0
    assert f(U, A, 1, A, A, 64, 64, A, None, 0, 0, None) == -3             # misaligned xq
    assert f(A, A, 1, A, A, 64, 64, U, None, 0, 0, None) == -3             # misaligned y
    assert f(A, A, 1, A, A, 64, 64, A, None, 7, 0, None) == -4             # unknown algo
    assert f(A, A, 129, A, A, 64, 64, A, None, 3, 0, None) == -4           # batched past 128 tokens
    assert f(A, A, 1, A, A, 64, 64, A, None, 0, 8, None) == -4             # unknown flag
    assert f(A, A, 1 << 20, A, A, 1 << 20, 64, A, None, 0, 0, None) == -2  # M * N >= 2^40
    # decode's grid holds at most 65535 token groups: of 16 tokens at K = 2560, of one token at
    # K = 65536 (a group's activations stay within 64 KB of shared memory)
    assert f(A, A, 16 * 65535 + 1, A, A, 64, 2560, A, None, 1, 0, None) == -4
    assert f(A, A, 65535 + 1, A, A, 8, 65536, A, None, 1, 0, None) == -4
    assert f(A, A, 1, A, A, 64, 65536 + 64, A, None, 1, 0, None) == -4   # decode past K = 65536
    assert f(A, A, 0, A, A, 64, 64, A, None, 0, 0, None) == 0              # empty batch


def test_forward_ws_argument_errors(lib):
    f = lib.bitlinear_forward_ws
    ws = bl.bitlinear_forward_workspace(17, 128)
    assert ws == 32 * 128 * 2 and bl.bitlinear_forward_workspace(0, 128) == 0
    assert bl.bitlinear_forward_workspace(2048, 10240) == 2048 * 10240 * 2
    assert f(A, A, 17, A, A, 64, 128, A, None, 4, 0, None, ws, None) == -7      # WIDE, no workspace
    assert f(A, A, 17, A, A, 64, 128, A, None, 4, 0, A, ws - 16, None) == -7    # too small
    assert f(A, A, 17, A, A, 64, 128, A, None, 4, 0, U, ws, None) == -3         # misaligned workspace
    assert f(A, A, 17, A, A, 64, 100, A, None, 4, 0, A, ws, None) == -2         # K % 64
    assert f(A, A, 17, A, A, 64, 128, A, None, 9, 0, A, ws, None) == -4         # unknown algo
    big = 1 << 28                                                                # 8 * M >= 2^31
    assert f(A, A, big, A, A, 64, 64, A, None, 4, 0, A, big * 64 * 2, None) == -4
    assert f(A, A, 0, A, A, 64, 128, A, None, 4, 0, None, 0, None) == 0         # empty batch
    assert lib.bitlinear_forward_ex(A, A, 17, A, A, 64, 128, A, None, 4, 0, None) == -7  # WIDE needs _ws


def test_linear_ws_argument_errors(lib):
    f = lib.bitlinear_linear_ws
    w = bl.BitLinearWeight(A, A, 64, A, None)
    arr = (bl.BitLinearWeight * 1)(w)
    ws = bl.bitlinear_forward_workspace(200, 128)
    assert f(A, None, 200, 128, None, 1e-6, arr, 1, A, A, 0, A, ws - 16, None) == -7   # too small
    assert f(A, None, 200, 128, None, 1e-6, arr, 1, A, A, 0, U, ws, None) == -3        # misaligned
    assert f(A, None, 0, 128, None, 1e-6, arr, 1, A, A, 0, None, 0, None) == 0         # empty batch
    assert f(A, None, 200, 100, None, 1e-6, arr, 1, A, A, 0, A, ws, None) == -2        # K % 64


def test_linear_gated_argument_errors(lib):
    f = lib.bitlinear_linear
    g = bl.BitLinearWeight(A, A, 64, A, None)
    one = (bl.BitLinearWeight * 1)(g)
    pair = (bl.BitLinearWeight * 2)(g, bl.BitLinearWeight(A, A, 128, A, None))
    three = (bl.BitLinearWeight * 3)(g, g, g)
    G = bl.FLAG_GATED
    assert f(A, None, 1, 128, None, 1e-6, one, 1, A, A, G, None) == -2       # one matrix
    assert f(A, None, 1, 128, None, 1e-6, three, 3, A, A, G, None) == -2     # three matrices
    assert f(A, None, 1, 128, None, 1e-6, pair, 2, A, A, G, None) == -2      # N differ
    assert f(A, None, 1, 128, None, 1e-6, one, 1, A, A, 4, None) == -4       # unknown flag bit
    same = (bl.BitLinearWeight * 2)(g, bl.BitLinearWeight(A, A, 64, None, None))
    assert f(A, None, 1, 128, None, 1e-6, same, 2, A, A, G, None) == -1      # the up output is required
    assert f(A, None, 0, 128, None, 1e-6, same, 2, A, A, G, None) == 0       # empty batch


def test_linear_matrix_count_errors(lib):
    f = lib.bitlinear_linear
    w = bl.BitLinearWeight(A, A, 64, A, None)
    five = (bl.BitLinearWeight * 5)(w, w, w, w, w)
    assert f(A, None, 1, 128, None, 1e-6, five, 5, A, A, 0, None) == -2      # more than four matrices
    assert f(A, None, 1, 128, None, 1e-6, five, 0, A, A, 0, None) == -2      # none
    assert f(A, None, 1, 128, None, 1e-6, None, 1, A, A, 0, None) == -1      # NULL array


def test_quant_act_argument_errors(lib):
    f = lib.bitlinear_quant_act
    assert f(None, None, 1, 64, None, 1e-6, A, A, None) == -1
    assert f(A, None, 1, 96, None, 1e-6, A, A, None) == -2                 # K % 64
    assert f(A, None, 1, 65536, None, 1e-6, A, A, None) == -2              # K too large
    assert f(A, U, 1, 64, None, 1e-6, A, A, None) == -3                    # misaligned mul
    assert f(A, None, 1, 64, A, -1.0, A, A, None) == -2                    # negative eps
    assert f(A, None, 0, 64, None, 1e-6, A, A, None) == 0                  # empty batch


def test_quantize_weights_argument_errors(lib):
    f = lib.bitlinear_quantize_weights
    assert f(A, 4, 64, A, A, None, 4096, None) == -7                       # no workspace
    assert f(A, 4, 64, A, A, A, 16, None) == -7                            # too small
    assert f(A, 4, 60, A, A, A, 4096, None) == -2                          # K % 64
    assert f(A, 1 << 21, 1 << 20, A, A, A, 4096, None) == -2               # N*K >= 2^40
    assert f(U, 4, 64, A, A, A, 4096, None) == -3
    assert f(None, 4, 64, A, A, A, 4096, None) == -1


def test_argmax_argument_errors(lib):
    f = lib.bitlinear_argmax
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    assert f(None, 1, 8, A, None) == -1                                     # NULL y
    assert f(A, 1, 8, None, None) == -1                                     # NULL index
    assert f(A, 1, 0, A, None) == -2                                        # N == 0
    assert f(A, -1, 8, A, None) == -2                                       # M < 0
    assert f(A, 1, 1 << 31, A, None) == -2                                  # N too large
    assert f(A + 2, 1, 8, A, None) == -3                                    # y not 4-byte aligned
    assert f(A, 0, 8, A, None) == 0                                         # empty batch
