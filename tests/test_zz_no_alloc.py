"""bitlinear_quantize_weights_noalloc against the oracle and the regular entry point.

The no-allocation entry point is for callers that cannot allocate device
memory when they quantise weights (a runtime with a fixed memory budget, a
plugin without an allocator): it keeps its scratch in a fixed array inside
the library instead of a caller workspace.  Its packed bytes and scale must
equal the oracle's weight_quant + pack exactly, and the regular entry point's,
on consecutive calls too (the shared scratch keeps the previous call's
contents and must be cleared).
This file is collected last so that a failure here does not hide the others.
"""
import numpy as np
import pytest
import torch

import bitlinear_w1_a8_gb300 as bl
import oracle
from bitlinear_w1_a8_gb300 import synth

pytestmark = pytest.mark.gpu


def _regular(W):
    N, K = W.shape
    packed = torch.empty(bl.bitlinear_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(bl.bitlinear_quantize_weights_workspace(N, K), dtype=torch.uint8, device="cuda")
    bl.bitlinear_quantize_weights(W, packed, sw, ws)
    return packed, sw


def _noalloc(W):
    N, K = W.shape
    packed = torch.full((bl.bitlinear_packed_bytes(N, K),), 0xEE, dtype=torch.uint8, device="cuda")
    sw = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    bl.bitlinear_quantize_weights_noalloc(W, packed, sw)
    return packed, sw


@pytest.mark.parametrize("N,K,seed", [(10240, 2560, 10), (300, 640, 3)])
def test_noalloc_matches_oracle_and_regular_on_two_calls(N, K, seed):
    bl.load_library()
    W1 = synth.weight(N, K, seed)
    W2 = synth.weight(N, K, seed + 1) * 3.0             # a different scale on the second call
    for W in (W1, W2):                                  # two calls in a row share the scratch
        Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
        packed_o = oracle.pack(Wq_o)
        Wd = W.cuda()
        p_na, s_na = _noalloc(Wd)
        p_ref, s_ref = _regular(Wd)
        assert bl.bitlinear_device_status() == 0
        # integer codes and the scale: identical (the bar of every byte-level parity test)
        assert s_na.item() == sw_o
        np.testing.assert_array_equal(p_na.cpu().numpy(), packed_o)
        assert s_na.item() == s_ref.item()
        np.testing.assert_array_equal(p_na.cpu().numpy(), p_ref.cpu().numpy())
