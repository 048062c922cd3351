"""The whole-block decode schedule replayed as one CUDA graph, against the oracle.

Two BitNet-3B layers of BitLinear calls ("Hesper.Models.BitNet" page, section
"Performance (BitNet-3B on A100)": the 32 layers' projections are the
per-token work) run as bitlinear_linear_ws calls with programmatic dependent
launch inside one CUDA graph, each call consuming the previous call's output:

    x -> [q || k || v] ; v -> o ; o -> RMSNorm -> [gate || up] ;
    ReLU^2(gate) * up -> sub-norm -> down ; down -> next layer's x

(with `gated`, the gate || up call writes ReLU^2(gate) * up itself,
BITLINEAR_FLAG_GATED, and the down call reads that product alone)

(the FFN structure of the "Transformer Block" page, sections "Feed-Forward
Network" and "Layer Structure"; attention itself is not part of this path, so
o reads v directly).  After two replays every call's int8 activations and
scales must equal the oracle's act_quant of the GPU's own fp32 input to that
call, its int32 accumulators the oracle's on sampled output columns, and its
outputs must lie within 1e-5 of the oracle's.  A PDL ordering fault (a call
reading its input before the producing kernel finished) shows up as a
mismatch here.
"""
import numpy as np
import pytest
import torch

import bitlinear_w1_a8_gb300 as bl
import oracle
from bitlinear_w1_a8_gb300 import synth
from harness import Y_RTOL, max_rel_err

pytestmark = pytest.mark.gpu

D, F = synth.DIM_3B, synth.FFN_3B
LAYERS = 2
SAMPLE_COLS = 192


def _quantize(N, K, seed):
    W = synth.weight(N, K, seed)
    packed = torch.empty(bl.bitlinear_packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    sw = torch.empty(1, dtype=torch.float32, device="cuda")
    ws = torch.empty(bl.bitlinear_quantize_weights_workspace(N, K), dtype=torch.uint8, device="cuda")
    bl.bitlinear_quantize_weights(W.cuda(), packed, sw, ws)
    Wq, sw_o, _ = oracle.weight_quant(W.numpy())
    assert sw.item() == sw_o
    return packed, sw, Wq


class Call:
    """One bitlinear_linear_ws call of the schedule with its own buffers."""

    def __init__(self, M, K, mats, x, mul=None, gamma=None, gated=False):
        self.M, self.K, self.x, self.mul, self.gamma, self.gated = M, K, x, mul, gamma, gated
        self.mats = mats  # list of (packed, sw, Wq)
        self.xq = torch.empty(M, K, dtype=torch.int8, device="cuda")
        self.sx = torch.empty(M, dtype=torch.float32, device="cuda")
        self.ys = [torch.empty(M, Wq.shape[0], dtype=torch.float32, device="cuda") for _, _, Wq in mats]
        self.accs = [torch.empty(M, Wq.shape[0], dtype=torch.int32, device="cuda") for _, _, Wq in mats]

    def run(self, ws, stream):
        bl.bitlinear_linear_ws(self.x, [(p, s, y, a) for (p, s, _), y, a in zip(self.mats, self.ys, self.accs)],
                               self.xq, self.sx, ws, mul=self.mul, rms_weight=self.gamma, rms_eps=1e-6,
                               flags=bl.FLAG_PDL | (bl.FLAG_GATED if self.gated else 0), stream=stream)

    def check(self, rng):
        x = self.x.cpu().numpy()
        mul = None if self.mul is None else self.mul.cpu().numpy()
        gamma = None if self.gamma is None else self.gamma.cpu().numpy()
        xq_o, sx_o = oracle.act_quant(x, mul=mul, gamma=gamma, eps=1e-6)
        np.testing.assert_array_equal(self.xq.cpu().numpy(), xq_o)
        np.testing.assert_array_equal(self.sx.cpu().numpy(), sx_o)
        N = self.mats[0][2].shape[0]
        cols = np.sort(rng.choice(N, size=min(SAMPLE_COLS, N), replace=False))
        cols[-1] = N - 1  # the last column (the ragged edge of any tile) always
        f32 = []
        for (_, sw, Wq), y, acc in zip(self.mats, self.ys, self.accs):
            if Wq.shape[0] != N:
                cols = np.sort(rng.choice(Wq.shape[0], size=min(SAMPLE_COLS, Wq.shape[0]), replace=False))
                cols[-1] = Wq.shape[0] - 1
            acc_o, y_o = oracle.forward(xq_o, sx_o, oracle.pack(np.ascontiguousarray(Wq[cols])), sw.item(),
                                        len(cols), self.K)
            np.testing.assert_array_equal(acc.cpu().numpy()[:, cols], acc_o)
            if not self.gated:
                assert max_rel_err(y.cpu().numpy()[:, cols], y_o) <= Y_RTOL
            # the rescale's fp32 steps: f32(acc) / f32(sx * sw)
            den = (sx_o.astype(np.float32)[:, None] * np.float32(sw.item())).astype(np.float32)
            f32.append((acc_o.astype(np.float32) / den).astype(np.float32))
        if self.gated:
            g, u = f32
            r = np.maximum(g, np.float32(0))
            h = ((r * r).astype(np.float32) * u).astype(np.float32)
            np.testing.assert_array_equal(self.ys[0].cpu().numpy()[:, cols], h)
            np.testing.assert_array_equal(self.ys[1].cpu().numpy()[:, cols], u)


@pytest.fixture(scope="module")
def weights():
    bl.load_library()
    layers = []
    for layer in range(LAYERS):
        shapes = [(D, D), (D, D), (D, D), (D, D), (F, D), (F, D), (D, F)]  # q k v o gate up down
        layers.append([_quantize(N, K, synth.weight_set_seed(layer, proj)) for proj, (N, K) in enumerate(shapes)])
    g_norm = synth.uniform((D,), 0.5, 1.5, synth.SEEDS["ffn_1b3"]["norm"]).cuda()
    g_sub = synth.uniform((F,), 0.5, 1.5, synth.SEEDS["ffn_1b3"]["subnorm"]).cuda()
    return layers, g_norm, g_sub


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("M", [1, 8, 16, 64])
def test_two_layer_schedule_in_one_graph(weights, M, gated):
    layers, g_norm, g_sub = weights
    x0 = synth.activations(M, D, synth.SEEDS["weight_set"]["x"]).cuda()
    calls = []
    x = x0
    for mats in layers:
        q, k, v, o, gate, up, down = mats
        qkv = Call(M, D, [q, k, v], x)
        c_o = Call(M, D, [o], qkv.ys[2])
        gu = Call(M, D, [gate, up], c_o.ys[0], gamma=g_norm, gated=gated)
        dn = Call(M, F, [down], gu.ys[0], mul=None if gated else gu.ys[1], gamma=g_sub)
        calls += [qkv, c_o, gu, dn]
        x = dn.ys[0]
    ws = torch.empty(bl.bitlinear_forward_workspace(M, F), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for c in calls:          # once eagerly: lazy set-up outside the capture
            c.run(ws, stream)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for c in calls:
                c.run(ws, stream)
        for c in calls:          # clear every output so the replay must write it
            for y in c.ys:
                y.fill_(float("nan"))
            c.xq.fill_(0)
        g.replay()
        g.replay()
    torch.cuda.synchronize()
    assert bl.bitlinear_device_status() == 0
    rng = np.random.default_rng(1000 + M + (7 if gated else 0))
    for c in calls:
        c.check(rng)
