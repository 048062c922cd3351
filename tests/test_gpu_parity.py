"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer and byte results (packed weights, xq, acc) and the scales (sw, sx)
must be identical; float outputs within 1e-5 relative error of the oracle's
fp64 value.  Sizes span several CTAs and ragged tails; the full-size cases
use the workloads' own shapes (BitNet-3B decode and prefill, BitNet-1.3B FFN).
"""
import numpy as np
import pytest
import torch

import bitlinear_w1_a8_gb300 as bl
import oracle
from bitlinear_w1_a8_gb300 import synth
from harness import (Y_RTOL, check_canary, full_parity, gpu_act_quant, gpu_forward, gpu_quantize_weights,
                     guarded, max_rel_err, rms_boundary_gamma, rms_boundary_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bl.load_library()
    torch.cuda.init()


ALGOS = [bl.ALGO_DECODE, bl.ALGO_PREFILL]


def test_small_bitlinear_m4_k256_n256():
    """The small single-BitLinear workload: M=4, K=N=256, W seed 0, x seed 1."""
    W = synth.weight(256, 256, synth.SEEDS["small"]["W"])
    x = synth.activations(4, 256, synth.SEEDS["small"]["x"])
    full_parity(W, x)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("M,N,K", [
    (1, 1, 64), (2, 1, 128), (1, 80, 64), (3, 300, 192), (5, 1000, 640), (8, 153, 128),
    (17, 2000, 256), (64, 512, 512), (65, 100, 256), (130, 257, 320), (1, 50000, 128),
])
def test_shapes(algo, M, N, K):
    W = synth.weight(N, K, 100 + N + K)
    x = synth.activations(M, K, 200 + M + K, outlier_seed=300 + K)
    full_parity(W, x, algo=algo)


@pytest.mark.parametrize("M,N,K", [
    (3, 1, 64),         # one weight row: every 16-row tile reads a clamped row
    (4, 17, 64),        # one k-block for all warps
    (5, 300, 64),       # one k-block on the MMA dots: most warps get no piece
    (16, 33, 64),       # the same with two column tiles
    (9, 7, 192),        # a 16-token group (two 8-token column tiles) holding 9 tokens
    (16, 2000, 2560),   # two full column tiles; the xs rows padded to an odd multiple of 64
    (12, 640, 10240),   # long K: 16 tokens, K split over a cluster of 4 CTAs
    (8, 300, 10240),    # K split over a cluster of 2
    (6, 129, 8256),     # a split into uneven K ranges (129 k-blocks: 64 + 65)
    (13, 1000, 8192),   # 16-token group, 4 ranges of 32 k-blocks
    (9, 50, 16384),     # 16-token group, a cluster of 8
    (16, 100, 32256),   # 8 ranges of 63 k-blocks: the largest split
    (33, 300, 1024),    # three token groups, the last with one token
    (8, 50000, 128),    # more CTAs than SMs
])
def test_decode_mma_shapes(M, N, K):
    """The decode kernel's warp-level MMA dots (3 tokens and more), forced, on ragged shapes."""
    W = synth.weight(N, K, 500 + N + K)
    x = synth.activations(M, K, 600 + M + K, outlier_seed=700 + K)
    full_parity(W, x, algo=bl.ALGO_DECODE)


@pytest.mark.parametrize("M,N,K", [(8, 300, 10240), (16, 33, 2560)])
def test_decode_mma_extreme_values(M, N, K):
    """int8 inputs at -128 and 127 (the contraction takes any int8, not only act_quant's
    [-127, 127]) against weights of all +-1: the largest sums the MMA dots meet, exact."""
    rng = np.random.default_rng(M * 1000 + K)
    xq = np.where(rng.random((M, K)) < 0.5, -128, 127).astype(np.int8)
    xq[0, :] = -128                                   # one row at the int8 minimum throughout
    Wq = np.where(rng.random((N, K)) < 0.5, -1, 1).astype(np.int8)
    Wq[0, :] = 1
    Wq[1 % N, :] = -1
    sx = np.full(M, 0.5, np.float32)
    sw = np.float32(1.0)
    packed = oracle.pack(Wq)
    acc_o, y_o = oracle.forward(xq, sx, packed, float(sw), N, K)
    assert acc_o[0, 0] == -128 * K
    acc_g, y_g = gpu_forward(torch.from_numpy(xq).cuda(), torch.from_numpy(sx).cuda(),
                             torch.from_numpy(packed).cuda(), torch.tensor([sw]).cuda(), N,
                             algo=bl.ALGO_DECODE)
    np.testing.assert_array_equal(acc_g, acc_o)
    assert max_rel_err(y_g, y_o) <= Y_RTOL


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 64), (2, 1, 128), (1, 80, 64), (3, 300, 192), (5, 1000, 640), (8, 153, 128),
    (17, 2000, 256), (64, 512, 512), (100, 257, 320), (128, 130, 64), (16, 50000, 128),
])
def test_shapes_batched(M, N, K):
    """The tensor-core kernel with weight rows on the MMA's M side (M <= 128)."""
    W = synth.weight(N, K, 100 + N + K)
    x = synth.activations(M, K, 200 + M + K, outlier_seed=300 + K)
    full_parity(W, x, algo=bl.ALGO_BATCHED)


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 64), (2, 1, 128), (1, 80, 64), (3, 300, 192), (5, 1000, 640), (8, 153, 128), (16, 128, 64),
    (17, 2000, 256), (33, 153, 128), (64, 512, 512), (100, 257, 320), (130, 257, 320), (197, 257, 640),
    (300, 2000, 1024), (16, 50000, 128), (3000, 96, 64),
])
def test_shapes_wide(M, N, K):
    """The tensor-core kernel fed by activations widened once into the
    workspace (bitlinear_forward_ws): ragged token and weight tiles, K splits,
    and a canary-guarded workspace."""
    W = synth.weight(N, K, 100 + N + K)
    x = synth.activations(M, K, 200 + M + K, outlier_seed=300 + K)
    full_parity(W, x, algo=bl.ALGO_WIDE)


@pytest.mark.parametrize("M,N,K", [(5, 300, 2048), (256, 640, 4096), (300, 2000, 1024)])
def test_forward_ws_auto_and_pdl(M, N, K):
    """AUTO through bitlinear_forward_ws, and the PDL flag on the WIDE path."""
    W = synth.weight(N, K, 120 + K)
    x = synth.activations(M, K, 121 + M)
    full_parity(W, x, workspace=True)
    full_parity(W, x, algo=bl.ALGO_WIDE, flags=bl.FLAG_PDL)


@pytest.mark.parametrize("algo,M,N,K", [
    (bl.ALGO_PREFILL, 130, 300, 2048), (bl.ALGO_PREFILL, 256, 640, 4096), (bl.ALGO_PREFILL, 40, 2560, 1024),
    (bl.ALGO_BATCHED, 64, 200, 8192), (bl.ALGO_BATCHED, 5, 1000, 4096),
    (bl.ALGO_WIDE, 130, 300, 2048), (bl.ALGO_WIDE, 200, 1000, 4096), (bl.ALGO_WIDE, 1, 1, 32768),
])
def test_split_k(algo, M, N, K):
    """Few tiles: K is split over the CTAs of a thread-block cluster, whose
    partial sums are added through distributed shared memory; acc and y must
    match the oracle as without a split."""
    W = synth.weight(N, K, 110 + K)
    x = synth.activations(M, K, 111 + M)
    full_parity(W, x, algo=algo)


@pytest.mark.parametrize("N,K", [(10240, 2560), (2560, 10240)])
def test_batched_bitnet3b_m32(N, K):
    """BitNet-3B FFN shapes at M = 32 through the batched kernel, every output."""
    W = synth.weight(N, K, 21)
    x = synth.activations(32, K, 22)
    full_parity(W, x, algo=bl.ALGO_BATCHED)


@pytest.mark.parametrize("M", [4, 5, 8, 9, 16, 17, 128, 129, 512, 513])
def test_auto_boundaries_with_workspace(M):
    """bitlinear_forward_ws with AUTO on both sides of every boundary of its rule at a long K
    (K = 8192, N = 300): dp4a decode | MMA decode (8-token groups, K split over a cluster) |
    16-token groups | the batched tensor-core kernel | WIDE | 128-token tiles."""
    W = synth.weight(300, 8192, 800 + M)
    x = synth.activations(M, 8192, 900 + M, outlier_seed=901)
    full_parity(W, x, algo=bl.ALGO_AUTO, flags=bl.FLAG_PDL, workspace=True)


@pytest.mark.parametrize("M", [1, 4, 64])
def test_pdl_flag(M):
    W = synth.weight(2000, 640, 7)
    x = synth.activations(M, 640, 8)
    full_parity(W, x, algo=bl.ALGO_AUTO, flags=bl.FLAG_PDL)


@pytest.mark.parametrize("M,K", [(1, 2048), (3, 2048), (7, 8192), (2, 64)])
def test_prologues(M, K):
    """ReLU^2 gating, RMSNorm, and both (gating first), bit-exact."""
    g = synth.activations(M, K, 40 + K)
    u = synth.activations(M, K, 41 + K)
    gamma = synth.uniform((K,), 0.5, 1.5, 42 + K)
    for mul, gm in ((u, None), (None, gamma), (u, gamma)):
        xq_o, sx_o = oracle.act_quant(g.numpy(), mul=None if mul is None else mul.numpy(),
                                      gamma=None if gm is None else gm.numpy(), eps=1e-6)
        xq_g, sx_g, _ = gpu_act_quant(g, mul, gm, 1e-6)
        np.testing.assert_array_equal(sx_g, sx_o)
        np.testing.assert_array_equal(xq_g, xq_o)


@pytest.mark.parametrize("kind", ["wide", "tiny_only", "zeros_and_subnormals", "window_edge", "just_below"])
@pytest.mark.parametrize("M", [1, 3])
def test_rmsnorm_exact_sum_paths(kind, M):
    """The RMSNorm sum of squares takes one 128-bit window when every value is
    within 2^31 of the row maximum's binade, three windows down to 2^96 below
    it, and an exponent-bucket path otherwise; all must give the oracle's
    codes (act_quant kernel and the fused M = 1 launch)."""
    K = 2048
    g = torch.Generator().manual_seed(90 + M)
    x = torch.randn(M, K, generator=g)
    if kind == "wide":            # a few values far below max/2^32: the bucket path
        x[:, 5] = 1e-12
        x[:, 77] = -3e-20
        x[:, 9] = 1e3
    elif kind == "tiny_only":     # every value tiny, within the window of each other
        x = x * 1e-30
    elif kind == "zeros_and_subnormals":  # exact zeros and fp32 subnormals next to normal values
        x[:, ::7] = 0.0
        x[:, 3] = 1e-40
        x[:, 11] = -7e-42
    elif kind == "window_edge":   # the row maximum in [2^10, 2^11), values in [2^-21, 2^-20): one window
        x[:, 3] = 1536.0
        x[:, 10] = float(np.float32(1.9999999) * np.float32(2.0 ** -21))
        x[:, 11] = -float(np.float32(1.0000001) * np.float32(2.0 ** -21))
    else:                         # one value a binade further down, [2^-22, 2^-21): three windows
        x[:, 3] = 1536.0
        x[:, 10] = 1.5 * 2.0 ** -22
    gamma = synth.uniform((K,), 0.5, 1.5, 91)
    xq_o, sx_o = oracle.act_quant(x.numpy(), gamma=gamma.numpy(), eps=1e-6)
    xq_g, sx_g, _ = gpu_act_quant(x, None, gamma, 1e-6)
    np.testing.assert_array_equal(sx_g, sx_o)
    np.testing.assert_array_equal(xq_g, xq_o)
    if M == 1:
        W = synth.weight(256, K, 92)
        _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
        y = torch.empty(1, 256, device="cuda")
        xq = torch.zeros(1, K, dtype=torch.int8, device="cuda")
        sx = torch.zeros(1, dtype=torch.float32, device="cuda")
        bl.bitlinear_linear(x.cuda(), [(packed_d, sw_d, y)], xq, sx, rms_weight=gamma.cuda(), rms_eps=1e-6)
        assert bl.bitlinear_device_status() == 0
        np.testing.assert_array_equal(xq.cpu().numpy(), xq_o)
        np.testing.assert_array_equal(sx.cpu().numpy(), sx_o)


@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_rmsnorm_scale_at_fp32_boundary(eps):
    """Rows whose RMSNorm scale lies within a few fp64 ulps of an fp32 rounding
    boundary: the kernels' fast estimate of the scale must step aside there and
    give the exact chain's value (act_quant kernel, the M = 1 fused launch and
    the fused few-token launch)."""
    x = torch.from_numpy(rms_boundary_rows(eps))
    gamma = torch.from_numpy(rms_boundary_gamma())
    M, K = x.shape
    xq_o, sx_o = oracle.act_quant(x.numpy(), gamma=gamma.numpy(), eps=eps)
    xq_g, sx_g, _ = gpu_act_quant(x, None, gamma, eps)
    np.testing.assert_array_equal(sx_g, sx_o)
    np.testing.assert_array_equal(xq_g, xq_o)
    W = synth.weight(256, K, 94)
    _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
    for rows in [slice(m, m + 1) for m in range(M)] + [slice(0, M)]:
        n = rows.stop - rows.start
        y = torch.empty(n, 256, device="cuda")
        xq = torch.zeros(n, K, dtype=torch.int8, device="cuda")
        sx = torch.zeros(n, dtype=torch.float32, device="cuda")
        bl.bitlinear_linear(x[rows].cuda(), [(packed_d, sw_d, y)], xq, sx, rms_weight=gamma.cuda(), rms_eps=eps)
        assert bl.bitlinear_device_status() == 0
        np.testing.assert_array_equal(sx.cpu().numpy(), sx_o[rows])
        np.testing.assert_array_equal(xq.cpu().numpy(), xq_o[rows])


def test_edge_values():
    """Zero rows, tiny rows (eps path), rounding ties, subnormals, huge values."""
    K, N = 128, 96
    x = torch.zeros(6, K)
    x[1, :4] = torch.tensor([1e-6, -2e-6, 0.0, 3e-7])
    x[2] = torch.linspace(-127, 127, K).round() + 0.5          # many .5 ties at sx = 127/127.5
    x[3, 0], x[3, 1:9] = 127.0, torch.tensor([-63.5, 0.5, 1.5, 2.5, -0.5, -1.5, 126.5, 62.5])
    x[4] = torch.tensor([1e-40, -3e-39] * (K // 2))            # subnormals only
    x[5] = torch.tensor([3e38, -1e-3] * (K // 2))              # near fp32 max
    W = synth.weight(N, K, 5)
    W[0] = 0.0
    W[1, :8] = torch.tensor([1e-41, -1e-42, 0.0, 1e-38, 3.0, -3.0, 0.01, -0.01])
    full_parity(W, x)
    full_parity(W, x, gamma=synth.uniform((K,), 0.5, 1.5, 6), eps=1e-6)


def test_zero_weight_matrix_and_ties():
    K = 64
    W = torch.zeros(10, K)
    full_parity(W, synth.activations(3, K, 9))
    # mean|W| = 1 exactly: entries at +-0.5, +-1.5 are rounding ties
    W = torch.tensor([[0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 0.375, -0.625] * 8,
                      [0.75] * 64], dtype=torch.float32)
    r = full_parity(W, synth.activations(2, K, 10))
    assert np.isfinite(r["y"]).all()


def test_empty_batch_is_noop():
    W = synth.weight(64, 64, 3)
    _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
    xq = torch.empty(0, 64, dtype=torch.int8, device="cuda")
    sx = torch.empty(0, dtype=torch.float32, device="cuda")
    y = torch.empty(0, 64, dtype=torch.float32, device="cuda")
    bl.bitlinear_forward(xq, sx, packed_d, sw_d, 64, y)
    bl.bitlinear_quant_act(torch.empty(0, 64, device="cuda"), xq, sx)
    assert bl.bitlinear_device_status() == 0


def test_misaligned_pointer_rejected():
    W = synth.weight(64, 64, 3)
    _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
    buf = torch.zeros(64 * 2 + 16, dtype=torch.int8, device="cuda")
    xq = buf[1:1 + 128].view(2, 64)  # 1-byte offset: not 16-byte aligned
    sx = torch.ones(2, device="cuda")
    y = torch.empty(2, 64, device="cuda")
    with pytest.raises(bl.BitLinearError) as e:
        bl.bitlinear_forward(xq, sx, packed_d, sw_d, 64, y)
    assert e.value.status == -3


# ---------------------------------------------------------------------------
# Full-size workloads.
# ---------------------------------------------------------------------------
DECODE_SHAPES = [("up_shape", synth.FFN_3B, synth.DIM_3B, "W_up_shape"),
                 ("down_shape", synth.DIM_3B, synth.FFN_3B, "W_down_shape")]


@pytest.mark.parametrize("name,N,K,seed_key", DECODE_SHAPES, ids=[s[0] for s in DECODE_SHAPES])
def test_decode_m1_full_size(name, N, K, seed_key):
    """BitNet-3B decode GEMV, M=1, 1% outlier channels x20: every output checked."""
    s = synth.SEEDS["decode"]
    W = synth.weight(N, K, s[seed_key])
    x = synth.activations(1, K, s["x"], outlier_seed=s["outliers"])
    full_parity(W, x, flags=bl.FLAG_PDL)


def _sampled_parity(W, x, rows, cols, algo, workspace=False):
    """Whole GPU path at full size; the oracle computes the sampled outputs only."""
    N, K = W.shape
    Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
    packed_g, sw_g, _, (packed_d, sw_d) = gpu_quantize_weights(W)
    assert sw_g == sw_o
    np.testing.assert_array_equal(packed_g, oracle.pack(Wq_o))
    xq_o, sx_o = oracle.act_quant(x.numpy())
    xq_g, sx_g, (xq_d, sx_d) = gpu_act_quant(x)
    np.testing.assert_array_equal(xq_g, xq_o)
    np.testing.assert_array_equal(sx_g, sx_o)
    acc_g, y_g = gpu_forward(xq_d, sx_d, packed_d, sw_d, N, algo=algo, workspace=workspace)
    acc_o, y_o = oracle.forward(xq_o[rows], sx_o[rows], oracle.pack(Wq_o[cols]), sw_o, len(cols), K)
    np.testing.assert_array_equal(acc_g[np.ix_(rows, cols)], acc_o)
    assert max_rel_err(y_g[np.ix_(rows, cols)], y_o) <= Y_RTOL
    return acc_g, y_g


@pytest.mark.parametrize("M", [12, 16])
def test_lm_head_few_tokens_decode(M):
    """The 50000 x 2560 LM head at 12 and 16 tokens: AUTO takes the decode kernel with
    MMA dots (16-token groups over 300+ CTAs in waves); sampled outputs and every
    token row's codes against the oracle."""
    W = synth.weight(50000, 2560, 4321)
    x = synth.activations(M, 2560, 4322, outlier_seed=4323)
    rng = np.random.default_rng(1)
    rows = np.arange(M)
    cols = np.unique(np.concatenate([rng.choice(50000, 200, replace=False), [0, 15, 16, 49999]]))
    _sampled_parity(W, x, rows, cols, bl.ALGO_AUTO)


@pytest.mark.parametrize("path", ["tiles128", "wide"])
@pytest.mark.parametrize("name,N,K,seed", [("up_shape", synth.FFN_3B, synth.DIM_3B, "W_up_shape"),
                                            ("down_shape", synth.DIM_3B, synth.FFN_3B, "W_down_shape")])
def test_prefill_m2048_sampled(name, N, K, seed, path):
    """BitNet-3B prefill GEMM, M=2048: sampled rows x columns against the oracle,
    spread over every output tile, plus the last row and column; through
    bitlinear_forward (AUTO: 128-token tiles) and through bitlinear_forward_ws
    with BITLINEAR_ALGO_WIDE (the activations widened once)."""
    s = synth.SEEDS["prefill"]
    W = synth.weight(N, K, s[seed])
    x = synth.activations(2048, K, s["x"])
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(2048, 24, replace=False), [0, 127, 128, 2047]]))
    cols = np.unique(np.concatenate([rng.choice(N, 160, replace=False), [0, 255, 256, N - 1]]))
    _sampled_parity(W, x, rows, cols, bl.ALGO_WIDE if path == "wide" else bl.ALGO_AUTO, workspace=(path == "wide"))


@pytest.mark.parametrize("M", [1, 512])
def test_ffn_1b3_chain(M):
    """BitNet-1.3B FFN sub-block: RMSNorm -> act_quant -> gate, up -> ReLU^2(gate)*up
    -> sub-norm -> act_quant -> down.  Stage-wise bit-exact (the oracle is fed
    the GPU's fp32 stage inputs), sampled columns at M = 512."""
    s = synth.SEEDS["ffn_1b3"]
    D, F = synth.DIM_1B3, synth.FFN_1B3
    gamma = synth.uniform((D,), 0.5, 1.5, s["norm"])
    gamma_sub = synth.uniform((F,), 0.5, 1.5, s["subnorm"])
    Wg, Wu, Wd = synth.weight(F, D, s["gate"]), synth.weight(F, D, s["up"]), synth.weight(D, F, s["down"])
    x = synth.activations(M, D, s["x"])
    rng = np.random.default_rng(1)
    cols_f = np.unique(rng.choice(F, 96 if M > 1 else F, replace=False))
    cols_d = np.unique(rng.choice(D, 96 if M > 1 else D, replace=False))
    rows = np.arange(M) if M <= 4 else np.unique(rng.choice(M, 12, replace=False))

    # stage 1: normed activations shared by gate and up
    xq_o, sx_o = oracle.act_quant(x.numpy(), gamma=gamma.numpy(), eps=1e-6)
    xq_g, sx_g, (xq_d, sx_d) = gpu_act_quant(x, None, gamma, 1e-6)
    np.testing.assert_array_equal(xq_g, xq_o)
    np.testing.assert_array_equal(sx_g, sx_o)
    outs = {}
    for name, W in (("gate", Wg), ("up", Wu)):
        Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
        packed_g, sw_g, _, (packed_d, sw_d) = gpu_quantize_weights(W)
        assert sw_g == sw_o
        acc_g, y_g = gpu_forward(xq_d, sx_d, packed_d, sw_d, F)
        acc_o, y_o = oracle.forward(xq_o[rows], sx_o[rows], oracle.pack(Wq_o[cols_f]), sw_o,
                                    len(cols_f), D)
        np.testing.assert_array_equal(acc_g[np.ix_(rows, cols_f)], acc_o)
        assert max_rel_err(y_g[np.ix_(rows, cols_f)], y_o) <= Y_RTOL
        outs[name] = torch.from_numpy(y_g)
    # stage 2: gating + sub-norm + act_quant, fed the GPU's fp32 gate/up outputs
    h_q_o, h_sx_o = oracle.act_quant(outs["gate"].numpy(), mul=outs["up"].numpy(),
                                     gamma=gamma_sub.numpy(), eps=1e-6)
    h_q_g, h_sx_g, (hq_d, hsx_d) = gpu_act_quant(outs["gate"], outs["up"], gamma_sub, 1e-6)
    np.testing.assert_array_equal(h_q_g, h_q_o)
    np.testing.assert_array_equal(h_sx_g, h_sx_o)
    # stage 3: down projection
    Wq_o, sw_o, _ = oracle.weight_quant(Wd.numpy())
    _, sw_g, _, (packed_d, sw_d) = gpu_quantize_weights(Wd)
    acc_g, y_g = gpu_forward(hq_d, hsx_d, packed_d, sw_d, D)
    acc_o, y_o = oracle.forward(h_q_o[rows], h_sx_o[rows], oracle.pack(Wq_o[cols_d]), sw_o,
                                len(cols_d), F)
    np.testing.assert_array_equal(acc_g[np.ix_(rows, cols_d)], acc_o)
    assert max_rel_err(y_g[np.ix_(rows, cols_d)], y_o) <= Y_RTOL


def test_repeat_calls_are_deterministic():
    W = synth.weight(3000, 1280, 12)
    x = synth.activations(3, 1280, 13)
    a = full_parity(W, x)
    b = full_parity(W, x, flags=bl.FLAG_PDL)
    np.testing.assert_array_equal(a["y"], b["y"])


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing satisfies gives up after its limit, records
    BITLINEAR_ERR_TIMEOUT, and the context keeps working."""
    assert bl.bitlinear_device_status(clear=True) == 0
    bl.bitlinear_selftest_wait_timeout(20_000_000)  # 20 ms
    assert bl.bitlinear_device_status(clear=True) == -6
    assert bl.bitlinear_device_status(clear=True) == 0
    W = synth.weight(64, 128, 4)
    x = synth.activations(2, 128, 5)
    full_parity(W, x)


@pytest.mark.parametrize("M,K,Ns,prolog", [
    (1, 2560, (10240, 10240), None),        # gate || up of a BitNet-3B decode step, one launch
    (1, 10240, (2560,), "gated"),           # down projection fed ReLU^2(gate)*up
    (1, 2048, (300, 1000, 64), "norm"),     # three matrices, RMSNorm prologue
    (1, 8192, (2048,), "gated+norm"),       # the 1.3B FFN sub-norm path
    (1, 128, (5,), None),                   # tiny
    (3, 640, (500, 77), None),              # M > 1: act_quant + one decode launch for both
    (130, 320, (257, 100), "norm"),         # tensor-core path per matrix
    (160, 8192, (300, 257, 64), None),      # WIDE region (with ws): three matrices, one pre-pass
    (200, 1024, (300, 1000, 2000), None),   # short K above 128 tokens: the tensor-core kernels
    (256, 8192, (2048,), "gated+norm"),     # a 1.3B FFN down call in the WIDE region
    (64, 8192, (2048, 300), "gated"),       # long K at M = 64: batched kernel, K split in a cluster
    (136, 8192, (1000, 300), "gated"),      # long K above 128 tokens: WIDE (with ws)
    (1, 2048, (300, 1000, 64, 7), "norm"),  # four matrices (the most one call takes), fused M = 1
    (40, 1024, (257, 100, 1000, 33), None), # four matrices on the batched kernel
    (5, 640, (500, 77, 1300, 16), "gated"), # four matrices on the decode kernel after act_quant
    (12, 10240, (2560, 640), None),         # two matrices, 16-token MMA group, K split over 4 CTAs
    (6, 8192, (300, 1000, 77), "norm"),     # three matrices, 8-token group, K split over 2 CTAs
    (16, 2560, (10240, 10240), None),       # 16 tokens, 20480 rows: one decode launch, MMA dots
])
@pytest.mark.parametrize("ws", [False, True])
def test_linear_matches_oracle(M, K, Ns, prolog, ws):
    """bitlinear_linear (act_quant + forward for matrices sharing one input) against the oracle;
    with ws, bitlinear_linear_ws with a canary-guarded workspace (the WIDE kernel takes the
    matrices its AUTO rule gives it, widening the activations once for all of them)."""
    x = synth.activations(M, K, 60 + K, outlier_seed=61 + K)
    mul = synth.activations(M, K, 62 + K) if prolog and "gated" in prolog else None
    gamma = synth.uniform((K,), 0.5, 1.5, 63 + K) if prolog and "norm" in prolog else None
    xq_o, sx_o = oracle.act_quant(x.numpy(), mul=None if mul is None else mul.numpy(),
                                  gamma=None if gamma is None else gamma.numpy(), eps=1e-6)
    mats, refs = [], []
    for i, N in enumerate(Ns):
        W = synth.weight(N, K, 70 + i + K)
        Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
        refs.append(oracle.forward(xq_o, sx_o, oracle.pack(Wq_o), sw_o, N, K))
        _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
        y = torch.full((M, N), 5.5, device="cuda")
        acc = torch.full((M, N), -3, dtype=torch.int32, device="cuda")
        mats.append((packed_d, sw_d, y, acc))
    xq = torch.zeros(M, K, dtype=torch.int8, device="cuda")
    sx = torch.zeros(M, dtype=torch.float32, device="cuda")
    kw = dict(mul=None if mul is None else mul.cuda(), rms_weight=None if gamma is None else gamma.cuda(),
              rms_eps=1e-6, flags=bl.FLAG_PDL)
    if ws:
        wsp, wfull = guarded(bl.bitlinear_forward_workspace(M, K), torch.uint8, 0x3C)
        bl.bitlinear_linear_ws(x.cuda(), mats, xq, sx, wsp, **kw)
    else:
        bl.bitlinear_linear(x.cuda(), mats, xq, sx, **kw)
    assert bl.bitlinear_device_status() == 0
    if ws:
        check_canary(wfull, 0x3C)
    np.testing.assert_array_equal(xq.cpu().numpy(), xq_o)
    np.testing.assert_array_equal(sx.cpu().numpy(), sx_o)
    for (packed_d, sw_d, y, acc), (acc_o, y_o) in zip(mats, refs):
        np.testing.assert_array_equal(acc.cpu().numpy(), acc_o)
        assert max_rel_err(y.cpu().numpy(), y_o) <= Y_RTOL


@pytest.mark.parametrize("M,K,Ns", [
    (2, 3072, (1300,)),            # at the register limit (3 float4 a thread)
    (2, 192, (1500, 401)),         # rows of 48 float4: warps straddle the two token rows
    (2, 2560, (2560, 2560, 640)),  # q || k || v widths
    (2, 704, (3100,)),             # ragged N
    (2, 2560, (10240, 10240)),     # gate || up widths
    (3, 2560, (10240, 10240)),     # 3 and 8 tokens take act_quant and the decode kernel
    (8, 2560, (10240, 10240)),
])
def test_linear_few_tokens_fused_quant(M, K, Ns):
    """Two tokens without a prologue and at least 8 rows a CTA: one decode launch in which
    every CTA quantises the token rows itself; codes, scales, accumulators and outputs
    against the oracle, with an all-zero row and an outlier row among the tokens."""
    x = synth.activations(M, K, 110 + K, outlier_seed=111 + K)
    x[M // 2] = 0.0
    x[M - 1, K // 3] = 3.0e4
    xq_o, sx_o = oracle.act_quant(x.numpy())
    mats, refs = [], []
    for i, N in enumerate(Ns):
        W = synth.weight(N, K, 112 + i + N)
        Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
        refs.append(oracle.forward(xq_o, sx_o, oracle.pack(Wq_o), sw_o, N, K))
        _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
        mats.append((packed_d, sw_d, torch.full((M, N), float("nan"), device="cuda"),
                     torch.full((M, N), -3, dtype=torch.int32, device="cuda")))
    xq_full = guarded(M * K, torch.int8, 77)
    sx_full = guarded(M, torch.float32, -3.0)
    xq, sx = xq_full[0].view(M, K), sx_full[0]
    for flags in (0, bl.FLAG_PDL):
        bl.bitlinear_linear(x.cuda(), mats, xq, sx, flags=flags)
        assert bl.bitlinear_device_status() == 0
        check_canary(xq_full[1], 77)
        check_canary(sx_full[1], -3.0)
        np.testing.assert_array_equal(xq.cpu().numpy(), xq_o)
        np.testing.assert_array_equal(sx.cpu().numpy(), sx_o)
        for (_, _, y, acc), (acc_o, y_o) in zip(mats, refs):
            np.testing.assert_array_equal(acc.cpu().numpy(), acc_o)
            assert max_rel_err(y.cpu().numpy(), y_o) <= Y_RTOL


def _f32_outputs(acc, sx, sw):
    """The rescale of the BitLinear definition in fp32 steps: f32(acc) / f32(sx * sw)."""
    den = (sx.astype(np.float32)[:, None] * np.float32(sw)).astype(np.float32)
    return (acc.astype(np.float32) / den).astype(np.float32)


@pytest.mark.parametrize("M,K,N,norm", [
    (1, 2560, 10240, False),    # BitNet-3B gate || up at M = 1: fused decode, gated in its epilogue
    (1, 2048, 5632, True),      # with the RMSNorm prologue
    (1, 128, 100, False),       # more CTAs than rows: one row of each matrix a CTA
    (3, 640, 500, False),       # act_quant, then the decode kernel (4-token groups)
    (8, 2560, 2048, False),     # 8-token groups
    (2, 2560, 5120, False),     # two tokens quantised in every CTA (no act_quant launch), gated pairs
    (2, 2560, 10240, False),    # the same at BitNet-3B gate || up widths
    (40, 1024, 1000, False),    # batched tensor-core kernel, then the elementwise gating
    (301, 512, 777, False),     # 128-token tiles; ragged M * N tail
    (200, 8192, 640, False),    # WIDE with a workspace, then the elementwise gating
    (16, 2560, 10240, False),   # 16 tokens, 20480 rows: decode (MMA dots), gated in its epilogue
    (8, 8192, 777, False),      # long K at 8 tokens: decode with K split over a cluster, gated
    (12, 10240, 2560, False),   # long K above 8 tokens: batched tensor-core kernel, then the gating
])
@pytest.mark.parametrize("ws", [False, True])
def test_linear_gated(M, K, N, norm, ws):
    """BITLINEAR_FLAG_GATED: the first output is ReLU^2(gate) * up in the fp32 steps of
    the gating prologue, the second the up output, bit for bit; a following call on that
    output without mul quantises exactly as one on the gate output with mul = up."""
    x = synth.activations(M, K, 100 + K, outlier_seed=101 + K)
    gamma = synth.uniform((K,), 0.5, 1.5, 102 + K) if norm else None
    xq_o, sx_o = oracle.act_quant(x.numpy(), gamma=None if gamma is None else gamma.numpy(), eps=1e-6)
    mats, accs_o, outs_o = [], [], []
    for i in range(2):
        W = synth.weight(N, K, 103 + i + K)
        Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
        acc_o, _ = oracle.forward(xq_o, sx_o, oracle.pack(Wq_o), sw_o, N, K)
        accs_o.append(acc_o)
        outs_o.append(_f32_outputs(acc_o, sx_o, sw_o))
        _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
        mats.append((packed_d, sw_d, torch.full((M, N), float("nan"), device="cuda"),
                     torch.full((M, N), -3, dtype=torch.int32, device="cuda")))
    g, u = outs_o
    r = np.maximum(g, np.float32(0))
    h = ((r * r).astype(np.float32) * u).astype(np.float32)
    xq = torch.zeros(M, K, dtype=torch.int8, device="cuda")
    sx = torch.zeros(M, dtype=torch.float32, device="cuda")
    kw = dict(rms_weight=None if gamma is None else gamma.cuda(), rms_eps=1e-6,
              flags=bl.FLAG_PDL | bl.FLAG_GATED)
    if ws:
        bl.bitlinear_linear_ws(x.cuda(), mats, xq, sx, torch.empty(bl.bitlinear_forward_workspace(M, K),
                                                                   dtype=torch.uint8, device="cuda"), **kw)
    else:
        bl.bitlinear_linear(x.cuda(), mats, xq, sx, **kw)
    assert bl.bitlinear_device_status() == 0
    np.testing.assert_array_equal(xq.cpu().numpy(), xq_o)
    np.testing.assert_array_equal(sx.cpu().numpy(), sx_o)
    for (_, _, _, acc), acc_o in zip(mats, accs_o):
        np.testing.assert_array_equal(acc.cpu().numpy(), acc_o)
    np.testing.assert_array_equal(mats[1][2].cpu().numpy(), u)
    np.testing.assert_array_equal(mats[0][2].cpu().numpy(), h)
    if N % 64 == 0 and M <= 8:
        # the down projection's input: h alone, against the oracle's gating prologue on g and u
        xq2_o, sx2_o = oracle.act_quant(g, mul=u)
        xq2, sx2, _ = gpu_act_quant(mats[0][2].cpu(), None, None)
        np.testing.assert_array_equal(xq2, xq2_o)
        np.testing.assert_array_equal(sx2, sx2_o)


# Matrices that the AUTO rule gives to the same tensor-core kernel share one
# grid whose column tiles span all of them; each case names the kernel(s) its
# shapes select (batched: M <= 128, N <= 4096, M >= 64 or K < 8192; the
# 128-token-tile kernel otherwise).  Ragged N puts a matrix boundary inside a
# wave and leaves partial tiles in the middle of the tile index space.
@pytest.mark.parametrize("M,K,Ns", [
    (32, 2560, (2560, 2560)),             # batched: two matrices (BitNet-3B q, k widths)
    (32, 2048, (300, 1000, 64)),          # batched: three ragged matrices
    (130, 1024, (257, 100, 1000)),        # 128-token tiles: three ragged matrices, ragged M
    (130, 12288, (300, 200)),             # 128-token tiles, split-K with two matrices
    (512, 512, (1000, 1500)),             # 128-token tiles: two matrices, four token tiles
    (512, 640, (130, 2000, 40)),          # 128-token tiles: three matrices
    (64, 12288, (300, 520, 96)),          # batched, split-K with three matrices
    (32, 1024, (5000, 2000, 700)),        # one 128-token-tile launch + one batched launch of two
], ids=lambda v: str(v))
def test_linear_tensor_core_groups(M, K, Ns):
    x = synth.activations(M, K, 80 + K, outlier_seed=81 + K)
    xq_o, sx_o = oracle.act_quant(x.numpy())
    mats, refs = [], []
    for i, N in enumerate(Ns):
        W = synth.weight(N, K, 90 + i + N)
        Wq_o, sw_o, _ = oracle.weight_quant(W.numpy())
        refs.append(oracle.forward(xq_o, sx_o, oracle.pack(Wq_o), sw_o, N, K))
        _, _, _, (packed_d, sw_d) = gpu_quantize_weights(W)
        y = torch.full((M, N), float("nan"), device="cuda")
        acc = torch.full((M, N), -3, dtype=torch.int32, device="cuda")
        mats.append((packed_d, sw_d, y, acc))
    xq = torch.zeros(M, K, dtype=torch.int8, device="cuda")
    sx = torch.zeros(M, dtype=torch.float32, device="cuda")
    for flags in (0, bl.FLAG_PDL):
        for (_, _, y, acc) in mats:
            y.fill_(float("nan"))
            acc.fill_(-3)
        bl.bitlinear_linear(x.cuda(), mats, xq, sx, flags=flags)
        assert bl.bitlinear_device_status() == 0
        np.testing.assert_array_equal(xq.cpu().numpy(), xq_o)
        for (packed_d, sw_d, y, acc), (acc_o, y_o) in zip(mats, refs):
            np.testing.assert_array_equal(acc.cpu().numpy(), acc_o)
            assert max_rel_err(y.cpu().numpy(), y_o) <= Y_RTOL


# --- greedy choice after the LM head -------------------------------------------
def _gpu_argmax(y):
    """y: numpy fp32 [M, N] -> int32 [M] through bitlinear_argmax (canary-guarded)."""
    M, N = y.shape
    idx, ifull = guarded(M, torch.int32, -5)
    bl.bitlinear_argmax(torch.from_numpy(np.ascontiguousarray(y)).cuda(), idx)
    assert bl.bitlinear_device_status() == 0
    check_canary(ifull, -5)
    return idx.cpu().numpy()


@pytest.mark.parametrize("M,N", [(1, 1), (3, 50000), (5, 257), (2, 4), (4, 3001), (65537, 8)])
def test_argmax_matches_oracle(M, N):
    g = torch.Generator().manual_seed(40 + N % 97)
    y = torch.randn(M, N, generator=g).numpy().astype(np.float32)
    # planted ties: the row maximum again, later in the row
    for m in range(min(M, 64)):
        j = int(np.argmax(y[m]))
        if j + 1 < N:
            y[m, N - 1] = y[m, j]
    np.testing.assert_array_equal(_gpu_argmax(y), oracle.argmax(y))


def test_argmax_special_rows():
    y = np.array([[0.0, -0.0, 0.0, -1.0], [-np.inf, -np.inf, -3.0, -np.inf],
                  [1.0, 1.0, 1.0, 1.0], [-2.0, 5.0, 5.0, 4.0]], np.float32)
    np.testing.assert_array_equal(_gpu_argmax(y), oracle.argmax(y))


def test_argmax_unaligned_rows():
    """N odd and a base that is only 4-byte aligned: the scalar scan."""
    M, N = 3, 1001
    g = torch.Generator().manual_seed(41)
    buf = torch.randn(M * N + 1, generator=g).cuda()
    y = buf[1:].view(M, N)
    idx = torch.empty(M, dtype=torch.int32, device="cuda")
    bl.bitlinear_argmax(y, idx)
    assert bl.bitlinear_device_status() == 0
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle.argmax(y.cpu().numpy()))


@pytest.mark.parametrize("M", [1, 3])
def test_lm_head_greedy_token(M):
    """LM head 2560 -> 50000 (BitNet-3B vocabulary) then the greedy token: the GPU
    index is the oracle's argmax of the GPU logits, and a maximum of the oracle's
    own fp64 logits up to the fp32 rescale's rounding."""
    N, K = synth.VOCAB, synth.DIM_3B
    W = synth.weight(N, K, synth.SEEDS["weight_set"]["lm_head"])
    x = synth.activations(M, K, synth.SEEDS["weight_set"]["x"])
    _, sw, _, (packed_d, sw_d) = gpu_quantize_weights(W)
    xq, sx, (xq_d, sx_d) = gpu_act_quant(x)
    acc_g, y_g = gpu_forward(xq_d, sx_d, packed_d, sw_d, N)
    idx = _gpu_argmax(y_g)
    np.testing.assert_array_equal(idx, oracle.argmax(y_g))
    Wq, sw_o, _ = oracle.weight_quant(W.numpy())
    assert sw == sw_o
    acc_o, y_o = oracle.forward(xq, sx, oracle.pack(Wq), sw_o, N, K)
    # the head's integer accumulators, every one of the 50000 per token
    np.testing.assert_array_equal(acc_g, acc_o)
    assert max_rel_err(y_g, y_o) <= Y_RTOL
    for m in range(M):
        best = y_o[m].max()
        assert y_o[m, idx[m]] >= best - Y_RTOL * abs(best)
