"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what it pins and which plausible mistake it would catch:
hand-worked values, the pages' printed weight sizes, exactly rounded sums
from the Python standard library, exact rational arithmetic, closed forms
and invariants.  CPU only.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from golden_io import as_array, read_kv, read_table


# --------------------------------------------------------------------------
# 1. The hand-worked 4x4 example (tests/golden/worked_4x4.txt).
#    Catches: wrong rounding mode, wrong eps path, transposed operands,
#    wrong rescale, wrong bit positions in the packed layout.
# --------------------------------------------------------------------------
def test_worked_4x4():
    g = read_kv("worked_4x4.txt")
    W = as_array(g["W"], np.float32)
    x = as_array(g["x"], np.float32)
    r = oracle.bitlinear(x, W)
    Wq, sw, mean = oracle.weight_quant(W)
    assert mean == float(g["mean"][0][0])
    assert r["sw"] == float(g["sw"][0][0])
    np.testing.assert_array_equal(r["Wq"], as_array(g["Wq"], np.int8))
    np.testing.assert_array_equal(r["sx"], as_array(g["sx"], np.float32).ravel())
    np.testing.assert_array_equal(r["xq"], as_array(g["xq"], np.int8))
    np.testing.assert_array_equal(r["acc"], as_array(g["acc"], np.int32))
    y_ref = as_array(g["y"], np.float64)
    np.testing.assert_allclose(r["y"], y_ref, rtol=1e-15, atol=0)
    words = r["packed"].view("<u4").reshape(4, 4)  # 4 rows x 4 words of one k-block
    np.testing.assert_array_equal(words[:, 0], as_array(g["packed_word0"], np.uint32).ravel())
    assert np.all(words[:, 1:] == int(g["packed_other_words"][0][0], 0))


# --------------------------------------------------------------------------
# 2. Packed sizes against the pages' printed figures.
#    Catches: a layout that is not 0.25 B/weight, wrong padding rule.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("row", read_table("page_sizes.txt"), ids=lambda r: r[0])
def test_packed_bytes_match_page_sizes(row):
    name, N, K, count, fig, unit, cite = row
    N, K, count = int(N), int(K), int(count)
    b = oracle.packed_bytes(N, K)
    assert b * 4 == N * K  # K % 64 == 0 here: exactly 2 bits per weight
    total_mb = count * b / 1e6
    dec = len(fig.split(".")[1]) if "." in fig else 0
    scale = 10 ** dec
    printed = float(fig)
    assert printed in (round(total_mb, dec), math.floor(total_mb * scale) / scale), (name, total_mb, cite)


def test_packed_bytes_padding():
    assert oracle.packed_bytes(3, 1) == 3 * 16
    assert oracle.packed_bytes(3, 64) == 3 * 16
    assert oracle.packed_bytes(3, 65) == 3 * 32
    assert oracle.packed_bytes(0, 64) == 0


# --------------------------------------------------------------------------
# 3. Exact sums against the standard library's exactly rounded math.fsum and
#    against Fraction arithmetic.  Catches: an fp32/fp64 running sum, a lost
#    carry, a wrong exponent bias, wrong subnormal handling, wrong rounding.
# --------------------------------------------------------------------------
def _wide_range_floats(rng, n):
    mant = rng.standard_normal(n)
    expo = rng.integers(-140, 100, n)
    v = (mant * np.exp2(expo)).astype(np.float32)
    v[rng.integers(0, n, n // 10)] = 0.0
    v[:8] = np.array([1e-45, -1e-45, 2e-40, -3e-39, 3.4e38, -1.7e38, 1.0, -1.0], np.float32)
    return v


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_exact_abs_sum_is_correctly_rounded(seed):
    rng = np.random.default_rng(seed)
    v = _wide_range_floats(rng, 4000)
    ref = math.fsum(abs(float(t)) for t in v)
    assert oracle.exact_abs_sum(v) == ref
    ref_frac = float(sum((abs(Fraction(float(t))) for t in v), Fraction(0)))
    assert oracle.exact_abs_sum(v) == ref_frac


@pytest.mark.parametrize("seed", [3, 4])
def test_exact_sq_sum_is_correctly_rounded(seed):
    rng = np.random.default_rng(seed)
    v = _wide_range_floats(rng, 3000)
    v[:6] = np.array([1e-45, 3.4e38, 2.0, 1e-20, -5e-39, 7.0], np.float32)
    ref = math.fsum(float(t) * float(t) for t in v)  # squares of floats are exact in fp64
    assert oracle.exact_sq_sum(v) == ref


def test_exact_sums_of_subnormals():
    # subnormals alone: |v| = frac * 2^-149 exactly (no hidden bit)
    v = np.array([1e-45, -1e-45, 1e-45, 2.5e-44, -1.1754942e-38, 5e-40], np.float32)
    ref = math.fsum(abs(float(t)) for t in v)
    assert ref > 0 and oracle.exact_abs_sum(v) == ref
    assert oracle.exact_abs_sum(np.array([1e-45] * 3, np.float32)) == 3 * 2.0 ** -149
    assert oracle.exact_sq_sum(np.array([1e-45, -1e-45], np.float32)) == 2 * 2.0 ** -298
    assert oracle.exact_sq_sum(v) == math.fsum(float(t) * float(t) for t in v)


def test_exact_sum_rounding_ties():
    # 2^53 + 1 (exact) must round to even 2^53; 2^53 + 3 rounds up to 2^53 + 4.
    big = np.float32(2.0 ** 52)
    one = np.float32(1.0)
    assert oracle.exact_abs_sum(np.array([big, big, one], np.float32)) == 2.0 ** 53
    assert oracle.exact_abs_sum(np.array([big, big, one, one, one], np.float32)) == 2.0 ** 53 + 4
    # A tiny term decides a tie: 2^53 + 1 + 2^-100 rounds up.
    tiny = np.float32(2.0 ** -100)
    assert oracle.exact_abs_sum(np.array([big, big, one, tiny], np.float32)) == 2.0 ** 53 + 2
    assert oracle.exact_abs_sum(np.zeros(5, np.float32)) == 0.0


# --------------------------------------------------------------------------
# 4. weight_quant: mean, scale, rounding ties, clamp, eps, fp32 decisions.
# --------------------------------------------------------------------------
def test_weight_quant_mean_matches_exact_mean():
    rng = np.random.default_rng(7)
    W = (rng.standard_normal((37, 91)) * 0.02).astype(np.float32)
    Wq, sw, mean = oracle.weight_quant(W)
    exact = sum((abs(Fraction(float(t))) for t in W.ravel()), Fraction(0)) / W.size
    # mean is the exact mean rounded via fp64 to fp32: within one fp32 ulp of it
    assert abs(Fraction(mean) - exact) <= Fraction(float(np.spacing(np.float32(mean))))
    assert sw == float(np.float32(1.0) / np.float32(mean))
    assert set(np.unique(Wq)) <= {-1, 0, 1}


def test_weight_quant_ties_round_to_even():
    # mean|W| = 1 -> sw = 1, so Wq = clamp(rne(W)).
    # sum|row 0| = 10, row 1 = 8 x 0.75 = 6: mean|W| = 16/16 = 1 exactly.
    W = np.array([[0.5, -0.5, 1.5, -1.5, 2.5, -2.5, 0.375, -0.625],
                  [0.75] * 8], np.float32)
    Wq, sw, mean = oracle.weight_quant(W)
    assert mean == 1.0 and sw == 1.0
    np.testing.assert_array_equal(Wq[0], [0, 0, 1, -1, 1, -1, 0, -1])
    np.testing.assert_array_equal(Wq[1], 1)


def test_weight_quant_eps_path():
    W = np.zeros((4, 8), np.float32)
    Wq, sw, mean = oracle.weight_quant(W)
    assert mean == 0.0 and sw == float(np.float32(1.0) / np.float32(1e-5))
    assert np.all(Wq == 0)
    W[0, 0] = 1e-7  # mean 3.1e-9 < eps: the eps clamp decides sw
    Wq, sw2, _ = oracle.weight_quant(W)
    assert sw2 == sw and Wq[0, 0] == 0  # 1e-7 * 1e5 = 0.01 -> 0


def test_weight_quant_ternary_is_fixed_point():
    # Any ternary W has mean|W| <= 1, hence sw >= 1 and |W*sw| >= 1 on nonzeros.
    rng = np.random.default_rng(11)
    W = rng.integers(-1, 2, (13, 70)).astype(np.float32)
    Wq, _, _ = oracle.weight_quant(W)
    np.testing.assert_array_equal(Wq, W.astype(np.int8))


def test_weight_quant_decides_in_fp32():
    # sum|W| = 24 over 8 entries: mean = 3, sw = fp32(1/3) = 0.33333334 (just above 1/3).
    # 1.5 * sw = 0.50000001 exactly, which rounds to the fp32 tie 0.5 -> 0 (even);
    # an fp64 product would round up to 1.  4.5 * sw rounds to 1.5 -> 2 -> clamp 1.
    W = np.array([[1.5, -1.5, 4.5, -4.5, 3, 3, 3, -3]], np.float32)
    Wq, sw, mean = oracle.weight_quant(W)
    assert mean == 3.0 and sw == float(np.float32(1) / np.float32(3))
    np.testing.assert_array_equal(Wq[0], [0, 0, 1, -1, 1, 1, 1, -1])


# --------------------------------------------------------------------------
# 5. act_quant: ties, eps path, clamp invariant, outliers.
# --------------------------------------------------------------------------
def test_act_quant_ties_and_scale():
    x = np.array([[127, -63.5, 0.5, 1.5, 2.5, -0.5, -1.5, 126.5]], np.float32)
    xq, sx = oracle.act_quant(x)
    assert sx[0] == 1.0
    np.testing.assert_array_equal(xq[0], [127, -64, 0, 2, 2, 0, -2, 126])


def test_act_quant_eps_rows():
    x = np.array([[0, 0, 0, 0], [1e-6, -2e-6, 0, 0], [1e-5, 0, 0, 0]], np.float32)
    xq, sx = oracle.act_quant(x)
    assert sx[0] == np.float32(127.0) / np.float32(1e-5) == np.float32(12700000.0)
    assert sx[1] == sx[0]
    np.testing.assert_array_equal(xq[0], 0)
    np.testing.assert_array_equal(xq[1], [13, -25, 0, 0])
    assert xq[2, 0] == 127


def test_act_quant_bound_never_reaches_minus_128():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[:, :3] *= 20
    x[7] = -np.abs(x[7])
    xq, sx = oracle.act_quant(x)
    assert np.abs(xq.astype(np.int32)).max() == 127
    assert xq.min() >= -127
    # the row maximum always maps to +-127 exactly
    amax_idx = np.abs(x).argmax(axis=1)
    np.testing.assert_array_equal(np.abs(xq[np.arange(64), amax_idx]), 127)


def test_act_quant_decides_in_fp32():
    # amax = 381 -> sx = fp32(127/381) = fp32(1/3) = 0.33333334.  1.5 * sx is
    # 0.50000001 exactly, an fp32 tie 0.5 after rounding -> 0 (an fp64 product
    # would give 1); 4.5 * sx -> 1.5 -> 2; -7.5 * sx -> -2.5 -> -2.
    x = np.array([[381.0, 1.5, 4.5, -7.5]], np.float32)
    xq, sx = oracle.act_quant(x)
    assert sx[0] == np.float32(1) / np.float32(3)
    np.testing.assert_array_equal(xq[0], [127, 0, 2, -2])


# --------------------------------------------------------------------------
# 6. Prologues: ReLU^2 * mul and RMSNorm closed forms.
# --------------------------------------------------------------------------
def test_relu_sq_mul_closed_form():
    g = np.array([[-1.0, 0.0, 2.0, 3.0, -0.0, 0.5]], np.float32)
    u = np.array([[5.0, 5.0, 0.5, -1.0, 9.0, 4.0]], np.float32)
    xq, sx, h = oracle.act_quant(g, mul=u, return_h=True)
    np.testing.assert_array_equal(h[0], [0, 0, 2, -9, 0, 1])


def test_rmsnorm_power_of_two_constants_are_exact():
    # eps = 0, x = c (a power of two): mean(x^2) = c^2, inv = 1/|c|, xn = sign * gamma
    for c in (1.0, 2.0, 0.25, -8.0):
        x = np.full((1, 16), c, np.float32)
        gamma = np.arange(1, 17, dtype=np.float32)
        _, _, h = oracle.act_quant(x, gamma=gamma, eps=0.0, return_h=True)
        np.testing.assert_array_equal(h[0], np.sign(c) * gamma)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((3, 100)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, 100).astype(np.float32)
    _, _, h1 = oracle.act_quant(x, gamma=gamma, eps=0.0, return_h=True)
    _, _, h2 = oracle.act_quant(x * np.float32(64.0), gamma=gamma, eps=0.0, return_h=True)
    np.testing.assert_array_equal(h1, h2)


def test_rmsnorm_unit_rms_and_eps():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 512)).astype(np.float32)
    _, _, h = oracle.act_quant(x, gamma=np.ones(512, np.float32), eps=0.0, return_h=True)
    np.testing.assert_allclose((h.astype(np.float64) ** 2).mean(axis=1), 1.0, rtol=1e-6)
    # a constant row c with eps: xn = c / sqrt(c^2 + eps) (exact value within 2 fp32 ulps)
    c, eps = 0.001, 1e-6
    x = np.full((1, 8), c, np.float32)
    _, _, h = oracle.act_quant(x, gamma=np.ones(8, np.float32), eps=eps, return_h=True)
    exact = float(np.float32(c)) / math.sqrt(float(np.float32(c)) ** 2 + eps)
    assert abs(h[0, 0] - exact) <= 2 * np.spacing(np.float32(exact))
    # all-zero row: inv = 1/sqrt(eps) is finite, the output is zero
    xq, sx, h = oracle.act_quant(np.zeros((1, 8), np.float32), gamma=np.ones(8, np.float32),
                                 eps=1e-6, return_h=True)
    assert np.all(h == 0) and np.all(xq == 0)


def test_gate_then_norm_order():
    # h = relu(g)^2 * u = [4, 4, 0, 4]; RMSNorm (eps 0): sqrt(48/4) = 2*sqrt(3),
    # so nonzero entries become 2/sqrt(3).  Norm-then-gate would give another value.
    g = np.array([[2.0, 2.0, -1.0, 2.0]], np.float32)
    u = np.array([[1.0, 1.0, 7.0, 1.0]], np.float32)
    _, _, h = oracle.act_quant(g, mul=u, gamma=np.ones(4, np.float32), eps=0.0, return_h=True)
    want = 2.0 / math.sqrt(3.0)
    for k in (0, 1, 3):
        assert abs(h[0, k] - want) <= 2 * np.spacing(np.float32(want))
    assert h[0, 2] == 0


# --------------------------------------------------------------------------
# 7. Pack / unpack: round trip, padding, invalid code, single-code positions.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("N,K", [(1, 1), (3, 64), (5, 100), (33, 130), (7, 256)])
def test_pack_roundtrip(N, K):
    rng = np.random.default_rng(N * 1000 + K)
    Wq = rng.integers(-1, 2, (N, K)).astype(np.int8)
    p = oracle.pack(Wq)
    np.testing.assert_array_equal(oracle.unpack(p, N, K), Wq)
    codes = np.stack([(p >> s) & 3 for s in (0, 2, 4, 6)])
    assert not np.any(codes == 3)


def test_pack_single_code_position():
    # One +1 (code 2) in an all-zero (code 1 = 0x55 bytes) matrix changes exactly
    # one byte: chunk (kb*N + n)*16, word (k%64)//16, byte i%4, bits 2*(i//4).
    N, K = 6, 192
    for n, k in [(0, 0), (5, 191), (2, 77), (3, 64 + 16 + 5)]:
        Wq = np.zeros((N, K), np.int8)
        Wq[n, k] = 1
        p = oracle.pack(Wq)
        diff = np.nonzero(p != 0x55)[0]
        i = k % 16
        want_byte = ((k // 64) * N + n) * 16 + 4 * ((k % 64) // 16) + (i % 4)
        assert list(diff) == [want_byte]
        assert p[want_byte] == (0x55 & ~(3 << 2 * (i // 4))) | (2 << 2 * (i // 4))


def test_pack_padding_and_invalid_code():
    Wq = np.ones((2, 10), np.int8)
    p = oracle.pack(Wq)
    assert p.size == 32
    # k >= 10 is padding: the unpacked padding weights are 0
    big = oracle.unpack(np.concatenate([p]), 2, 10)
    np.testing.assert_array_equal(big, Wq)
    bad = p.copy()
    bad[0] |= 0x03  # code 3 at k = 0 of row 0
    with pytest.raises(oracle.OracleError):
        oracle.unpack(bad, 2, 10)
    with pytest.raises(oracle.OracleError):
        oracle.pack(np.full((1, 4), 2, np.int8))


# --------------------------------------------------------------------------
# 8. Contraction and rescale: brute force in exact arithmetic, closed forms.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_forward_bruteforce_exact(seed):
    rng = np.random.default_rng(100 + seed)
    M, N, K = rng.integers(1, 9, 3)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    r = oracle.bitlinear(x, W)
    acc64 = r["xq"].astype(np.int64) @ r["Wq"].astype(np.int64).T
    np.testing.assert_array_equal(r["acc"], acc64)
    for m in range(M):
        for n in range(N):
            exact = Fraction(int(acc64[m, n])) / (Fraction(float(r["sx"][m])) * Fraction(r["sw"]))
            assert r["y"][m, n] == float(exact)  # one correctly rounded division
            # and the fake-quant form sum_k (xq/sx)(Wq/sw) is the same number
            fq = sum(Fraction(int(r["xq"][m, k])) / Fraction(float(r["sx"][m]))
                     * Fraction(int(r["Wq"][n, k])) / Fraction(r["sw"]) for k in range(K))
            assert fq == exact


def test_forward_packed_equals_unpacked():
    rng = np.random.default_rng(21)
    M, N, K = 5, 40, 200
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal((M, K)).astype(np.float32)
    Wq, sw, _ = oracle.weight_quant(W)
    xq, sx = oracle.act_quant(x)
    a1, y1 = oracle.forward(xq, sx, oracle.pack(Wq), sw, N, K)
    a2, y2 = oracle.forward_unpacked(xq, sx, Wq, sw)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(y1, y2)


def test_integer_inputs_are_fixed_points():
    # ternary W with mean 1 and integer x with row max 127: both quantisers are
    # identities and y is the exact integer matmul.
    rng = np.random.default_rng(22)
    M, N, K = 6, 9, 64
    W = rng.choice([-1.0, 1.0], (N, K)).astype(np.float32)
    x = rng.integers(-127, 128, (M, K)).astype(np.float32)
    x[:, 0] = 127.0
    r = oracle.bitlinear(x, W)
    assert r["sw"] == 1.0 and np.all(r["sx"] == 1.0)
    want = x.astype(np.int64) @ W.astype(np.int64).T
    np.testing.assert_array_equal(r["acc"], want)
    np.testing.assert_array_equal(r["y"], want.astype(np.float64))


def test_constant_weights_closed_form():
    # W == c > 1e-5: mean = c, Wq == 1, y = sum_k xq / (sx * (1/c)).
    c = np.float32(0.25)
    W = np.full((3, 64), c, np.float32)
    rng = np.random.default_rng(23)
    x = rng.standard_normal((2, 64)).astype(np.float32)
    r = oracle.bitlinear(x, W)
    assert np.all(r["Wq"] == 1) and r["sw"] == 4.0
    s = r["xq"].astype(np.int64).sum(axis=1)
    np.testing.assert_array_equal(r["acc"], np.repeat(s[:, None], 3, axis=1))
    np.testing.assert_allclose(r["y"], (s / r["sx"].astype(np.float64) / 4.0)[:, None].repeat(3, 1), rtol=1e-15)


def test_one_hot_activation_closed_form():
    # x = a e_k0 with a >= 1e-5: xq = 127 e_k0, sx = 127/a, y = a * Wq[:, k0] / sw
    rng = np.random.default_rng(24)
    W = (rng.standard_normal((10, 64)) * 0.02).astype(np.float32)
    a, k0 = np.float32(3.0), 17
    x = np.zeros((1, 64), np.float32)
    x[0, k0] = a
    r = oracle.bitlinear(x, W)
    np.testing.assert_array_equal(r["xq"][0], 127 * (np.arange(64) == k0))
    want = float(a) * r["Wq"][:, k0].astype(np.float64) / r["sw"]
    np.testing.assert_allclose(r["y"][0], want, rtol=1e-6)


def test_zero_weights_give_zero():
    W = np.zeros((4, 64), np.float32)
    x = np.random.default_rng(25).standard_normal((3, 64)).astype(np.float32)
    r = oracle.bitlinear(x, W)
    assert r["sw"] == float(np.float32(1) / np.float32(1e-5))
    assert np.all(r["y"] == 0) and np.all(r["acc"] == 0)


# --- greedy choice after the LM head ------------------------------------------
# Hand-worked rows with known answers: the first index of the row maximum.
@pytest.mark.parametrize("row, want", [
    ([1.0, 3.0, 3.0, 2.0], 1),            # tie: the earlier index
    ([-5.0, -1.0, -1.0, -7.0], 1),        # all negative
    ([0.0, -0.0, 0.0, -1.0], 0),          # -0 and +0 are equal
    ([7.5], 0),                           # one element
    ([-np.inf, -3.0], 1),
    ([2.0, 1.0, 1.0, 2.0, 2.5], 4),       # maximum last
    ([1e30, 1e30 * 1.0000001, 1e30], 1),  # one ulp apart in fp32
])
def test_argmax_hand_rows(row, want):
    y = np.array([row], np.float32)
    assert oracle.argmax(y)[0] == want


def test_argmax_rows_are_independent_one_hot():
    M, N = 3, 50000
    y = np.zeros((M, N), np.float32)
    hot = [31337, 0, N - 1]
    for m, h in enumerate(hot):
        y[m, h] = 1.0
    assert list(oracle.argmax(y)) == hot


# --- RMSNorm scale next to an fp32 rounding boundary ----------------------------
# The boundary rows (one repeated value c per row, K = 2560) must sit where
# their table says: the fp64 chain 1/sqrt(c^2 + eps), each step rounded, lies
# that many fp64 ulps from the midpoint between two fp32 values.  numpy's fp64
# sqrt and division round correctly, so this recomputes the chain exactly.
def test_rms_boundary_rows_sit_on_the_boundary():
    from harness import RMS_BOUNDARY_ROWS
    for eps, bits, dist in RMS_BOUNDARY_ROWS:
        c = float(np.array([bits], dtype=np.uint32).view(np.float32)[0])
        y = np.float64(1.0) / np.sqrt(np.float64(c) * np.float64(c) + np.float64(eps))
        low = int(np.array([y]).view(np.uint64)[0]) & ((1 << 29) - 1)
        assert low - (1 << 28) == dist, (eps, hex(bits))


# With eps = 0 the chain collapses (sqrt(c^2) = |c| exactly), so the oracle's
# normalised row is a closed form: inv = fp32(fp64(1/|c|)), h = fp32(fp32(x*inv)*gamma).
def test_rms_boundary_rows_closed_form():
    from harness import RMS_BOUNDARY_ROWS, rms_boundary_gamma, rms_boundary_rows
    gamma = rms_boundary_gamma()
    x = rms_boundary_rows(0.0)
    _, sx, h = oracle.act_quant(x, gamma=gamma, eps=0.0, return_h=True)
    for m in range(x.shape[0]):
        c = abs(float(x[m, 0]))
        inv = np.float32(np.float64(1.0) / np.float64(c))
        want = ((x[m] * inv).astype(np.float32) * gamma).astype(np.float32)
        np.testing.assert_array_equal(h[m], want)
        assert sx[m] == np.float32(127.0) / np.abs(want).max()
