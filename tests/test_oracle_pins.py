"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: hand-worked
values from the formulas (tests/golden), brute force with exact fractions or
plain integer loops, closed forms, library routines that the oracle does not
use, and invariants the pages state. Every oracle function has at least one
pin that a plausible slip (dropped eps, wrong rounding mode, swapped operand,
wrong bit order, wrong sign) would fail.
"""
import math
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as O
from tests.golden import as_array, load
from ternary_weight_linear_06_b300 import workloads as WL

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------- rounding
def test_round_rational_matches_numpy_double_to_float():
    # numpy's float64 -> float32 conversion is IEEE round-to-nearest-even; for
    # a double d the exact rational is d itself.
    rng = random.Random(1)
    for _ in range(3000):
        d = rng.uniform(-1, 1) * 2.0 ** rng.randint(-160, 120)
        d = abs(d)
        fr = Fraction(d)
        got = O.round_rational_to_f32(fr.numerator, fr.denominator)
        want = np.float32(d)
        assert got.view(np.uint32) == want.view(np.uint32), d


def test_round_rational_ties_and_subnormals():
    two = Fraction(2)
    cases = [
        (Fraction(2 ** 24 + 1), 2.0 ** 24),             # tie -> even (down)
        (Fraction(2 ** 24 + 3), 2.0 ** 24 + 4),         # tie -> even (up)
        (Fraction(3, 2) * two ** -149, 2.0 ** -148),    # subnormal tie -> even
        (Fraction(1, 2) * two ** -149, 0.0),            # below half the min -> 0
        (Fraction(5, 8) * two ** -149, 2.0 ** -149),
        (Fraction(1, 3), float(np.float32(1.0) / np.float32(3.0))),
    ]
    for x, want in cases:
        got = O.round_rational_to_f32(x.numerator, x.denominator)
        assert float(got) == want, (x, got, want)


# ------------------------------------------------------------------- gamma
def _gamma_bruteforce(W):
    a = np.abs(np.asarray(W, np.float32)).ravel()
    s = sum(Fraction(float(v)) for v in a)
    r = s / a.size
    return O.round_rational_to_f32(r.numerator, r.denominator)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_gamma_equals_exact_fraction_bruteforce(seed):
    rng = np.random.default_rng(seed)
    # mixed magnitudes incl. subnormals and large values, both signs
    W = (rng.standard_normal(300) * 10.0 ** rng.uniform(-44, 30, 300)).astype(np.float32)
    W[:5] = np.array([1e-45, -3e-45, 0.0, -0.0, 1e30], np.float32)
    assert O.absmean_gamma(W).view(np.uint32) == _gamma_bruteforce(W).view(np.uint32)


def test_gamma_config1_bruteforce():
    W, _ = WL.tiny_case(0)
    assert O.absmean_gamma(W).view(np.uint32) == _gamma_bruteforce(W).view(np.uint32)


def test_gamma_hand_values_and_ties():
    g = load("hand_rounding.txt")
    assert O.absmean_gamma(np.array([1, 2, 3, 4], np.float32)) == np.float32(2.5)
    assert O.absmean_gamma(np.array([-1, 2, -3, 4], np.float32)) == np.float32(2.5)
    for key in ("a", "b"):
        W = as_array(g[f"gamma_tie_{key}_w"], np.float64).astype(np.float32)
        want = as_array(g[f"gamma_tie_{key}"], np.float64).astype(np.float32)[0]
        assert O.absmean_gamma(W) == want


def test_gamma_is_order_independent_where_naive_fp32_is_not():
    W = np.array([2.0 ** 24] + [1.0] * 64, np.float32)
    g1 = O.absmean_gamma(W)
    g2 = O.absmean_gamma(W[::-1].copy())
    assert g1.view(np.uint32) == g2.view(np.uint32)
    exact = Fraction(2 ** 24 + 64, 65)
    assert g1 == O.round_rational_to_f32(exact.numerator, exact.denominator)
    naive = np.float32(0)
    for v in W:
        naive = np.float32(naive + v)
    assert np.float32(naive / np.float32(65)) != g1   # 2^24 + 1.0 loses each 1.0


def test_gamma_closed_form_gaussian():
    # E|W| = sigma * sqrt(2/pi) for W ~ N(0, sigma^2); SE = sigma*sqrt(1-2/pi)/sqrt(n)
    sigma, n = 0.02, 1 << 20
    W = WL.gaussian_weights(1024, 1024, sigma, seed=11)
    want = sigma * math.sqrt(2 / math.pi)
    se = sigma * math.sqrt(1 - 2 / math.pi) / math.sqrt(n)
    assert abs(float(O.absmean_gamma(W)) - want) < 5 * se


def test_weight_scale_adds_eps_in_fp32():
    assert O.weight_scale(np.float32(0.0)) == np.float32(1e-5)
    g = np.float32(0.10875)
    assert O.weight_scale(g) == np.float32(g + np.float32(1e-5))
    assert O.weight_scale(g) != g                       # eps not dropped
    _, s_w, t = O.pack_weights(np.zeros((4, 8), np.float32))
    assert s_w == np.float32(1e-5) and not t.any()      # all-zero W stays zero


# --------------------------------------------------------------- ternarize
def test_hand_example_weights():
    g = load("hand_bitlinear.txt")
    W = as_array(g["W"], np.float64).astype(np.float32)
    gamma = O.absmean_gamma(W)
    assert abs(float(gamma) - 0.10875) < 2e-7 * 0.10875
    packed, s_w, t = O.pack_weights(W)
    assert abs(float(s_w) - 0.10876) < 2e-7
    np.testing.assert_array_equal(t, as_array(g["t"], np.int8))
    np.testing.assert_array_equal(packed.ravel(), as_array(g["packed"], np.uint8).ravel())


def test_roundclip_ties_hand():
    g = load("hand_rounding.txt")
    W = as_array(g["ternary_w"], np.float64).astype(np.float32)[None, :]
    np.testing.assert_array_equal(O.ternarize(W, np.float32(1.0))[0],
                                  as_array(g["ternary_t"], np.int8))


def test_ternary_invariants():
    W = WL.gaussian_weights(512, 512, 0.02, seed=3, outlier_frac=0.001)
    _, s_w, t = O.pack_weights(W)
    assert set(np.unique(t)) <= {-1, 0, 1}
    # sign symmetry: t(-W) = -t(W) (gamma is unchanged by the sign)
    _, s_w2, t2 = O.pack_weights(-W)
    assert s_w2 == s_w
    np.testing.assert_array_equal(t2, -t)
    # a constant matrix maps to all ones: W/s_w = c/(c+eps) in (0.5, 1]
    _, _, tc = O.pack_weights(np.full((3, 8), 0.37, np.float32))
    assert (tc == 1).all()
    # positive entries never map to -1 and vice versa
    assert not ((W > 0) & (t < 0)).any() and not ((W < 0) & (t > 0)).any()


def test_zero_fraction_closed_form():
    # t = 0 iff |W| <= s_w/2 ~ sigma*sqrt(2/pi)/2, so P(t=0) = 2*Phi(sqrt(2/pi)/2) - 1
    W = WL.gaussian_weights(1024, 1024, 0.02, seed=5)
    _, _, t = O.pack_weights(W)
    p = math.erf(math.sqrt(2 / math.pi) / 2 / math.sqrt(2))
    assert abs(float((t == 0).mean()) - p) < 0.003
    assert abs(p - 0.3101) < 1e-3


def test_pack_codes_hand_and_roundtrip():
    g = load("hand_rounding.txt")
    t = as_array(g["pack_t"], np.int8)
    np.testing.assert_array_equal(O.pack_codes(t).ravel(), as_array(g["pack_bytes"], np.uint8))
    rng = np.random.default_rng(9)
    t = rng.integers(-1, 2, size=(7, 64)).astype(np.int8)
    np.testing.assert_array_equal(O.unpack_codes(O.pack_codes(t), 64), t)
    # bit order: column k=4b+j sits in bits [2j, 2j+1] of byte b
    t = np.zeros((1, 8), np.int8) - 1
    t[0, 5] = 1                       # byte 1, slot 1 -> code 2 << 2
    assert O.pack_codes(t)[0, 1] == (2 << 2) and O.pack_codes(t)[0, 0] == 0


# -------------------------------------------------------------- act quant
def test_act_quant_hand_and_ties():
    g = load("hand_bitlinear.txt")
    q, m = O.quant_act(as_array(g["X"], np.float64).astype(np.float32)[None, :])
    np.testing.assert_array_equal(q[0], as_array(g["q"], np.int8))
    assert m[0] == np.float32(2.0)
    r = load("hand_rounding.txt")
    q, m = O.quant_act(as_array(r["act_x"], np.float64).astype(np.float32)[None, :])
    np.testing.assert_array_equal(q[0], as_array(r["act_q"], np.int8))


def test_act_quant_invariants():
    _, X = WL.tiny_case(0)
    q, m = O.quant_act(X)
    # the absmax element maps to +-127
    for i in (0, 1, 3):
        j = int(np.argmax(np.abs(X[i])))
        assert abs(int(q[i, j])) == 127 and np.sign(q[i, j]) == np.sign(X[i, j])
    # an all-zero token stays zero with m = eps
    assert not q[2].any() and m[2] == np.float32(1e-5)
    # the 50x outlier row: outlier -> +-127, most others small
    j = int(np.argmax(np.abs(X[3])))
    assert abs(X[3, j]) == 50.0 and abs(int(q[3, j])) == 127
    others = np.delete(q[3], j)
    assert np.mean(np.abs(others) <= 3) > 0.7
    # odd symmetry and power-of-two scale invariance (m scales, q does not)
    q2, m2 = O.quant_act(-X)
    np.testing.assert_array_equal(q2, -q)
    q3, m3 = O.quant_act(X[[0, 1, 3]] * np.float32(8.0))
    np.testing.assert_array_equal(q3, q[[0, 1, 3]])
    np.testing.assert_array_equal(m3, m[[0, 1, 3]] * np.float32(8.0))
    # range
    assert q.min() >= -128 and q.max() <= 127


def test_act_quant_matches_torch_formula_reading():
    # torch (a different library) evaluating the same fp32 expression
    X = WL.student_t(16, 512, seed=4)
    q, m = O.quant_act(X)
    xt = torch.from_numpy(X)
    mt = torch.clamp(xt.abs().amax(dim=1), min=1e-5)
    qt = torch.clamp(torch.round((xt * 127.0) / mt[:, None]), -128, 127).to(torch.int8)
    np.testing.assert_array_equal(q, qt.numpy())
    np.testing.assert_array_equal(m, mt.numpy())


def test_bf16_widening():
    u = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x0000, 0x8000], np.uint16)
    f = O.bf16_bits_to_f32(u)
    assert f[0] == 1.0 and f[1] == -2.0 and f[2] == np.float32(2.0 ** -133)
    assert f[4] == 0.0 and np.signbit(f[5])
    t = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(f.view(np.uint32), t.view(np.uint32))


# ------------------------------------------------------------- int matmul
def test_int_matmul_bruteforce_loops():
    rng = np.random.default_rng(2)
    q = rng.integers(-128, 128, size=(3, 40)).astype(np.int8)
    t = rng.integers(-1, 2, size=(5, 40)).astype(np.int8)
    acc = O.int_matmul(q, t)
    assert acc.shape == (3, 5)
    for i in range(3):
        for j in range(5):
            s = 0
            for k in range(40):
                if t[j, k] == 1:
                    s += int(q[i, k])
                elif t[j, k] == -1:
                    s -= int(q[i, k])
            assert acc[i, j] == s


def test_int_matmul_float64_library_and_invariants():
    rng = np.random.default_rng(3)
    q = rng.integers(-128, 128, size=(6, 2048)).astype(np.int8)
    t = rng.integers(-1, 2, size=(9, 2048)).astype(np.int8)
    acc = O.int_matmul(q, t)
    ref = torch.from_numpy(q.astype(np.float64)) @ torch.from_numpy(t.astype(np.float64)).T
    np.testing.assert_array_equal(acc, ref.numpy().astype(np.int32))
    nnz = (t != 0).sum(axis=1)
    assert (np.abs(acc) <= 128 * nnz[None, :]).all()
    perm = rng.permutation(2048)
    np.testing.assert_array_equal(O.int_matmul(q[:, perm], t[:, perm]), acc)
    # zero weights contribute nothing
    t0 = t.copy()
    t0[:, ::2] = 0
    np.testing.assert_array_equal(O.int_matmul(q, t0), O.int_matmul(q[:, 1::2], t[:, 1::2]))


# ---------------------------------------------------------------- dequant
def test_dequant_hand_and_fp64():
    g = load("hand_bitlinear.txt")
    W = as_array(g["W"], np.float64).astype(np.float32)
    X = as_array(g["X"], np.float64).astype(np.float32)[None, :]
    _, s_w, t = O.pack_weights(W)
    Y, acc, q, m = O.forward(X, t, s_w)
    np.testing.assert_array_equal(acc[0], as_array(g["acc"], np.int32))
    want = as_array(g["y"], np.float64)
    assert np.max(np.abs(Y[0] - want) / np.abs(want)) < 1e-6
    # exact case: s_w = 2, m = 127 gives c = 2 and y = 2 * acc
    y = O.dequant(np.array([[3, -5, 1 << 20]]), np.float32(2.0), np.array([127.0], np.float32))
    np.testing.assert_array_equal(y[0], np.array([6, -10, 2 << 20], np.float32))
    # fp64 recompute
    rng = np.random.default_rng(4)
    acc = rng.integers(-3_000_000, 3_000_000, size=(5, 7))
    m = (10.0 ** rng.uniform(-3, 2, 5)).astype(np.float32)
    y = O.dequant(acc, np.float32(0.0161), m)
    ref = acc * (np.float64(np.float32(0.0161)) * m.astype(np.float64)[:, None] / 127.0)
    assert np.max(np.abs(y - ref) / np.maximum(np.abs(ref), 1e-30)) < 1e-6


def test_forward_zero_token_and_packed_path():
    W, X = WL.tiny_case(0)
    packed, s_w, t = O.pack_weights(W)
    Y, acc, q, m = O.forward(X, t, s_w)
    assert not Y[2].any() and not acc[2].any()
    Y2 = O.forward_packed(X, packed, s_w)[0]
    np.testing.assert_array_equal(Y, Y2)


# -------------------------------------------------------------------- FFN
def test_relu2_and_ffn_composition():
    y = np.array([[-2.0, -0.0, 0.0, 0.5, 3.0]], np.float32)
    np.testing.assert_array_equal(O.relu2(y), np.array([[0, 0, 0, 0.25, 9.0]], np.float32))
    rng = np.random.default_rng(6)
    Wu = WL.gaussian_weights(64, 32, 0.02, seed=7)
    Wd = WL.gaussian_weights(32, 64, 0.02, seed=8)
    X = rng.standard_normal((5, 32)).astype(np.float32)
    _, su, tu = O.pack_weights(Wu)
    _, sd, td = O.pack_weights(Wd)
    Y, h = O.ffn(X, tu, su, td, sd)
    assert (h >= 0).all() and h.shape == (5, 64)
    y_up = O.forward(X, tu, su)[0]
    np.testing.assert_array_equal(h, np.where(y_up > 0, y_up * y_up, 0).astype(np.float32))
    np.testing.assert_array_equal(Y, O.forward(h, td, sd)[0])
    # requant of h is non-negative
    qh, _ = O.quant_act(h)
    assert qh.min() >= 0


def test_gated_ffn_sign_flip_and_zero_gate():
    # Flipping the sign of the gate weights flips the sign of every gate output
    # exactly (the quantizers are odd), so for each element exactly one of the
    # two gated h values is ReLU^2(+-y_gate) * y_up and the other is +-0; their
    # sum is fp32(fp32(y_gate^2) * y_up), computed here from y alone.
    rng = np.random.default_rng(9)
    Wu = WL.gaussian_weights(48, 64, 0.02, seed=10)
    Wg = WL.gaussian_weights(48, 64, 0.02, seed=11)
    Wd = WL.gaussian_weights(64, 48, 0.02, seed=12)
    X = rng.standard_normal((6, 64)).astype(np.float32)
    _, su, tu = O.pack_weights(Wu)
    _, sg, tg = O.pack_weights(Wg)
    _, sgn, tgn = O.pack_weights(-Wg)
    assert sgn == sg and np.array_equal(tgn, -tg)
    _, sd, td = O.pack_weights(Wd)
    _, h1 = O.ffn_gated(X, tu, su, tg, sg, td, sd)
    _, h2 = O.ffn_gated(X, tu, su, tgn, sgn, td, sd)
    y_up = O.forward(X, tu, su)[0].astype(np.float64)
    y_g = O.forward(X, tg, sg)[0].astype(np.float64)
    sq = np.array(y_g * y_g, np.float32).astype(np.float64)          # fp32(y_g^2), exact product in fp64
    expect = np.array(sq * y_up, np.float32)                           # one fp32 rounding of the product
    np.testing.assert_array_equal((h1.astype(np.float64) + h2.astype(np.float64)).astype(np.float32), expect)
    assert np.all((h1 == 0) | (h2 == 0))
    # where the gate is not positive, h is a zero (of either sign) whatever up is
    assert np.all(h1[y_g <= 0] == 0)
    # a gate equal to up gives h = ReLU(y)^2 * y: non-negative, zero for y <= 0
    _, h3 = O.ffn_gated(X, tu, su, tu, su, td, sd)
    assert np.all(h3 >= 0) and np.all(h3[y_up <= 0] == 0)


def test_tie_count_diagnostic():
    s = np.float32(1.0)
    W = np.array([[0.5, np.nextafter(np.float32(0.5), np.float32(1)), 0.3, -0.5]], np.float32)
    assert O.tie_count(W, s) == 3


# ----------------------------------------------------------------- SubLN RMSNorm
def test_rmsnorm_constant_rows_closed_form():
    # x = c in every column: mean x^2 = c^2, so every normalized value is
    # sign(c) * |c| / sqrt(c^2 + e); every code is +-127 and the scale is that
    # magnitude. A sum in place of the mean (1/sqrt(K) off), eps outside the
    # root, or a missing root each miss it by far more than an fp32 step.
    K = 256
    for c in (3.0, -0.75, 1024.0):
        for e in (0.0, 0.5, 1e-5):
            X = np.full((1, K), c, np.float32)
            q, m = O.rmsnorm_quant(X, eps_norm=e)
            assert np.all(q == (127 if c > 0 else -127))
            want = abs(c) / math.sqrt(c * c + float(np.float32(e)))
            assert abs(float(m[0]) - want) <= 2.0 ** -23 * want, (c, e, m[0], want)


def test_rmsnorm_one_hot_gain():
    # A gain that keeps one column j: u has one non-zero entry, so its code is
    # +-127 (sign of x_j * gain) and every other code is 0. The scale is
    # |x_j * gain| / sqrt(rms(x)^2 + e): the statistic is over x, not over the
    # gained row (which would give sqrt(K) / |gain| instead).
    rng = np.random.default_rng(21)
    K, j, gam, e = 128, 37, np.float32(-2.5), 0.25
    X = rng.standard_normal((5, K)).astype(np.float32)
    g = np.zeros(K, np.float32)
    g[j] = gam
    q, m = O.rmsnorm_quant(X, g, eps_norm=e)
    want_q = np.zeros_like(q)
    want_q[:, j] = np.where(X[:, j] * gam > 0, 127, -127)
    np.testing.assert_array_equal(q, want_q)
    rms = np.linalg.norm(X.astype(np.float64), axis=1) / math.sqrt(K)
    want = np.abs(X[:, j].astype(np.float64) * float(gam)) / np.sqrt(rms ** 2 + e)
    np.testing.assert_allclose(m.astype(np.float64), want, rtol=2.5e-7)


def test_rmsnorm_scale_invariance_without_eps():
    # With eps_norm = 0 the norm removes any per-row factor; for powers of two
    # every step is exact, so codes and scales are bit-identical.
    rng = np.random.default_rng(24)
    X = rng.standard_normal((7, 320)).astype(np.float32)
    g = rng.uniform(-2, 2, 320).astype(np.float32)
    q0, m0 = O.rmsnorm_quant(X, g, eps_norm=0.0)
    for k in (-6, -1, 3, 20):
        q, m = O.rmsnorm_quant((X * np.float32(2.0 ** k)).astype(np.float32), g, eps_norm=0.0)
        np.testing.assert_array_equal(q, q0)
        np.testing.assert_array_equal(m.view(np.uint32), m0.view(np.uint32))
    # eps_norm > 0 does change the scale of a small row (sqrt(rms^2 + e) > rms)
    _, m_small = O.rmsnorm_quant((X * np.float32(2.0 ** -6)).astype(np.float32), g, eps_norm=0.5)
    _, m_unit = O.rmsnorm_quant(X, g, eps_norm=0.5)
    assert np.all(m_small < m_unit)


def test_rmsnorm_forward_matches_literal_normalize_then_quantize():
    # The definition read literally, in fp64: n = x * g / sqrt(mean x^2 + e),
    # codes rint(127 n / max|n|), Y = s_w * (codes . t) * max|n| / 127. The
    # oracle takes the codes from fp32(x * g) instead: they may differ only
    # where 127 n / max|n| lies within fp32 rounding of a half-integer, and the
    # oracle's scale m must equal max|n| up to that rounding.
    rng = np.random.default_rng(22)
    M, K, N, e = 48, 512, 40, 1e-5
    X = (rng.standard_normal((M, K)) * rng.uniform(0.1, 30, (M, 1))).astype(np.float32)
    g = rng.uniform(-1.5, 1.5, K).astype(np.float32)
    _, s_w, t = O.pack_weights(WL.gaussian_weights(N, K, 0.02, seed=23))
    Y, acc, q, m = O.forward_rmsnorm(X, t, s_w, g, eps_norm=e)
    x = X.astype(np.float64)
    n = x * g.astype(np.float64) / np.sqrt((x * x).mean(axis=1, keepdims=True) + float(np.float32(e)))
    amax = np.abs(n).max(axis=1)
    v = 127.0 * n / amax[:, None]
    q_lit = np.clip(np.rint(v), -128, 127)
    near_tie = np.abs(np.abs(v - np.floor(v)) - 0.5) < 1e-4
    assert np.all((q == q_lit) | near_tie)
    np.testing.assert_allclose(m.astype(np.float64), amax, rtol=2.5e-7)
    y_lit = float(s_w) * acc.astype(np.float64) * amax[:, None] / 127.0
    nz = acc != 0
    assert np.all(np.abs(Y[nz] - y_lit[nz]) <= 6e-7 * np.abs(y_lit[nz]))
    assert np.all(Y[~nz] == 0)


def test_ffn_subln_norms_remove_scales():
    # eps_norm = 0: the input norm makes Y independent of a power-of-two scale
    # of X, and the norm on h makes it independent of a power-of-two scale of
    # s_up (h scales by 16 ungated, by 4 gated) or of s_gate. Without the norm
    # on h the second check fails: the plain FFN is not invariant.
    rng = np.random.default_rng(25)
    D, F, M = 64, 96, 5
    X = rng.standard_normal((M, D)).astype(np.float32)
    _, su, tu = O.pack_weights(WL.gaussian_weights(F, D, 0.02, seed=26))
    _, sg, tg = O.pack_weights(WL.gaussian_weights(F, D, 0.02, seed=27))
    _, sd, td = O.pack_weights(WL.gaussian_weights(D, F, 0.02, seed=28))
    g_in = rng.uniform(0.5, 1.5, D).astype(np.float32)
    g_sub = rng.uniform(-1.5, 1.5, F).astype(np.float32)
    four, two = np.float32(4), np.float32(2)
    for gated in (False, True):
        kw = dict(g_in=g_in, g_sub=g_sub, eps_norm=0.0)
        if gated:
            kw.update(t_gate=tg, s_gate=sg)
        Y0, _ = O.ffn_subln(X, tu, su, td, sd, **kw)
        Y1, _ = O.ffn_subln((X * np.float32(8)).astype(np.float32), tu, su, td, sd, **kw)
        Y2, _ = O.ffn_subln(X, tu, su * four, td, sd, **kw)
        np.testing.assert_array_equal(Y1.view(np.uint32), Y0.view(np.uint32))
        np.testing.assert_array_equal(Y2.view(np.uint32), Y0.view(np.uint32))
        if gated:
            kw.update(s_gate=sg * two)
            Y3, _ = O.ffn_subln(X, tu, su, td, sd, **kw)
            np.testing.assert_array_equal(Y3.view(np.uint32), Y0.view(np.uint32))
    P0, _ = O.ffn(X, tu, su, td, sd)
    P2, _ = O.ffn(X, tu, su * four, td, sd)
    assert not np.array_equal(P0, P2)
