"""Host-side checks of the arithmetic arguments the CUDA kernels rest on (no GPU).

The kernels take a few shortcuts that are exact by an error bound rather than
by construction. Each is restated here step by step in IEEE fp32 / fp64 with
numpy (round to nearest even, the same as the `_rn` intrinsics) and compared
with the plain definition on many values, including values built to sit on
the decision boundaries. Nothing here is shared with the CUDA sources or the
oracle.
"""
import math

import numpy as np

import oracle as O
from ternary_weight_linear_06_b300 import workloads as WL

F = np.float32


def _defined_code(x, m):
    """clamp(rint(fp32(fp32(x*127)/m)), -128, 127)."""
    return np.clip(np.rint((x * F(127)) / m), -128, 127)


def _division_free_code(x, m):
    """The kernels' rule: c = fp32(x * fp32(127 * fp32(1/m))) rounded by rint,
    with the defined quotient deciding when c is within 1e-4 of a half-integer."""
    s127 = F(127) * (F(1) / m)
    c = x * s127
    r = np.rint(c)
    near = np.abs(c - r) > F(0.4999)
    return np.where(near, np.rint((x * F(127)) / m), r), near


def test_division_free_code_matches_the_definition():
    rng = np.random.default_rng(0)
    n = 400_000
    m = np.exp(rng.uniform(-30, 30, n)).astype(F)
    x = (rng.uniform(-1, 1, n).astype(F) * m).astype(F)
    x[: n // 20] = m[: n // 20] * np.sign(rng.uniform(-1, 1, n // 20)).astype(F)   # |x| = m
    k = rng.integers(-127, 127, n)
    ties = (((k + 0.5) / 127.0) * m.astype(np.float64)).astype(F)                  # 127 x / m near k + 1/2
    ties = np.where(np.abs(ties) <= m, ties, x)
    total_near = 0
    for X in (x, ties, np.nextafter(ties, F(np.inf)), np.nextafter(ties, F(-np.inf))):
        X = np.where(np.abs(X) <= m, X, x).astype(F)
        want = _defined_code(X, m)
        got, near = _division_free_code(X, m)
        np.testing.assert_array_equal(got, want)
        assert np.abs(want).max() <= 127          # the definition's clamp never binds for |x| <= m
        c = X * (F(127) * (F(1) / m))
        assert np.abs(c.astype(np.float64) - (X * F(127)) / m).max() < 3.5e-5
        total_near += int(near.sum())
    assert total_near > 0                         # the boundary cases did reach the division


def test_integer_shift_gives_the_twos_complement_byte():
    r = np.arange(-127, 128).astype(F)
    bits = (r + F(12582912.0)).view(np.uint32)    # + 1.5 * 2^23
    np.testing.assert_array_equal(bits & 0xFF, r.astype(np.int64) & 0xFF)


def _two_sum(a, b):
    t = (a + b).astype(F)
    z = (t - a).astype(F)
    return t, ((a - (t - z)).astype(F) + (b - z).astype(F)).astype(F)


def _pair_add(ah, al, bh, bl):
    sh, sl = _two_sum(ah, bh)
    e = (sl + (al + bl).astype(F)).astype(F)
    hi = (sh + e).astype(F)
    return hi, (e - (hi - sh)).astype(F)


def _kernel_rms_factor(X, eps_norm, bf16, threads=256):
    """Sum of x^2 as the kernels take it for one-CTA rows (two Dot2 chains per
    thread over its 16-column groups, pairs combined across lanes by a
    butterfly and across warps in order), then two Newton steps for 1/sqrt in
    fp64 from an fp32 estimate taken two ulp off, rsqrtf's worst case."""
    M, K = X.shape
    G = K // 16
    p = np.zeros((M, threads, 2), F)
    s = np.zeros((M, threads, 2), F)
    for g in range(G):
        t = g % threads
        for j in range(16):
            x = X[:, 16 * g + j]
            c = j & 1
            h = (x * x).astype(F)
            th, tl = _two_sum(p[:, t, c], h)
            p[:, t, c] = th
            if bf16:
                s[:, t, c] = (s[:, t, c] + tl).astype(F)
            else:
                e = (x.astype(np.float64) * x - h).astype(F)            # the FMA remainder, exact
                s[:, t, c] = (s[:, t, c] + (tl + e).astype(F)).astype(F)
    vh, vl = _pair_add(p[:, :, 0], s[:, :, 0], p[:, :, 1], s[:, :, 1])
    vh = vh.reshape(M, threads // 32, 32)
    vl = vl.reshape(M, threads // 32, 32)
    for o in (16, 8, 4, 2, 1):
        idx = np.arange(32) ^ o
        vh, vl = _pair_add(vh, vl, vh[:, :, idx], vl[:, :, idx])
    Sh, Sl = vh[:, 0, 0], vl[:, 0, 0]
    for w in range(1, threads // 32):
        Sh, Sl = _pair_add(Sh, Sl, vh[:, w, 0], vl[:, w, 0])
    S = Sh.astype(np.float64) + Sl.astype(np.float64)
    a = S * (1.0 / K) + float(F(eps_norm))
    # the fp32 estimate at rsqrtf's documented worst case, two ulp off
    y = ((F(1) / np.sqrt(a.astype(F))).astype(F) * F(1 + 2.0 ** -22)).astype(F).astype(np.float64)
    for _ in range(2):
        y = y * (-0.5 * ((a * y) * y) + 1.5)
    return y


def test_compensated_sum_of_squares_gives_the_oracles_scale():
    # Rows with scales over 16 orders of magnitude, fp32 and bf16 inputs: the
    # token scale m = fp32(max(max|u|, eps) * r) from the kernels' r equals the
    # one from the exact sum of squares (readings allow one fp32 step; none
    # is expected at this accuracy).
    rng = np.random.default_rng(3)
    for K, bf16 in ((512, False), (2560, True), (1024, False)):
        X = WL.prefill_activations(96, K, seed=910 + K)
        X = (X * np.exp(rng.uniform(-18, 18, (96, 1)))).astype(F)
        if bf16:
            X = O.bf16_bits_to_f32(WL.f32_to_bf16_bits(X))
        r_kernel = _kernel_rms_factor(X, 1e-5, bf16)
        r_exact = O.rms_factor(X, 1e-5)
        assert np.max(np.abs(r_kernel / r_exact - 1.0)) < 2e-14
        _, m_u = O.quant_act(X)
        np.testing.assert_array_equal((m_u.astype(np.float64) * r_kernel).astype(F),
                                      (m_u.astype(np.float64) * r_exact).astype(F))


def test_pack_partials_fit_in_128_bits():
    # abs_sum_kernel adds mant << (e - 86) for biased exponents e in [86, 158]:
    # each term is below 2^24 * 2^72 = 2^96, and N*K < 2^31 terms keep any
    # subset of the block partials below 2^127, so a CTA may add them in
    # unsigned 128-bit arithmetic without overflow.
    term_max = ((1 << 24) - 1) << (158 - 86)
    assert term_max < 2 ** 96
    assert term_max * ((1 << 31) - 1) < 2 ** 127
    assert math.log2(term_max * ((1 << 31) - 1)) < 127
