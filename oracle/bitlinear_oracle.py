"""Plain CPU oracle for the BitLinear forward of BitNet b1.58.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
this module. The product path (the CUDA library and its Python binding) never
does, and this module imports nothing from the product.

It is written for a reader checking it against the pages by eye: every step is
the definition, in the order the pages give it, with numpy as the only library
(IEEE fp32 arithmetic where the method fixes fp32, Python integers where the
method asks for an exact value). No blocking, fusion or reordering.

Sources (page title, section, equation):
  [P3] "BitNet解读" (markgoyens.top), section 模型架构 / 权重量化函数:
       eq. (3) gamma = (1/nm) * sum |W_ij|; W' = W / (gamma + eps);
       eqs. (1),(2) W~ = RoundClip(W', -1, 1), round to nearest then clip;
       activation quantization: per token, scaled into [-Qb, Qb], symmetric,
       no zero point.
  [P1] "BitNet b1.58 2B4T Technical Report" (Chinese translation,
       developer.volcengine.com), section 2 架构: BitLinear replaces
       torch.nn.Linear; weights absmean-ternary, activations per-token absmax
       int8; section 2 FFN uses squared ReLU; no bias terms anywhere.
  [P1 §5.1] / [P4 §5.1] "BitNet b1.58 2B4T Technical Report | Summary",
       section 5.1 GPU Inference: four ternary values are packed into one
       8-bit value for storage.
  [P3 革命性的效率提升] the matmul becomes integer additions: +1 adds the
       activation, -1 subtracts it, 0 skips it.
  [P5 §1.1] (gitcode.csdn.net bitnet.cpp intro, 1.1 1.58-bit 三值量化): the
       integer result is brought back to range with the scaling factor.

Readings where the pages are silent (each repeated in the design notes):
  * eps = 1e-5 for both weights and activations; Qb = 127, clamp to [-128, 127].
  * gamma is the exact mean of |W| rounded once to fp32 (ties to even);
    s_w = fp32(gamma + eps) is the one per-matrix scale, used for the
    ternarization and again for the dequantization.
  * "round to nearest" is rint (ties to even).
  * activation quant: m = max(max_k |x_k|, eps); q = clamp(rint(fp32(fp32(x*127)/m))).
  * dequant: c = fp32(fp32(s_w * m) / 127); y = fp32(float(acc) * c).
  * storage code of a ternary value t is t + 1 in {0, 1, 2}; byte b of a row
    holds k = 4b + j in bits [2j, 2j+1] (little end first).
  * FFN: ungated up -> ReLU^2 -> requant (same eps) -> down; no norm between.
  * gated FFN: h = fp32(fp32(ReLU(gate)^2) * up), then requant and down.
  * SubLN is an RMSNorm with a per-feature gain g and no bias, applied to the
    input of a BitLinear before its activation quantization:
    n_ik = x_ik * g_k * r_i, r_i = 1 / sqrt(mean_k x_ik^2 + eps_norm),
    eps_norm = 1e-5. In the FFN it sits on the block input and on h before
    the down projection. Absmax codes do not change when a row is multiplied
    by the positive factor r_i, so the codes are taken from u = fp32(x * g)
    and r_i goes into the per-token scale: m_i = fp32(max(max|u|, eps) * r_i).
    r_i is computed in fp64 from the exact sum of squares.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

EPS = np.float32(1e-5)
EPS_NORM = np.float32(1e-5)
QB = 127
FLT_MAX = Fraction(int(np.finfo(np.float32).max))

__all__ = [
    "EPS", "QB",
    "round_rational_to_f32", "abs_sum_exact", "absmean_gamma", "weight_scale",
    "ternarize", "pack_codes", "unpack_codes", "pack_weights",
    "bf16_bits_to_f32", "quant_act", "int_matmul", "dequant", "forward",
    "forward_packed", "relu2", "ffn", "ffn_gated", "tie_count",
    "EPS_NORM", "rms_factor", "rmsnorm_quant", "forward_rmsnorm", "ffn_subln",
]


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


# --------------------------------------------------------------------------
# exact rounding helper
# --------------------------------------------------------------------------
def round_rational_to_f32(num: int, den: int) -> np.float32:
    """The fp32 value nearest to num/den (num >= 0, den > 0), ties to even.

    IEEE 754 roundTiesToEven, written out with Python fractions: find the
    binade, take the 24 significant bits (fewer in the subnormal range, where
    the last bit weighs 2^-149), round on the exact remainder.
    """
    if den <= 0 or num < 0:
        raise ValueError("round_rational_to_f32 needs num >= 0 and den > 0")
    if num == 0:
        return np.float32(0.0)
    x = Fraction(num, den)
    e = num.bit_length() - den.bit_length()          # floor(log2 x) is e-1 or e
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    lsb = max(e - 23, -149)                          # weight of the last kept bit
    scaled = x / Fraction(2) ** lsb
    q = scaled.numerator // scaled.denominator
    rem = scaled - q
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and q % 2 == 1):
        q += 1
    value = Fraction(q) * Fraction(2) ** lsb
    if value > FLT_MAX:
        return np.float32(np.inf)
    return np.float32(float(value))                  # exact: value is an fp32 number


# --------------------------------------------------------------------------
# weights: absmean -> ternary -> 2-bit codes   [P3 eqs. (1)-(3)], [P1 §5.1]
# --------------------------------------------------------------------------
def abs_sum_exact(W) -> int:
    """sum |W_ij| as an exact integer in units of 2^-149 (the fp32 quantum).

    Every finite fp32 |w| equals mant * 2^(s - 149) with integer mant < 2^24
    and s = max(exponent_field - 1, 0). Mantissas are summed per s (each bucket
    sum is an integer below 2^53 as long as the matrix has fewer than 2^29
    entries, so the float64 accumulation inside np.bincount is exact), then
    the buckets are combined with Python integers.
    """
    a = np.abs(_f32(W)).ravel()
    if a.size >= (1 << 29):
        raise ValueError("matrix too large for the exact bucket sum")
    total = 0
    chunk = 1 << 24
    for start in range(0, a.size, chunk):
        bits = a[start:start + chunk].view(np.uint32)
        exp_field = (bits >> 23) & 0xFF
        if np.any(exp_field == 0xFF):
            raise ValueError("non-finite weight")
        frac = (bits & 0x7FFFFF).astype(np.int64)
        mant = np.where(exp_field == 0, frac, frac | 0x800000)
        s = np.where(exp_field == 0, 0, exp_field.astype(np.int64) - 1)
        sums = np.bincount(s, weights=mant.astype(np.float64), minlength=254)
        for si in np.nonzero(sums)[0]:
            total += int(sums[si]) << int(si)
    return total


def absmean_gamma(W) -> np.float32:
    """gamma = (1/nm) * sum |W_ij|   [P3 eq. (3)], rounded once to fp32."""
    W = _f32(W)
    if W.size == 0:
        raise ValueError("empty weight matrix")
    return round_rational_to_f32(abs_sum_exact(W), W.size << 149)


def weight_scale(gamma, eps=EPS) -> np.float32:
    """s_w = gamma + eps in fp32   [P3, W' = W / (gamma + eps)]."""
    return np.float32(np.float32(gamma) + np.float32(eps))


def ternarize(W, s_w) -> np.ndarray:
    """W~ = RoundClip(W / s_w, -1, 1)   [P3 eqs. (1), (2)]: fp32 division,
    round to nearest (ties to even), clip. Returns int8 in {-1, 0, 1}."""
    Wn = _f32(W) / np.float32(s_w)
    return np.clip(np.rint(Wn), -1, 1).astype(np.int8)


def pack_codes(t) -> np.ndarray:
    """Four ternary values per byte   [P1 §5.1]. Code = t + 1; byte b of a row
    holds columns 4b..4b+3, column 4b+j in bits [2j, 2j+1]. Shape [N, K/4]."""
    t = np.asarray(t, dtype=np.int8)
    N, K = t.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    c = (t.astype(np.int16) + 1).astype(np.uint8).reshape(N, K // 4, 4)
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def unpack_codes(packed, K: int) -> np.ndarray:
    """Inverse of pack_codes: [N, K/4] bytes -> int8 [N, K]. Code 3 is not a
    valid code; it is returned as 2 (t = +2) so that a test sees it."""
    p = np.asarray(packed, dtype=np.uint8)
    N = p.shape[0]
    c = np.stack([(p >> (2 * j)) & 3 for j in range(4)], axis=-1).reshape(N, K)
    return (c.astype(np.int16) - 1).astype(np.int8)


def pack_weights(W, eps=EPS):
    """The whole weight path: (packed [N, K/4] uint8, s_w fp32, t int8 [N, K])."""
    gamma = absmean_gamma(W)
    s_w = weight_scale(gamma, eps)
    t = ternarize(W, s_w)
    return pack_codes(t), s_w, t


def tie_count(W, s_w) -> int:
    """Diagnostic: entries with |W/s_w| within one fp32 ulp of 0.5 (the
    ternary ties), which a different division or rounding would flip."""
    r = np.abs(_f32(W) / np.float32(s_w))
    half = np.float32(0.5)
    lo = np.nextafter(half, np.float32(0))
    hi = np.nextafter(half, np.float32(1))
    return int(np.count_nonzero((r >= lo) & (r <= hi)))


# --------------------------------------------------------------------------
# activations: per-token absmax int8   [P3 activation quantization], [P1 §2]
# --------------------------------------------------------------------------
def bf16_bits_to_f32(u16) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 exactly (append 16 zero bits)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def quant_act(X, eps=EPS):
    """Per token i: m_i = max(max_k |x_ik|, eps); q_ik = clamp(rint(fp32(fp32(
    x_ik * 127) / m_i)), -128, 127). Returns (q int8 [M, K], m fp32 [M])."""
    X = _f32(X)
    if X.ndim != 2 or X.shape[1] == 0:
        raise ValueError("X must be [M, K] with K > 0")
    absmax = np.max(np.abs(X), axis=1) if X.shape[0] else np.zeros(0, np.float32)
    m = np.maximum(absmax, np.float32(eps)).astype(np.float32)
    scaled = (X * np.float32(QB)) / m[:, None]
    q = np.clip(np.rint(scaled), -QB - 1, QB).astype(np.int8)
    return q, m


# --------------------------------------------------------------------------
# integer matmul and dequant   [P3 革命性的效率提升], [P5 §1.1]
# --------------------------------------------------------------------------
def int_matmul(q, t) -> np.ndarray:
    """acc[i, j] = sum_k q[i, k] * t[j, k], exact (int64), returned as int32."""
    acc = np.asarray(q, dtype=np.int64) @ np.asarray(t, dtype=np.int64).T
    if acc.size and np.max(np.abs(acc)) >= (1 << 31):
        raise OverflowError("accumulator exceeds int32")
    return acc.astype(np.int32)


def dequant(acc, s_w, m) -> np.ndarray:
    """y_ij = fp32(float(acc_ij) * c_i) with c_i = fp32(fp32(s_w * m_i) / 127)."""
    acc = np.asarray(acc, dtype=np.int64)
    if acc.size and np.max(np.abs(acc)) > (1 << 24):
        raise OverflowError("accumulator not exact in fp32")
    c = (np.float32(s_w) * _f32(m)) / np.float32(QB)
    return (acc.astype(np.float32) * c.astype(np.float32)[:, None]).astype(np.float32)


def forward(X, t, s_w, eps=EPS):
    """BitLinear forward with ternary weights t [N, K] and scale s_w:
    returns (Y fp32 [M, N], acc int32 [M, N], q int8 [M, K], m fp32 [M])."""
    q, m = quant_act(X, eps)
    acc = int_matmul(q, t)
    return dequant(acc, s_w, m), acc, q, m


def forward_packed(X, packed, s_w, eps=EPS):
    """forward() taking the packed [N, K/4] codes."""
    K = _f32(X).shape[1]
    return forward(X, unpack_codes(packed, K), s_w, eps)


def relu2(y) -> np.ndarray:
    """Squared ReLU   [P1 §2 FFN]: y*y (fp32) where y > 0, else 0."""
    y = _f32(y)
    return np.where(y > 0, y * y, np.float32(0)).astype(np.float32)


def ffn(X, t_up, s_up, t_down, s_down, eps=EPS):
    """Ungated FFN block: up -> ReLU^2 -> requant -> down. Returns (Y, h)."""
    y_up = forward(X, t_up, s_up, eps)[0]
    h = relu2(y_up)
    return forward(h, t_down, s_down, eps)[0], h


def ffn_gated(X, t_up, s_up, t_gate, s_gate, t_down, s_down, eps=EPS):
    """Gated FFN block (squared ReLU in place of SwiGLU's SiLU, [P1 §2]):
    h = fp32(ReLU^2(gate(X)) * up(X)), requantized per token, then down.
    gate and up are BitLinears on the same input. Returns (Y, h)."""
    y_up = forward(X, t_up, s_up, eps)[0]
    y_gate = forward(X, t_gate, s_gate, eps)[0]
    h = (relu2(y_gate) * y_up).astype(np.float32)
    return forward(h, t_down, s_down, eps)[0], h


# --------------------------------------------------------------------------
# SubLN: RMSNorm before the activation quantization
#   [P1 §2 架构, 归一化 and 偏置移除], [P2 架构上的关键修改, 归一化 row],
#   [P3 模型架构, 组件兼容性: RMSNorm]
# --------------------------------------------------------------------------
def rms_factor(X, eps_norm=EPS_NORM) -> np.ndarray:
    """r_i = 1 / sqrt(S_i / K + eps_norm) in fp64, S_i = sum_k x_ik^2.

    Each square of an fp32 value is exact in fp64, and math.fsum rounds their
    exact sum once, so S_i is the correctly rounded sum. The division, the
    addition of eps_norm (an fp32 value), the square root and the reciprocal
    are then fp64 operations, each rounded once, in that order."""
    X = _f32(X)
    M, K = X.shape
    e = float(np.float32(eps_norm))
    r = np.empty(M, np.float64)
    for i in range(M):
        S = math.fsum((X[i].astype(np.float64) ** 2).tolist())
        r[i] = 1.0 / math.sqrt(S / K + e)
    return r


def rmsnorm_quant(X, g=None, eps_norm=EPS_NORM, eps=EPS):
    """RMSNorm (gain g [K], no bias) followed by the per-token absmax quant.

    Codes come from u = fp32(x * g) (u = x without a gain) because absmax
    codes ignore the positive per-token factor r_i; the factor goes into the
    scale: (q, m_u) = quant_act(u); m_i = fp32(fp64(m_u_i) * r_i).
    Returns (q int8 [M, K], m fp32 [M])."""
    X = _f32(X)
    u = X if g is None else (X * _f32(g)[None, :]).astype(np.float32)
    q, m_u = quant_act(u, eps)
    r = rms_factor(X, eps_norm)
    m = (m_u.astype(np.float64) * r).astype(np.float32)
    return q, m


def forward_rmsnorm(X, t, s_w, g=None, eps_norm=EPS_NORM, eps=EPS):
    """BitLinear forward on RMSNorm(X): returns (Y, acc, q, m) like forward()."""
    q, m = rmsnorm_quant(X, g, eps_norm, eps)
    acc = int_matmul(q, t)
    return dequant(acc, s_w, m), acc, q, m


def ffn_subln(X, t_up, s_up, t_down, s_down, g_in=None, g_sub=None, t_gate=None, s_gate=None,
              eps_norm=EPS_NORM, eps=EPS):
    """FFN block with SubLN: RMSNorm(g_in) on X, up (and gate) on that one
    quantization, ReLU^2 (times up when gated), RMSNorm(g_sub) on h, down.
    Returns (Y, h)."""
    q, m = rmsnorm_quant(X, g_in, eps_norm, eps)
    y_up = dequant(int_matmul(q, t_up), s_up, m)
    if t_gate is None:
        h = relu2(y_up)
    else:
        y_gate = dequant(int_matmul(q, t_gate), s_gate, m)
        h = (relu2(y_gate) * y_up).astype(np.float32)
    return forward_rmsnorm(h, t_down, s_down, g_sub, eps_norm, eps)[0], h
