"""CPU oracle of the MXFP8 variant of the SwiGLU expert layer.

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: only ``tests/``, the smoke check and the
benchmark's CPU-baseline leg may import it; it imports numpy alone and shares no code with the
CUDA path.

"Section 09: Grouped GEMM" (§9.5, last paragraph) describes a routed MXFP8 path: scaled grouped
GEMM for the forward and the Dgrad, BF16 grouped GEMM for the Wgrad. The pages do not define
the format; the plain reading is the OCP Microscaling (MX) format MXFP8 (OCP "Microscaling
Formats (MX) Specification" v1.0): blocks of 32 consecutive elements along the contraction
dimension share one power-of-two scale X stored as E8M0 (an exponent with bias 127), and each
element is stored as FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, largest finite 448). The value of element i of a block is X * e4m3(code_i).

Readings (each also listed in the design notes):
  m1  the shared exponent of a block is floor(log2(max |v|)) - 8 (8 = the exponent of E4M3's
      largest normal, the spec's emax_elem), clamped to the E8M0 range [-127, 127]; an all-zero
      block takes -127. Elements are v / X rounded to the nearest E4M3 value, ties to the even
      code, and saturated to +-448 (values between 448 * X and 512 * X clamp).
  m2  every operand is quantized along its contraction dimension: x and dy along d, the
      SwiGLU output along h, dU along 2h, each weight along the dimension its product
      contracts (so a weight is quantized twice, once per orientation).
  m3  operands that the BF16 path holds as bf16 are quantized from those bf16 values: the
      SwiGLU output P = w * A and the SwiGLU-backward output dU are rounded to bf16 (nearest,
      ties to even) first, as the BF16 path stores them.
  m4  the routing weight multiplies the SwiGLU output before its quantization, and the Dgrad
      scales dA by it, as in the BF16 path (reading c5 of the bf16 oracle: an exact
      reordering of a linear sum in exact arithmetic; here it fixes which values are
      quantized).
  m5  the Wgrads stay BF16 (§9.5): dW_ug = dU^T xp and dW_down = P^T dy with the
      unquantized P and dU of this path.
The products of dequantized operands are exact in float64 sums (no rounding of products).
"""
from __future__ import annotations

from typing import Callable, Sequence, Union

import numpy as np

ArrayOrFn = Union[np.ndarray, Callable[[int], np.ndarray]]

BLOCK = 32          # elements per shared scale (OCP MX)
E4M3_MAX = 448.0
EMAX_ELEM = 8       # exponent of the largest normal E4M3 value (448 = 1.75 * 2^8)
SCALE_BIAS = 127    # E8M0 bias
SCALE_MIN, SCALE_MAX = -127, 127


def _slice(w: ArrayOrFn, e: int) -> np.ndarray:
    return np.asarray(w(e) if callable(w) else w[e], dtype=np.float64)


def segments(offsets: np.ndarray):
    """Expert e owns rows [offsets[e-1], offsets[e]) (inclusive offsets, Fig. 37)."""
    off = np.asarray(offsets, dtype=np.int64)
    starts = np.concatenate([[0], off[:-1]])
    return [(int(s), int(t)) for s, t in zip(starts, off)]


# ---------------------------------------------------------------------------------------------
# FP8 E4M3 and E8M0 (OCP 8-bit floating point; OCP MX v1.0)
# ---------------------------------------------------------------------------------------------
def e4m3_value(code: int) -> float:
    """Value of an E4M3 code from the format definition: sign bit 7, exponent bits 6..3 (bias
    7), mantissa bits 2..0; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there
    are no infinities."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def e4m3_table() -> np.ndarray:
    """Values of all 256 codes (NaN for the two NaN codes)."""
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


_POS_CODES = np.arange(0, 0x7F)                      # +0 ... +448, increasing values
_POS_VALUES = np.array([e4m3_value(int(c)) for c in _POS_CODES])


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Round each value to the nearest E4M3 value (ties to the code with an even mantissa, i.e.
    an even code), saturating magnitudes above 448 to 448 (reading m1). Returns uint8 codes;
    zero and values that round to zero get +0 or -0 by sign."""
    v = np.asarray(v, np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first grid value >= a
    hi = np.minimum(hi, _POS_VALUES.size - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    return np.where(v < 0, code | 0x80, code).astype(np.uint8)


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    return e4m3_table()[np.asarray(code, np.int64)]


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even (reading m3), from float64 values in the
    float32 range: float64 -> nearest float32 is not the same as nearest bf16, so the rounding
    is done on the float64 value's bf16 grid directly."""
    v = np.asarray(v, np.float64)
    out = np.zeros_like(v)
    nz = v != 0
    m, e = np.frexp(v[nz])                      # v = m * 2^e, 0.5 <= |m| < 1
    scaled = m * 256.0                          # 8 significant bits: 128 <= |scaled| < 256
    r = np.round(scaled)                        # numpy rounds half to even
    out[nz] = np.ldexp(r, e - 8)
    return out


# ---------------------------------------------------------------------------------------------
# MX quantization along the last axis (reading m1)
# ---------------------------------------------------------------------------------------------
def mx_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """Shared exponent of each block: floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for an
    all-zero block."""
    amax = np.asarray(amax, np.float64)
    _, e = np.frexp(np.where(amax > 0, amax, 1.0))   # amax = m * 2^e with 0.5 <= m < 1
    exp = (e - 1) - EMAX_ELEM                          # floor(log2(amax)) = e - 1
    exp = np.where(amax > 0, exp, SCALE_MIN)
    return np.clip(exp, SCALE_MIN, SCALE_MAX).astype(np.int64)


def mx_quantize(x: np.ndarray):
    """Quantize along the last axis in blocks of 32 (a partial last block is padded with zeros,
    which do not change its maximum). Returns (codes uint8 [..., K], scale exponents int64
    [..., ceil(K/32)])."""
    x = np.asarray(x, np.float64)
    K = x.shape[-1]
    nb = -(-K // BLOCK)
    pad = nb * BLOCK - K
    xp = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1) if pad else x
    blocks = xp.reshape(x.shape[:-1] + (nb, BLOCK))
    exp = mx_scale_exponent(np.abs(blocks).max(axis=-1))
    scaled = blocks / np.ldexp(1.0, exp)[..., None]
    codes = e4m3_encode(scaled).reshape(x.shape[:-1] + (nb * BLOCK,))[..., :K]
    return codes, exp


def mx_dequantize(codes: np.ndarray, exp: np.ndarray) -> np.ndarray:
    """X * e4m3(code) for every element (X = 2^exp of its block)."""
    codes = np.asarray(codes)
    K = codes.shape[-1]
    scale = np.repeat(np.ldexp(1.0, np.asarray(exp)), BLOCK, axis=-1)[..., :K]
    return e4m3_decode(codes) * scale


def mx_round_trip(x: np.ndarray, axis: int = -1) -> np.ndarray:
    """The values an MXFP8 operand carries: x quantized in blocks along `axis`, dequantized."""
    x = np.moveaxis(np.asarray(x, np.float64), axis, -1)
    return np.moveaxis(mx_dequantize(*mx_quantize(x)), -1, axis)


# ---------------------------------------------------------------------------------------------
# The MXFP8 expert layer (Eq. 13 forward, Eq. 15 dgrad through scaled GEMMs; BF16 wgrad)
# ---------------------------------------------------------------------------------------------
def _silu(z):
    return z / (1.0 + np.exp(-z))


def mx_expert_forward(xp: np.ndarray, offsets: np.ndarray, w_ug: ArrayOrFn, w_down: ArrayOrFn,
                      row_weight: np.ndarray | None = None, experts: Sequence[int] | None = None):
    """Eq. 13 per expert with MXFP8 operands (readings m1-m4):
        U_e = q(X_e) q(W_ug,e)^T                  (both quantized along d)
        P_e = w * silu(U_e[:, :h]) * U_e[:, h:]   (w = row_weight of each row, 1 when None)
        Y_e = q(bf16(P_e)) q(W_down,e)            (P along h; W_down [h, d] along h)
    Returns (y [n, d], u [n, 2h], p [n, h]) in float64; rows of experts not computed stay 0."""
    xp = np.asarray(xp, np.float64)
    n, d = xp.shape
    h = _slice(w_down, 0).shape[0]
    y, u, p = np.zeros((n, d)), np.zeros((n, 2 * h)), np.zeros((n, h))
    segs = segments(offsets)
    for e in (range(len(segs)) if experts is None else experts):
        s, t = segs[e]
        if t == s:
            continue
        ue = mx_round_trip(xp[s:t]) @ mx_round_trip(_slice(w_ug, e)).T
        w = np.ones(t - s) if row_weight is None else np.asarray(row_weight, np.float64)[s:t]
        pe = w[:, None] * (_silu(ue[:, :h]) * ue[:, h:])
        y[s:t] = mx_round_trip(bf16_round(pe)) @ mx_round_trip(_slice(w_down, e), axis=0)
        u[s:t], p[s:t] = ue, pe
    return y, u, p


def mx_expert_backward(dy: np.ndarray, xp: np.ndarray, u: np.ndarray, p: np.ndarray,
                       offsets: np.ndarray, w_ug: ArrayOrFn, w_down: ArrayOrFn,
                       row_weight: np.ndarray | None = None, experts: Sequence[int] | None = None):
    """Eq. 15 per expert: scaled Dgrads, BF16 Wgrads (readings m1-m5). With g, v = U[:, :h],
    U[:, h:], s = sigmoid(g):
        dA  = w * (q(dY_e) q(W_down,e)^T)         (dY along d; W_down [h, d] along d)
        dU  = [dA v s (1 + g (1 - s)), dA silu(g)]
        dX  = q(bf16(dU)) q(W_ug,e)               (dU along 2h; W_ug [2h, d] along 2h)
        dW_ug = dU^T X_e,  dW_down = P^T dY_e     (BF16 wgrads of the unquantized operands)
    and, per row, the routing-weight term <SwiGLU(U)_p, (q(dY_e) q(W_down,e)^T)_p>: the gradient of
    the combine with respect to the row's routing weight, <y~_p, dOut[t]> with the unweighted
    expert output y~, evaluated through the scaled Dgrad product (dY the plain gather of dOut).
    Returns (dxp [n, d], dw_ug [E, 2h, d], dw_down [E, h, d], du [n, 2h], g_dot [n])."""
    dy = np.asarray(dy, np.float64)
    xp = np.asarray(xp, np.float64)
    u = np.asarray(u, np.float64)
    p = np.asarray(p, np.float64)
    n, d = xp.shape
    h = u.shape[1] // 2
    segs = segments(offsets)
    E = len(segs)
    dxp, du, g_dot = np.zeros((n, d)), np.zeros((n, 2 * h)), np.zeros(n)
    dw_ug, dw_down = np.zeros((E, 2 * h, d)), np.zeros((E, h, d))
    for e in (range(E) if experts is None else experts):
        s, t = segs[e]
        if t == s:
            continue
        wu, wd = _slice(w_ug, e), _slice(w_down, e)
        w = np.ones(t - s) if row_weight is None else np.asarray(row_weight, np.float64)[s:t]
        g, v = u[s:t, :h], u[s:t, h:]
        sg = 1.0 / (1.0 + np.exp(-g))
        ge = mx_round_trip(dy[s:t]) @ mx_round_trip(wd).T
        da = w[:, None] * ge
        g_dot[s:t] = np.einsum("ph,ph->p", g * sg * v, ge)
        due = np.concatenate([da * v * sg * (1.0 + g * (1.0 - sg)), da * g * sg], axis=1)
        dxp[s:t] = mx_round_trip(bf16_round(due)) @ mx_round_trip(wu, axis=0)
        dw_ug[e] = due.T @ xp[s:t]
        dw_down[e] = p[s:t].T @ dy[s:t]
        du[s:t] = due
    return dxp, dw_ug, dw_down, du, g_dot
