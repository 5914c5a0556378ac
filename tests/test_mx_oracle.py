"""Pins for the MXFP8 oracle (oracle/mx_oracle.py).

The E4M3 code table is checked against PyTorch's float8_e4m3fn type (a library reading of the
same OCP format) and the values the format definition fixes; the rounding against PyTorch's
conversion and hand-worked ties; the scale rule against hand-evaluated exponents; the axis of
quantization with rows of very different magnitudes; and the MXFP8 layer against the plain
fp64 oracle: exactly where the operands are MX-representable, and within the quantization error
bound where they are not. A planted mistake in each part fails at least one of these.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import mx_oracle as X
from ragged_grouped_gemm_device_gb300 import workloads as W


# ------------------------------------------------------------------------------ E4M3 and E8M0
def test_e4m3_table_matches_the_format_and_torch():
    tab = X.e4m3_table()
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    ok = ~np.isnan(tab)
    assert np.array_equal(tab[ok], ref[ok])
    # values fixed by the definition: largest finite, smallest normal, smallest subnormal, one
    assert tab[0x7E] == 448.0 and tab[0x08] == 2.0 ** -6 and tab[0x01] == 2.0 ** -9 and tab[0x38] == 1.0
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF]) and tab[0xFE] == -448.0
    assert np.isnan(tab).sum() == 2 and not np.isinf(tab).any()


def test_e4m3_encode_round_trips_every_finite_code():
    tab = X.e4m3_table()
    codes = np.array([c for c in range(256) if not np.isnan(tab[c]) and c != 0x80])
    assert np.array_equal(X.e4m3_encode(tab[codes]), codes.astype(np.uint8))


def test_e4m3_encode_ties_to_even_and_saturates():
    cases = {
        1.0625: 0x38,            # halfway 1.0 (even) / 1.125 (odd)
        1.1875: 0x3A,            # halfway 1.125 (odd) / 1.25 (even)
        2.0 ** -10: 0x00,        # halfway 0 / smallest subnormal (odd)
        3 * 2.0 ** -10: 0x02,    # halfway 2^-9 (odd) / 2^-8 (even)
        464.0: 0x7E,             # halfway 448 / the missing 480: saturates
        449.0: 0x7E, 1e9: 0x7E,
        -500.0: 0xFE,
        0.0: 0x00,
    }
    for v, c in cases.items():
        assert int(X.e4m3_encode(np.array([v]))[0]) == c, v


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.1, 1.0, 30.0)])
    v = np.clip(v, -448, 448).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = X.e4m3_encode(v)
    # torch keeps the sign of values that round to zero; the oracle gives them +0 or -0 by sign
    # as well, so the codes agree everywhere
    assert np.array_equal(got, ref)


def test_scale_exponent_rule():
    amax = np.array([1.0, 448.0, 511.9, 512.0, 0.75, 0.0, 2.0 ** -130, 2.0 ** 120, 3.0 * 2 ** -20])
    want = np.array([-8, 0, 0, 1, -9, -127, -127, 112, -19 - 8])
    assert np.array_equal(X.mx_scale_exponent(amax), want)


def test_mx_quantize_blocks_are_exact_for_representable_values_and_clamp_above_448():
    rng = np.random.default_rng(1)
    tab = X.e4m3_table()
    finite = tab[(~np.isnan(tab)) & (np.abs(tab) <= 448)]
    blk = rng.choice(finite, size=(5, 96))
    blk[:, ::32] = 448.0                                     # each block's max maps to 448
    scale = np.ldexp(1.0, rng.integers(-20, 20, size=(5, 1)))
    x = blk * scale
    codes, exp = X.mx_quantize(x)
    assert np.array_equal(X.mx_dequantize(codes, exp), x)
    # the floor rule maps 500 to 448 (clamp), not to a larger scale
    c, e = X.mx_quantize(np.array([[500.0] + [1.0] * 31]))
    assert e[0, 0] == 0 and X.e4m3_decode(c)[0, 0] == 448.0


def test_mx_quantize_partial_block_and_error_bound():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((64, 72)) * np.ldexp(1.0, rng.integers(-10, 10, size=(64, 1)))
    codes, exp = X.mx_quantize(x)
    assert codes.shape == (64, 72) and exp.shape == (64, 3)   # 72 = 2 blocks + 8 elements
    deq = X.mx_dequantize(codes, exp)
    # each element: half an E4M3 step of its binade (at least half the smallest subnormal step),
    # or, above 448 X, the clamp to 448 X
    ex = np.repeat(exp, 32, axis=1)[:, :72]
    step = np.maximum(np.ldexp(1.0, np.floor(np.log2(np.abs(x) + 1e-300)).astype(int) - 3), np.ldexp(1.0, ex - 9))
    clamp = np.abs(x) - 448.0 * np.ldexp(1.0, ex)
    assert (np.abs(deq - x) <= np.maximum(0.5 * step, clamp) * (1 + 1e-12)).all()
    assert (clamp > 0).any()                                 # some block maxima did clamp


def test_mx_round_trip_axis():
    # rows of very different magnitudes: exact along each row (one scale per row block), lossy
    # along columns, where a block mixes magnitudes 2^0 .. 2^93
    tab = X.e4m3_table()
    vals = np.random.default_rng(3).choice(tab[(tab > 2 ** -3) & (tab <= 448)], size=(32, 64))
    x = vals * np.ldexp(1.0, 3 * np.arange(32))[:, None]
    assert np.array_equal(X.mx_round_trip(x, axis=1), x)
    assert not np.array_equal(X.mx_round_trip(x, axis=0), x)
    assert np.array_equal(X.mx_round_trip(x.T, axis=0), x.T)


def test_bf16_round_matches_float32_bf16_rounding():
    rng = np.random.default_rng(4)
    v = (rng.standard_normal(50000) * np.ldexp(1.0, rng.integers(-30, 30, 50000))).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
    assert np.array_equal(X.bf16_round(v.astype(np.float64)), want)


# ------------------------------------------------------------------------------ the layer
def _representable(rng, shape, scale):
    """Values of the form +-(1 + m/8) 2^k, m <= 6, with small k, times `scale`: exact in bf16
    and in MXFP8 along any axis (every block's max is within 2^8 of its min, and a block max
    of mantissa 1.875 would clamp)."""
    m = rng.integers(0, 7, size=shape)
    k = rng.integers(-3, 2, size=shape)
    s = rng.choice([-1.0, 1.0], size=shape)
    return s * (1 + m / 8.0) * np.ldexp(1.0, k) * scale


def _quant_bound(pe, w):
    """Bound of |q(bf16(P)) W - P W| per output: sum over k of |P~_k - P_k| |W_kj|, with
    |P~ - P| <= 2^-9 |P| (bf16) + max(2^-4 |b|, |b| - 448 X) (E4M3 step or clamp, b = bf16(P))
    + 2^-10 X (half the smallest subnormal step), X = 2^exp of the element's block."""
    b = X.bf16_round(pe)
    _, ex = X.mx_quantize(b)
    xs = np.repeat(np.ldexp(1.0, ex), 32, axis=1)[:, : pe.shape[1]]
    dp = 2.0 ** -9 * np.abs(pe) + np.maximum(2.0 ** -4 * np.abs(b), np.abs(b) - 448.0 * xs) + 2.0 ** -10 * xs
    return dp @ np.abs(w)


def _case(seed):
    wl = W.custom(T=150, k=3, E=6, d=64, h=96, seed=seed, invalid_frac=0.05, empty_experts=(2,))
    rng = np.random.default_rng(seed)
    x = _representable(rng, (wl.T, wl.d), 1.0)
    wug = _representable(rng, (wl.E, 2 * wl.h, wl.d), 0.125)
    wdn = _representable(rng, (wl.E, wl.h, wl.d), 0.125)
    r = O.route_offsets(wl.ids, wl.E)
    xp = O.permute(x, r["sorted_src"], r["M"], wl.k)
    w_row = np.zeros(wl.n)
    w_row[: r["M"]] = wl.weights.reshape(-1)[r["sorted_src"][: r["M"]]]
    return wl, r, xp, wug, wdn, w_row


def test_mx_forward_exact_where_representable_and_within_the_quantization_bound():
    wl, r, xp, wug, wdn, w_row = _case(5)
    M = r["M"]
    y, u, p = X.mx_expert_forward(xp, r["offsets"], wug, wdn, w_row)
    y0, u0, a0, _ = O.expert_forward(xp, r["offsets"], wug, wdn)
    # x and W_ug are MX-representable: U is the plain product, P = w * SwiGLU(U)
    assert np.allclose(u[:M], u0[:M], rtol=1e-13, atol=1e-13)
    assert np.allclose(p[:M], w_row[:M, None] * a0[:M], rtol=1e-13, atol=1e-15)
    # P is quantized: |y - w y0| <= sum_k |P~_k - P_k| |W_kj| with |P~ - P| <= (2^-9 + 2^-4 (1 + 2^-8))|P|
    # plus the smallest scaled step of its block
    yw = w_row[:M, None] * y0[:M]
    segs = O.segments(r["offsets"])
    for e, (s, t) in enumerate(segs):
        if t == s:
            continue
        bound = _quant_bound(p[s:t], wdn[e])
        assert (np.abs(y[s:t] - yw[s:t]) <= bound * (1 + 1e-9)).all()
        assert np.abs(y[s:t] - yw[s:t]).max() > 0      # P really was quantized


def test_mx_backward_dgrad_exact_where_representable_and_bf16_wgrads():
    wl, r, xp, wug, wdn, w_row = _case(6)
    M = r["M"]
    rng = np.random.default_rng(7)
    dy = np.zeros((wl.n, wl.d))
    dy[:M] = _representable(rng, (M, wl.d), 1.0)
    y, u, p = X.mx_expert_forward(xp, r["offsets"], wug, wdn, w_row)
    dxp, dwu, dwd, du, g_dot = X.mx_expert_backward(dy, xp, u, p, r["offsets"], wug, wdn, w_row)
    # dy and W_down are representable: dU is the plain oracle's with dY = w * dy at the boundary
    dxp0, dwu0, dwd0, du0 = O.expert_backward(w_row[:, None] * dy, xp, u, r["offsets"], wug, wdn)
    assert np.allclose(du[:M], du0[:M], rtol=1e-12, atol=1e-14)
    # the wgrads are BF16 products of the unquantized operands
    assert np.allclose(dwu, dwu0, rtol=1e-12, atol=1e-12)
    wd_ref = np.zeros_like(dwd)
    for e, (s, t) in enumerate(O.segments(r["offsets"])):
        wd_ref[e] = p[s:t].T @ dy[s:t]
    assert np.allclose(dwd, wd_ref, rtol=1e-13, atol=1e-13)
    # dU is quantized for the up dgrad: dxp within the quantization bound of bf16(dU)
    for e, (s, t) in enumerate(O.segments(r["offsets"])):
        if t == s:
            continue
        bound = _quant_bound(du[s:t], wug[e])
        assert (np.abs(dxp[s:t] - dxp0[s:t]) <= bound * (1 + 1e-9)).all()
    # empty experts: no arithmetic, zero gradients
    assert not dwu[2].any() and not dwd[2].any()
    # the routing-weight term through the exact (representable) dgrad is the plain oracle's
    # routing-weight gradient <y~, dOut> (dy is the unweighted gather of dOut here)
    y0, _, _, _ = O.expert_forward(xp, r["offsets"], wug, wdn)
    T, k = wl.T, wl.k
    dout = np.zeros((T, wl.d))
    src = r["sorted_src"][:M]
    dout[src // k] = dy[:M]          # a dOut whose gather is dy (each token's slots share one row)
    dwr_plain = O.routing_weight_grad(dout, y0, r["inv_map"], T, k)
    dwr = np.where(r["inv_map"] >= 0, g_dot[np.maximum(r["inv_map"], 0)], 0.0).reshape(T, k)
    tok = np.unique(src // k)
    one_slot = np.bincount(src // k, minlength=T)[tok] == 1
    assert np.allclose(dwr[tok[one_slot]], dwr_plain[tok[one_slot]], rtol=1e-12, atol=1e-12)


def test_mx_forward_planted_mistakes_fail_the_bound():
    """Weights whose magnitudes change by 2^5 from one output row (W_ug) or column (W_down) to
    the next are MX-exact along the contraction axis only. The MXFP8 forward must then give the
    plain U exactly and stay within the bound of the P quantization; quantizing a weight along
    the other axis, or dropping the routing weight, breaks one of these."""
    wl, r, xp, _, _, w_row = _case(8)
    rng = np.random.default_rng(9)
    mag_rows = np.ldexp(1.0, 5 * (np.arange(2 * wl.h) % 5) - 20)[None, :, None]
    mag_cols = np.ldexp(1.0, 5 * (np.arange(wl.d) % 5) - 20)[None, None, :]
    wug = _representable(rng, (wl.E, 2 * wl.h, wl.d), 1.0) * mag_rows      # exact along d only
    wdn = _representable(rng, (wl.E, wl.h, wl.d), 1.0) * mag_cols          # exact along h only
    assert not np.array_equal(X.mx_round_trip(wug[0], axis=0), wug[0])
    assert not np.array_equal(X.mx_round_trip(wdn[0], axis=1), wdn[0])
    s0, t0 = O.segments(r["offsets"])[0]
    y, u, p = X.mx_expert_forward(xp, r["offsets"], wug, wdn, w_row)
    y0, u0, a0, _ = O.expert_forward(xp, r["offsets"], wug, wdn)
    assert np.allclose(u[s0:t0], u0[s0:t0], rtol=1e-13, atol=0)
    pe = p[s0:t0]
    yw = w_row[s0:t0, None] * y0[s0:t0]
    bound = _quant_bound(pe, wdn[0])
    assert (np.abs(y[s0:t0] - yw) <= bound * (1 + 1e-9)).all()
    # planted: W_ug quantized along 2h (its other axis) changes U
    u_wrong = X.mx_round_trip(xp[s0:t0]) @ X.mx_round_trip(wug[0], axis=0).T
    assert not np.allclose(u_wrong, u0[s0:t0], rtol=1e-6, atol=0)
    # planted: W_down quantized along d leaves the bound
    y_wrong = X.mx_round_trip(X.bf16_round(pe)) @ X.mx_round_trip(wdn[0], axis=1)
    assert not (np.abs(y_wrong - yw) <= bound * (1 + 1e-9)).all()
    # planted: the routing weight dropped leaves the bound
    y_now = X.mx_round_trip(X.bf16_round(a0[s0:t0])) @ X.mx_round_trip(wdn[0], axis=0)
    assert not (np.abs(y_now - yw) <= bound).all()
