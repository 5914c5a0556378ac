"""CPU fp64 oracle for the ragged grouped SwiGLU expert layer.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, the smoke check and the benchmark's CPU-baseline leg
import this module; the library's product path never calls it, and it shares no code with the
CUDA path (it imports numpy alone).

What it computes is the plain definition of the method, written out per expert in float64:
no blocking, fusion or reordering beyond what the definitions state. Every function names the
passage it follows. Pages cited:

* "Section 09: Grouped GEMM" (OLMo-core MoE report, §9) -- Eq. 13 (SwiGLU expert), Eq. 14
  (padding fraction), Fig. 35 (capacity rule and toy layout), Fig. 37 (device offsets, problem
  list, toy tiles), Eq. 15 and Table 15 (dgrad / wgrad), Eq. 16 (aligned capacity), Eq. 17
  (column partition), Eq. 18 (load imbalance).
* "Grouped expert GEMM: schedule irregular rows without changing the experts" -- FLOP
  convention for a gated expert, distinct expert parameters, empty groups.
* "grouped_mm" agent doc (halo) -- sort by expert dropping ids outside [0, E), int32
  cumulative offsets, scatter back with routing weights, atomic-free inverse map.

Readings where the pages are silent (each also listed in the design notes):
  c1  SwiGLU(U) = silu(U[:, :h]) * U[:, h:], gate rows first in W_ug.
  c2  offsets are inclusive segment ends, length E, int32.
  c3  rows inside an expert segment keep the order of the flat slot index t*k + j.
  c4  ids outside [0, E) are dropped: not counted, inverse map entry -1.
  c5  routing weights are applied at the combine, after the down projection.
  c10 a capacity-padded expert keeps its first C rows in placement order; later rows drop.

Parity status: every function here is pinned by tests/test_oracle.py against page values,
closed forms, brute-force loops or library special cases (torch autograd, np.add.at).
"""
from __future__ import annotations

import math
from typing import Callable, Sequence, Union

import numpy as np

ArrayOrFn = Union[np.ndarray, Callable[[int], np.ndarray]]


def _slice(w: ArrayOrFn, e: int) -> np.ndarray:
    return np.asarray(w(e) if callable(w) else w[e], dtype=np.float64)


# ---------------------------------------------------------------------------------------------
# a1-a3: histogram, offsets, stable placement, inverse map
# ---------------------------------------------------------------------------------------------
def route_offsets(ids: np.ndarray, E: int) -> dict:
    """Route histogram, inclusive int32 cumulative offsets, placement and inverse map.

    "Section 09: Grouped GEMM", Fig. 37 steps 1-2: the per-expert row counts live on the device
    and a prefix sum turns them into cumulative offsets whose each value ends one expert's
    segment (counts (1,4,3,2) -> [1,5,8,10]). The agent doc: tokens are sorted by expert into
    contiguous blocks after dropping ids outside [0, E); an inverse map [N, top_k] records the
    sorted position that feeds each (token, slot), sentinel-padded.

    Returns counts [E], offsets [E] (inclusive), sorted_src [n] (flat slot index placed at each
    position, -1 past M), inv_map [n] (position of each flat slot, -1 when dropped), M.
    """
    flat = np.asarray(ids).reshape(-1).astype(np.int64)
    n = flat.size
    valid = (flat >= 0) & (flat < E)
    counts = np.bincount(flat[valid], minlength=E).astype(np.int64)
    offsets = np.cumsum(counts)
    M = int(offsets[-1]) if E > 0 else 0
    slots = np.nonzero(valid)[0]
    # stable sort by expert keeps flat-index order inside each segment (reading c3)
    order = np.argsort(flat[slots], kind="stable")
    sorted_src = np.full(n, -1, np.int64)
    sorted_src[:M] = slots[order]
    inv_map = np.full(n, -1, np.int64)
    inv_map[sorted_src[:M]] = np.arange(M)
    return dict(counts=counts.astype(np.int32), offsets=offsets.astype(np.int32),
                sorted_src=sorted_src.astype(np.int32), inv_map=inv_map.astype(np.int32), M=M)


def segments(offsets: np.ndarray):
    """Problem list of Fig. 37 step 3: expert e owns rows [offsets[e-1], offsets[e])."""
    off = np.asarray(offsets, dtype=np.int64)
    starts = np.concatenate([[0], off[:-1]])
    return [(int(s), int(t)) for s, t in zip(starts, off)]


# ---------------------------------------------------------------------------------------------
# a5 / a9: permute (gather), optionally scaled per row
# ---------------------------------------------------------------------------------------------
def permute(x: np.ndarray, sorted_src: np.ndarray, M: int, k: int, row_scale=None) -> np.ndarray:
    """Gather token rows into expert-contiguous order (the forward gather x[idx] of the agent
    doc). Row p < M is x[sorted_src[p] // k], times row_scale[sorted_src[p]] when given (the
    combine's backward, Eq. 15 applied to the weighted sum). Rows p >= M are zero here; the
    device path leaves them untouched."""
    x = np.asarray(x, dtype=np.float64)
    n = sorted_src.size
    xp = np.zeros((n, x.shape[1]), np.float64)
    src = sorted_src[:M].astype(np.int64)
    xp[:M] = x[src // k]
    if row_scale is not None:
        xp[:M] *= np.asarray(row_scale, np.float64).reshape(-1)[src][:, None]
    return xp


# ---------------------------------------------------------------------------------------------
# a6-a7: the SwiGLU expert per segment (Eq. 13)
# ---------------------------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu(u: np.ndarray, h: int) -> np.ndarray:
    """SwiGLU(U) = silu(gate) * up with gate = U[:, :h], up = U[:, h:] (reading c1)."""
    return silu(u[:, :h]) * u[:, h:]


def expert_forward(xp: np.ndarray, offsets: np.ndarray, w_ug: ArrayOrFn, w_down: ArrayOrFn,
                   experts: Sequence[int] | None = None):
    """Eq. 13 per expert: U_e = X_e W_ug,e^T, Y_e = SwiGLU(U_e) W_down,e.

    Each row is multiplied by its own expert's matrices ("Grouped expert GEMM" page: grouping
    is not averaging or concatenating experts). Empty experts do no arithmetic. ``experts``
    restricts the loop to a sample of experts (rows of other experts stay zero).

    Returns (y [n, d], u [n, 2h], a [n, h], macs) with macs the multiply-adds performed.
    """
    xp = np.asarray(xp, dtype=np.float64)
    n, d = xp.shape
    w0 = _slice(w_down, 0)
    h = w0.shape[0]
    y = np.zeros((n, d), np.float64)
    u = np.zeros((n, 2 * h), np.float64)
    a = np.zeros((n, h), np.float64)
    macs = 0
    segs = segments(offsets)
    for e in (range(len(segs)) if experts is None else experts):
        s, t = segs[e]
        if t == s:
            continue
        ue = xp[s:t] @ _slice(w_ug, e).T
        ae = swiglu(ue, h)
        y[s:t] = ae @ _slice(w_down, e)
        u[s:t], a[s:t] = ue, ae
        macs += (t - s) * d * 2 * h + (t - s) * h * d
    return y, u, a, macs


# ---------------------------------------------------------------------------------------------
# a8 / a14: combine through the inverse map
# ---------------------------------------------------------------------------------------------
def combine(y: np.ndarray, inv_map: np.ndarray, weights, T: int, k: int) -> np.ndarray:
    """Scatter expert outputs back to tokens and apply routing weights (agent doc), expressed
    as a gather + reduction over the inverse map: out[t] = sum_j w[t,j] * y[inv[t,j]] over the
    slots j with inv >= 0. weights=None means all ones (the permute's backward)."""
    y = np.asarray(y, dtype=np.float64)
    inv = np.asarray(inv_map).reshape(T, k).astype(np.int64)
    w = np.ones((T, k)) if weights is None else np.asarray(weights, np.float64).reshape(T, k)
    out = np.zeros((T, y.shape[1]), np.float64)
    for j in range(k):
        ok = inv[:, j] >= 0
        out[ok] += w[ok, j][:, None] * y[inv[ok, j]]
    return out


def routing_weight_grad(dout: np.ndarray, y: np.ndarray, inv_map: np.ndarray, T: int,
                        k: int) -> np.ndarray:
    """Gradient of the combine (agent doc: scatter back with routing weights) with respect to
    the routing weights. out[t] = sum_j w[t,j] * y[inv[t,j]] is linear in w, so
    dL/dw[t,j] = <dOut[t], y[inv[t,j]]> with y the unweighted expert output; 0 for a dropped
    slot. Returns float64 [T, k]."""
    dout = np.asarray(dout, np.float64)
    y = np.asarray(y, np.float64)
    inv = np.asarray(inv_map).reshape(T, k).astype(np.int64)
    dw = np.zeros((T, k), np.float64)
    for j in range(k):
        ok = inv[:, j] >= 0
        dw[ok, j] = np.einsum("td,td->t", dout[ok], y[inv[ok, j]])
    return dw


# ---------------------------------------------------------------------------------------------
# a10-a13: backward (Eq. 15, Table 15) of the SwiGLU expert
# ---------------------------------------------------------------------------------------------
def expert_backward(dy: np.ndarray, xp: np.ndarray, u: np.ndarray, offsets: np.ndarray,
                    w_ug: ArrayOrFn, w_down: ArrayOrFn, experts: Sequence[int] | None = None):
    """Dgrad and wgrad of Eq. 13 per expert, each projection following Eq. 15:
    grad X = grad Y W^T and grad W = X^T grad Y, with M_e as output rows (dgrad) and as the
    contraction length (wgrad), Table 15.

    With g, v = U[:, :h], U[:, h:], s = sigmoid(g), A = silu(g) * v:
      dA = dY W_down^T;  dg = dA * v * s * (1 + g (1 - s));  dv = dA * silu(g)
      dU = [dg dv];  dX = dU W_ug;  dW_ug = dU^T X;  dW_down = A^T dY.
    Empty experts get dW = 0. Returns (dxp [n, d], dw_ug [E, 2h, d], dw_down [E, h, d], du).
    """
    dy = np.asarray(dy, np.float64)
    xp = np.asarray(xp, np.float64)
    u = np.asarray(u, np.float64)
    n, d = xp.shape
    h = u.shape[1] // 2
    segs = segments(offsets)
    E = len(segs)
    dxp = np.zeros((n, d), np.float64)
    du = np.zeros((n, 2 * h), np.float64)
    dw_ug = np.zeros((E, 2 * h, d), np.float64)
    dw_down = np.zeros((E, h, d), np.float64)
    for e in (range(E) if experts is None else experts):
        s, t = segs[e]
        if t == s:
            continue
        wu, wd = _slice(w_ug, e), _slice(w_down, e)
        g, v = u[s:t, :h], u[s:t, h:]
        sg = 1.0 / (1.0 + np.exp(-g))
        ae = g * sg * v
        da = dy[s:t] @ wd.T
        due = np.concatenate([da * v * sg * (1.0 + g * (1.0 - sg)), da * g * sg], axis=1)
        dxp[s:t] = due @ wu
        dw_ug[e] = due.T @ xp[s:t]
        dw_down[e] = ae.T @ dy[s:t]
        du[s:t] = due
    return dxp, dw_ug, dw_down, du


# ---------------------------------------------------------------------------------------------
# One grouped projection (Eq. 15 / Eq. 17): Y_e = X_e W_e over row segments
# ---------------------------------------------------------------------------------------------
def grouped_linear(x: np.ndarray, offsets: np.ndarray, w: ArrayOrFn) -> np.ndarray:
    """Forward row of Table 15: Y_e = X_e W_e with W_e [d_in, d_out], per row segment."""
    x = np.asarray(x, np.float64)
    segs = segments(offsets)
    d_out = _slice(w, 0).shape[1]
    y = np.zeros((x.shape[0], d_out))
    for e, (s, t) in enumerate(segs):
        if t > s:
            y[s:t] = x[s:t] @ _slice(w, e)
    return y


# ---------------------------------------------------------------------------------------------
# Comparison variant: capacity-padded BMM (Eq. 14, Fig. 35)
# ---------------------------------------------------------------------------------------------
def capacity_ceil(c: float, M: int, n_local: int) -> int:
    """C = ceil(c * M_bar) with M_bar = M / N_local (Fig. 35 sweep rule; footnote 1 of §9)."""
    return int(math.ceil(c * M / n_local - 1e-12))


def capacity_eq16(c: float, M: int, n_local: int, ep_ranks: int = 1) -> int:
    """Eq. 16: C = M_E * 8 * ceil(floor(c * M_bar / M_E) / 8)."""
    mbar = M / n_local
    return ep_ranks * 8 * int(math.ceil(math.floor(c * mbar / ep_ranks) / 8))


def rho_pad(counts: np.ndarray, C: int) -> float:
    """Eq. 14: padding fraction 1 - sum(M_e) / (N_local * C), over routed rows that fit."""
    counts = np.asarray(counts, np.int64)
    return 1.0 - float(np.minimum(counts, C).sum()) / float(counts.size * C)


def padded_bmm_forward(xp: np.ndarray, offsets: np.ndarray, C: int, w_ug: ArrayOrFn,
                       w_down: ArrayOrFn):
    """Fig. 35: pad every expert to capacity C, run one regular batched product, discard the
    padding. Each expert keeps its first C rows in placement order (reading c10); a row beyond
    C is dropped and its output is zero. Returns (y [n, d], stats)."""
    xp = np.asarray(xp, np.float64)
    n, d = xp.shape
    segs = segments(offsets)
    E = len(segs)
    h = _slice(w_down, 0).shape[0]
    xpad = np.zeros((E, C, d))
    for e, (s, t) in enumerate(segs):
        keep = min(t - s, C)
        xpad[e, :keep] = xp[s:s + keep]
    ypad = np.zeros((E, C, d))
    for e in range(E):   # the batched product touches every padded row
        ypad[e] = swiglu(xpad[e] @ _slice(w_ug, e).T, h) @ _slice(w_down, e)
    y = np.zeros((n, d))
    dropped = 0
    for e, (s, t) in enumerate(segs):
        keep = min(t - s, C)
        y[s:s + keep] = ypad[e, :keep]
        dropped += (t - s) - keep
    counts = np.array([t - s for s, t in segs])
    stats = dict(rows_multiplied=E * C, padding_rows=int(E * C - np.minimum(counts, C).sum()),
                 dropped_rows=dropped, rho_pad=rho_pad(counts, C))
    return y, stats


# ---------------------------------------------------------------------------------------------
# Closed forms used by the measurement
# ---------------------------------------------------------------------------------------------
def flops_fwd(M: int, d: int, h: int) -> int:
    """Gated expert, two-FLOP multiply-add convention: 6 * n_e * d * h ("Grouped expert GEMM"
    page); excludes the nonlinearity, routing and backward."""
    return 6 * M * d * h


def flops_fwd_bwd(M: int, d: int, h: int) -> int:
    """Forward plus dgrad and wgrad of both projections (each the m*n*k of its forward,
    Table 15): 18 * M * d * h."""
    return 18 * M * d * h


def imbalance_IH(counts: np.ndarray) -> float:
    """Eq. 18: I_H = 1 - H(p) / log N_local with p_e = M_e / M (0 log 0 = 0)."""
    counts = np.asarray(counts, np.float64)
    p = counts / counts.sum()
    p = p[p > 0]
    return 1.0 + float((p * np.log(p)).sum()) / math.log(counts.size)


def toy_tiles(counts: Sequence[int], tile_rows: int, col_blocks: int) -> int:
    """Fig. 37 step 4: tiles of ``tile_rows`` rows over ``col_blocks`` column blocks for every
    expert of the problem list: sum_e ceil(M_e / tile_rows) * col_blocks."""
    return int(sum(-(-int(c) // tile_rows) * col_blocks for c in counts))


def roofline_ceiling(intensity: float, bandwidth: float, peak: float) -> float:
    """Attainable rate of the roofline lab: min(peak, intensity * bandwidth)."""
    return min(peak, intensity * bandwidth)
