"""Helpers for the GPU parity tests: run the library pipeline and the oracle pipeline on the same
seeded inputs, and compare with the tolerance the float results must meet:
    ||got - ref|| / ||ref|| <= 5e-3   and   max |got - ref| <= 2e-2 * (1 + |ref|)  elementwise.
The oracle is fp64 throughout; the library rounds A, U, y, dU, dxp and out to bf16 once each and
accumulates in fp32, so the bound is a few bf16 half-ulps (2^-9) of accumulated rounding."""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import _lib

REL_NORM_TOL = 5e-3
MAX_ABS_TOL = 2e-2

_WEIGHT_CACHE: dict = {}


def dev_bf16(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).cuda()


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_f32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def device_weights(wl):
    """W_ug [E, 2h, d] and W_down [E, h, d] on the device, built expert by expert."""
    key = (wl.name, wl.seed, wl.E, wl.d, wl.h)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE.clear()
        wug = torch.empty(wl.E, 2 * wl.h, wl.d, dtype=torch.bfloat16, device="cuda")
        wdn = torch.empty(wl.E, wl.h, wl.d, dtype=torch.bfloat16, device="cuda")
        for e in range(wl.E):
            wug[e].copy_(torch.from_numpy(wl.w_ug(e)).to(torch.bfloat16))
            wdn[e].copy_(torch.from_numpy(wl.w_down(e)).to(torch.bfloat16))
        _WEIGHT_CACHE[key] = (wug, wdn)
    return _WEIGHT_CACHE[key]


def nan_filled(shape, dtype=torch.bfloat16) -> torch.Tensor:
    """A buffer whose unwritten rows would poison any result that read them."""
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def assert_close(got, ref, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = got - ref
    denom = max(np.linalg.norm(ref), 1e-30)
    rel = np.linalg.norm(err) / denom
    assert rel <= REL_NORM_TOL, f"{what}: normalised error {rel:.3e} > {REL_NORM_TOL}"
    bound = MAX_ABS_TOL * (1.0 + np.abs(ref))
    worst = np.argmax(np.abs(err) - bound)
    assert (np.abs(err) <= bound).all(), (
        f"{what}: |err| {np.abs(err).flat[worst]:.3e} > bound {bound.flat[worst]:.3e} at {np.unravel_index(worst, err.shape)}")


def unblock_u(u_bytes: torch.Tensor, offsets: np.ndarray, h: int) -> torch.Tensor:
    """Rows [M, 2h] (fp32) of the saved U from its blocked 24-bit layout, as the header states it:
    row p of expert e (the segment starting at s_e) is row r = p - s_e of row tile G = (row tiles
    of the experts before e) + r // 128, lane l = r % 32 of quadrant q = (r % 128) // 32; column
    c is in 16-column chunk ci = c // 16 for gate columns and ceil(h/16) + (c - h) // 16 for up
    columns, position j = c % 16 in it. The chunk's block starts at byte ((G*4 + q)*C2 + ci)*1536
    (C2 = 2 ceil(h/16)); the upper 16 bits of value j are the little-endian 16-bit word
    (j // 8)*256 + l*8 + j % 8 of the block, its lower 8 bits byte 1024 + l*16 + j, and the fp32
    value is those 24 bits followed by 8 zero bits."""
    h16 = (h + 15) // 16
    c2 = 2 * h16
    starts = np.concatenate([[0], offsets[:-1]])
    tiles = (offsets - starts + 127) // 128
    tile0 = np.concatenate([[0], np.cumsum(tiles)[:-1]])
    M = int(offsets[-1])
    p = np.arange(M)
    e = np.searchsorted(offsets, p, side="right")
    r = p - starts[e]
    g = tile0[e] + r // 128
    q = (r % 128) // 32
    lane = r % 32
    c = np.arange(2 * h)
    cc = np.where(c < h, c, c - h)
    ci = cc // 16 + np.where(c < h, 0, h16)
    j = cc % 16
    block = ((g[:, None] * 4 + q[:, None]) * c2 + ci[None, :]) * 1536
    hi_at = block + (j // 8)[None, :] * 512 + lane[:, None] * 16 + (j % 8)[None, :] * 2
    lo_at = block + 1024 + lane[:, None] * 16 + j[None, :]
    b = u_bytes.reshape(-1).view(torch.uint8)
    dev = b.device
    hi = b[torch.from_numpy(hi_at).to(dev)].to(torch.int64) | (b[torch.from_numpy(hi_at + 1).to(dev)].to(torch.int64) << 8)
    lo = b[torch.from_numpy(lo_at).to(dev)].to(torch.int64)
    v = (hi << 16) | (lo << 8)
    bits = torch.where(v >= 2 ** 31, v - 2 ** 32, v).to(torch.int32)  # the same 32 bits as int32
    return bits.view(torch.float32)


class DevicePipeline:
    """The library pipeline (route, permute, grouped forward, optional backward, combine) on
    a workload, with NaN-filled row buffers so that rows past M cannot leak into results."""

    def __init__(self, wl, with_u=True):
        self.wl = wl
        T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
        self.ids = dev_i32(wl.ids)
        self.x = dev_bf16(wl.x())
        self.weights = dev_f32(wl.weights)
        self._w = None
        self.counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        self.offsets = torch.full((E,), -7, dtype=torch.int32, device="cuda")
        self.sorted_src = torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")
        self.inv_map = torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")
        ws = _lib.moe_workspace_bytes(_lib.OP_ROUTE, T, k, E)
        self.route_ws = torch.empty(max(ws, 1), dtype=torch.uint8, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.cap = n
        self.xp = nan_filled((max(n, 1), d))
        self.y = nan_filled((max(n, 1), d))
        self.a = nan_filled((max(n, 1), h))
        # saved state for the backward: the low half of P [n, h], then U (24 bits, blocked)
        sv = _lib.moe_workspace_bytes(_lib.OP_SAVED, T, k, E, d, h)
        self.saved = nan_filled((max(sv, 4) // 4,), torch.float32) if with_u else None

    @property
    def w_ug(self):
        if self._w is None:
            self._w = device_weights(self.wl)
        return self._w[0]

    @property
    def w_down(self):
        if self._w is None:
            self._w = device_weights(self.wl)
        return self._w[1]

    def route(self):
        wl = self.wl
        _lib.moe_route_offsets(self.ids, wl.T, wl.k, wl.E, self.counts, self.offsets, self.sorted_src,
                               self.inv_map, self.route_ws)
        return self

    def permute(self):
        wl = self.wl
        _lib.moe_permute(self.x, self.sorted_src, self.offsets, None, wl.T, wl.k, wl.E, wl.d, self.xp)
        return self

    def forward(self):
        wl = self.wl
        fw = _lib.moe_workspace_bytes(_lib.OP_FWD, wl.T, wl.k, wl.E, wl.d, wl.h)
        ws = torch.empty(fw, dtype=torch.uint8, device="cuda") if fw > 0 else None
        _lib.moe_grouped_swiglu_fwd(self.xp, self.offsets, None, None, wl.E, self.cap, wl.d, wl.h, self.w_ug,
                                    self.w_down, self.y, self.a, self.saved, ws, self.status)
        return self

    @property
    def u(self):
        """The U the forward saved (24 bits of each fp32 value), as [M, 2h] fp32 rows (unblocked)."""
        h = self.wl.h
        h8 = (h + 7) // 8 * 8  # widths that are not multiples of 8 are stored zero-padded
        u_flat, _ = _lib.saved_views(self.saved, max(self.cap, 1), h)
        u8 = unblock_u(u_flat, self.offsets.cpu().numpy().astype(np.int64), h8)
        return torch.cat([u8[:, :h], u8[:, h8:h8 + h]], dim=1)

    def combine(self):
        wl = self.wl
        self.out = torch.empty(wl.T, wl.d, dtype=torch.bfloat16, device="cuda")
        _lib.moe_unpermute_combine(self.y, self.inv_map, self.weights, wl.T, wl.k, wl.d, self.out)
        return self

    def backward(self, dy):
        wl = self.wl
        n, d, h, E = self.cap, wl.d, wl.h, wl.E
        self.dy = dy
        self.dxp = nan_filled((max(n, 1), d))
        self.dw_ug = torch.full((E, 2 * h, d), float("nan"), dtype=torch.float32, device="cuda")
        self.dw_down = torch.full((E, h, d), float("nan"), dtype=torch.float32, device="cuda")
        ws = _lib.moe_workspace_bytes(_lib.OP_BWD, wl.T, wl.k, E, d, h)
        self.bwd_ws = torch.full((max(ws, 2) // 2,), float("nan"), dtype=torch.bfloat16, device="cuda")
        _lib.moe_grouped_bwd(dy, self.xp, self.a, self.saved, self.offsets, None, None, E, n, d, h, self.w_ug,
                             self.w_down,
                             self.dxp, self.dw_ug, self.dw_down, self.bwd_ws, self.status)
        return self


_ORACLE_CACHE: dict = {}


def oracle_run(wl, experts=None):
    """The oracle pipeline on the same inputs: route, permute, expert forward. The last result is
    kept, so the forward and backward tests of one (costly) workload compute it once."""
    key = (wl.name, wl.seed, wl.T, wl.k, wl.E, wl.d, wl.h, wl.ids.tobytes(),
           None if experts is None else tuple(experts))
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE.clear()
        r = O.route_offsets(wl.ids, wl.E)
        xp = O.permute(wl.x(), r["sorted_src"], r["M"], wl.k)
        y, u, a, _ = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down, experts)
        _ORACLE_CACHE[key] = (r, xp, y, u, a)
    return _ORACLE_CACHE[key]


def sample_experts(counts, n_pick=6, seed=0):
    """First, last, largest, smallest non-empty and a few random experts."""
    counts = np.asarray(counts)
    nz = np.nonzero(counts)[0]
    pick = {int(nz[0]), int(nz[-1]), int(nz[np.argmax(counts[nz])]), int(nz[np.argmin(counts[nz])])}
    rng = np.random.default_rng(seed)
    while len(pick) < min(n_pick, nz.size):
        pick.add(int(rng.choice(nz)))
    return sorted(pick)


def rows_of(offsets, experts):
    segs = O.segments(offsets)
    return np.concatenate([np.arange(*segs[e]) for e in experts]) if experts else np.zeros(0, int)
