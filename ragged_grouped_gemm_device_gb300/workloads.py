"""Seeded synthetic inputs for the ragged grouped SwiGLU expert layer.

This module draws random numbers and rounds them to bf16. It holds none of the method's
arithmetic (no histogram, offsets, placement, GEMM, SwiGLU or combine), so both the CUDA path
and the CPU oracle can consume what it produces.

Five workloads, named for what they are:

* ``toy``       -- the four-expert worked example of Figs. 35-37 of "Section 09: Grouped GEMM"
                   (rows per expert 1, 4, 3, 2; M = 10), d = 64, h = 128.
* ``balanced``  -- T = 2048 tokens, E = 8, top-2 over N(0,1) router logits, d = 1024, h = 2048.
* ``finegrained`` -- T = 4096, E = 128, top-8 over N(0,1) logits plus a per-expert N(0, 0.5)
                   bias, d = 2048, h = 768 (the Qwen3-30B-A3B expert shape quoted in the
                   grouped_mm agent doc's isolated-kernel benchmark).
* ``skew``      -- E = 64, M = 20000 rows, k = 1, Zipf(1.2) counts over a random expert
                   permutation with 13 experts empty and no count a multiple of 8,
                   d = h = 1000 (not tile aligned).
* ``large``     -- T = 16384, E = 256, top-8 over N(0,1) logits, d = 2048, h = 512.

Weights are N(0, std = 1/sqrt(fan_in)) with fan_in = d for W_ug and h for W_down. Every
per-expert weight slice comes from its own seeded stream, so a sample of experts can be drawn
without generating the rest. Routing weights are the softmax over the k selected logits
(uniform(0,1) for the toy; 1 for k = 1 skew).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# stream tags: each tensor family draws from its own SeedSequence branch
_TAG_IDS, _TAG_X, _TAG_WUG, _TAG_WDOWN, _TAG_DOUT, _TAG_DY, _TAG_W = 1, 2, 3, 4, 5, 6, 7


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32 holding them."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """uint16 bit patterns of bf16-exact float32 values (for copying to a bf16 device tensor)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def _rng(seed: int, tag: int, *extra: int) -> np.random.Generator:
    return np.random.default_rng([seed, tag, *extra])


def _normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return round_to_bf16(a)


def _topk_softmax(logits: np.ndarray, k: int):
    """Router used only to generate inputs: top-k by logit (ties -> lower expert id), softmax
    over the k selected logits."""
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    sel = sel - sel.max(axis=1, keepdims=True)
    p = np.exp(sel)
    p /= p.sum(axis=1, keepdims=True)
    return order.astype(np.int32), p.astype(np.float32)


def skew_counts(seed: int, E: int = 64, M: int = 20000, n_empty: int = 13, s: float = 1.2):
    """Per-expert counts for the skew workload.

    1. permute the experts with a seeded permutation; 2. the last ``n_empty`` get zero rows;
    3. the others get weights r^-s (rank r = 1..), apportioned to M by largest remainder;
    4. counts that are multiples of 8 are nudged by one row, conserving the sum, so no count
    is a multiple of 8 (hence none of 128).
    """
    rng = _rng(seed, _TAG_IDS, 4)
    perm = rng.permutation(E)
    active = perm[: E - n_empty]
    r = np.arange(1, active.size + 1, dtype=np.float64)
    wts = r ** (-s)
    quota = M * wts / wts.sum()
    base = np.floor(quota).astype(np.int64)
    rem = M - int(base.sum())
    frac_order = np.argsort(-(quota - base), kind="stable")
    base[frac_order[:rem]] += 1
    counts = np.zeros(E, dtype=np.int64)
    counts[active] = base

    def bad(c):
        return c % 8 == 0

    for e in active:
        if not bad(counts[e]):
            continue
        ranked = active[np.argsort(-counts[active], kind="stable")]
        partner = ranked[0] if ranked[0] != e else ranked[1]
        counts[e] += 1
        counts[partner] -= 1
        if bad(counts[partner]):
            counts[e] += 1
            counts[partner] -= 1
    assert counts.sum() == M
    assert all(not bad(counts[e]) and counts[e] > 0 for e in active)
    return counts.astype(np.int32), active


@dataclass
class Workload:
    name: str
    T: int
    k: int
    E: int
    d: int
    h: int
    seed: int = 0
    ids: np.ndarray = field(default=None, repr=False)      # int32 [T, k]
    weights: np.ndarray = field(default=None, repr=False)  # float32 [T, k]
    has_bwd: bool = True
    bwd_from_dout: bool = False   # True: upstream grad is dOut [T, d] through the combine

    @property
    def n(self) -> int:
        """Fixed physical capacity in rows: one per (token, slot)."""
        return self.T * self.k

    def x(self) -> np.ndarray:
        """Token activations X, float32 [T, d] holding bf16 values, N(0, 1)."""
        return _normal_bf16(_rng(self.seed, _TAG_X), (self.T, self.d))

    def w_ug(self, e: int) -> np.ndarray:
        """Expert e's up/gate weight [2h, d] (gate rows first), N(0, 1/sqrt(d))."""
        return _normal_bf16(_rng(self.seed, _TAG_WUG, e), (2 * self.h, self.d), 1.0 / np.sqrt(self.d))

    def w_down(self, e: int) -> np.ndarray:
        """Expert e's down weight [h, d], N(0, 1/sqrt(h))."""
        return _normal_bf16(_rng(self.seed, _TAG_WDOWN, e), (self.h, self.d), 1.0 / np.sqrt(self.h))

    def w_ug_all(self) -> np.ndarray:
        return np.stack([self.w_ug(e) for e in range(self.E)])

    def w_down_all(self) -> np.ndarray:
        return np.stack([self.w_down(e) for e in range(self.E)])

    def dout(self) -> np.ndarray:
        """Upstream gradient of the combined output, [T, d], N(0, 1)."""
        return _normal_bf16(_rng(self.seed, _TAG_DOUT), (self.T, self.d))

    def dy(self, rows: int) -> np.ndarray:
        """Upstream gradient at the grouped-GEMM boundary, [rows, d], N(0, 1)."""
        return _normal_bf16(_rng(self.seed, _TAG_DY), (rows, self.d))


def make(name: str, seed: int = 0) -> Workload:
    """Build one of the five named workloads (routing drawn here; weights drawn lazily)."""
    if name == "toy":
        wl = Workload("toy", T=10, k=1, E=4, d=64, h=128, seed=seed)
        rng = _rng(seed, _TAG_IDS, 1)
        wl.ids = rng.permutation(np.array([0, 1, 1, 1, 1, 2, 2, 2, 3, 3], np.int32)).reshape(10, 1)
        wl.weights = rng.uniform(0.0, 1.0, size=(10, 1)).astype(np.float32)
        return wl
    if name == "toy_sorted":
        wl = make("toy", seed)
        wl.name = "toy_sorted"
        wl.ids = np.array([0, 1, 1, 1, 1, 2, 2, 2, 3, 3], np.int32).reshape(10, 1)
        return wl
    if name == "balanced":
        wl = Workload("balanced", T=2048, k=2, E=8, d=1024, h=2048, seed=seed, has_bwd=False)
        logits = _rng(seed, _TAG_IDS, 2).standard_normal((wl.T, wl.E))
        wl.ids, wl.weights = _topk_softmax(logits, wl.k)
        return wl
    if name == "finegrained":
        wl = Workload("finegrained", T=4096, k=8, E=128, d=2048, h=768, seed=seed)
        rng = _rng(seed, _TAG_IDS, 3)
        logits = rng.standard_normal((wl.T, wl.E)) + rng.normal(0.0, 0.5, size=(1, wl.E))
        wl.ids, wl.weights = _topk_softmax(logits, wl.k)
        return wl
    if name == "skew":
        wl = Workload("skew", T=20000, k=1, E=64, d=1000, h=1000, seed=seed)
        counts, _ = skew_counts(seed)
        rows = np.repeat(np.arange(wl.E, dtype=np.int32), counts)
        wl.ids = _rng(seed, _TAG_IDS, 5).permutation(rows).reshape(wl.T, 1)
        wl.weights = np.ones((wl.T, 1), np.float32)
        return wl
    if name == "large":
        wl = Workload("large", T=16384, k=8, E=256, d=2048, h=512, seed=seed, bwd_from_dout=True)
        logits = _rng(seed, _TAG_IDS, 6).standard_normal((wl.T, wl.E))
        wl.ids, wl.weights = _topk_softmax(logits, wl.k)
        return wl
    if name == "medium":
        # the large workload's expert shape with a quarter of the tokens and experts: a few GB on
        # the device, still above the 129 MB L2 (used for detailed profiler captures)
        wl = Workload("medium", T=4096, k=8, E=64, d=2048, h=512, seed=seed, bwd_from_dout=True)
        logits = _rng(seed, _TAG_IDS, 7).standard_normal((wl.T, wl.E))
        wl.ids, wl.weights = _topk_softmax(logits, wl.k)
        return wl
    raise ValueError(f"unknown workload {name!r}")


def custom(T: int, k: int, E: int, d: int, h: int, seed: int = 0, invalid_frac: float = 0.0,
           empty_experts=(), name: str = "custom") -> Workload:
    """A small seeded workload for edge cases: uniform random expert ids, optional -1/E padding
    ids (a fraction ``invalid_frac`` of slots) and experts that receive no rows."""
    rng = _rng(seed, _TAG_IDS, 99, T, k, E)
    allowed = np.array([e for e in range(E) if e not in set(empty_experts)], np.int32)
    ids = allowed[rng.integers(0, allowed.size, size=(T, k))] if allowed.size else np.full((T, k), -1, np.int32)
    if invalid_frac > 0:
        mask = rng.uniform(size=(T, k)) < invalid_frac
        bad = np.where(rng.uniform(size=(T, k)) < 0.5, -1, E).astype(np.int32)
        ids = np.where(mask, bad, ids).astype(np.int32)
    wl = Workload(name, T=T, k=k, E=E, d=d, h=h, seed=seed)
    wl.ids = ids.astype(np.int32)
    wl.weights = _rng(seed, _TAG_W, T, k).uniform(0.0, 1.0, size=(T, k)).astype(np.float32)
    return wl


def exact_counts(counts, d: int, h: int, seed: int = 0, name: str = "exact_counts") -> Workload:
    """top_k = 1 and expert e receives exactly counts[e] tokens, in a seeded random token order:
    segment lengths chosen around the tile and K-step boundaries of the kernels."""
    counts = np.asarray(counts, np.int64)
    rng = _rng(seed, _TAG_IDS, 7, counts.size, int(counts.sum()))
    ids = np.repeat(np.arange(counts.size, dtype=np.int32), counts)
    ids = ids[rng.permutation(ids.size)]
    T = int(ids.size)
    wl = Workload(name, T=T, k=1, E=int(counts.size), d=d, h=h, seed=seed)
    wl.ids = ids.reshape(T, 1).astype(np.int32)
    wl.weights = _rng(seed, _TAG_W, T, 1).uniform(0.0, 1.0, size=(T, 1)).astype(np.float32)
    return wl


NAMES = ("toy", "balanced", "finegrained", "skew", "large")


# ---------------------------------------------------------------------------------------------
# One square expert projection (Figs. 38 and 40 of "Section 09: Grouped GEMM"): 16 local
# experts, Y_e = X_e W_e with W_e [K, N], K = N = 4096.
_TAG_PROJ_W, _TAG_PROJ_X, _TAG_HIST, _TAG_PERM = 8, 9, 10, 11


def projection_weight(e: int, K: int, N: int, seed: int = 0) -> np.ndarray:
    """Expert e's projection weight [K, N], N(0, 1/sqrt(K)), bf16 values in float32."""
    return _normal_bf16(_rng(seed, _TAG_PROJ_W, e, K, N), (K, N), 1.0 / np.sqrt(K))


def projection_x(rows: int, K: int, seed: int = 0) -> np.ndarray:
    """Projection input rows [rows, K], N(0, 1), bf16 values in float32."""
    return _normal_bf16(_rng(seed, _TAG_PROJ_X, rows, K), (rows, K))


def balanced_counts(M: int, E: int) -> np.ndarray:
    """M rows over E experts as evenly as possible (the first M mod E experts get one more)."""
    c = np.full(E, M // E, np.int64)
    c[: M % E] += 1
    return c


def _entropy_imbalance(counts: np.ndarray) -> float:
    """Eq. 18 of "Section 09" for a drawn histogram, used only to stratify the draws:
    1 + sum_e p_e log p_e / log E over the experts with rows."""
    p = np.asarray(counts, np.float64) / float(np.sum(counts))
    p = p[p > 0]
    return 1.0 + float(np.sum(p * np.log(p))) / float(np.log(len(counts)))


def dirichlet_histograms(M: int = 65536, E: int = 16, n_bins: int = 10, per_bin: int = 10,
                         tile: int = 128, align: int = 8, seed: int = 0,
                         max_draws: int = 400000) -> list:
    """Fig. 40's fixed-work histograms: symmetric-Dirichlet proposals (concentration drawn
    log-uniformly from 10^-2.5 to 10^2) turned into exact counts that are multiples of `align`,
    hold at least one `tile` of rows per expert and sum to M (each expert gets one tile, the
    remaining (M - E*tile)/align units of `align` rows go by largest remainder of the
    proposal, ties to the lower expert). Kept: `per_bin` histograms with distinct sorted counts
    in each of `n_bins` equal-width ranges of I_H between 0 and the largest admissible I_H
    (one expert holding everything but the other experts' single tiles).

    Returns a list of (counts int64 [E], I_H), bin by bin."""
    units = M - E * tile
    if units < 0 or units % align:
        raise ValueError("M - E*tile must be a non-negative multiple of align")
    units //= align
    top = np.full(E, tile, np.int64)
    top[0] += units * align
    i_max = _entropy_imbalance(top)
    rng = _rng(seed, _TAG_HIST, M, E, n_bins, per_bin)
    bins = [[] for _ in range(n_bins)]
    seen = set()
    for _ in range(max_draws):
        if all(len(b) >= per_bin for b in bins):
            break
        alpha = 10.0 ** rng.uniform(-2.5, 2.0)
        p = rng.dirichlet(np.full(E, alpha))
        if not np.all(np.isfinite(p)) or p.sum() <= 0:
            continue
        quota = p / p.sum() * units
        alloc = np.floor(quota).astype(np.int64)
        rest = int(units - alloc.sum())
        order = np.argsort(-(quota - alloc), kind="stable")
        alloc[order[:rest]] += 1
        counts = tile + align * alloc
        key = tuple(sorted(counts.tolist()))
        if key in seen:
            continue
        ih = _entropy_imbalance(counts)
        b = min(int(ih / i_max * n_bins), n_bins - 1)
        if len(bins[b]) < per_bin:
            bins[b].append((counts, ih))
            seen.add(key)
    if not all(len(b) >= per_bin for b in bins):
        raise RuntimeError("could not fill every I_H range; raise max_draws")
    return [item for b in bins for item in b]


def expert_permutations(E: int, n: int, seed: int = 0) -> list:
    """n seeded permutations of the expert indices (the first is the identity)."""
    rng = _rng(seed, _TAG_PERM, E, n)
    return [np.arange(E)] + [rng.permutation(E) for _ in range(n - 1)]
