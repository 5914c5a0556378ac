"""The seeded input generators of the projection studies hold what they promise."""
import numpy as np

from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import workloads as W


def test_dirichlet_histograms_are_fixed_work_and_stratified():
    hists = W.dirichlet_histograms()
    assert len(hists) == 100
    keys = set()
    i_max = None
    for counts, ih in hists:
        assert counts.shape == (16,) and counts.sum() == 65536
        assert (counts % 8 == 0).all() and (counts >= 128).all()
        assert abs(ih - O.imbalance_IH(counts)) < 1e-12  # Eq. 18, from the oracle
        keys.add(tuple(sorted(counts.tolist())))
    assert len(keys) == 100  # distinct histograms
    # the most concentrated admissible histogram bounds the ranges; ten per equal-width range
    top = np.full(16, 128)
    top[0] = 65536 - 15 * 128
    i_max = O.imbalance_IH(top)
    ih = np.array([h[1] for h in hists])
    b = np.minimum((ih / i_max * 10).astype(int), 9)
    assert np.bincount(b, minlength=10).tolist() == [10] * 10
    assert W.dirichlet_histograms()[37][0].tolist() == hists[37][0].tolist()  # seeded


def test_balanced_counts_and_permutations():
    assert W.balanced_counts(64, 16).tolist() == [4] * 16
    assert W.balanced_counts(21, 4).tolist() == [6, 5, 5, 5]
    perms = W.expert_permutations(16, 4)
    assert perms[0].tolist() == list(range(16))
    assert all(sorted(p.tolist()) == list(range(16)) for p in perms)
    assert len({tuple(p.tolist()) for p in perms}) == 4


def test_exact_counts_workload():
    counts = [1, 15, 0, 513, 64]
    wl = W.exact_counts(counts, d=64, h=32, seed=5)
    assert (wl.T, wl.k, wl.E) == (sum(counts), 1, len(counts))
    r = O.route_offsets(wl.ids, wl.E)
    assert list(r["counts"]) == counts and r["M"] == sum(counts)
    again = W.exact_counts(counts, d=64, h=32, seed=5)
    assert np.array_equal(again.ids, wl.ids) and np.array_equal(again.weights, wl.weights)
    # the token order is shuffled, not grouped by expert
    assert not np.array_equal(wl.ids[:, 0], np.sort(wl.ids[:, 0]))
    assert ((wl.weights >= 0) & (wl.weights < 1)).all()
