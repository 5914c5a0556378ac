"""Pins for the CPU oracle: page values, closed forms, brute force and library special cases.

Each test fixes something the pages or the mathematics determine independently of the oracle's
own code, so that a dropped term, a swapped gate/up, a wrong index or a transposed operand in
the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import brute
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _layer(wl, experts=None):
    """The oracle's forward pipeline: route -> permute -> experts -> combine."""
    r = O.route_offsets(wl.ids, wl.E)
    x = wl.x()
    xp = O.permute(x, r["sorted_src"], r["M"], wl.k)
    y, u, a, macs = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down, experts)
    out = O.combine(y, r["inv_map"], wl.weights, wl.T, wl.k)
    return r, x, xp, y, u, a, out, macs


# ------------------------------------------------------------------------------ page values
def test_toy_offsets_and_problem_list():
    g = _gold("toy_fig35_37.json")
    for name in ("toy", "toy_sorted"):
        wl = W.make(name)
        r = O.route_offsets(wl.ids, wl.E)
        assert r["counts"].tolist() == g["counts"]
        assert r["offsets"].tolist() == g["offsets_inclusive"]
        assert r["M"] == g["M"]
        assert [list(s) for s in O.segments(r["offsets"])] == g["problem_list"]
        assert r["offsets"].dtype == np.int32


def test_toy_capacity_padding_and_tiles():
    g = _gold("toy_fig35_37.json")
    counts = np.array(g["counts"])
    C = O.capacity_ceil(g["capacity_factor"], g["M"], g["n_local"])
    assert C == g["C"]
    assert O.rho_pad(counts, C) == pytest.approx(g["rho_pad"], abs=0)
    assert O.toy_tiles(counts, g["toy_tile_rows"], g["toy_col_blocks"]) == g["toy_tiles"]
    wl = W.make("toy")
    r = O.route_offsets(wl.ids, wl.E)
    xp = O.permute(wl.x(), r["sorted_src"], r["M"], wl.k)
    y_pad, st = O.padded_bmm_forward(xp, r["offsets"], C, wl.w_ug, wl.w_down)
    assert st["rows_multiplied"] == g["rows_multiplied_bmm"]
    assert st["padding_rows"] == g["padding_rows"]
    assert st["dropped_rows"] == 0
    # with no row dropped the padded path reproduces the exact-row grouped result
    y, *_ = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down)
    np.testing.assert_allclose(y_pad, y, rtol=1e-12, atol=1e-12)


def test_capacity_rules_against_page_numbers():
    g = _gold("measured_pages.json")
    f = g["fig38_capacity"]
    C = O.capacity_ceil(f["c"], f["M"], f["n_local"])
    assert C == f["C"] and f["n_local"] * C == f["rows_multiplied"]
    # Eq. 16 by hand: floor(1.25 * 2.5) = 3 -> 8 * ceil(3 / 8) = 8 (one EP rank);
    # two ranks: floor(1.25 * 2.5 / 2) = 1 -> 2 * 8 * ceil(1 / 8) = 16
    assert O.capacity_eq16(1.25, 10, 4, 1) == 8
    assert O.capacity_eq16(1.25, 10, 4, 2) == 16
    # balanced load of 8 rows at 1.25x capacity (10 rows) pads 20% of the scheduled rows
    assert O.rho_pad(np.full(16, 8), 10) == pytest.approx(g["eq16_padding_fraction"]["rho_pad"])
    e = g["eq17_flops"]
    assert round(2 * e["T"] * e["d_in"] * e["d_out"] / 1e12, 2) == e["tflop_rounded"]


def test_roofline_lab_units():
    g = _gold("measured_pages.json")["roofline_lab"]
    for inten, want in g["cases"]:
        assert O.roofline_ceiling(inten, g["bandwidth"], g["peak_gflops"]) == want


# ------------------------------------------------------------------------------ closed forms
def test_flop_convention_and_empty_experts_do_no_work():
    wl = W.custom(T=24, k=2, E=6, d=16, h=24, seed=3, empty_experts=(1, 4))
    r, x, xp, y, u, a, out, macs = _layer(wl)
    assert r["counts"][1] == 0 and r["counts"][4] == 0
    assert 2 * macs == O.flops_fwd(r["M"], wl.d, wl.h) == 6 * r["M"] * wl.d * wl.h
    assert O.flops_fwd_bwd(r["M"], wl.d, wl.h) == 3 * O.flops_fwd(r["M"], wl.d, wl.h)
    dy = W._normal_bf16(np.random.default_rng(1), (wl.n, wl.d))
    _, dw_ug, dw_down, _ = O.expert_backward(dy, xp, u, r["offsets"], wl.w_ug, wl.w_down)
    for e in (1, 4):
        assert not dw_ug[e].any() and not dw_down[e].any()


def test_imbalance_closed_forms():
    assert O.imbalance_IH(np.full(16, 7)) == pytest.approx(0.0, abs=1e-15)
    assert O.imbalance_IH(np.array([100, 0, 0, 0])) == pytest.approx(1.0, abs=1e-15)
    want = 1.0 + (0.75 * math.log(0.75) + 0.25 * math.log(0.25)) / math.log(2)
    assert O.imbalance_IH(np.array([3, 1])) == pytest.approx(want, rel=1e-14)


# ------------------------------------------------------------------------------ brute force
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_route_matches_brute_force_and_invariants(seed):
    wl = W.custom(T=37, k=3, E=5, d=8, h=8, seed=seed, invalid_frac=0.15, empty_experts=(2,))
    r = O.route_offsets(wl.ids, wl.E)
    counts, offsets, placed, inv = brute.route(wl.ids.tolist(), wl.E)
    assert r["counts"].tolist() == counts
    assert r["offsets"].tolist() == offsets
    M = r["M"]
    assert r["sorted_src"][:M].tolist() == placed
    assert (r["sorted_src"][M:] == -1).all()
    assert r["inv_map"].tolist() == inv
    flat = wl.ids.reshape(-1)
    for p in range(M):
        assert r["inv_map"][r["sorted_src"][p]] == p
    for e, (s, t) in enumerate(O.segments(r["offsets"])):
        seg = r["sorted_src"][s:t]
        assert (flat[seg] == e).all()
        assert (np.diff(seg) > 0).all()          # stable: flat-index order inside a segment
    dropped = (flat < 0) | (flat >= wl.E)
    assert (r["inv_map"][dropped] == -1).all()


@pytest.mark.parametrize("name,seed", [("toy", 0), ("custom", 5)])
def test_forward_matches_per_row_brute_force(name, seed):
    if name == "toy":
        wl = W.make("toy")
    else:
        wl = W.custom(T=9, k=2, E=4, d=8, h=16, seed=seed, invalid_frac=0.2, empty_experts=(3,))
    x = wl.x()
    wug, wdn = wl.w_ug_all(), wl.w_down_all()
    want = np.array(brute.layer_forward(x.tolist(), wl.ids.tolist(), wl.weights.tolist(),
                                        wug.tolist(), wdn.tolist(), wl.E))
    *_, out, _ = _layer(wl)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------ special cases
def test_single_expert_is_dense_swiglu_mlp():
    torch = pytest.importorskip("torch")
    wl = W.custom(T=17, k=1, E=1, d=32, h=48, seed=7)
    wl.weights = np.ones_like(wl.weights)
    *_, out, _ = _layer(wl)
    xt = torch.from_numpy(wl.x().astype(np.float64))
    wu = torch.from_numpy(wl.w_ug(0).astype(np.float64))
    wd = torch.from_numpy(wl.w_down(0).astype(np.float64))
    g, v = (xt @ wu.T).split(wl.h, dim=1)
    want = (torch.nn.functional.silu(g) * v) @ wd
    np.testing.assert_allclose(out, want.numpy(), rtol=1e-12, atol=1e-12)


def test_eq17_column_partition_equals_dense_product():
    rng = np.random.default_rng(11)
    T, din, n_exp, width = 13, 24, 4, 10
    X = W.round_to_bf16(rng.standard_normal((T, din)).astype(np.float32)).astype(np.float64)
    Wd = W.round_to_bf16(rng.standard_normal((din, n_exp * width)).astype(np.float32)).astype(np.float64)
    blocks = np.stack([Wd[:, e * width:(e + 1) * width] for e in range(n_exp)])
    x_rep = np.concatenate([X] * n_exp)
    offsets = np.arange(1, n_exp + 1) * T
    y = O.grouped_linear(x_rep, offsets, blocks)
    got = np.concatenate([y[e * T:(e + 1) * T] for e in range(n_exp)], axis=1)
    np.testing.assert_allclose(got, X @ Wd, rtol=1e-13, atol=1e-13)


def _torch_layer_grads(wl, dout):
    torch = pytest.importorskip("torch")
    x = torch.tensor(wl.x(), dtype=torch.float64, requires_grad=True)
    wu = torch.tensor(wl.w_ug_all(), dtype=torch.float64, requires_grad=True)
    wd = torch.tensor(wl.w_down_all(), dtype=torch.float64, requires_grad=True)
    wr = torch.tensor(wl.weights.astype(np.float64), requires_grad=True)
    rows = []
    for t in range(wl.T):
        acc = torch.zeros(wl.d, dtype=torch.float64)
        for j in range(wl.k):
            e = int(wl.ids[t, j])
            if 0 <= e < wl.E:
                g, v = (wu[e] @ x[t]).split(wl.h)
                acc = acc + wr[t, j] * ((torch.nn.functional.silu(g) * v) @ wd[e])
        rows.append(acc)
    out = torch.stack(rows)
    (out * torch.from_numpy(dout.astype(np.float64))).sum().backward()
    dwr = wr.grad.numpy() if wr.grad is not None else np.zeros_like(wl.weights, np.float64)
    return out.detach().numpy(), x.grad.numpy(), wu.grad.numpy(), wd.grad.numpy(), dwr


def _oracle_layer_grads(wl, dout):
    r, x, xp, y, u, a, out, _ = _layer(wl)
    dy = O.permute(dout, r["sorted_src"], r["M"], wl.k, row_scale=wl.weights)
    dxp, dw_ug, dw_down, _ = O.expert_backward(dy, xp, u, r["offsets"], wl.w_ug, wl.w_down)
    dx = O.combine(dxp, r["inv_map"], None, wl.T, wl.k)
    dwr = O.routing_weight_grad(dout, y, r["inv_map"], wl.T, wl.k)
    return out, dx, dw_ug, dw_down, dwr


def test_backward_matches_torch_autograd_fp64():
    wl = W.custom(T=11, k=3, E=5, d=12, h=20, seed=4, invalid_frac=0.1, empty_experts=(0,))
    dout = W._normal_bf16(np.random.default_rng(2), (wl.T, wl.d))
    want = _torch_layer_grads(wl, dout)
    got = _oracle_layer_grads(wl, dout)
    for g_, w_ in zip(got, want):
        np.testing.assert_allclose(g_, w_, rtol=1e-11, atol=1e-11)
    # dropped slots (ids outside [0, E)) carry no gradient
    assert not got[4][(wl.ids < 0) | (wl.ids >= wl.E)].any()


def test_routing_weight_grad_central_differences_on_toy():
    """The layer loss <dOut, out> is linear in each routing weight: a central difference is
    exact up to rounding."""
    wl = W.custom(T=7, k=2, E=3, d=8, h=12, seed=12, invalid_frac=0.15)
    dout = W._normal_bf16(np.random.default_rng(9), (wl.T, wl.d)).astype(np.float64)
    r, x, xp, y, u, a, out, _ = _layer(wl)
    dwr = O.routing_weight_grad(dout, y, r["inv_map"], wl.T, wl.k)

    def loss(w):
        return float((O.combine(y, r["inv_map"], w, wl.T, wl.k) * dout).sum())

    w0 = wl.weights.astype(np.float64)
    for t in range(wl.T):
        for j in range(wl.k):
            plus, minus = w0.copy(), w0.copy()
            plus[t, j] += 0.5
            minus[t, j] -= 0.5
            assert loss(plus) - loss(minus) == pytest.approx(dwr[t, j], rel=1e-12, abs=1e-12)


def test_backward_central_differences_on_toy():
    wl = W.make("toy")
    dout = W._normal_bf16(np.random.default_rng(3), (wl.T, wl.d)).astype(np.float64)
    _, dx, dw_ug, dw_down, _ = _oracle_layer_grads(wl, dout)
    x0, wu0, wd0 = wl.x().astype(np.float64), wl.w_ug_all().astype(np.float64), wl.w_down_all().astype(np.float64)
    r = O.route_offsets(wl.ids, wl.E)

    def loss(x, wu, wd):
        xp = O.permute(x, r["sorted_src"], r["M"], wl.k)
        y, *_ = O.expert_forward(xp, r["offsets"], wu, wd)
        return float((O.combine(y, r["inv_map"], wl.weights, wl.T, wl.k) * dout).sum())

    eps = 1e-6
    rng = np.random.default_rng(0)
    for arr, grad, which in ((x0, dx, 0), (wu0, dw_ug, 1), (wd0, dw_down, 2)):
        for _ in range(4):
            idx = tuple(rng.integers(0, s) for s in arr.shape)
            plus, minus = [a.copy() for a in (x0, wu0, wd0)], [a.copy() for a in (x0, wu0, wd0)]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            fd = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert fd == pytest.approx(grad[idx], rel=1e-6, abs=1e-7)


# ------------------------------------------------------------------------------ invariants
@pytest.mark.parametrize("k", [1, 2, 8])
def test_permute_then_combine_is_k_times_identity(k):
    wl = W.custom(T=33, k=k, E=7, d=24, h=8, seed=k)
    x = wl.x()
    r = O.route_offsets(wl.ids, wl.E)
    xp = O.permute(x, r["sorted_src"], r["M"], k)
    back = O.combine(xp, r["inv_map"], None, wl.T, k)
    assert np.array_equal(back, k * x.astype(np.float64))


def test_combine_equals_scatter_add_reference():
    wl = W.custom(T=29, k=4, E=6, d=16, h=8, seed=9, invalid_frac=0.2)
    r = O.route_offsets(wl.ids, wl.E)
    y = np.random.default_rng(5).standard_normal((wl.n, wl.d))
    got = O.combine(y, r["inv_map"], wl.weights, wl.T, wl.k)
    want = np.zeros((wl.T, wl.d))
    M = r["M"]
    src = r["sorted_src"][:M]
    w = wl.weights.reshape(-1)[src]
    np.add.at(want, src // wl.k, w[:, None] * y[:M])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)


def test_results_invariant_to_expert_relabelling():
    wl = W.custom(T=21, k=2, E=5, d=8, h=12, seed=6, invalid_frac=0.1, empty_experts=(2,))
    dout = W._normal_bf16(np.random.default_rng(8), (wl.T, wl.d))
    out, dx, dw_ug, dw_down, dwr = _oracle_layer_grads(wl, dout)
    pi = np.array([3, 0, 4, 1, 2])
    wu, wd = wl.w_ug_all(), wl.w_down_all()
    wl2 = W.custom(T=21, k=2, E=5, d=8, h=12, seed=6, invalid_frac=0.1, empty_experts=(2,))
    valid = (wl.ids >= 0) & (wl.ids < wl.E)
    wl2.ids = np.where(valid, pi[np.clip(wl.ids, 0, wl.E - 1)], wl.ids).astype(np.int32)
    inv_pi = np.argsort(pi)
    wl2.w_ug = lambda e: wu[inv_pi[e]]
    wl2.w_down = lambda e: wd[inv_pi[e]]
    wl2.w_ug_all = lambda: wu[inv_pi]
    wl2.w_down_all = lambda: wd[inv_pi]
    out2, dx2, dw_ug2, dw_down2, dwr2 = _oracle_layer_grads(wl2, dout)
    assert np.array_equal(out, out2) and np.array_equal(dx, dx2) and np.array_equal(dwr, dwr2)
    assert np.array_equal(dw_ug2, dw_ug[inv_pi]) and np.array_equal(dw_down2, dw_down[inv_pi])


def test_padded_bmm_drops_rows_beyond_capacity():
    wl = W.custom(T=20, k=1, E=3, d=8, h=8, seed=12)
    r = O.route_offsets(wl.ids, wl.E)
    xp = O.permute(wl.x(), r["sorted_src"], r["M"], wl.k)
    y, *_ = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down)
    C = 4
    yb, st = O.padded_bmm_forward(xp, r["offsets"], C, wl.w_ug, wl.w_down)
    for e, (s, t) in enumerate(O.segments(r["offsets"])):
        np.testing.assert_allclose(yb[s:s + min(C, t - s)], y[s:s + min(C, t - s)], rtol=1e-12, atol=1e-12)
        assert not yb[s + C:t].any()
    assert st["dropped_rows"] == int(np.maximum(r["counts"] - C, 0).sum())


# ------------------------------------------------------------------------------ planted mistakes
def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle and check a pin above catches each one."""
    wl = W.custom(T=9, k=2, E=4, d=8, h=16, seed=5, invalid_frac=0.2, empty_experts=(3,))
    x, wug, wdn = wl.x(), wl.w_ug_all(), wl.w_down_all()
    want = np.array(brute.layer_forward(x.tolist(), wl.ids.tolist(), wl.weights.tolist(),
                                        wug.tolist(), wdn.tolist(), wl.E))
    good = O.swiglu
    monkeypatch.setattr(O, "swiglu", lambda u, h: O.silu(u[:, h:]) * u[:, :h])   # gate/up swapped
    *_, out, _ = _layer(wl)
    assert not np.allclose(out, want, rtol=1e-6)
    monkeypatch.setattr(O, "swiglu", good)
    real_combine = O.combine
    monkeypatch.setattr(O, "combine", lambda y, inv, w, T, k: real_combine(y, inv, None, T, k))  # weights dropped
    *_, out, _ = _layer(wl)
    assert not np.allclose(out, want, rtol=1e-6)
    monkeypatch.setattr(O, "combine", real_combine)
    # routing-weight gradient taken against the weighted output, or against the wrong slot
    dout = W._normal_bf16(np.random.default_rng(4), (wl.T, wl.d))
    want_dwr = _torch_layer_grads(wl, dout)[4]
    real_rwg = O.routing_weight_grad
    w2 = wl.weights.astype(np.float64)
    for bad in (lambda do, y, inv, T, k: real_rwg(do, y, inv, T, k) * w2,
                lambda do, y, inv, T, k: real_rwg(do, y, np.roll(np.asarray(inv).reshape(T, k), 1, axis=1), T, k)):
        monkeypatch.setattr(O, "routing_weight_grad", bad)
        assert not np.allclose(_oracle_layer_grads(wl, dout)[4], want_dwr, rtol=1e-6)
