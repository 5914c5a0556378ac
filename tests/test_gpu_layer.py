"""The whole expert layer through the public Python layer (route -> permute -> grouped forward ->
combine, then the backward), checked end to end against the oracle pipeline."""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import workloads as W
from ragged_grouped_gemm_device_gb300.layer import ExpertLayer

pytestmark = pytest.mark.gpu


def _oracle_layer(wl, dout):
    r = O.route_offsets(wl.ids, wl.E)
    xp = O.permute(wl.x(), r["sorted_src"], r["M"], wl.k)
    y, u, a, _ = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down)
    out = O.combine(y, r["inv_map"], wl.weights, wl.T, wl.k)
    dy = O.permute(dout, r["sorted_src"], r["M"], wl.k, row_scale=wl.weights)
    dxp, dw_ug, dw_down, _ = O.expert_backward(dy, xp, u, r["offsets"], wl.w_ug, wl.w_down)
    dx = O.combine(dxp, r["inv_map"], None, wl.T, wl.k)
    dwr = O.routing_weight_grad(dout, y, r["inv_map"], wl.T, wl.k)
    return out, dx, dw_ug, dw_down, dwr


@pytest.mark.parametrize("name", ["toy", "edge", "edge_odd_width", "edge_top32", "finegrained"])
def test_layer_forward_backward(lib, name):
    if name == "edge":
        wl = W.custom(T=211, k=4, E=11, d=72, h=40, seed=21, invalid_frac=0.1, empty_experts=(2, 7))
    elif name == "edge_odd_width":
        wl = W.custom(T=120, k=3, E=5, d=60, h=37, seed=22, invalid_frac=0.05, empty_experts=(3,))
    elif name == "edge_top32":
        # the largest top_k: 32 slots per token, combined and routing-weight gradients of 32 slots
        wl = W.custom(T=96, k=32, E=40, d=64, h=64, seed=23, invalid_frac=0.05, empty_experts=(5,))
    else:
        wl = W.make(name)
    w_ug, w_down = G.device_weights(wl)
    layer = ExpertLayer(w_ug, w_down)
    doutn = wl.dout()
    out = layer.forward(G.dev_bf16(wl.x()), G.dev_i32(wl.ids), G.dev_f32(wl.weights))
    dx, dw_ug, dw_down, dwr = layer.backward(G.dev_bf16(doutn))
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    o_out, o_dx, o_ug, o_dn, o_dwr = _oracle_layer(wl, doutn)
    G.assert_close(G.host(dwr), o_dwr, f"d_weights[{name}]")
    dropped = (wl.ids < 0) | (wl.ids >= wl.E)
    assert not G.host(dwr)[dropped].any()
    G.assert_close(G.host(out), o_out, f"out[{name}]")
    G.assert_close(G.host(dx), o_dx, f"dx[{name}]")
    nz = np.bincount(wl.ids[(wl.ids >= 0) & (wl.ids < wl.E)], minlength=wl.E) > 0
    G.assert_close(G.host(dw_ug)[nz], o_ug[nz], f"dW_ug[{name}]")
    G.assert_close(G.host(dw_down)[nz], o_dn[nz], f"dW_down[{name}]")


@pytest.mark.slow
def test_large_layer_sampled_tokens(lib):
    """Full-size large workload through the layer; the oracle recomputes a sample of tokens (a
    token's output and input gradient depend only on its own row and its experts)."""
    wl = W.make("large")
    w_ug, w_down = G.device_weights(wl)
    layer = ExpertLayer(w_ug, w_down)
    doutn = wl.dout()
    out = layer.forward(G.dev_bf16(wl.x()), G.dev_i32(wl.ids), G.dev_f32(wl.weights))
    dx, _, _, dwr = layer.backward(G.dev_bf16(doutn))
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    toks = np.sort(np.random.default_rng(3).choice(wl.T, size=48, replace=False))
    sub = W.Workload("large_sub", T=toks.size, k=wl.k, E=wl.E, d=wl.d, h=wl.h, seed=wl.seed)
    sub.ids, sub.weights = wl.ids[toks], wl.weights[toks]
    xs, ds = wl.x()[toks], doutn[toks]
    sub.x = lambda: xs
    sub.w_ug, sub.w_down = wl.w_ug, wl.w_down
    o_out, o_dx, _, _, o_dwr = _oracle_layer(sub, ds)
    G.assert_close(G.host(out)[toks], o_out, "out[large]")
    G.assert_close(G.host(dx)[toks], o_dx, "dx[large]")
    G.assert_close(G.host(dwr)[toks], o_dwr, "d_weights[large]")


def test_layer_is_deterministic(lib):
    """Stable placement, the atomic-free combine and fixed-slot partial sums make every output of
    the layer bit-identical from one run to the next."""
    wl = W.custom(T=700, k=4, E=24, d=256, h=192, seed=23, invalid_frac=0.05, empty_experts=(5,))
    w_ug, w_down = G.device_weights(wl)
    x, ids, wts, dout = G.dev_bf16(wl.x()), G.dev_i32(wl.ids), G.dev_f32(wl.weights), G.dev_bf16(wl.dout())
    runs = []
    for _ in range(2):
        layer = ExpertLayer(w_ug, w_down)
        out = layer.forward(x, ids, wts).clone()
        grads = [g.clone() for g in layer.backward(dout)]
        torch.cuda.synchronize()
        assert layer.status.item() == 0
        runs.append([out] + grads)
    for a, b in zip(*runs):
        assert torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.uint8) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def test_zero_stride_upstream_gradient(lib):
    """A scalar loss broadcasts its gradient back as an expanded [T, d] view with strides (0, 0)
    ("Grouped expert GEMM": zero-stride gradients from .sum() reach the grouped GEMM's backward).
    The layer takes it and gives the same bits as for the dense tensor of the same values; a
    transposed (non-contiguous) input x likewise."""
    wl = W.custom(T=96, k=2, E=5, d=128, h=64, seed=31, empty_experts=(1,))
    w_ug, w_down = G.device_weights(wl)
    ids, w = G.dev_i32(wl.ids), G.dev_f32(wl.weights)
    x = G.dev_bf16(wl.x())
    results = []
    for variant in ("dense", "strided"):
        layer = ExpertLayer(w_ug, w_down)
        xin = x if variant == "dense" else x.t().contiguous().t()  # same values, column-major
        assert variant == "dense" or not xin.is_contiguous()
        out = layer.forward(xin, ids, w).clone()
        g = torch.full((), 0.75, dtype=torch.bfloat16, device="cuda").expand(wl.T, wl.d)
        assert g.stride() == (0, 0)
        dout = g.contiguous() if variant == "dense" else g
        res = [t.clone() for t in layer.backward(dout)]
        torch.cuda.synchronize()
        assert layer.status.item() == 0
        results.append([out] + res)
    for a, b in zip(*results):
        assert torch.equal(a, b)
    # and the values are the oracle's for that constant gradient
    doutn = np.full((wl.T, wl.d), 0.75, np.float32)
    o_out, o_dx, o_ug, o_dn, o_dwr = _oracle_layer(wl, doutn)
    out, dx, dw_ug, dw_down, dwr = results[1]
    G.assert_close(G.host(out), o_out, "out[zero-stride]")
    G.assert_close(G.host(dx), o_dx, "dx[zero-stride]")
    G.assert_close(G.host(dwr), o_dwr, "d_weights[zero-stride]")
    nz = np.bincount(wl.ids.ravel(), minlength=wl.E) > 0
    G.assert_close(G.host(dw_ug)[nz], o_ug[nz], "dW_ug[zero-stride]")
    G.assert_close(G.host(dw_down)[nz], o_dn[nz], "dW_down[zero-stride]")
