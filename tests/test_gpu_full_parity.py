"""Full-size parity of the benchmarked workload, and invariance of every result to the order of
the expert groups.

The large workload (T = 16384 tokens, E = 256 experts, top-8, d = 2048, h = 512) runs through
the public layer (route -> permute -> grouped forward with the routing weights -> combine, then
the backward), and through the benchmark's own sequence of single-kernel calls, which must give
the same bits. Every routed row of the saved SwiGLU output, the expert output and the
input-row gradient, every expert's two weight gradients and every token's output, input
gradient and routing-weight gradient are compared with the oracle at the task tolerance. The
oracle runs expert chunk by expert chunk: a chunk is the sub-problem made of the chunk's
experts and their (contiguous) row segments, which is the plain definition restricted to those
experts.

"Grouped expert GEMM: schedule irregular rows without changing the experts" asks that output
and gradient agreement be checked after reordering the groups. Relabelling the experts with a
permutation (ids and weight slices together) must leave the layer's outputs bit-identical and
permute its weight gradients exactly: a segment keeps its rows in flat-index order whatever
its expert's index, tiles start at segment starts, and every sum runs in a fixed order.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import workloads as W
from ragged_grouped_gemm_device_gb300.layer import ExpertLayer

pytestmark = pytest.mark.gpu

CHUNK_EXPERTS = 32


def _rows_f32(t: torch.Tensor, M: int) -> np.ndarray:
    return t[:M].float().cpu().numpy()


def _bench_step_matches_layer(wl, w_ug, w_down, layer, out, dx, dw_ug, dw_down, dwr):
    """The benchmark times the step as one C-ABI call per kernel (`bench.TrainingStep`); the layer
    runs the composite forward and backward. On the same inputs every result of the timed calls
    equals the layer's bit for bit, so the parity below holds for the benchmarked sequence too."""
    import bench
    from ragged_grouped_gemm_device_gb300 import _lib as L
    step = bench.TrainingStep(L, wl.T, wl.k, wl.E, wl.d, wl.h, w_ug, w_down, w_ug.device)
    for _, _, fn in step.calls(G.dev_bf16(wl.x()), G.dev_i32(wl.ids), G.dev_f32(wl.weights),
                               G.dev_bf16(wl.dout())):
        fn()
    torch.cuda.synchronize()
    assert step.status.item() == 0
    M = int(layer.offsets[-1].item())
    assert torch.equal(step.offsets, layer.offsets) and torch.equal(step.inv_map, layer.inv_map[: wl.n])
    assert torch.equal(step.sorted_src[:M], layer.sorted_src[:M])
    for got, want, what in ((step.a[:M], layer.a[:M], "a"), (step.y[:M], layer.y[:M], "y"),
                            (step.dxp[:M], layer.dxp[:M], "dxp"), (step.out, out, "out"), (step.dx, dx, "dx"),
                            (step.dw_ug, dw_ug, "dW_ug"), (step.dw_down, dw_down, "dW_down"),
                            (step.dw_route, dwr, "d_weights")):
        assert torch.equal(got, want), what
    del step
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_large_workload_full_parity(lib):
    wl = W.make("large")
    T, k, E, d, h = wl.T, wl.k, wl.E, wl.d, wl.h
    w_ug, w_down = G.device_weights(wl)
    layer = ExpertLayer(w_ug, w_down)
    doutn = wl.dout()
    out = layer.forward(G.dev_bf16(wl.x()), G.dev_i32(wl.ids), G.dev_f32(wl.weights))
    dx, dw_ug, dw_down, dwr = layer.backward(G.dev_bf16(doutn))
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    _bench_step_matches_layer(wl, w_ug, w_down, layer, out, dx, dw_ug, dw_down, dwr)

    r = O.route_offsets(wl.ids, E)
    M = r["M"]
    assert np.array_equal(layer.offsets.cpu().numpy(), r["offsets"])
    assert np.array_equal(layer.sorted_src[:M].cpu().numpy(), r["sorted_src"][:M])
    assert np.array_equal(layer.inv_map[: wl.n].cpu().numpy(), r["inv_map"])
    x = wl.x()
    w_row = wl.weights.reshape(-1).astype(np.float64)[r["sorted_src"][:M]]  # routing weight of row p

    got_a, got_y, got_dxp = _rows_f32(layer.a, M), _rows_f32(layer.y, M), _rows_f32(layer.dxp, M)
    got_ug, got_dn = dw_ug.cpu().numpy(), dw_down.cpu().numpy()
    y_ref = np.zeros((M, d))          # unweighted expert output of every row (for the combine)
    dxp_ref = np.zeros((M, d))
    segs = O.segments(r["offsets"])
    for c0 in range(0, E, CHUNK_EXPERTS):
        ex = list(range(c0, min(E, c0 + CHUNK_EXPERTS)))
        s0, s1 = segs[ex[0]][0], segs[ex[-1]][1]
        if s1 == s0:
            continue
        off_c = r["offsets"][ex].astype(np.int64) - s0
        wu = lambda i, ex=ex: wl.w_ug(ex[i])
        wd = lambda i, ex=ex: wl.w_down(ex[i])
        src_c = r["sorted_src"][s0:s1]
        xp_c = O.permute(x, src_c, s1 - s0, k)
        dy_c = O.permute(doutn, src_c, s1 - s0, k, row_scale=wl.weights)
        y_c, u_c, a_c, _ = O.expert_forward(xp_c, off_c, wu, wd)
        dxp_c, dwu_c, dwd_c, _ = O.expert_backward(dy_c, xp_c, u_c, off_c, wu, wd)
        wr = w_row[s0:s1, None]
        # the layer folds the routing weight into the SwiGLU output: a_save = w*A, y = (w*A) W_down
        G.assert_close(got_a[s0:s1], wr * a_c, f"A rows {s0}:{s1}")
        G.assert_close(got_y[s0:s1], wr * y_c, f"y rows {s0}:{s1}")
        G.assert_close(got_dxp[s0:s1], dxp_c, f"dxp rows {s0}:{s1}")
        nz = [i for i, e in enumerate(ex) if segs[e][1] > segs[e][0]]
        z = [i for i, e in enumerate(ex) if segs[e][1] == segs[e][0]]
        G.assert_close(got_ug[ex][nz], dwu_c[nz], f"dW_ug experts {ex[0]}..{ex[-1]}")
        G.assert_close(got_dn[ex][nz], dwd_c[nz], f"dW_down experts {ex[0]}..{ex[-1]}")
        assert not got_ug[ex][z].any() and not got_dn[ex][z].any()
        y_ref[s0:s1], dxp_ref[s0:s1] = y_c, dxp_c
    del got_a, got_y, got_dxp, got_ug, got_dn

    inv = r["inv_map"]
    G.assert_close(G.host(out), O.combine(y_ref, inv, wl.weights, T, k), "out (every token)")
    G.assert_close(G.host(dx), O.combine(dxp_ref, inv, None, T, k), "dx (every token)")
    G.assert_close(G.host(dwr), O.routing_weight_grad(doutn, y_ref, inv, T, k), "d_weights (every slot)")


def _layer_run(wl, ids, w_ug, w_down):
    layer = ExpertLayer(w_ug, w_down)
    out = layer.forward(G.dev_bf16(wl.x()), G.dev_i32(ids), G.dev_f32(wl.weights)).clone()
    grads = [g.clone() for g in layer.backward(G.dev_bf16(wl.dout()))]
    torch.cuda.synchronize()
    assert layer.status.item() == 0
    return [out] + grads


@pytest.mark.parametrize("case", ["ragged", "finegrained"])
def test_results_invariant_to_expert_order(lib, case):
    if case == "ragged":
        # several row tiles per expert with ragged tails, empty experts and dropped ids
        wl = W.custom(T=900, k=4, E=13, d=136, h=200, seed=51, invalid_frac=0.05, empty_experts=(2, 9))
    else:
        wl = W.make("finegrained")
    E = wl.E
    pi = np.random.default_rng(52).permutation(E)       # expert e is relabelled pi[e]
    ids = wl.ids.astype(np.int64)
    valid = (ids >= 0) & (ids < E)
    ids_p = np.where(valid, pi[np.clip(ids, 0, E - 1)], ids).astype(np.int32)
    w_ug, w_down = G.device_weights(wl)
    order = torch.from_numpy(np.argsort(pi)).cuda()      # slot pi[e] holds expert e's weights
    w_ug_p, w_down_p = w_ug[order].contiguous(), w_down[order].contiguous()

    base = _layer_run(wl, wl.ids, w_ug, w_down)
    perm = _layer_run(wl, ids_p, w_ug_p, w_down_p)
    out0, dx0, dwu0, dwd0, dwr0 = base
    out1, dx1, dwu1, dwd1, dwr1 = perm
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
    assert torch.equal(bits(out1), bits(out0))
    assert torch.equal(bits(dx1), bits(dx0))
    assert torch.equal(bits(dwr1), bits(dwr0))
    pit = torch.from_numpy(pi).cuda()
    assert torch.equal(bits(dwu1[pit]), bits(dwu0))
    assert torch.equal(bits(dwd1[pit]), bits(dwd0))

    # and the relabelled run agrees with the oracle on the relabelled problem
    r = O.route_offsets(ids_p, E)
    wu_p = lambda e: wl.w_ug(int(np.argsort(pi)[e]))
    wd_p = lambda e: wl.w_down(int(np.argsort(pi)[e]))
    xp = O.permute(wl.x(), r["sorted_src"], r["M"], wl.k)
    y, u, _, _ = O.expert_forward(xp, r["offsets"], wu_p, wd_p)
    G.assert_close(G.host(out1), O.combine(y, r["inv_map"], wl.weights, wl.T, wl.k), f"out[{case}, relabelled]")
