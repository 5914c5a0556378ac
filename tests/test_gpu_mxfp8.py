"""GPU parity of the MXFP8 variant ("Section 09: Grouped GEMM", §9.5: scaled grouped GEMMs for
the forward and the Dgrad, BF16 Wgrad) against the MXFP8 oracle (oracle/mx_oracle.py).

Quantized codes and scales are integers decided from bf16 inputs, so they are compared bit for
bit (activations through moe_mx_quantize_rows, weights through moe_mx_prepare_weights in all
four orientations). The layer's float results use the task tolerance against the oracle's
MXFP8 layer, which quantizes the same bf16 values: the only differences left are fp32
accumulation and the rare quantization decisions that the GPU's fp32 SwiGLU output and the
oracle's fp64 one take on opposite sides of a rounding boundary.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from oracle import mx_oracle as X
from ragged_grouped_gemm_device_gb300 import _lib as L
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    "toy": lambda: W.make("toy"),                      # d = 64: half of one 128-element chunk
    # ragged tiles, empty experts, dropped ids, d = 96 (three 32-blocks in the last chunk)
    "edge": lambda: W.custom(T=300, k=3, E=9, d=96, h=256, seed=61, invalid_frac=0.05, empty_experts=(0, 4)),
    # several 128-row tiles per expert with tails
    "edge_tiles": lambda: W.custom(T=700, k=2, E=5, d=160, h=384, seed=62),
    "finegrained": lambda: W.make("finegrained"),
}


def _round256(n):
    return (n + 255) // 256 * 256


def _ntp(N):
    return 2 * (((N + 127) // 128 + 1) // 2)


def _kc(K):
    return (K + 127) // 128


def _atom_index(G, r, b, K):
    """Byte of the scale of row r (0..127) of tile G, 32-block b, in the atom layout."""
    return (G * _kc(K) + b // 4) * 512 + (r % 32) * 16 + (r // 32) * 4 + b % 4


def _activation_scales(sf, offsets, M, K):
    """[M, K/32] scale codes of rows p < M from the problem list's tile atoms."""
    offs = np.asarray(offsets, np.int64)
    starts = np.concatenate([[0], offs[:-1]])
    tile0 = np.concatenate([[0], np.cumsum((offs - starts + 127) // 128)[:-1]])
    p = np.arange(M)
    e = np.searchsorted(offs, p, side="right")
    rr = p - starts[e]
    Gt = tile0[e] + rr // 128
    b = np.arange(K // 32)
    idx = _atom_index(Gt[:, None], (rr % 128)[:, None], b[None, :], K)
    return sf[idx]


def _weight_scales(sf, E, N, K):
    """[E, N, K/32] scale codes of a weight's codes [E, N, K]."""
    e = np.arange(E)[:, None, None]
    n = np.arange(N)[None, :, None]
    b = np.arange(K // 32)[None, None, :]
    return sf[_atom_index(e * _ntp(N) + n // 128, n % 128, b, K)]


def _prepared(wl):
    w_ug, w_down = G.device_weights(wl)
    E, d, h = wl.E, wl.d, wl.h
    nb = L.moe_workspace_bytes(L.OP_MX_WEIGHTS, 0, 1, E, d, h)
    assert nb > 0
    mxw = torch.empty(nb, dtype=torch.uint8, device="cuda")
    L.moe_mx_prepare_weights(w_ug, w_down, E, d, h, mxw)
    return mxw


def _weight_parts(mxw, E, d, h):
    """(codes, scales) of the four prepared orientations, as the header lays them out."""
    host = mxw.cpu().numpy()
    parts, off = [], 0
    for N, K in ((2 * h, d), (d, h), (h, d), (d, 2 * h)):
        qb = _round256(E * N * K)
        sb = _round256(E * _ntp(N) * _kc(K) * 512)
        parts.append((host[off:off + E * N * K].reshape(E, N, K), host[off + qb:off + qb + sb]))
        off += qb + sb
    return parts


@pytest.mark.parametrize("name", ["toy", "edge", "finegrained"])
def test_mx_quantize_rows_bit_exact(lib, name):
    wl = CASES[name]()
    run = G.DevicePipeline(wl, with_u=False).route().permute()
    torch.cuda.synchronize()
    r = O.route_offsets(wl.ids, wl.E)
    M, n, d = r["M"], wl.n, wl.d
    q = torch.full((n, d), 0xEE, dtype=torch.uint8, device="cuda")
    sf = torch.full((L.moe_workspace_bytes(L.OP_MX_ROW_SCALES, wl.T, wl.k, wl.E, d, 128),), 0xEE,
                    dtype=torch.uint8, device="cuda")
    L.moe_mx_quantize_rows(run.xp, run.offsets, wl.E, n, d, q, sf, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    xp = O.permute(wl.x(), r["sorted_src"], M, wl.k)
    codes, exp = X.mx_quantize(xp[:M])
    got_q = q.cpu().numpy()
    assert np.array_equal(got_q[:M], codes)
    assert (got_q[M:] == 0xEE).all()                      # rows past M untouched
    got_s = _activation_scales(sf.cpu().numpy(), r["offsets"], M, d)
    assert np.array_equal(got_s.astype(np.int64), exp + 127)
    if (d // 32) % 4:                                     # scales past K in the last chunk: 2^0
        tail = _activation_scales(sf.cpu().numpy(), r["offsets"], M, _kc(d) * 128)[:, d // 32:]
        assert (tail == 127).all()


@pytest.mark.parametrize("name", ["toy", "edge", "edge_tiles"])
def test_mx_prepare_weights_bit_exact(lib, name):
    wl = CASES[name]()
    E, d, h = wl.E, wl.d, wl.h
    mxw = _prepared(wl)
    torch.cuda.synchronize()
    wug = np.stack([wl.w_ug(e) for e in range(E)]).astype(np.float64)
    wdn = np.stack([wl.w_down(e) for e in range(E)]).astype(np.float64)
    refs = [wug, np.transpose(wdn, (0, 2, 1)), wdn, np.transpose(wug, (0, 2, 1))]
    for (q, sf), ref in zip(_weight_parts(mxw, E, d, h), refs):
        codes, exp = X.mx_quantize(ref)
        assert np.array_equal(q, codes)
        N, K = ref.shape[1], ref.shape[2]
        assert np.array_equal(_weight_scales(sf, E, N, K).astype(np.int64), exp + 127)


def _mx_run(wl, backward):
    """The MXFP8 layer on device: route, permute, scaled forward (routing weights folded), and
    optionally the backward from the plain gather of dOut."""
    run = G.DevicePipeline(wl).route().permute()
    E, d, h, n = wl.E, wl.d, wl.h, wl.n
    mxw = _prepared(wl)
    ws = torch.empty(L.moe_workspace_bytes(L.OP_MX_FWD, wl.T, wl.k, E, d, h), dtype=torch.uint8, device="cuda")
    L.moe_grouped_swiglu_fwd_mxfp8(run.xp, run.offsets, run.sorted_src, run.weights, E, n, d, h, mxw, run.y,
                                   run.a, run.saved, ws, run.status)
    out = {}
    if backward:
        dout = wl.dout()
        dy = G.nan_filled((n, d))
        L.moe_permute(G.dev_bf16(dout), run.sorted_src, run.offsets, None, wl.T, wl.k, E, d, dy)
        dxp = G.nan_filled((n, d))
        dwu = torch.full((E, 2 * h, d), float("nan"), device="cuda")
        dwd = torch.full((E, h, d), float("nan"), device="cuda")
        dwr = torch.full((n,), float("nan"), device="cuda")
        bws = torch.empty(L.moe_workspace_bytes(L.OP_MX_BWD, wl.T, wl.k, E, d, h), dtype=torch.uint8, device="cuda")
        L.moe_grouped_bwd_mxfp8(dy, run.xp, run.a, run.saved, run.offsets, run.sorted_src, run.weights, E, n, d, h,
                                mxw, dxp, dwu, dwd, bws, run.status, inv_map=run.inv_map, dw_route=dwr)
        out.update(dout=dout, dxp=dxp, dwu=dwu, dwd=dwd, dwr=dwr)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    return run, out


def _oracle(wl, backward, dout=None, experts=None):
    r = O.route_offsets(wl.ids, wl.E)
    M = r["M"]
    xp = O.permute(wl.x(), r["sorted_src"], M, wl.k)
    w_row = np.zeros(wl.n)
    w_row[:M] = wl.weights.reshape(-1)[r["sorted_src"][:M]]
    y, u, p = X.mx_expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down, w_row, experts)
    res = dict(r=r, y=y, u=u, p=p)
    if backward:
        dy = O.permute(dout, r["sorted_src"], M, wl.k)
        res.update(zip(("dxp", "dwu", "dwd", "du", "g_dot"),
                       X.mx_expert_backward(dy, xp, u, p, r["offsets"], wl.w_ug, wl.w_down, w_row, experts)))
    return res


@pytest.mark.parametrize("name", list(CASES))
def test_mx_forward_backward_match_oracle(lib, name):
    wl = CASES[name]()
    run, g = _mx_run(wl, backward=True)
    o = _oracle(wl, True, g["dout"])
    M = o["r"]["M"]
    G.assert_close(G.host(run.a)[:M], o["p"][:M], f"P[{name}]")
    G.assert_close(G.host(run.u)[:M], o["u"][:M], f"U[{name}]")
    G.assert_close(G.host(run.y)[:M], o["y"][:M], f"y[{name}]")
    assert np.isnan(G.host(run.y)[M:]).all()
    G.assert_close(G.host(g["dxp"])[:M], o["dxp"][:M], f"dxp[{name}]")
    nz = o["r"]["counts"] > 0
    G.assert_close(G.host(g["dwu"])[nz], o["dwu"][nz], f"dW_ug[{name}]")
    G.assert_close(G.host(g["dwd"])[nz], o["dwd"][nz], f"dW_down[{name}]")
    assert not G.host(g["dwu"])[~nz].any() and not G.host(g["dwd"])[~nz].any()
    inv = o["r"]["inv_map"]
    dwr_ref = np.where(inv >= 0, o["g_dot"][np.maximum(inv, 0)], 0.0)
    G.assert_close(G.host(g["dwr"]), dwr_ref, f"d_weights[{name}]")


def test_mx_forward_is_closer_to_mx_oracle_than_to_bf16_oracle(lib):
    """The scaled path really computes with MXFP8 operands: against the unquantized fp64 forward
    its error is the quantization's (percent level), against the MXFP8 oracle the fp32 one."""
    wl = CASES["edge_tiles"]()
    run, _ = _mx_run(wl, backward=False)
    o = _oracle(wl, False)
    M = o["r"]["M"]
    xp = O.permute(wl.x(), o["r"]["sorted_src"], M, wl.k)
    y0, _, _, _ = O.expert_forward(xp, o["r"]["offsets"], wl.w_ug, wl.w_down)
    w_row = wl.weights.reshape(-1)[o["r"]["sorted_src"][:M]].astype(np.float64)
    got = G.host(run.y)[:M]
    e_mx = np.linalg.norm(got - o["y"][:M]) / np.linalg.norm(o["y"][:M])
    e_bf = np.linalg.norm(got - w_row[:, None] * y0[:M]) / np.linalg.norm(w_row[:, None] * y0[:M])
    assert e_mx < 5e-3 < e_bf


@pytest.mark.slow
def test_mx_large_sampled_experts(lib):
    wl = W.make("large")
    run, g = _mx_run(wl, backward=True)
    r = O.route_offsets(wl.ids, wl.E)
    experts = G.sample_experts(r["counts"], n_pick=6)
    o = _oracle(wl, True, g["dout"], experts)
    rows = G.rows_of(r["offsets"], experts)
    G.assert_close(G.host(run.a)[rows], o["p"][rows], "P[large]")
    G.assert_close(G.host(run.y)[rows], o["y"][rows], "y[large]")
    G.assert_close(G.host(g["dxp"])[rows], o["dxp"][rows], "dxp[large]")
    G.assert_close(G.host(g["dwu"][experts]), o["dwu"][experts], "dW_ug[large]")
    G.assert_close(G.host(g["dwd"][experts]), o["dwd"][experts], "dW_down[large]")


@pytest.mark.parametrize("name", ["toy", "edge", "finegrained"])
def test_mx_permute_equals_permute_then_quantize(lib, name):
    """The gather fused with the quantization writes the same bytes as the gather followed by
    the standalone quantizer: bf16 rows, codes and every scale atom byte."""
    wl = CASES[name]()
    run = G.DevicePipeline(wl, with_u=False).route().permute()
    n, d, E = wl.n, wl.d, wl.E
    sfb = L.moe_workspace_bytes(L.OP_MX_ROW_SCALES, wl.T, wl.k, E, d, 128)
    q1 = torch.full((n, d), 0xEE, dtype=torch.uint8, device="cuda")
    sf1 = torch.full((sfb,), 0xEE, dtype=torch.uint8, device="cuda")
    L.moe_mx_quantize_rows(run.xp, run.offsets, E, n, d, q1, sf1, run.status)
    xp2 = G.nan_filled((n, d))
    q2, sf2 = torch.full_like(q1, 0xEE), torch.full_like(sf1, 0xEE)
    L.moe_permute_mxfp8(run.x, run.sorted_src, run.offsets, wl.T, wl.k, E, d, xp2, q2, sf2, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    M = int(run.offsets[-1].item())
    assert torch.equal(xp2[:M].view(torch.int16), run.xp[:M].view(torch.int16))
    assert torch.equal(q2, q1) and torch.equal(sf2, sf1)


def test_mx_layer_with_fused_gathers_is_bit_identical(lib):
    """The scaled forward fed with the codes of moe_permute_mxfp8, and the scaled backward fed
    with the codes of the dOut gather, give exactly what the calls that quantize internally give."""
    wl = CASES["edge_tiles"]()
    run, g = _mx_run(wl, backward=True)
    E, d, h, n, T, k = wl.E, wl.d, wl.h, wl.n, wl.T, wl.k
    mxw = _prepared(wl)
    sfb = L.moe_workspace_bytes(L.OP_MX_ROW_SCALES, T, k, E, d, h)
    xq = torch.empty(n, d, dtype=torch.uint8, device="cuda")
    xsf = torch.empty(sfb, dtype=torch.uint8, device="cuda")
    L.moe_permute_mxfp8(run.x, run.sorted_src, run.offsets, T, k, E, d, None, xq, xsf, run.status)
    y2, a2 = G.nan_filled((n, d)), G.nan_filled((n, h))
    sv2 = torch.full_like(run.saved, float("nan"))
    ws = torch.empty(L.moe_workspace_bytes(L.OP_MX_FWD, T, k, E, d, h), dtype=torch.uint8, device="cuda")
    L.moe_grouped_swiglu_fwd_mxfp8(None, run.offsets, run.sorted_src, run.weights, E, n, d, h, mxw, y2, a2, sv2, ws,
                                   run.status, xq=xq, xsf=xsf)
    dy = G.nan_filled((n, d))
    dyq = torch.empty(n, d, dtype=torch.uint8, device="cuda")
    dysf = torch.empty(sfb, dtype=torch.uint8, device="cuda")
    L.moe_permute_mxfp8(G.dev_bf16(g["dout"]), run.sorted_src, run.offsets, T, k, E, d, dy, dyq, dysf, run.status)
    dxp2 = G.nan_filled((n, d))
    dwu2, dwd2 = torch.empty_like(g["dwu"]), torch.empty_like(g["dwd"])
    dwr2 = torch.full_like(g["dwr"], float("nan"))
    bws = torch.empty(L.moe_workspace_bytes(L.OP_MX_BWD, T, k, E, d, h), dtype=torch.uint8, device="cuda")
    L.moe_grouped_bwd_mxfp8(dy, run.xp, a2, sv2, run.offsets, run.sorted_src, run.weights, E, n, d, h, mxw, dxp2,
                            dwu2, dwd2, bws, run.status, inv_map=run.inv_map, dw_route=dwr2, dyq=dyq, dysf=dysf)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    M = int(run.offsets[-1].item())
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)
    assert torch.equal(bits(y2[:M]), bits(run.y[:M])) and torch.equal(bits(a2[:M]), bits(run.a[:M]))
    assert torch.equal(bits(dxp2[:M]), bits(g["dxp"][:M]))
    assert torch.equal(bits(dwu2), bits(g["dwu"])) and torch.equal(bits(dwd2), bits(g["dwd"]))
    assert torch.equal(bits(dwr2), bits(g["dwr"]))


def test_mx_edge_problem_lists(lib):
    """The largest expert count (1024 experts of a few rows, every 37th empty: one ragged tile
    per expert, scale atoms indexed up to the problem list's last tile) and a problem with no
    routed rows at all (nothing launched, zero gradients)."""
    wl = W.custom(T=400, k=4, E=1024, d=64, h=128, seed=63, invalid_frac=0.02,
                  empty_experts=tuple(range(0, 1024, 37)))
    run, g = _mx_run(wl, backward=True)
    o = _oracle(wl, True, g["dout"])
    M = o["r"]["M"]
    G.assert_close(G.host(run.y)[:M], o["y"][:M], "y[E=1024]")
    G.assert_close(G.host(g["dxp"])[:M], o["dxp"][:M], "dxp[E=1024]")
    nz = o["r"]["counts"] > 0
    G.assert_close(G.host(g["dwu"])[nz], o["dwu"][nz], "dW_ug[E=1024]")
    assert not G.host(g["dwd"])[~nz].any()

    wl0 = W.custom(T=0, k=2, E=5, d=64, h=128, seed=64)
    E, d, h = wl0.E, wl0.d, wl0.h
    offs = torch.zeros(E, dtype=torch.int32, device="cuda")
    mxw = _prepared(wl0)
    one = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")
    dwu = torch.full((E, 2 * h, d), float("nan"), device="cuda")
    dwd = torch.full((E, h, d), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(L.moe_workspace_bytes(L.OP_MX_BWD, 0, 2, E, d, h), 256), dtype=torch.uint8, device="cuda")
    sv = torch.zeros(max(L.moe_workspace_bytes(L.OP_SAVED, 0, 2, E, d, h), 256), dtype=torch.uint8, device="cuda")
    L.moe_grouped_swiglu_fwd_mxfp8(one(1, d), offs, None, None, E, 0, d, h, mxw, one(1, d), one(1, h), sv, ws, status)
    L.moe_grouped_bwd_mxfp8(one(1, d), one(1, d), one(1, h), sv, offs, None, None, E, 0, d, h, mxw, one(1, d), dwu,
                            dwd, ws, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert not dwu.any() and not dwd.any()
