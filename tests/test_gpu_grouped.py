"""GPU parity of the grouped SwiGLU expert forward and backward (tcgen05 kernels) against the
fp64 oracle, on the full small and mid-size workloads and on sampled experts of the large one.

Row buffers start NaN-filled, so a tile that read or wrote past its expert's segment (or past
M) would show up as a non-finite or mismatched value."""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FWD_CASES = {
    "toy": lambda: W.make("toy"),
    "toy_sorted": lambda: W.make("toy_sorted"),
    # K tail (d = 40 < 64), column tail (h = 24: half of a 16-column chunk), empty experts
    "edge_small": lambda: W.custom(T=77, k=3, E=9, d=40, h=24, seed=7, invalid_frac=0.05, empty_experts=(0, 4)),
    # several row tiles per expert with ragged tails, K = 136 (tail of 8), h = 200
    "edge_wide": lambda: W.custom(T=300, k=2, E=5, d=136, h=200, seed=8),
    # one expert over many row tiles
    "edge_one_expert": lambda: W.custom(T=700, k=1, E=1, d=64, h=64, seed=9),
    # most experts empty, the last one non-empty
    "edge_sparse": lambda: W.custom(T=100, k=1, E=64, d=64, h=72, seed=10, empty_experts=tuple(range(0, 62))),
    # the largest problem list (E = 1024 experts of ~12 rows, every 41st empty): the in-kernel
    # offsets and tile prefix at their maximum size, one ragged tile per expert
    "edge_max_experts": lambda: W.custom(T=3000, k=4, E=1024, d=64, h=64, seed=11,
                                         empty_experts=tuple(range(0, 1024, 41))),
    # widths whose bf16 rows are not 16-byte multiples: zero-padded copies inside the composites
    "edge_odd_width": lambda: W.custom(T=150, k=3, E=6, d=60, h=44, seed=13, invalid_frac=0.05,
                                       empty_experts=(1,)),
    "edge_odd_width2": lambda: W.custom(T=90, k=2, E=5, d=77, h=33, seed=14),
    # the widest rows the header allows: d = 2^20 (a contraction of 16384 K blocks in one tile,
    # 4096 column tiles in the down projection and the wgrads) and h = 2^20 (8192 column tiles of
    # the up/gate projection, a 2 GB saved U, 16384 gradient row tiles per expert). With
    # W_down ~ N(0, 1/sqrt(h)) the down dgrad's sums over d = 2^20 products have an rms of
    # sqrt(d/h); h = 64 keeps them at ~128, where fp32 accumulation (even rounded to nearest at
    # every step) still meets the elementwise bound on the gradients' near-zero elements -- at
    # h = 16 (sums of ~256) it does not, whatever the order of the additions.
    "edge_max_d": lambda: W.custom(T=24, k=1, E=2, d=1 << 20, h=64, seed=15),
    "edge_max_h": lambda: W.custom(T=24, k=2, E=1, d=32, h=1 << 20, seed=16),
    # the narrowest rows: d = h = 8 (one 16-byte row pitch, a K block mostly zero fill) and
    # d = h = 1 (zero-padded to 8 inside the composite calls)
    "edge_min_width": lambda: W.custom(T=40, k=2, E=3, d=8, h=8, seed=18, empty_experts=(2,)),
    "edge_width_1": lambda: W.custom(T=30, k=2, E=3, d=1, h=1, seed=19),
    # one expert with 20000 rows: a wgrad contraction of 313 K blocks, accumulated in segments
    "edge_long_expert": lambda: W.custom(T=20000, k=1, E=2, d=64, h=64, seed=17, empty_experts=(1,)),
    "balanced": lambda: W.make("balanced"),
    "finegrained": lambda: W.make("finegrained"),
    "skew": lambda: W.make("skew"),
}

BWD_CASES = ["toy", "edge_small", "edge_wide", "edge_one_expert", "edge_sparse", "edge_max_experts",
             "edge_odd_width", "edge_odd_width2", "edge_max_d", "edge_max_h", "edge_min_width", "edge_width_1",
             "edge_long_expert", "finegrained", "skew"]


def _dy(wl, M):
    """Upstream gradient at the grouped boundary: N(0,1) rows < M, NaN past M."""
    dyh = wl.dy(max(wl.n, 1))
    dy = G.dev_bf16(dyh)
    dy[M:] = float("nan")
    dyh = dyh.astype(np.float64)
    dyh[M:] = 0.0
    return dy, dyh


@pytest.mark.parametrize("name", list(FWD_CASES))
def test_grouped_forward(lib, name):
    wl = FWD_CASES[name]()
    run = G.DevicePipeline(wl).route().permute().forward()
    torch.cuda.synchronize()
    assert run.status.item() == 0
    r, xp, y, u, a = G.oracle_run(wl)
    M = r["M"]
    G.assert_close(G.host(run.a)[:M], a[:M], f"A[{name}]")
    G.assert_close(G.host(run.u)[:M], u[:M], f"U[{name}]")
    G.assert_close(G.host(run.y)[:M], y[:M], f"y[{name}]")
    # unused capacity stays outside the final offset: never written
    assert np.isnan(G.host(run.y)[M:]).all() and np.isnan(G.host(run.a)[M:]).all()


@pytest.mark.parametrize("name", BWD_CASES)
def test_grouped_backward(lib, name):
    wl = FWD_CASES[name]()
    run = G.DevicePipeline(wl).route().permute().forward()
    r, xp, y, u, a = G.oracle_run(wl)
    M = r["M"]
    dy, dyh = _dy(wl, M)
    run.backward(dy)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    dxp, dw_ug, dw_down, du = O.expert_backward(dyh, xp, u, r["offsets"], wl.w_ug, wl.w_down)
    G.assert_close(G.host(run.dxp)[:M], dxp[:M], f"dxp[{name}]")
    got_ug, got_dn = G.host(run.dw_ug), G.host(run.dw_down)
    nz = r["counts"] > 0
    G.assert_close(got_ug[nz], dw_ug[nz], f"dW_ug[{name}]")
    G.assert_close(got_dn[nz], dw_down[nz], f"dW_down[{name}]")
    assert not got_ug[~nz].any() and not got_dn[~nz].any(), "empty experts must get zero gradients"
    assert np.isnan(G.host(run.dxp)[M:]).all()


# Segment lengths around the CTA-pair wgrad's boundaries: an expert's last K block holds 1..64
# rows and its rows end exactly on a 16-row K step (16, 48, 64, 128, 256) or inside one (1, 15,
# 17, 63, 65, ...); one expert is empty. The gradient heights (h and 2h: 72/144, 160/320,
# 256/512 rows) leave the odd CTA of the last 256-row pair tile none of the gradient's rows, part
# of them or all of them, and the widths d (200, 384, 136) end inside a 256-column tile.
EXACT_COUNTS = [1, 15, 16, 17, 48, 63, 64, 65, 100, 128, 0, 200, 255, 256, 257, 513]


@pytest.mark.parametrize("d,h", [(200, 72), (384, 160), (136, 256)])
def test_wgrad_pair_expert_boundaries(lib, d, h):
    wl = W.exact_counts(EXACT_COUNTS, d=d, h=h, seed=21)
    run = G.DevicePipeline(wl).route().permute().forward()
    r, xp, y, u, a = G.oracle_run(wl)
    M = r["M"]
    assert list(r["counts"]) == EXACT_COUNTS
    dy, dyh = _dy(wl, M)
    run.backward(dy)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    dxp, dw_ug, dw_down, du = O.expert_backward(dyh, xp, u, r["offsets"], wl.w_ug, wl.w_down)
    got_ug, got_dn = G.host(run.dw_ug), G.host(run.dw_down)
    nz = r["counts"] > 0
    G.assert_close(got_ug[nz], dw_ug[nz], f"dW_ug[{d}x{h}]")
    G.assert_close(got_dn[nz], dw_down[nz], f"dW_down[{d}x{h}]")
    assert not got_ug[~nz].any() and not got_dn[~nz].any(), "empty experts must get zero gradients"
    G.assert_close(G.host(run.dxp)[:M], dxp[:M], f"dxp[{d}x{h}]")


@pytest.mark.slow
def test_large_forward_backward_sampled_experts(lib):
    """The large workload at full size; the oracle checks every row and gradient of a sample of
    experts (first, last, largest, smallest and random ones)."""
    wl = W.make("large")
    run = G.DevicePipeline(wl).route().permute().forward()
    r = O.route_offsets(wl.ids, wl.E)
    M = r["M"]
    experts = G.sample_experts(r["counts"], n_pick=8)
    xp = O.permute(wl.x(), r["sorted_src"], M, wl.k)
    y, u, a, _ = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down, experts)
    dy, dyh = _dy(wl, M)
    run.backward(dy)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    rows = G.rows_of(r["offsets"], experts)
    G.assert_close(G.host(run.a)[rows], a[rows], "A[large]")
    G.assert_close(G.host(run.y)[rows], y[rows], "y[large]")
    dxp, dw_ug, dw_down, _ = O.expert_backward(dyh, xp, u, r["offsets"], wl.w_ug, wl.w_down, experts)
    G.assert_close(G.host(run.dxp)[rows], dxp[rows], "dxp[large]")
    G.assert_close(G.host(run.dw_ug[experts]), dw_ug[experts], "dW_ug[large]")
    G.assert_close(G.host(run.dw_down[experts]), dw_down[experts], "dW_down[large]")
    assert np.isfinite(G.host(run.y)[:M]).all() and np.isfinite(G.host(run.dxp)[:M]).all()


def test_bad_offsets_flag_and_no_work(lib):
    """Decreasing offsets, or a final offset beyond the buffer, set MOE_DEV_BAD_OFFSETS and the
    kernels compute nothing."""
    from ragged_grouped_gemm_device_gb300 import _lib
    wl = FWD_CASES["edge_small"]()
    run = G.DevicePipeline(wl)
    for bad in ([5, 3, 9, 9, 9, 9, 9, 9, 9], [1, 2, 3, 4, 5, 6, 7, 8, wl.n + 1]):
        run.offsets.copy_(torch.tensor(bad, dtype=torch.int32))
        run.status.zero_()
        _lib.moe_grouped_swiglu_fwd(run.xp, run.offsets, None, None, wl.E, run.cap, wl.d, wl.h, run.w_ug,
                                    run.w_down, run.y, run.a, run.saved, None, run.status)
        torch.cuda.synchronize()
        assert run.status.item() & _lib.MOE_DEV_BAD_OFFSETS
        assert np.isnan(G.host(run.y)).all()


def test_single_kernel_entry_points_equal_composites(lib):
    """The per-step entry points (one kernel each) reproduce the composite forward and backward
    bit for bit, with routing weights folded in (the composite backward runs both wgrads in one
    launch, as moe_grouped_wgrad_dual does); the bf16-only wgrad (no low half) stays within the
    normalised tolerance."""
    from ragged_grouped_gemm_device_gb300 import _lib as L
    wl = W.custom(T=300, k=4, E=7, d=136, h=200, seed=31, invalid_frac=0.05, empty_experts=(3,))
    run = G.DevicePipeline(wl).route().permute()
    n, d, h, E = run.cap, wl.d, wl.h, wl.E
    y1, a1 = G.nan_filled((n, d)), G.nan_filled((n, h))
    sv1 = torch.zeros_like(run.saved)
    L.moe_grouped_swiglu_fwd(run.xp, run.offsets, run.sorted_src, run.weights, E, n, d, h, run.w_ug, run.w_down,
                             y1, a1, sv1, None, run.status)
    y2, a2 = G.nan_filled((n, d)), G.nan_filled((n, h))
    sv2 = torch.zeros_like(run.saved)
    L.moe_grouped_up_swiglu(run.xp, run.offsets, run.sorted_src, run.weights, E, n, d, h, run.w_ug, a2, sv2,
                            run.status)
    L.moe_grouped_down(a2, run.offsets, E, n, d, h, run.w_down, y2, run.status)
    dy = G.dev_bf16(wl.dy(n))
    ws = torch.zeros(L.moe_workspace_bytes(L.OP_BWD, wl.T, wl.k, E, d, h), dtype=torch.uint8, device="cuda")
    dxp1 = G.nan_filled((n, d))
    dwu1 = torch.zeros(E, 2 * h, d, device="cuda")
    dwd1 = torch.zeros(E, h, d, device="cuda")
    dwr1 = torch.full((n,), float("nan"), device="cuda")
    L.moe_grouped_bwd(dy, run.xp, a1, sv1, run.offsets, run.sorted_src, run.weights, E, n, d, h, run.w_ug,
                      run.w_down, dxp1, dwu1, dwd1, ws, run.status, inv_map=run.inv_map, dw_route=dwr1)
    du_hi, du_lo = G.nan_filled((n, 2 * h)), G.nan_filled((n, 2 * h))
    dxp2 = G.nan_filled((n, d))
    dwu2, dwd2, dwu3 = (torch.zeros_like(dwu1), torch.zeros_like(dwd1), torch.zeros_like(dwu1))
    _, p_lo = L.saved_views(sv2, n, h)
    part = torch.full((n, L.routing_grad_parts(h)), float("nan"), device="cuda")
    L.moe_grouped_down_dgrad_swiglu(dy, sv2, run.offsets, run.sorted_src, run.weights, E, n, d, h, run.w_down,
                                    du_hi, du_lo, run.status, dw_part=part)
    dwr2 = torch.full((n,), float("nan"), device="cuda")
    L.moe_routing_weight_grad(part, run.inv_map, wl.T, wl.k, h, dwr2)
    L.moe_grouped_up_dgrad(du_hi, run.offsets, E, n, d, h, run.w_ug, dxp2, run.status)
    L.moe_grouped_wgrad(a2, p_lo, h, dy, d, run.offsets, E, n, dwd2, run.status)
    L.moe_grouped_wgrad(du_hi, du_lo, 2 * h, run.xp, d, run.offsets, E, n, dwu2, run.status)
    L.moe_grouped_wgrad(du_hi, None, 2 * h, run.xp, d, run.offsets, E, n, dwu3, run.status)
    # both gradients from one launch, with and without the low halves
    dwd4, dwu4 = torch.full_like(dwd1, float("nan")), torch.full_like(dwu1, float("nan"))
    L.moe_grouped_wgrad_dual(a2, p_lo, h, dy, d, dwd4, du_hi, du_lo, 2 * h, run.xp, d, dwu4, run.offsets, E, n,
                             run.status)
    dwd5, dwu5 = torch.full_like(dwd1, float("nan")), torch.full_like(dwu1, float("nan"))
    L.moe_grouped_wgrad_dual(a2, None, h, dy, d, dwd5, du_hi, None, 2 * h, run.xp, d, dwu5, run.offsets, E, n,
                             run.status)
    dwd6 = torch.full_like(dwd1, float("nan"))
    L.moe_grouped_wgrad(a2, None, h, dy, d, run.offsets, E, n, dwd6, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    M = int(run.offsets[-1].item())
    for got, want in ((y2, y1), (a2, a1), (dxp2, dxp1)):
        assert torch.equal(got[:M], want[:M])
    # saved compared as bytes: bit for bit, whatever values it holds
    assert torch.equal(sv2.view(torch.uint8), sv1.view(torch.uint8))
    assert torch.equal(dwu2, dwu1) and torch.equal(dwd2, dwd1)
    assert torch.equal(dwu4, dwu1) and torch.equal(dwd4, dwd1)
    assert torch.equal(dwu5, dwu3) and torch.equal(dwd5, dwd6)
    assert torch.equal(dwr2, dwr1) and torch.isfinite(dwr1).all()
    err = (dwu3 - dwu1).double().norm() / dwu1.double().norm()
    assert err <= G.REL_NORM_TOL, f"bf16-only wgrad normalised error {err:.2e}"


def test_outputs_at_16_byte_alignment_match_32_byte_aligned(lib):
    """Row outputs whose base is 16- but not 32-byte aligned take the 16-byte store path of the
    up/gate and dgrad epilogues; the results are bit-identical to the 32-byte path."""
    from ragged_grouped_gemm_device_gb300 import _lib as L
    wl = W.custom(T=200, k=2, E=5, d=128, h=256, seed=41, empty_experts=(2,))
    run = G.DevicePipeline(wl).route().permute()
    n, d, h, E = run.cap, wl.d, wl.h, wl.E
    M = int(run.offsets[-1].item())

    def shifted(rows, cols, shift):
        """A [rows, cols] bf16 view whose first element sits `shift` elements into a NaN buffer."""
        buf = G.nan_filled((rows * cols + 16,))
        return buf[shift:shift + rows * cols].view(rows, cols)

    sv = torch.zeros(L.moe_workspace_bytes(L.OP_SAVED, wl.T, wl.k, E, d, h) + 32, dtype=torch.uint8, device="cuda")
    results = []
    for shift in (0, 8):  # 8 bf16 = 16 bytes
        a = shifted(n, h, shift)
        saved = sv[2 * shift:2 * shift + L.moe_workspace_bytes(L.OP_SAVED, wl.T, wl.k, E, d, h)]
        saved.zero_()
        L.moe_grouped_up_swiglu(run.xp, run.offsets, run.sorted_src, run.weights, E, n, d, h, run.w_ug, a, saved,
                                run.status)
        dy = G.dev_bf16(wl.dy(n))
        du_hi, du_lo = shifted(n, 2 * h, shift), shifted(n, 2 * h, shift)
        L.moe_grouped_down_dgrad_swiglu(dy, saved, run.offsets, run.sorted_src, run.weights, E, n, d, h,
                                        run.w_down, du_hi, du_lo, run.status)
        torch.cuda.synchronize()
        assert run.status.item() == 0
        results.append((a[:M].clone(), saved.clone(), du_hi[:M].clone(), du_lo[:M].clone()))
    for x0, x1 in zip(*results):
        assert torch.equal(x0.view(torch.uint8), x1.view(torch.uint8))


def test_long_contraction_keeps_fp32_accuracy(lib):
    """A contraction of 2^20 products in one tile (the wgrad over one expert's 2^20 rows, fp32
    out). The tensor core's accumulator does not round each addition to nearest: left alone, its
    error grows like a truncating sum (rms 1.2 on sums of rms ~1000 here). Contractions longer
    than 8192 are accumulated in segments folded in round-to-nearest fp32, which keeps the error
    at the level of an fp32 sum."""
    from ragged_grouped_gemm_device_gb300 import _lib as L
    K, P, Q = 1 << 20, 16, 16
    rng = np.random.default_rng(5)
    a = torch.from_numpy(rng.standard_normal((K, P)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy(rng.standard_normal((K, Q)).astype(np.float32)).to(torch.bfloat16)
    ref = a.double().numpy().T @ b.double().numpy()
    offs = torch.tensor([K], dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dw = torch.full((1, P, Q), float("nan"), device="cuda")
    L.moe_grouped_wgrad(a.cuda(), None, P, b.cuda(), Q, offs, 1, K, dw, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    err = dw[0].cpu().double().numpy() - ref
    rms_ref = np.sqrt((ref ** 2).mean())
    assert rms_ref > 500
    # an fp32 sum rounded to nearest at every step has an rms error of ~0.005 here
    assert np.sqrt((err ** 2).mean()) < 0.05 and np.abs(err).max() < 0.25, (np.sqrt((err ** 2).mean()), np.abs(err).max())
