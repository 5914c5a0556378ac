"""The combine fused into the down projection for top_k = 1 ("Section 09: Grouped GEMM", §9.4:
the down projection writes straight into the combine buffer). With one slot per token there is
nothing to reduce, so the fused call must give bit for bit what the grouped forward followed by
the combine gives (weights folded, combine with weights = NULL), with zero rows for tokens whose
slot was dropped, and agree with the oracle's weighted combine."""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import _lib as L
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    "toy": lambda: W.make("toy"),
    "skew": lambda: W.make("skew"),
    # dropped ids (zero rows), empty experts, ragged tiles
    "edge": lambda: W.custom(T=500, k=1, E=7, d=72, h=136, seed=71, invalid_frac=0.1, empty_experts=(2,)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_top1_fused_combine_equals_forward_then_combine(lib, name):
    wl = CASES[name]()
    assert wl.k == 1
    run = G.DevicePipeline(wl).route().permute()
    T, E, d, h = wl.T, wl.E, wl.d, wl.h
    y = G.nan_filled((T, d))
    a1, a2 = G.nan_filled((T, h)), G.nan_filled((T, h))
    sv1, sv2 = torch.zeros_like(run.saved), torch.zeros_like(run.saved)
    L.moe_grouped_swiglu_fwd(run.xp, run.offsets, run.sorted_src, run.weights, E, T, d, h, run.w_ug, run.w_down, y,
                             a1, sv1, None, run.status)
    out1 = G.nan_filled((T, d))
    L.moe_unpermute_combine(y, run.inv_map, None, T, 1, d, out1)
    out2 = G.nan_filled((T, d))
    L.moe_grouped_swiglu_fwd_top1_combine(run.xp, run.offsets, run.sorted_src, run.inv_map, run.weights, E, T, d,
                                          h, run.w_ug, run.w_down, out2, a2, sv2, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    M = int(run.offsets[-1].item())
    assert torch.equal(out2.view(torch.int16), out1.view(torch.int16))
    assert torch.equal(a2[:M].view(torch.int16), a1[:M].view(torch.int16))
    assert torch.equal(sv2.view(torch.uint8), sv1.view(torch.uint8))
    dropped = (wl.ids.reshape(-1) < 0) | (wl.ids.reshape(-1) >= E)
    assert not G.host(out2)[dropped].any()
    r, xp, yo, u, a = G.oracle_run(wl)
    G.assert_close(G.host(out2), O.combine(yo, r["inv_map"], wl.weights, T, 1), f"out[{name}]")


def test_top1_fused_combine_max_experts_and_no_tokens(lib):
    wl = W.custom(T=900, k=1, E=1024, d=64, h=64, seed=72, invalid_frac=0.05,
                  empty_experts=tuple(range(0, 1024, 29)))
    run = G.DevicePipeline(wl).route().permute()
    T, E, d, h = wl.T, wl.E, wl.d, wl.h
    out = G.nan_filled((T, d))
    L.moe_grouped_swiglu_fwd_top1_combine(run.xp, run.offsets, run.sorted_src, run.inv_map, run.weights, E, T, d, h,
                                          run.w_ug, run.w_down, out, G.nan_filled((T, h)), None, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    r, xp, yo, u, a = G.oracle_run(wl)
    G.assert_close(G.host(out), O.combine(yo, r["inv_map"], wl.weights, T, 1), "out[E=1024]")
    # no tokens: nothing to launch, status OK
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.moe_grouped_swiglu_fwd_top1_combine(run.xp, run.offsets, run.sorted_src, run.inv_map, None, E, 0, d, h,
                                          run.w_ug, run.w_down, out, G.nan_filled((1, h)), None, z)
