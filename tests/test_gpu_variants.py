"""GPU parity of the two comparison variants built in the same library: the capacity-padded BMM
("Section 09: Grouped GEMM", Eq. 14 and Fig. 35) and the host-scheduled per-expert loop
(Fig. 36)."""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import _lib
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,C", [("toy", 4), ("toy", 2), ("edge", None), ("balanced", None), ("skew", None)])
def test_padded_bmm_matches_oracle(lib, name, C):
    wl = W.custom(T=300, k=2, E=5, d=136, h=200, seed=8) if name == "edge" else W.make(name)
    run = G.DevicePipeline(wl).route().permute()
    r = O.route_offsets(wl.ids, wl.E)
    M = r["M"]
    if C is None:
        C = O.capacity_ceil(1.25, M, wl.E)
    ws = torch.empty(_lib.moe_workspace_bytes(_lib.OP_PADDED_BMM, wl.T, wl.k, wl.E, wl.d, wl.h, C),
                     dtype=torch.uint8, device="cuda")
    _lib.moe_padded_bmm_swiglu_fwd(run.xp, run.offsets, wl.E, run.cap, wl.d, wl.h, C, run.w_ug, run.w_down,
                                   run.y, ws, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    xp = O.permute(wl.x(), r["sorted_src"], M, wl.k)
    want, stats = O.padded_bmm_forward(xp, r["offsets"], C, wl.w_ug, wl.w_down)
    got = G.host(run.y)
    kept = np.ones(M, bool)
    for e, (s, t) in enumerate(O.segments(r["offsets"])):
        kept[s + min(C, t - s):t] = False
    G.assert_close(got[:M][kept], want[:M][kept], f"bmm[{name},C={C}]")
    assert not got[:M][~kept].any(), "rows beyond the capacity are dropped (zero output)"
    if name == "toy" and C == 4:
        assert stats["rows_multiplied"] == 16 and stats["padding_rows"] == 6


@pytest.mark.parametrize("name", ["toy", "edge_sparse", "skew"])
def test_host_loop_matches_oracle(lib, name):
    if name == "edge_sparse":
        wl = W.custom(T=100, k=1, E=64, d=64, h=72, seed=10, empty_experts=tuple(range(0, 62)))
    else:
        wl = W.make(name)
    run = G.DevicePipeline(wl).route().permute()
    _lib.moe_loop_swiglu_fwd(run.xp, run.offsets, wl.E, run.cap, wl.d, wl.h, run.w_ug, run.w_down, run.y,
                             run.a, run.saved, run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    r, xp, y, u, a = G.oracle_run(wl)
    M = r["M"]
    G.assert_close(G.host(run.y)[:M], y[:M], f"loop y[{name}]")
    G.assert_close(G.host(run.a)[:M], a[:M], f"loop A[{name}]")
    # the saved U of expert e lands in the row tiles the grouped kernels give it
    G.assert_close(G.host(run.u)[:M], u[:M], f"loop U[{name}]")
    assert np.isnan(G.host(run.y)[M:]).all()
