"""What the wgrads' precision scheme buys, measured against the oracle.

The library keeps the wgrads' activation operand (P = w*A for the down projection, dU for the
up/gate projection) as a bf16 high + low pair and contracts both halves. The same operands
through the one-half (plain bf16) wgrad are compared here with the oracle on the workloads with
a backward, at the task tolerance: normalised error <= 5e-3 and |err| <= 2e-2 (1 + |ref|)
elementwise. Each case prints one line (prefix PRECISION) with, for both schemes, the
normalised error, the worst |err| / bound, the share of elements over the bound and the largest
|ref| among them. The hi/lo scheme must meet both bounds; the bf16 one must meet the normalised
bound (it is the elementwise bound on long expert segments that it can miss).
"""
import json

import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import _lib as L
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _stats(got, ref):
    err = got - ref
    bound = G.MAX_ABS_TOL * (1.0 + np.abs(ref))
    over = np.abs(err) > bound
    return {"rel": float(np.linalg.norm(err) / np.linalg.norm(ref)),
            "worst_err_over_bound": float((np.abs(err) / bound).max()),
            "share_over_bound": float(over.mean()),
            "max_ref_over_bound": float(np.abs(ref)[over].max()) if over.any() else None}


@pytest.mark.parametrize("name", ["finegrained", "skew", pytest.param("large", marks=pytest.mark.slow)])
def test_wgrad_precision_scheme(lib, name):
    wl = W.make(name)
    run = G.DevicePipeline(wl).route().permute().forward()
    r = O.route_offsets(wl.ids, wl.E)
    M, n, E, d, h = r["M"], wl.n, wl.E, wl.d, wl.h
    dyh = wl.dy(max(n, 1))
    dy = G.dev_bf16(dyh)
    run.backward(dy)
    # the same operands through the one-half wgrad: dU high half from the backward's workspace
    half = (n * 2 * h * 2 + 255) // 256 * 256
    du_hi = run.bwd_ws.view(torch.uint8)[:n * 2 * h * 2].view(torch.bfloat16).view(n, 2 * h)
    assert half >= n * 2 * h * 2
    dwu1 = torch.empty(E, 2 * h, d, device="cuda")
    dwd1 = torch.empty(E, h, d, device="cuda")
    L.moe_grouped_wgrad_dual(run.a, None, h, dy, d, dwd1, du_hi, None, 2 * h, run.xp, d, dwu1, run.offsets, E, n,
                             run.status)
    torch.cuda.synchronize()
    assert run.status.item() == 0
    experts = G.sample_experts(r["counts"], n_pick=8) if name == "large" else [e for e in range(E) if r["counts"][e]]
    xp = O.permute(wl.x(), r["sorted_src"], M, wl.k)
    y, u, a, _ = O.expert_forward(xp, r["offsets"], wl.w_ug, wl.w_down, experts)
    dyo = dyh.astype(np.float64)
    dyo[M:] = 0.0
    _, dw_ug, dw_down, _ = O.expert_backward(dyo, xp, u, r["offsets"], wl.w_ug, wl.w_down, experts)
    line = {"workload": name, "M": M, "max_rows_per_expert": int(r["counts"].max()), "experts_checked": len(experts)}
    for tag, (gu, gd) in (("hi_lo", (run.dw_ug, run.dw_down)), ("bf16", (dwu1, dwd1))):
        line[tag] = {"dW_ug": _stats(G.host(gu[experts]), dw_ug[experts]),
                     "dW_down": _stats(G.host(gd[experts]), dw_down[experts])}
    print("PRECISION " + json.dumps(line))
    for g in ("dW_ug", "dW_down"):
        assert line["hi_lo"][g]["rel"] <= G.REL_NORM_TOL and line["hi_lo"][g]["share_over_bound"] == 0.0
        assert line["bf16"][g]["rel"] <= G.REL_NORM_TOL
