"""The debug build (libmoe_gg_debug.so, compiled with MOE_GG_DEBUG) in place of a memory checker.

Each run is a child process that loads one build before anything else (the binding keeps the
first library it loads) and checks which one it got:
- "release" / "debug": the layer forward and backward on small edge cases (the toy workload, one
  expert, all experts empty but one, ragged tiles with dropped ids and an empty expert, widths
  that are not multiples of 8), the MXFP8 forward and backward, and one call captured into a CUDA
  graph. The debug build must report no failed bounds check, and both builds must give the same
  bits: the checks change no arithmetic.
- "planted": the debug build only. Out-of-range rows and slots are written into the inverse map
  and the slot map on the device; the debug kernels' own checks must catch them, skip the access
  and report the site, the index and its bound. (A release build would read out of bounds here,
  so the child stops unless the debug build is the one loaded.)
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, os, sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from ragged_grouped_gemm_device_gb300 import _lib as L
mode, outdir = sys.argv[2], sys.argv[3]
want_debug = mode != "release"
L.load(L.DEBUG_LIB_PATH if want_debug else L.LIB_PATH)
if L.moe_debug_build() != want_debug:
    sys.exit("wrong build loaded")
from ragged_grouped_gemm_device_gb300 import workloads as W
from ragged_grouped_gemm_device_gb300.layer import ExpertLayer

dev, i32, u8, bf16 = "cuda", torch.int32, torch.uint8, torch.bfloat16
bf = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(bf16).to(dev)
bits = lambda t: (t.view(torch.int16) if t.dtype == bf16 else t).cpu().numpy()
L.moe_debug_report(reset=True)
out = {}

def layer_case(name, wl):
    layer = ExpertLayer(bf(wl.w_ug_all()), bf(wl.w_down_all()))
    y = layer.forward(bf(wl.x()), torch.from_numpy(wl.ids).to(dev), torch.from_numpy(wl.weights).to(dev))
    res = layer.backward(bf(wl.dout()))
    torch.cuda.synchronize()
    assert layer.status.item() == 0, (name, layer.status.item())
    for key, t in zip(("out", "dx", "dw_ug", "dw_down", "dw_route"), (y,) + tuple(res)):
        out[name + "/" + key] = bits(t)

def route(wl):
    T, k, E, n = wl.T, wl.k, wl.E, wl.n
    counts, offs = torch.empty(E, dtype=i32, device=dev), torch.empty(E, dtype=i32, device=dev)
    ss, inv = torch.empty(n, dtype=i32, device=dev), torch.empty(n, dtype=i32, device=dev)
    ws = torch.empty(max(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), 1), dtype=u8, device=dev)
    L.moe_route_offsets(torch.from_numpy(wl.ids).to(dev), T, k, E, counts, offs, ss, inv, ws)
    return offs, ss, inv

def mx_case(name, wl):
    T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
    st = torch.zeros(1, dtype=i32, device=dev)
    offs, ss, inv = route(wl)
    w = torch.from_numpy(wl.weights).to(dev)
    mxw = torch.empty(L.moe_workspace_bytes(L.OP_MX_WEIGHTS, T, k, E, d, h), dtype=u8, device=dev)
    L.moe_mx_prepare_weights(bf(wl.w_ug_all()), bf(wl.w_down_all()), E, d, h, mxw)
    xp = torch.empty(n, d, dtype=bf16, device=dev)
    xq = torch.empty(n, d, dtype=u8, device=dev)
    xsf = torch.empty(L.moe_workspace_bytes(L.OP_MX_ROW_SCALES, T, k, E, d, h), dtype=u8, device=dev)
    L.moe_permute_mxfp8(bf(wl.x()), ss, offs, T, k, E, d, xp, xq, xsf, st)
    y, a = torch.empty(n, d, dtype=bf16, device=dev), torch.empty(n, h, dtype=bf16, device=dev)
    sv = torch.empty(L.moe_workspace_bytes(L.OP_SAVED, T, k, E, d, h), dtype=u8, device=dev)
    fws = torch.empty(L.moe_workspace_bytes(L.OP_MX_FWD, T, k, E, d, h), dtype=u8, device=dev)
    L.moe_grouped_swiglu_fwd_mxfp8(None, offs, ss, w, E, n, d, h, mxw, y, a, sv, fws, st, xq=xq, xsf=xsf)
    dy = bf(wl.dy(n))
    dxp = torch.empty(n, d, dtype=bf16, device=dev)
    dwu = torch.empty(E, 2 * h, d, device=dev)
    dwd = torch.empty(E, h, d, device=dev)
    dwr = torch.empty(n, device=dev)
    bws = torch.empty(L.moe_workspace_bytes(L.OP_MX_BWD, T, k, E, d, h), dtype=u8, device=dev)
    L.moe_grouped_bwd_mxfp8(dy, xp, a, sv, offs, ss, w, E, n, d, h, mxw, dxp, dwu, dwd, bws, st,
                            inv_map=inv, dw_route=dwr)
    torch.cuda.synchronize()
    assert st.item() == 0, (name, st.item())
    M = int(offs[-1].item())
    for key, t in (("y", y[:M]), ("a", a[:M]), ("dxp", dxp[:M]), ("dw_ug", dwu), ("dw_down", dwd), ("dw_route", dwr)):
        out[name + "/" + key] = bits(t)

def graph_case(name, wl):
    # a call queued while its stream is captured: the debug build must not wait on that stream
    T, k, E, d = wl.T, wl.k, wl.E, wl.d
    offs, ss, inv = route(wl)
    x = bf(wl.x())
    xp = torch.zeros(wl.n, d, dtype=bf16, device=dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        L.moe_permute(x, ss, offs, None, T, k, E, d, xp)
    g.replay()
    torch.cuda.synchronize()
    out[name + "/xp"] = bits(xp[: int(offs[-1].item())])

if mode in ("release", "debug"):
    layer_case("toy", W.make("toy"))
    layer_case("one_expert", W.custom(T=200, k=1, E=1, d=128, h=128, seed=71))
    layer_case("one_nonempty", W.custom(T=150, k=2, E=8, d=128, h=256, seed=72,
                                        empty_experts=(0, 1, 2, 3, 5, 6, 7)))
    layer_case("ragged", W.custom(T=333, k=4, E=16, d=256, h=384, seed=73, invalid_frac=0.05,
                                  empty_experts=(3,)))
    layer_case("odd_width", W.custom(T=64, k=2, E=4, d=60, h=44, seed=74))
    mx_case("mx", W.custom(T=300, k=4, E=8, d=256, h=256, seed=75, invalid_frac=0.03))
    graph_case("graph", W.custom(T=100, k=2, E=4, d=128, h=128, seed=76))
    np.savez(os.path.join(outdir, mode + ".npz"), **out)
    m, s, i, l = L.moe_debug_report(reset=True)
    print(json.dumps({"mask": m, "site": s, "index": i, "limit": l, "n": len(out)}), flush=True)
else:
    found = {}
    wl = W.custom(T=96, k=2, E=4, d=128, h=128, seed=77)
    T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
    offs, ss, inv = route(wl)
    w = torch.from_numpy(wl.weights).to(dev)
    # (1) the combine meets an inverse-map row past the T*top_k permuted rows
    y = bf(np.ones((n, d), np.float32))
    res = torch.empty(T, d, dtype=bf16, device=dev)
    bad_inv = inv.clone()
    bad_inv[5] = n + 5
    L.moe_unpermute_combine(y, bad_inv, None, T, k, d, res)
    found["combine"] = L.moe_debug_report(reset=True)
    # (2) the up/gate epilogue meets a slot past cap in the slot map, where it reads the weight
    bad_ss = ss.clone()
    bad_ss[0] = n + 7
    xp = torch.empty(n, d, dtype=bf16, device=dev)
    L.moe_permute(bf(wl.x()), ss, offs, None, T, k, E, d, xp)
    yy, a = torch.empty(n, d, dtype=bf16, device=dev), torch.empty(n, h, dtype=bf16, device=dev)
    L.moe_grouped_swiglu_fwd(xp, offs, bad_ss, w, E, n, d, h, bf(wl.w_ug_all()), bf(wl.w_down_all()), yy, a,
                             None, None, None)
    found["slot"] = L.moe_debug_report(reset=True)
    # (3) the routing-weight gradient meets an inverse-map row past the slots
    part = torch.zeros(n, 2, device=dev)
    dw = torch.empty(n, device=dev)
    L.moe_routing_weight_grad(part, bad_inv, T, k, 128, dw)
    found["rwg"] = L.moe_debug_report(reset=True)
    # (4) top_k = 1: the down projection meets a destination token row past T (and the up/gate
    # epilogue, reading the same slot map for the weight, a slot past cap = T)
    w1 = W.custom(T=80, k=1, E=4, d=128, h=128, seed=78)
    offs1, ss1, inv1 = route(w1)
    bad1 = ss1.clone()
    bad1[3] = w1.T + 9
    xp1 = torch.empty(w1.n, w1.d, dtype=bf16, device=dev)
    L.moe_permute(bf(w1.x()), ss1, offs1, None, w1.T, 1, w1.E, w1.d, xp1)
    o1 = torch.empty(w1.T, w1.d, dtype=bf16, device=dev)
    a1 = torch.empty(w1.T, w1.h, dtype=bf16, device=dev)
    L.moe_grouped_swiglu_fwd_top1_combine(xp1, offs1, bad1, inv1, torch.from_numpy(w1.weights).to(dev), w1.E,
                                          w1.T, w1.d, w1.h, bf(w1.w_ug_all()), bf(w1.w_down_all()), o1, a1)
    found["dst"] = L.moe_debug_report(reset=True)
    found["clean"] = L.moe_debug_report(reset=True)
    print(json.dumps({k: list(v) for k, v in found.items()}), flush=True)
"""


def _run(mode, outdir):
    os.makedirs(outdir, exist_ok=True)
    res = subprocess.run([sys.executable, "-c", CHILD, ROOT, mode, str(outdir)], capture_output=True, text=True,
                         timeout=900)
    assert res.returncode == 0, res.stderr[-3000:]
    return json.loads([ln for ln in res.stdout.splitlines() if ln.startswith("{")][-1])


@pytest.fixture(scope="module")
def debug_lib(lib):
    from ragged_grouped_gemm_device_gb300 import build
    return build.build(debug=True)


def test_debug_build_passes_its_checks_and_matches_release(debug_lib, tmp_path):
    rel = _run("release", tmp_path)
    dbg = _run("debug", tmp_path)
    assert rel == {"mask": 0, "site": -1, "index": 0, "limit": 0, "n": rel["n"]}
    assert dbg["mask"] == 0 and dbg["site"] == -1, f"failed bounds check: {dbg}"
    a, b = np.load(tmp_path / "release.npz"), np.load(tmp_path / "debug.npz")
    assert sorted(a.files) == sorted(b.files) and len(a.files) == rel["n"] == dbg["n"]
    for key in a.files:
        assert np.array_equal(a[key], b[key]), key


def test_debug_build_catches_planted_indices(debug_lib, tmp_path):
    from ragged_grouped_gemm_device_gb300 import _lib as L
    got = _run("planted", tmp_path)
    n, cap = 96 * 2, 96 * 2
    sites = {name: i for i, name in enumerate(["gg_row", "gg_tile", "gg_slot", "gg_dst", "gg_sfa", "gg_sfb",
                                                "gg_mxsf", "combine_row", "rwg_row", "route_pos", "mx_tile"])}
    assert got["combine"] == [1 << sites["combine_row"], sites["combine_row"], n + 5, n]
    assert got["slot"] == [1 << sites["gg_slot"], sites["gg_slot"], n + 7, cap]
    assert got["rwg"] == [1 << sites["rwg_row"], sites["rwg_row"], n + 5, n]
    # both the slot read for the weight (up/gate) and the destination row (down) are caught; the
    # up/gate launch runs first, so its site is the first failure
    assert got["dst"] == [(1 << sites["gg_slot"]) | (1 << sites["gg_dst"]), sites["gg_slot"], 80 + 9, 80]
    assert got["clean"] == [0, -1, 0, 0]
    assert L.moe_debug_site_name(sites["combine_row"]).startswith("combine")
