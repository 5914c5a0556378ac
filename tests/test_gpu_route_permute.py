"""GPU parity of the integer and data-movement steps against the oracle: route histogram,
offsets, placement and inverse map bit-exact; permute bit-exact; combine within tolerance and
the permute/combine identity bit-exact."""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import _lib
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = {
    "toy": lambda: W.make("toy"),
    "toy_sorted": lambda: W.make("toy_sorted"),
    "balanced": lambda: W.make("balanced"),
    "finegrained": lambda: W.make("finegrained"),
    "skew": lambda: W.make("skew"),
    "large": lambda: W.make("large"),
    "invalid_ids": lambda: W.custom(T=1000, k=4, E=37, d=16, h=8, seed=1, invalid_frac=0.1, empty_experts=(3, 5)),
    "single_expert": lambda: W.custom(T=300, k=2, E=1, d=16, h=8, seed=2),
    "max_experts": lambda: W.custom(T=5000, k=8, E=1024, d=16, h=8, seed=3),
    "all_dropped": lambda: W.custom(T=50, k=2, E=4, d=16, h=8, seed=4, invalid_frac=1.0),
    "one_token": lambda: W.custom(T=1, k=8, E=16, d=16, h=8, seed=5),
    "top32": lambda: W.custom(T=129, k=32, E=40, d=16, h=8, seed=6, invalid_frac=0.05),
    # rows of 154 bytes: the element-wise gather and combine
    "odd_width": lambda: W.custom(T=333, k=3, E=7, d=77, h=8, seed=15, invalid_frac=0.05),
}


@pytest.mark.parametrize("name", list(CASES))
def test_route_offsets_bit_exact(lib, name):
    wl = CASES[name]()
    run = G.DevicePipeline(wl, with_u=False).route()
    torch.cuda.synchronize()
    r = O.route_offsets(wl.ids, wl.E)
    assert np.array_equal(run.counts.cpu().numpy(), r["counts"])
    assert np.array_equal(run.offsets.cpu().numpy(), r["offsets"])
    n = wl.n
    assert np.array_equal(run.sorted_src[:n].cpu().numpy(), r["sorted_src"])
    assert np.array_equal(run.inv_map[:n].cpu().numpy(), r["inv_map"])


def test_route_zero_tokens(lib):
    E = 6
    counts = torch.full((E,), 5, dtype=torch.int32, device="cuda")
    offsets = torch.full((E,), 5, dtype=torch.int32, device="cuda")
    dummy = torch.empty(1, dtype=torch.int32, device="cuda")
    _lib.moe_route_offsets(dummy, 0, 2, E, counts, offsets, dummy, dummy, None)
    torch.cuda.synchronize()
    assert not counts.any() and not offsets.any()


@pytest.mark.parametrize("name", ["toy", "balanced", "finegrained", "skew", "invalid_ids", "single_expert", "top32"])
def test_permute_bit_exact_and_tail_untouched(lib, name):
    wl = CASES[name]()
    run = G.DevicePipeline(wl, with_u=False).route().permute()
    torch.cuda.synchronize()
    r = O.route_offsets(wl.ids, wl.E)
    M = r["M"]
    want = O.permute(wl.x(), r["sorted_src"], M, wl.k)
    got = G.host(run.xp)
    assert np.array_equal(got[:M], want[:M])
    assert np.isnan(got[M:]).all()


def test_permute_row_scale_rounds_once(lib):
    wl = CASES["invalid_ids"]()
    run = G.DevicePipeline(wl, with_u=False).route()
    _lib.moe_permute(run.x, run.sorted_src, run.offsets, run.weights, wl.T, wl.k, wl.E, wl.d, run.xp)
    torch.cuda.synchronize()
    r = O.route_offsets(wl.ids, wl.E)
    M = r["M"]
    want = O.permute(wl.x(), r["sorted_src"], M, wl.k, row_scale=wl.weights)[:M]
    got = G.host(run.xp)[:M]
    # one rounding of an fp32 product to bf16: within half a bf16 ulp (2^-9 relative) plus fp32
    assert (np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-30).all()


@pytest.mark.parametrize("name", ["toy", "balanced", "finegrained", "invalid_ids", "all_dropped", "top32"])
def test_combine_matches_oracle(lib, name):
    wl = CASES[name]()
    run = G.DevicePipeline(wl, with_u=False).route()
    yh = W._normal_bf16(np.random.default_rng(7), (max(wl.n, 1), wl.d))
    y = G.dev_bf16(yh)
    out = torch.full((wl.T, wl.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    _lib.moe_unpermute_combine(y, run.inv_map, run.weights, wl.T, wl.k, wl.d, out)
    torch.cuda.synchronize()
    r = O.route_offsets(wl.ids, wl.E)
    want = O.combine(yh[: wl.n], r["inv_map"], wl.weights, wl.T, wl.k)
    got = G.host(out)
    if r["M"] == 0:
        assert not got.any()
    else:
        G.assert_close(got, want, f"combine[{name}]")


@pytest.mark.parametrize("k", [1, 2, 8])
def test_permute_then_combine_is_k_times_identity(lib, k):
    wl = W.custom(T=1000, k=k, E=13, d=264, h=8, seed=k)
    run = G.DevicePipeline(wl, with_u=False).route().permute()
    out = torch.empty(wl.T, wl.d, dtype=torch.bfloat16, device="cuda")
    _lib.moe_unpermute_combine(run.xp, run.inv_map, None, wl.T, k, wl.d, out)
    torch.cuda.synchronize()
    assert torch.equal(out, run.x * k)


@pytest.mark.slow
def test_route_permute_combine_at_the_slot_limit(lib):
    """T*top_k = 2^31 - 8, just below the header's limit of 2^31 slots (int32 indices): routing,
    the gather and the combine keep every index in range. Checked on the device: the counts
    against a direct count, the placement and the inverse map on a million sampled rows, the
    gathered rows bit for bit, and the combine of small integers (exact in bf16) against
    top_k * x. About 75 GB of device memory."""
    from ragged_grouped_gemm_device_gb300 import _lib as L
    k, E, d = 8, 4, 8
    T = (1 << 28) - 1
    n = T * k
    assert n == (1 << 31) - 8
    dev, i32 = "cuda", torch.int32
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    ids = torch.randint(0, E, (n,), dtype=i32, device=dev, generator=gen)
    counts, offsets = torch.empty(E, dtype=i32, device=dev), torch.empty(E, dtype=i32, device=dev)
    sorted_src, inv = torch.empty(n, dtype=i32, device=dev), torch.empty(n, dtype=i32, device=dev)
    ws = torch.empty(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), dtype=torch.uint8, device=dev)
    L.moe_route_offsets(ids, T, k, E, counts, offsets, sorted_src, inv, ws)
    ref_counts = torch.stack([(ids == e).sum() for e in range(E)])
    assert torch.equal(counts.long(), ref_counts)
    assert torch.equal(offsets.long(), ref_counts.cumsum(0)) and int(offsets[-1]) == n
    p = torch.randint(0, n, (1 << 20,), dtype=torch.int64, device=dev, generator=gen)
    p = torch.cat([p, torch.tensor([0, n - 2, n - 1], device=dev)])
    src = sorted_src[p].long()
    assert torch.equal(ids[src].long(), torch.searchsorted(offsets.long(), p, right=True))
    assert torch.equal(inv[src].long(), p)
    # stable placement: within a segment the slots keep increasing flat-index order
    q = p[p + 1 < n]
    same = torch.searchsorted(offsets.long(), q, right=True) == torch.searchsorted(offsets.long(), q + 1, right=True)
    assert (sorted_src[q[same]] < sorted_src[q[same] + 1]).all()
    del ids, ws
    x = torch.randint(-3, 4, (T, d), dtype=i32, device=dev, generator=gen).to(torch.bfloat16)
    xp = torch.empty(n, d, dtype=torch.bfloat16, device=dev)
    L.moe_permute(x, sorted_src, offsets, None, T, k, E, d, xp)
    assert torch.equal(xp[p], x[src // k])
    out = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    L.moe_unpermute_combine(xp, inv, None, T, k, d, out)
    assert torch.equal(out, x * k)
