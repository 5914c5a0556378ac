"""The routing entry point that allocates nothing.

moe_route_offsets_noalloc serves callers that cannot hand the library a device workspace (code
where cudaMalloc is not allowed or not safe, or a binding with no device allocator): its
scratch is one fixed array inside the library. Here it is called through the C ABI and its
outputs are compared with moe_route_offsets (which uses a caller workspace). Routing results are
integers, so the tolerance is bit-exact. Problems of different shapes are routed one after the
other (and the first again), so that contents the shared array keeps from an earlier call
cannot leak into a later one. The edge cases are no slots at all, the largest expert count,
and the largest problem the array holds, next to one a warp chunk larger, which is refused.
This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import gpu_util as G
from ragged_grouped_gemm_device_gb300 import _lib
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SCRATCH = 1 << 20  # MOE_NOALLOC_ROUTE_SCRATCH_BYTES


def _scratch_bytes(T, k, E):
    return -(-(T * k) // 256) * E * 4


def _route(wl, noalloc):
    run = G.DevicePipeline(wl, with_u=False)
    if noalloc:
        _lib.moe_route_offsets_noalloc(run.ids, wl.T, wl.k, wl.E, run.counts, run.offsets, run.sorted_src,
                                       run.inv_map)
    else:
        run.route()
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (run.counts, run.offsets, run.sorted_src[: wl.n], run.inv_map[: wl.n])]


def test_noalloc_route_matches_workspace_route_on_consecutive_calls(lib):
    cases = [W.make("large"),  # 131072 slots, 256 experts: 512 KiB of scratch
             W.custom(T=1000, k=4, E=37, d=16, h=8, seed=1, invalid_frac=0.1, empty_experts=(3, 5)),
             # no slots: counts and offsets are zero
             W.custom(T=0, k=4, E=11, d=16, h=8, seed=2),
             # the largest expert count, a few tokens (most experts empty)
             W.custom(T=300, k=8, E=1024, d=16, h=8, seed=3, invalid_frac=0.02),
             # exactly the array's size: ceil(65536 / 256) warps x 1024 experts x 4 bytes = 1 MiB
             W.custom(T=8192, k=8, E=1024, d=16, h=8, seed=4),
             W.make("large")]
    assert _scratch_bytes(8192, 8, 1024) == SCRATCH
    for wl in cases:
        want = _route(wl, noalloc=False)
        got = _route(wl, noalloc=True)
        for g, w in zip(got, want):
            assert np.array_equal(g, w)
        if wl.T == 0:
            assert not got[0].any() and not got[1].any()


def test_noalloc_route_rejects_problems_beyond_its_scratch(lib):
    dummy = torch.empty(1, dtype=torch.int32, device="cuda")
    call = lambda T, k, E: _lib.load().moe_route_offsets_noalloc(
        _lib._ptr(dummy), T, k, E, _lib._ptr(dummy), _lib._ptr(dummy), _lib._ptr(dummy), _lib._ptr(dummy), None)
    # one slot past the 1 MiB problem needs a 257th warp chunk: refused before any launch
    assert _scratch_bytes(8193, 8, 1024) > SCRATCH
    assert call(8193, 8, 1024) == 3  # MOE_ERR_WORKSPACE_TOO_SMALL
    # ceil(262144 / 256) warps x 1024 experts x 4 bytes = 4 MiB
    assert call(32768, 8, 1024) == 3
