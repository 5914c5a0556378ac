"""A wait bound that runs out becomes MOE_DEV_TIMEOUT in the caller's status word, not a hung GPU.

A child process sets MOE_GG_WAIT_TIMEOUT_NS to 1 ns, far below any wait of a real tile, so
the first wait of every grouped kernel that is not satisfied at its first try runs out. The kernel
raises its abort flag, every role leaves its loop, the teardown waits (bounded separately, by
seconds) let in-flight copies and MMAs finish, tensor memory is freed and the kernel returns.
The test checks the status bit, that the whole layer returned within a bounded time, and that
the CUDA context still runs ordinary work afterwards."""
import os
import subprocess
import sys
import time

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from ragged_grouped_gemm_device_gb300 import workloads as W
from ragged_grouped_gemm_device_gb300.layer import ExpertLayer

wl = W.custom(T=1024, k=4, E=8, d=1024, h=512, seed=3)  # 16 K blocks per up/gate tile
bf = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).cuda()
layer = ExpertLayer(bf(wl.w_ug_all()), bf(wl.w_down_all()))
layer.forward(bf(wl.x()), torch.from_numpy(wl.ids).cuda(), torch.from_numpy(wl.weights).cuda())
layer.backward(bf(wl.dout()))
torch.cuda.synchronize()
status = layer.status.item()
check = (torch.ones(4096, device="cuda") * 2).sum().item()  # the context is still usable
print("STATUS", status, "CHECK", check, flush=True)
"""


def test_expired_wait_bound_reports_timeout_and_returns(lib):
    from ragged_grouped_gemm_device_gb300 import _lib
    env = dict(os.environ, MOE_GG_WAIT_TIMEOUT_NS="1")
    t0 = time.monotonic()
    res = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True,
                         timeout=300)
    elapsed = time.monotonic() - t0
    assert res.returncode == 0, res.stderr[-2000:]
    line = [ln for ln in res.stdout.splitlines() if ln.startswith("STATUS")][-1].split()
    status, check = int(line[1]), float(line[3])
    assert status & _lib.MOE_DEV_TIMEOUT, f"status {status}: no wait ran out"
    assert check == 8192.0
    # six grouped launches, each bounded by its teardown waits (seconds), plus process start-up
    assert elapsed < 240, f"took {elapsed:.0f} s"


CHILD_MX = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
from ragged_grouped_gemm_device_gb300 import _lib as L
from ragged_grouped_gemm_device_gb300 import workloads as W

wl = W.custom(T=1024, k=4, E=8, d=1024, h=512, seed=3)
T, k, E, d, h, n = wl.T, wl.k, wl.E, wl.d, wl.h, wl.n
bf = lambda a: torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).cuda()
dev, i32, u8 = "cuda", torch.int32, torch.uint8
st = torch.zeros(1, dtype=i32, device=dev)
counts, offs = torch.empty(E, dtype=i32, device=dev), torch.empty(E, dtype=i32, device=dev)
ss, inv = torch.empty(n, dtype=i32, device=dev), torch.empty(n, dtype=i32, device=dev)
rws = torch.empty(L.moe_workspace_bytes(L.OP_ROUTE, T, k, E), dtype=u8, device=dev)
L.moe_route_offsets(torch.from_numpy(wl.ids).cuda(), T, k, E, counts, offs, ss, inv, rws)
mxw = torch.empty(L.moe_workspace_bytes(L.OP_MX_WEIGHTS, T, k, E, d, h), dtype=u8, device=dev)
L.moe_mx_prepare_weights(bf(wl.w_ug_all()), bf(wl.w_down_all()), E, d, h, mxw)
sfb = L.moe_workspace_bytes(L.OP_MX_ROW_SCALES, T, k, E, d, h)
xp, xq, xsf = torch.empty(n, d, dtype=torch.bfloat16, device=dev), torch.empty(n, d, dtype=u8, device=dev), torch.empty(sfb, dtype=u8, device=dev)
L.moe_permute_mxfp8(bf(wl.x()), ss, offs, T, k, E, d, xp, xq, xsf, st)
y, a = torch.empty(n, d, dtype=torch.bfloat16, device=dev), torch.empty(n, h, dtype=torch.bfloat16, device=dev)
sv = torch.empty(L.moe_workspace_bytes(L.OP_SAVED, T, k, E, d, h), dtype=u8, device=dev)
fws = torch.empty(L.moe_workspace_bytes(L.OP_MX_FWD, T, k, E, d, h), dtype=u8, device=dev)
L.moe_grouped_swiglu_fwd_mxfp8(None, offs, None, None, E, n, d, h, mxw, y, a, sv, fws, st, xq=xq, xsf=xsf)
dy = bf(wl.dy(n))
dxp = torch.empty(n, d, dtype=torch.bfloat16, device=dev)
dwu, dwd = torch.empty(E, 2 * h, d, device=dev), torch.empty(E, h, d, device=dev)
bws = torch.empty(L.moe_workspace_bytes(L.OP_MX_BWD, T, k, E, d, h), dtype=u8, device=dev)
L.moe_grouped_bwd_mxfp8(dy, xp, a, sv, offs, None, None, E, n, d, h, mxw, dxp, dwu, dwd, bws, st)
torch.cuda.synchronize()
check = (torch.ones(4096, device="cuda") * 2).sum().item()
print("STATUS", st.item(), "CHECK", check, flush=True)
"""


def test_expired_wait_bound_in_the_mxfp8_kernels(lib):
    """The block-scaled kernels (scale copies to tensor memory and scaled MMAs in flight) leave
    through the same bounded teardown when a wait runs out."""
    from ragged_grouped_gemm_device_gb300 import _lib
    env = dict(os.environ, MOE_GG_WAIT_TIMEOUT_NS="1")
    t0 = time.monotonic()
    res = subprocess.run([sys.executable, "-c", CHILD_MX, ROOT], env=env, capture_output=True, text=True,
                         timeout=300)
    elapsed = time.monotonic() - t0
    assert res.returncode == 0, res.stderr[-2000:]
    line = [ln for ln in res.stdout.splitlines() if ln.startswith("STATUS")][-1].split()
    status, check = int(line[1]), float(line[3])
    assert status & _lib.MOE_DEV_TIMEOUT, f"status {status}: no wait ran out"
    assert check == 8192.0
    assert elapsed < 240, f"took {elapsed:.0f} s"
