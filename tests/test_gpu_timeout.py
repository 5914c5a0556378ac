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
