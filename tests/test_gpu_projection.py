"""GPU parity of one square grouped expert projection at the shape of the capacity and
load-histogram studies ("Section 09: Grouped GEMM", Figs. 38 and 40: 16 experts, d = h = 4096):
sampled rows against the fp64 oracle, and the capacity-padded layout (the same kernel over a
uniform problem list) bit-identical to the exact-row grouped result on every valid row."""
import numpy as np
import pytest
import torch

import gpu_util as G
from oracle import moe_oracle as O
from ragged_grouped_gemm_device_gb300 import _lib as L
from ragged_grouped_gemm_device_gb300 import workloads as W

pytestmark = pytest.mark.gpu

E, K, N, M = 16, 4096, 4096, 8192


@pytest.fixture(scope="module")
def proj():
    # a concentrated histogram (8-row aligned, one 128-row tile at least per expert)
    hists = W.dirichlet_histograms(M=M, E=E, n_bins=3, per_bin=1, seed=3)
    counts = hists[-1][0]
    w_host = [W.projection_weight(e, K, N) for e in range(E)]
    w = torch.stack([torch.from_numpy(a) for a in w_host]).to(torch.bfloat16).cuda()
    x_host = W.projection_x(M, K)
    return counts, x_host, w_host, w


def test_square_projection_sampled_rows_match_oracle(lib, proj):
    counts, x_host, w_host, w = proj
    offsets = np.cumsum(counts).astype(np.int32)
    x = G.dev_bf16(x_host)
    y = G.nan_filled((M, N))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.moe_grouped_down(x, G.dev_i32(offsets), E, M, N, K, w, y, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = G.host(y)
    starts = np.concatenate([[0], offsets[:-1]])
    rng = np.random.default_rng(5)
    rows, want = [], []
    for e in range(E):
        s, t = int(starts[e]), int(offsets[e])
        pick = sorted({s, t - 1, *rng.integers(s, t, 2).tolist()})
        seg = O.grouped_linear(x_host[pick], np.array([len(pick)]), lambda i, e=e: w_host[e])
        rows += pick
        want.append(seg)
    G.assert_close(got[rows], np.concatenate(want), "square projection")


def test_padded_layout_equals_grouped_rows(lib, proj):
    counts, x_host, _, w = proj
    offsets = np.cumsum(counts).astype(np.int32)
    starts = np.concatenate([[0], offsets[:-1]])
    x = G.dev_bf16(x_host)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = G.nan_filled((M, N))
    L.moe_grouped_down(x, G.dev_i32(offsets), E, M, N, K, w, y, status)
    # capacity layout: every expert's rows, then zero rows, up to C = max count
    C = int(counts.max())
    xpad = torch.zeros(E * C, K, dtype=torch.bfloat16, device="cuda")
    for e in range(E):
        xpad[e * C:e * C + int(counts[e])] = x[int(starts[e]):int(offsets[e])]
    ypad = G.nan_filled((E * C, N))
    uoffs = torch.arange(1, E + 1, dtype=torch.int32, device="cuda") * C
    L.moe_grouped_down(xpad, uoffs, E, E * C, N, K, w, ypad, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    for e in range(E):
        c = int(counts[e])
        assert torch.equal(ypad[e * C:e * C + c], y[int(starts[e]):int(offsets[e])])
        assert not ypad[e * C + c:(e + 1) * C].any()


def test_column_partition_equals_dense_product(lib):
    """Eq. 17 (Fig. 39's split): E expert GEMMs over the column blocks of one weight, each fed the
    same rows, reproduce the dense product; checked against the oracle's dense fp64 product."""
    T, K, N, E = 96, 512, 2048, 4
    x_host = W.projection_x(T, K, seed=7)
    w_host = W.projection_weight(0, K, N, seed=7)
    w = torch.from_numpy(w_host).to(torch.bfloat16).cuda()
    wg = w.view(K, E, N // E).permute(1, 0, 2).contiguous()
    xr = G.dev_bf16(x_host).repeat(E, 1)
    yg = G.nan_filled((E * T, N // E))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    offs = torch.arange(1, E + 1, dtype=torch.int32, device="cuda") * T
    L.moe_grouped_down(xr, offs, E, E * T, N // E, K, wg, yg, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    got = G.host(yg).reshape(E, T, N // E).transpose(1, 0, 2).reshape(T, N)
    want = O.grouped_linear(x_host, np.array([T]), lambda e: w_host)
    G.assert_close(got, want, "column partition")
