"""One SwiGLU expert layer driven through the C ABI: route -> permute -> grouped forward ->
combine, and the backward pass. PyTorch only allocates device memory and supplies the stream;
every step is a library kernel. Buffers are allocated once per shape and reused, so repeated
calls with new routing allocate nothing ("Section 09: Grouped GEMM" §9.4: fixed physical
shapes, unpadded compute)."""
from __future__ import annotations

import torch

from . import _lib


def _dense(t: torch.Tensor) -> torch.Tensor:
    """The library reads row-major contiguous rows. A view with other strides -- notably the
    zero-stride gradient a scalar loss broadcasts back (`out.sum().backward()` hands over an
    expanded [T, d] tensor with strides (0, 0)), which "Grouped expert GEMM" lists as an edge case
    of the grouped GEMM's backward -- is materialised once here; dense tensors pass through."""
    return t if t.is_contiguous() else t.contiguous()


class ExpertLayer:
    """Holds the expert weights W_ug [E, 2h, d] and W_down [E, h, d] (bf16, on the device)."""

    def __init__(self, w_ug: torch.Tensor, w_down: torch.Tensor):
        E, two_h, d = w_ug.shape
        assert w_down.shape == (E, two_h // 2, d)
        assert w_ug.dtype == torch.bfloat16 and w_down.dtype == torch.bfloat16
        self.E, self.d, self.h = E, d, two_h // 2
        self.w_ug, self.w_down = w_ug.contiguous(), w_down.contiguous()
        self.device = w_ug.device
        self._key = None
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def _buffers(self, T: int, k: int):
        if self._key == (T, k):
            return
        dev, E, d, h, n = self.device, self.E, self.d, self.h, T * k
        i32, bf = torch.int32, torch.bfloat16
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E, dtype=i32, device=dev)
        self.sorted_src = torch.empty(max(n, 1), dtype=i32, device=dev)
        self.inv_map = torch.empty(max(n, 1), dtype=i32, device=dev)
        rw = _lib.moe_workspace_bytes(_lib.OP_ROUTE, T, k, E, d, h)
        self.route_ws = torch.empty(max(rw, 1), dtype=torch.uint8, device=dev)
        self.xp = torch.empty(max(n, 1), d, dtype=bf, device=dev)
        self.y = torch.empty(max(n, 1), d, dtype=bf, device=dev)
        self.a = torch.empty(max(n, 1), h, dtype=bf, device=dev)
        sv = _lib.moe_workspace_bytes(_lib.OP_SAVED, T, k, E, d, h)
        self.saved = torch.empty(max(sv, 1), dtype=torch.uint8, device=dev)
        self.out = torch.empty(T, d, dtype=bf, device=dev)
        self.dy = torch.empty(max(n, 1), d, dtype=bf, device=dev)
        self.dxp = torch.empty(max(n, 1), d, dtype=bf, device=dev)
        self.dx = torch.empty(T, d, dtype=bf, device=dev)
        self.dw_ug = torch.empty(E, 2 * h, d, dtype=torch.float32, device=dev)
        self.dw_down = torch.empty(E, h, d, dtype=torch.float32, device=dev)
        self.dw_route = torch.empty(T, k, dtype=torch.float32, device=dev)
        fw = _lib.moe_workspace_bytes(_lib.OP_FWD, T, k, E, d, h)
        self.fwd_ws = torch.empty(fw, dtype=torch.uint8, device=dev) if fw > 0 else None
        bw = _lib.moe_workspace_bytes(_lib.OP_BWD, T, k, E, d, h)
        self.bwd_ws = torch.empty(max(bw, 1), dtype=torch.uint8, device=dev)
        self._key = (T, k)

    def forward(self, x: torch.Tensor, ids: torch.Tensor, weights: torch.Tensor, stream=None):
        """x [T, d] bf16, ids [T, k] int32, weights [T, k] fp32 -> out [T, d] bf16."""
        x, ids, weights = _dense(x), _dense(ids), _dense(weights)
        T, k = ids.shape
        self._buffers(T, k)
        self.T, self.k, self.weights = T, k, weights
        E, d, h, n = self.E, self.d, self.h, T * k
        _lib.moe_route_offsets(ids, T, k, E, self.counts, self.offsets, self.sorted_src, self.inv_map,
                               self.route_ws, stream)
        _lib.moe_permute(x, self.sorted_src, self.offsets, None, T, k, E, d, self.xp, stream)
        if k == 1 and d % 8 == 0 and h % 8 == 0:
            # one slot per token: the down projection writes the token rows itself (no y, no
            # combine pass); the routing weight is folded into the SwiGLU output
            _lib.moe_grouped_swiglu_fwd_top1_combine(self.xp, self.offsets, self.sorted_src, self.inv_map, weights,
                                                     E, T, d, h, self.w_ug, self.w_down, self.out, self.a,
                                                     self.saved, self.status, stream)
            return self.out
        # the routing weight is applied in the up/gate projection's epilogue; the combine sums
        _lib.moe_grouped_swiglu_fwd(self.xp, self.offsets, self.sorted_src, weights, E, n, d, h, self.w_ug,
                                    self.w_down, self.y, self.a, self.saved, self.fwd_ws, self.status, stream)
        _lib.moe_unpermute_combine(self.y, self.inv_map, None, T, k, d, self.out, stream)
        return self.out

    def backward(self, dout: torch.Tensor, stream=None):
        """dout [T, d] bf16 -> (dx [T, d] bf16, dW_ug [E, 2h, d] fp32, dW_down [E, h, d] fp32,
        d_weights [T, k] fp32: the gradient of the routing weights, 0 for dropped slots)."""
        T, k, E, d, h, n = self.T, self.k, self.E, self.d, self.h, self.T * self.k
        dout = _dense(dout)
        _lib.moe_permute(dout, self.sorted_src, self.offsets, None, T, k, E, d, self.dy, stream)
        _lib.moe_grouped_bwd(self.dy, self.xp, self.a, self.saved, self.offsets, self.sorted_src, self.weights,
                             E, n, d, h, self.w_ug,
                             self.w_down, self.dxp, self.dw_ug, self.dw_down, self.bwd_ws, self.status,
                             stream, inv_map=self.inv_map, dw_route=self.dw_route)
        _lib.moe_unpermute_combine(self.dxp, self.inv_map, None, T, k, d, self.dx, stream)
        return self.dx, self.dw_ug, self.dw_down, self.dw_route
