"""ctypes binding of libmoe_gg.so (declared in include/moe_gg.h).

Argument marshalling only: each function takes torch tensors (or None for nullable pointers),
passes their device pointers and the current CUDA stream to the C entry point of the same name,
and raises MoEError on a non-OK status. Every step runs in the library's CUDA kernels; there is
no fallback of any kind, and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gg.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "libmoe_gg_debug.so")  # same ABI, built with MOE_GG_DEBUG
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe_gg.h")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
          3: "MOE_ERR_WORKSPACE_TOO_SMALL", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT",
          6: "MOE_ERR_UNSUPPORTED_DEVICE"}
MOE_DEV_TIMEOUT = 0x1
MOE_DEV_BAD_OFFSETS = 0x2
OP_ROUTE, OP_FWD, OP_BWD, OP_PADDED_BMM, OP_LOOP, OP_SAVED, OP_MX_WEIGHTS, OP_MX_FWD, OP_MX_BWD, OP_MX_ROW_SCALES = \
    range(10)

_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_PI32, _PI64 = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_longlong)
SIGNATURES = {
    "moe_workspace_bytes": (_S, [_I, _I, _I, _I, _I, _I, _I]),
    "moe_route_offsets": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P]),
    "moe_permute": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P]),
    "moe_grouped_swiglu_fwd": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _S, _P, _P]),
    "moe_grouped_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _S, _P,
                             _P]),
    "moe_unpermute_combine": (_I, [_P, _P, _P, _I, _I, _I, _P, _P]),
    "moe_padded_bmm_swiglu_fwd": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _S, _P, _P]),
    "moe_loop_swiglu_fwd": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_grouped_up_swiglu": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_grouped_down": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_grouped_down_dgrad_swiglu": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "moe_routing_weight_grad": (_I, [_P, _P, _I, _I, _I, _P, _P]),
    "moe_grouped_up_dgrad": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
    "moe_grouped_wgrad": (_I, [_P, _P, _I, _P, _I, _P, _I, _I, _P, _P, _P]),
    "moe_grouped_wgrad_dual": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _I, _P, _I, _P, _P, _I, _I, _P, _P]),
    "moe_mx_prepare_weights": (_I, [_P, _P, _I, _I, _I, _P, _S, _P]),
    "moe_mx_quantize_rows": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "moe_permute_mxfp8": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_grouped_swiglu_fwd_mxfp8": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _S, _P, _P]),
    "moe_grouped_bwd_mxfp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                   _S, _P, _P]),
    "moe_grouped_swiglu_fwd_top1_combine": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                                 _P]),
    "moe_route_offsets_noalloc": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_cuda_error": (ctypes.c_char_p, []),
    "moe_abi_version": (_I, []),
    "moe_debug_build": (_I, []),
    "moe_debug_report": (_I, [_PI32, _PI32, _PI64, _PI64, _I]),
    "moe_debug_site_name": (ctypes.c_char_p, [_I]),
}
MOE_DEBUG_CALL_ERROR_BIT = 30

_lib = None


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == 4 and _lib is not None:
            detail = ": " + _lib.moe_last_cuda_error().decode()
        super().__init__(f"{fn} returned {STATUS.get(status, status)}{detail}")


def header_functions(path: str = HEADER):
    """Names of the functions include/moe_gg.h declares."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def open_library(path: str):
    """A ctypes handle of a build of the library at `path`, every entry point declared."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run __graft_entry__.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load(path: str = None):
    """Load the library (once; the first call's path wins, so a process that wants the debug
    build calls load(DEBUG_LIB_PATH) before anything else) and return its handle. Without a
    path: the release build, or the debug build when MOE_GG_DEBUG_LIB=1 is set in the
    environment (to run a whole program or test suite with the debug build's bounds checks)."""
    global _lib
    if _lib is None:
        if path is None:
            path = DEBUG_LIB_PATH if os.environ.get("MOE_GG_DEBUG_LIB") == "1" else LIB_PATH
        _lib = open_library(path)
    return _lib


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def moe_workspace_bytes(op: int, T: int, top_k: int, E: int, d: int = 0, h: int = 0, capacity_C: int = 0) -> int:
    return int(load().moe_workspace_bytes(op, T, top_k, E, d, h, capacity_C))


def moe_route_offsets(ids, T, top_k, E, counts, offsets, sorted_src, inv_map, ws, stream=None):
    L = load()
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("moe_route_offsets", L.moe_route_offsets(_ptr(ids), T, top_k, E, _ptr(counts), _ptr(offsets),
                                                    _ptr(sorted_src), _ptr(inv_map), _ptr(ws), ws_bytes,
                                                    _stream(stream)))


def moe_route_offsets_noalloc(ids, T, top_k, E, counts, offsets, sorted_src, inv_map, stream=None):
    """moe_route_offsets without a workspace: for callers that cannot allocate device memory; the
    scratch is one fixed 1 MiB array inside the library (calls that overlap on the GPU race)."""
    _check("moe_route_offsets_noalloc", load().moe_route_offsets_noalloc(
        _ptr(ids), T, top_k, E, _ptr(counts), _ptr(offsets), _ptr(sorted_src), _ptr(inv_map), _stream(stream)))


def moe_permute(x, sorted_src, offsets, row_scale, T, top_k, E, d, xp, stream=None):
    _check("moe_permute", load().moe_permute(_ptr(x), _ptr(sorted_src), _ptr(offsets), _ptr(row_scale),
                                             T, top_k, E, d, _ptr(xp), _stream(stream)))


def moe_grouped_swiglu_fwd(xp, offsets, sorted_src, weights, E, cap, d, h, w_ug, w_down, y, a_save,
                           saved=None, ws=None, dev_status=None, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("moe_grouped_swiglu_fwd", load().moe_grouped_swiglu_fwd(
        _ptr(xp), _ptr(offsets), _ptr(sorted_src), _ptr(weights), E, cap, d, h, _ptr(w_ug), _ptr(w_down),
        _ptr(y), _ptr(a_save), _ptr(saved), _ptr(ws), ws_bytes, _ptr(dev_status), _stream(stream)))


def moe_grouped_bwd(dy, xp, a_save, saved, offsets, sorted_src, weights, E, cap, d, h, w_ug, w_down, dxp,
                    dw_ug, dw_down, ws, dev_status=None, stream=None, inv_map=None, dw_route=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("moe_grouped_bwd", load().moe_grouped_bwd(
        _ptr(dy), _ptr(xp), _ptr(a_save), _ptr(saved), _ptr(offsets), _ptr(sorted_src), _ptr(weights), E,
        cap, d, h, _ptr(w_ug),
        _ptr(w_down), _ptr(dxp), _ptr(dw_ug), _ptr(dw_down), _ptr(inv_map), _ptr(dw_route), _ptr(ws), ws_bytes,
        _ptr(dev_status), _stream(stream)))


def moe_grouped_up_swiglu(xp, offsets, sorted_src, weights, E, cap, d, h, w_ug, a_save, saved=None,
                          dev_status=None, stream=None):
    _check("moe_grouped_up_swiglu", load().moe_grouped_up_swiglu(
        _ptr(xp), _ptr(offsets), _ptr(sorted_src), _ptr(weights), E, cap, d, h, _ptr(w_ug), _ptr(a_save),
        _ptr(saved), _ptr(dev_status), _stream(stream)))


def moe_grouped_down(a, offsets, E, cap, d, h, w_down, y, dev_status=None, stream=None):
    _check("moe_grouped_down", load().moe_grouped_down(
        _ptr(a), _ptr(offsets), E, cap, d, h, _ptr(w_down), _ptr(y), _ptr(dev_status), _stream(stream)))


def moe_grouped_down_dgrad_swiglu(dy, saved, offsets, sorted_src, weights, E, cap, d, h, w_down, du_hi, du_lo,
                                  dev_status=None, stream=None, dw_part=None):
    _check("moe_grouped_down_dgrad_swiglu", load().moe_grouped_down_dgrad_swiglu(
        _ptr(dy), _ptr(saved), _ptr(offsets), _ptr(sorted_src), _ptr(weights), E, cap, d, h, _ptr(w_down),
        _ptr(du_hi), _ptr(du_lo), _ptr(dw_part), _ptr(dev_status), _stream(stream)))


def routing_grad_parts(h):
    """Partial sums per row the dgrad leaves for the routing-weight gradient: 2 ceil(h/256)."""
    return 2 * ((h + 255) // 256)


def moe_routing_weight_grad(dw_part, inv_map, T, top_k, h, dw_route, stream=None):
    _check("moe_routing_weight_grad", load().moe_routing_weight_grad(
        _ptr(dw_part), _ptr(inv_map), T, top_k, h, _ptr(dw_route), _stream(stream)))


def moe_grouped_up_dgrad(du_hi, offsets, E, cap, d, h, w_ug, dxp, dev_status=None, stream=None):
    _check("moe_grouped_up_dgrad", load().moe_grouped_up_dgrad(
        _ptr(du_hi), _ptr(offsets), E, cap, d, h, _ptr(w_ug), _ptr(dxp), _ptr(dev_status), _stream(stream)))


def moe_grouped_wgrad(p_hi, p_lo, p_cols, q, q_cols, offsets, E, cap, dw, dev_status=None, stream=None):
    _check("moe_grouped_wgrad", load().moe_grouped_wgrad(
        _ptr(p_hi), _ptr(p_lo), p_cols, _ptr(q), q_cols, _ptr(offsets), E, cap, _ptr(dw), _ptr(dev_status),
        _stream(stream)))


def moe_grouped_wgrad_dual(p1_hi, p1_lo, p1_cols, q1, q1_cols, dw1, p2_hi, p2_lo, p2_cols, q2, q2_cols, dw2,
                           offsets, E, cap, dev_status=None, stream=None):
    _check("moe_grouped_wgrad_dual", load().moe_grouped_wgrad_dual(
        _ptr(p1_hi), _ptr(p1_lo), p1_cols, _ptr(q1), q1_cols, _ptr(dw1), _ptr(p2_hi), _ptr(p2_lo), p2_cols,
        _ptr(q2), q2_cols, _ptr(dw2), _ptr(offsets), E, cap, _ptr(dev_status), _stream(stream)))


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def moe_mx_prepare_weights(w_ug, w_down, E, d, h, mxw, stream=None):
    _check("moe_mx_prepare_weights", load().moe_mx_prepare_weights(
        _ptr(w_ug), _ptr(w_down), E, d, h, _ptr(mxw), _nbytes(mxw), _stream(stream)))


def moe_permute_mxfp8(x, sorted_src, offsets, T, top_k, E, d, xp, q, sf, dev_status=None, stream=None):
    _check("moe_permute_mxfp8", load().moe_permute_mxfp8(
        _ptr(x), _ptr(sorted_src), _ptr(offsets), T, top_k, E, d, _ptr(xp), _ptr(q), _ptr(sf), _ptr(dev_status),
        _stream(stream)))


def moe_mx_quantize_rows(x, offsets, E, cap, K, q, sf, dev_status=None, stream=None):
    _check("moe_mx_quantize_rows", load().moe_mx_quantize_rows(
        _ptr(x), _ptr(offsets), E, cap, K, _ptr(q), _ptr(sf), _ptr(dev_status), _stream(stream)))


def moe_grouped_swiglu_fwd_mxfp8(xp, offsets, sorted_src, weights, E, cap, d, h, mxw, y, a_save, saved, ws,
                                 dev_status=None, stream=None, xq=None, xsf=None):
    _check("moe_grouped_swiglu_fwd_mxfp8", load().moe_grouped_swiglu_fwd_mxfp8(
        _ptr(xp), _ptr(xq), _ptr(xsf), _ptr(offsets), _ptr(sorted_src), _ptr(weights), E, cap, d, h, _ptr(mxw), _ptr(y), _ptr(a_save),
        _ptr(saved), _ptr(ws), _nbytes(ws), _ptr(dev_status), _stream(stream)))


def moe_grouped_bwd_mxfp8(dy, xp, a_save, saved, offsets, sorted_src, weights, E, cap, d, h, mxw, dxp, dw_ug,
                          dw_down, ws, dev_status=None, stream=None, inv_map=None, dw_route=None, dyq=None, dysf=None):
    _check("moe_grouped_bwd_mxfp8", load().moe_grouped_bwd_mxfp8(
        _ptr(dy), _ptr(dyq), _ptr(dysf), _ptr(xp), _ptr(a_save), _ptr(saved), _ptr(offsets), _ptr(sorted_src), _ptr(weights), E, cap, d,
        h, _ptr(mxw), _ptr(dxp), _ptr(dw_ug), _ptr(dw_down), _ptr(inv_map), _ptr(dw_route), _ptr(ws), _nbytes(ws),
        _ptr(dev_status), _stream(stream)))


def saved_views(saved, cap, h):
    """The parts of the forward's `saved` buffer (a contiguous tensor of any dtype, read as bytes):
    the low half of P = w*A (bf16 [cap, h8]; the high half is a_save) at byte 0, then U rounded to
    24 bits in the kernels' blocked layout (a flat byte view; see the header for the block
    order). h8 = h rounded up to a multiple of 8: widths that are not are stored zero-padded."""
    import torch
    saved = saved.reshape(-1).view(torch.uint8)
    h = (h + 7) // 8 * 8
    pb = cap * h * 2
    off = (pb + 255) // 256 * 256
    p_lo = saved[:pb].view(torch.bfloat16).view(cap, h)
    u = saved[off:]
    return u, p_lo


def moe_unpermute_combine(y, inv_map, weights, T, top_k, d, out, stream=None):
    _check("moe_unpermute_combine", load().moe_unpermute_combine(
        _ptr(y), _ptr(inv_map), _ptr(weights), T, top_k, d, _ptr(out), _stream(stream)))


def moe_grouped_swiglu_fwd_top1_combine(xp, offsets, sorted_src, inv_map, weights, E, T, d, h, w_ug, w_down, out,
                                        a_save, saved=None, dev_status=None, stream=None):
    _check("moe_grouped_swiglu_fwd_top1_combine", load().moe_grouped_swiglu_fwd_top1_combine(
        _ptr(xp), _ptr(offsets), _ptr(sorted_src), _ptr(inv_map), _ptr(weights), E, T, d, h, _ptr(w_ug),
        _ptr(w_down), _ptr(out), _ptr(a_save), _ptr(saved), _ptr(dev_status), _stream(stream)))


def moe_padded_bmm_swiglu_fwd(xp, offsets, E, cap, d, h, capacity_C, w_ug, w_down, y, ws,
                              dev_status=None, stream=None):
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check("moe_padded_bmm_swiglu_fwd", load().moe_padded_bmm_swiglu_fwd(
        _ptr(xp), _ptr(offsets), E, cap, d, h, capacity_C, _ptr(w_ug), _ptr(w_down), _ptr(y), _ptr(ws),
        ws_bytes, _ptr(dev_status), _stream(stream)))


def moe_loop_swiglu_fwd(xp, offsets, E, cap, d, h, w_ug, w_down, y, a_save, saved=None, dev_status=None,
                        stream=None):
    _check("moe_loop_swiglu_fwd", load().moe_loop_swiglu_fwd(
        _ptr(xp), _ptr(offsets), E, cap, d, h, _ptr(w_ug), _ptr(w_down), _ptr(y), _ptr(a_save),
        _ptr(saved), _ptr(dev_status), _stream(stream)))


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_abi_version() -> int:
    return int(load().moe_abi_version())


def moe_debug_build() -> bool:
    return bool(load().moe_debug_build())


def moe_debug_report(reset: bool = True, lib=None):
    """(site_mask, first_site, index, limit) of the debug build's bounds checks since the last
    reset (waits for the device); (0, -1, 0, 0) from a release build."""
    L = lib if lib is not None else load()
    m, s, i, l = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_longlong(), ctypes.c_longlong()
    _check("moe_debug_report", L.moe_debug_report(ctypes.byref(m), ctypes.byref(s), ctypes.byref(i),
                                                  ctypes.byref(l), int(reset)))
    return m.value, s.value, i.value, l.value


def moe_debug_site_name(site: int) -> str:
    return load().moe_debug_site_name(site).decode()
