"""CPU-only checks of the C-ABI library: it builds for sm_103a, loads, exports every function the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes

import pytest

from ragged_grouped_gemm_device_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_functions_all_exported(lib):
    names = _lib.header_functions()
    assert "moe_grouped_swiglu_fwd" in names and len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"


def test_abi_version_and_status_strings(lib):
    assert lib.moe_abi_version() == 2
    for code in _lib.STATUS:
        assert lib.moe_status_string(code)
    assert b"unknown" in lib.moe_status_string(99)


def test_workspace_sizes_are_host_arithmetic(lib):
    # route: one int32 per (warp chunk of 256 slots, expert), rounded to 256 bytes
    assert _lib.moe_workspace_bytes(_lib.OP_ROUTE, 16384, 8, 256) == (16384 * 8 // 256) * 256 * 4
    assert _lib.moe_workspace_bytes(_lib.OP_FWD, 16384, 8, 256, 2048, 512) == 0
    # odd pitches: zero-padded copies (xp, y [n, d8], a [n, h8], W_ug [E, 2 h8, d8], W_down
    # [E, h8, d8]), each rounded to 256 bytes
    r256 = lambda b: (b + 255) // 256 * 256
    n, E, d8, h8 = 10 * 3, 6, 64, 48
    assert _lib.moe_workspace_bytes(_lib.OP_FWD, 10, 3, E, 60, 44) == \
        2 * r256(n * d8 * 2) + r256(n * h8 * 2) + r256(E * 2 * h8 * d8 * 2) + r256(E * h8 * d8 * 2)
    assert _lib.moe_workspace_bytes(_lib.OP_SAVED, 10, 3, E, 60, 44) == \
        _lib.moe_workspace_bytes(_lib.OP_SAVED, 10, 3, E, 64, 48)
    # backward: dU high and low halves, [n, 2h] bf16 each, then the routing-gradient partials,
    # [n, 2 ceil(h/256)] fp32
    assert _lib.moe_workspace_bytes(_lib.OP_BWD, 16384, 8, 256, 2048, 512) == \
        2 * 16384 * 8 * 1024 * 2 + 16384 * 8 * 4 * 4
    assert _lib.routing_grad_parts(512) == 4 and _lib.routing_grad_parts(1000) == 8
    # saved state: the low bf16 half of P [n, h], then U at 24 bits in 1536-byte blocks (32 rows
    # x 16 columns x 3 bytes) for each of at most (n + 127 E) / 128 row tiles, 4 lane quadrants and
    # 2 ceil(h/16) column chunks
    n = 16384 * 8
    tiles = (n + 127 * 256) // 128
    assert tiles == 1278
    assert _lib.moe_workspace_bytes(_lib.OP_SAVED, 16384, 8, 256, 2048, 512) == n * 512 * 2 + tiles * 4 * 64 * 1536
    tiles = (20000 + 127 * 64) // 128  # h = 1000: 63 chunks per half, the last one partial
    assert _lib.moe_workspace_bytes(_lib.OP_SAVED, 20000, 1, 64, 1000, 1000) == 20000 * 1000 * 2 + tiles * 4 * 126 * 1536
    bmm = _lib.moe_workspace_bytes(_lib.OP_PADDED_BMM, 10, 1, 4, 64, 128, 4)
    assert bmm == 2 * (16 * 64 * 2) + 16 * 128 * 2  # [16, 64] bf16 x2 and [16, 128] bf16
    assert _lib.moe_workspace_bytes(_lib.OP_ROUTE, 10, 1, 0) == 0      # invalid E
    assert _lib.moe_workspace_bytes(_lib.OP_ROUTE, 10, 33, 4) == 0     # top_k above 32


def test_invalid_arguments_rejected_before_any_cuda_call(lib):
    p = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    INVALID, SHAPE, WS = 1, 2, 3
    assert lib.moe_route_offsets(p, 10, 1, 0, p, p, p, p, p, 1 << 20, None) == SHAPE      # E = 0
    assert lib.moe_route_offsets(p, 10, 1, 2000, p, p, p, p, p, 1 << 20, None) == SHAPE   # E > 1024
    assert lib.moe_route_offsets(p, -1, 1, 4, p, p, p, p, p, 1 << 20, None) == INVALID
    assert lib.moe_route_offsets(p, 10, 1, 4, None, p, p, p, p, 1 << 20, None) == INVALID
    assert lib.moe_route_offsets(p, 100000, 8, 256, p, p, p, p, p, 16, None) == WS
    assert lib.moe_permute(p, p, p, None, 10, 1, 4, (1 << 20) + 8, p, None) == SHAPE      # d too wide
    assert lib.moe_permute(p, p, p, None, 10, 1, 4, 0, p, None) == INVALID                 # d = 0
    assert lib.moe_permute(ctypes.c_void_p(18), p, p, None, 10, 1, 4, 16, p, None) == INVALID  # misaligned
    fwd = lib.moe_grouped_swiglu_fwd
    # h % 8 != 0: run on zero-padded copies, which need the forward workspace
    assert fwd(p, p, None, None, 4, 10, 64, 100, p, p, p, p, None, None, 0, None, None) == WS
    assert lib.moe_grouped_up_swiglu(p, p, None, None, 4, 10, 64, 100, p, p, None, None, None) == SHAPE
    assert fwd(p, p, None, None, 4, 10, 64, 128, p, p, p, None, None, None, 0, None, None) == INVALID  # a_save
    assert fwd(p, p, None, None, 4, -1, 64, 128, p, p, p, p, None, None, 0, None, None) == INVALID
    assert fwd(p, p, None, p, 4, 10, 64, 128, p, p, p, p, None, None, 0, None, None) == INVALID  # weights w/o src
    bwd = lib.moe_grouped_bwd
    assert bwd(p, p, p, p, p, None, None, 4, 10, 64, 128, p, p, p, p, p, None, None, p, 0, None, None) == WS
    assert bwd(p, p, p, None, p, None, None, 4, 10, 64, 128, p, p, p, p, p, None, None, p, 1 << 20, None,
               None) == INVALID
    # dw_route without inv_map; a workspace large enough for dU but not for the partials
    assert bwd(p, p, p, p, p, None, None, 4, 10, 64, 128, p, p, p, p, p, None, p, p, 1 << 20, None,
               None) == INVALID
    need = _lib.moe_workspace_bytes(_lib.OP_BWD, 10, 1, 4, 64, 128)
    assert bwd(p, p, p, p, p, None, None, 4, 10, 64, 128, p, p, p, p, p, p, p, p, need - 256, None,
               None) == WS
    rwg = lib.moe_routing_weight_grad
    assert rwg(p, p, 10, 0, 128, p, None) == INVALID                                       # top_k = 0
    assert rwg(p, p, 10, 40, 128, p, None) == SHAPE                                        # top_k > 32
    assert rwg(None, p, 10, 2, 128, p, None) == INVALID
    assert rwg(None, None, 0, 2, 128, None, None) == 0                                     # no slots: no-op
    assert lib.moe_grouped_wgrad(p, None, 12, p, 64, p, 4, 10, p, None, None) == SHAPE        # p_cols % 8
    assert lib.moe_grouped_up_dgrad(p, p, 0, 10, 64, 128, p, p, None, None) == INVALID       # E = 0
    assert lib.moe_unpermute_combine(p, p, None, 10, 40, 64, p, None) == SHAPE            # top_k > 32
    assert lib.moe_padded_bmm_swiglu_fwd(p, p, 4, 10, 64, 128, 0, p, p, p, p, 1 << 20, None, None) == INVALID
    assert lib.moe_padded_bmm_swiglu_fwd(p, p, 4, 10, 64, 128, 4, p, p, p, p, 16, None, None) == WS
    assert lib.moe_loop_swiglu_fwd(p, p, 4, 10, 64, 128, p, p, None, None, p, None, None) == INVALID
    # the two wgrads of one launch must agree on the low half
    assert lib.moe_grouped_wgrad_dual(p, p, 64, p, 64, p, p, None, 64, p, 64, p, p, 4, 10, None, None) == INVALID
    # MXFP8: d a multiple of 32, h of 128; 256-byte aligned prepared weights and workspace
    p256 = ctypes.c_void_p(256)
    mxf = lambda *a: lib.moe_grouped_swiglu_fwd_mxfp8(a[0], None, None, *a[1:])
    assert mxf(p, p, None, None, 4, 10, 64, 96, p256, p, p, None, p256, 1 << 30, None, None) == SHAPE   # h % 128
    assert mxf(p, p, None, None, 4, 10, 48, 128, p256, p, p, None, p256, 1 << 30, None, None) == SHAPE  # d % 32
    assert mxf(p, p, None, None, 4, 10, 64, 128, p, p, p, None, p256, 1 << 30, None, None) == INVALID   # mxw align
    need = _lib.moe_workspace_bytes(_lib.OP_MX_FWD, 10, 1, 4, 64, 128)
    assert need > 0 and mxf(p, p, None, None, 4, 10, 64, 128, p256, p, p, None, p256, need - 1, None, None) == WS
    # codes without their scales, or neither xp nor codes
    assert lib.moe_grouped_swiglu_fwd_mxfp8(None, p, None, p, None, None, 4, 10, 64, 128, p256, p, p, None, p256,
                                            1 << 30, None, None) == INVALID
    assert lib.moe_grouped_swiglu_fwd_mxfp8(None, None, None, p, None, None, 4, 10, 64, 128, p256, p, p, None, p256,
                                            1 << 30, None, None) == INVALID
    assert lib.moe_permute_mxfp8(p, p, p, 10, 1, 4, 40, None, p, p, None, None) == SHAPE               # d % 32
    assert lib.moe_mx_prepare_weights(p, p, 4, 64, 128, p256, 16, None) == WS
    assert lib.moe_mx_quantize_rows(p, p, 4, 10, 40, p, p, None, None) == SHAPE                     # K % 32
    mxb = lib.moe_grouped_bwd_mxfp8
    assert mxb(p, None, None, p, p, None, p, None, None, 4, 10, 64, 128, p256, p, p, p, None, None, p256, 1 << 30,
               None, None) == INVALID                                                                # saved


def test_binding_argument_counts_match_header():
    """Every ctypes signature of the binding has as many arguments as the header declares."""
    import re
    text = re.sub(r"/\*.*?\*/", "", open(_lib.HEADER).read(), flags=re.S)
    for name, (_, args) in _lib.SIGNATURES.items():
        m = re.search(r"\b" + name + r"\s*\(([^;]*?)\)\s*;", text)
        assert m, name
        params = m.group(1).strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(args) == n, (name, len(args), n)


def test_debug_build_loads_with_the_same_abi(lib):
    """libmoe_gg_debug.so (MOE_GG_DEBUG: device-side bounds checks, a wait at the end of each
    call) exports the same functions, says it is the debug build, and validates arguments on the
    host exactly as the release build does. A release build reports no failed check without
    touching CUDA."""
    dbg = _lib.open_library(build.build(debug=True))
    rel = _lib.open_library(_lib.LIB_PATH)
    for name in _lib.header_functions():
        assert hasattr(dbg, name), name
    assert dbg.moe_debug_build() == 1 and rel.moe_debug_build() == 0
    assert dbg.moe_abi_version() == rel.moe_abi_version()
    assert _lib.moe_debug_report(lib=rel) == (0, -1, 0, 0)
    p = ctypes.c_void_p(16)
    for L in (rel, dbg):
        assert L.moe_route_offsets(p, 10, 1, 0, p, p, p, p, p, 1 << 20, None) == 2      # E = 0
        assert L.moe_permute(ctypes.c_void_p(18), p, p, None, 10, 1, 4, 16, p, None) == 1  # misaligned
    names = [dbg.moe_debug_site_name(s).decode() for s in range(11)]
    assert len(set(names)) == 11 and "?" not in names and dbg.moe_debug_site_name(11) == b"?"
