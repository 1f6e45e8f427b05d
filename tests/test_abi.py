"""The C ABI library loads and exports every entry point include/moe.h
declares; host-side argument checks reject bad calls before any CUDA work
(these calls never reach the device, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s+(moe_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from mixture_experts_routed_softmax_gb300.build import build
    from mixture_experts_routed_softmax_gb300 import _lib
    build()
    return _lib.load()


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_fwd", "moe_expert_bwd", "moe_combine",
              "moe_route_bwd", "moe_decode_fwd", "moe_decode_workspace_size",
              "moe_workspace_size", "moe_status", "moe_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from mixture_experts_routed_softmax_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no binding"


def test_capacity_and_workspace_sizes(lib):
    assert lib.moe_row_capacity(16384, 4, 32, 128) == 16384 * 4 + 32 * 127
    assert lib.moe_workspace_size(1, 8192, 2560, 512, 10, 128) > 0
    assert lib.moe_workspace_size(2, 8192, 2560, 512, 10, 128) > 0
    assert lib.moe_workspace_size(99, 8192, 2560, 512, 10, 128) == 0
    assert lib.moe_status_str(0) == b"MOE_OK"


def test_host_argument_checks(lib):
    from mixture_experts_routed_softmax_gb300 import _lib as L
    P = 0x1000  # a non-null, 16-byte aligned stand-in; these calls return before touching it
    # null required pointers
    wr = lib.moe_workspace_size(3, 4, 8, 4, 2, 16)
    assert wr >= 3 * 8 * 8 * 2
    assert lib.moe_route(None, P, None, None, 4, 8, 4, 2, P, P, P, P, wr, None) == L.MOE_ERR_ARG
    # k > E
    assert lib.moe_route(P, P, None, None, 4, 8, 4, 5, P, P, P, P, wr, None) == L.MOE_ERR_ARG
    # d not a multiple of 8
    assert lib.moe_route(P, P, None, None, 4, 12, 4, 2, P, P, P, P, wr, None) == L.MOE_ERR_UNSUPPORTED
    # E above the limit
    assert lib.moe_route(P, P, None, None, 4, 8, 2048, 2, P, P, P, P, wr, None) == L.MOE_ERR_UNSUPPORTED
    # workspace too small
    assert lib.moe_route(P, P, None, None, 4, 8, 4, 2, P, P, P, P, wr - 1, None) == L.MOE_ERR_ARG
    ws = lib.moe_workspace_size(1, 4, 8, 4, 2, 16)
    cap = lib.moe_row_capacity(4, 2, 4, 16)
    # align not a power of two / out of range
    for align in (0, 24, 8, 512):
        assert lib.moe_permute(P, 4, 2, 4, 0, align, P, 8, cap, P, P, P, P, P, P, ws, None) == L.MOE_ERR_ARG
    # capacity too small
    assert lib.moe_permute(P, 4, 2, 4, 0, 16, P, 8, cap - 1, P, P, P, P, P, P, ws, None) == L.MOE_ERR_CAPACITY
    # with a shared expert the capacity counts its T rows and group
    cap1 = lib.moe_row_capacity(4, 3, 5, 16)
    assert lib.moe_permute(P, 4, 2, 4, 1, 16, P, 8, cap, P, P, P, P, P, P, ws, None) == L.MOE_ERR_CAPACITY
    assert lib.moe_permute(P, 4, 2, 4, -1, 16, P, 8, cap1, P, P, P, P, P, P, ws, None) == L.MOE_ERR_ARG
    # workspace too small
    assert lib.moe_permute(P, 4, 2, 4, 0, 16, P, 8, cap, P, P, P, P, P, P, ws - 1, None) == L.MOE_ERR_ARG
    # misaligned activation pointer
    assert lib.moe_permute(P, 4, 2, 4, 0, 16, P + 2, 8, cap, P, P, P, P, P, P, ws, None) == L.MOE_ERR_ARG
    # expert GEMMs: f not a multiple of 8
    assert lib.moe_expert_fwd(P, P, None, None, 4, 2, 4, 0, 8, 12, cap, P, P, P, P, P, P, P, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_expert_fwd(P, None, None, None, 4, 2, 4, 0, 8, 16, cap, P, P, P, P, P, P, P, None) == L.MOE_ERR_ARG
    # a clamped SwiGLU needs a positive limit
    bad = L.Swiglu(0.0, 1.702, 1.0)
    assert lib.moe_expert_fwd(P, P, None, ctypes.addressof(bad), 4, 2, 4, 0, 8, 16, cap, P, P, P, P, P, P, P, None) == L.MOE_ERR_ARG
    # fused expert forward: T = 0 does nothing; a missing map, a short
    # workspace, f not a multiple of 8
    wsf = lib.moe_expert_fwd_fused_workspace_size(cap, 4, 0)
    assert wsf >= 4 * (cap // 128 + 4)
    assert lib.moe_expert_fwd_fused(None, None, None, None, None, 0, 2, 4, 0, 8, 16, cap,
                                    None, None, None, None, None, None, 0, None) == L.MOE_OK
    assert lib.moe_expert_fwd_fused(P, None, P, P, None, 4, 2, 4, 0, 8, 16, cap, P, P, P, P,
                                    P, P, wsf, None) == L.MOE_ERR_ARG
    assert lib.moe_expert_fwd_fused(P, P, P, P, None, 4, 2, 4, 0, 8, 16, cap, P, P, P, P,
                                    P, P, wsf - 1, None) == L.MOE_ERR_ARG
    assert lib.moe_expert_fwd_fused(P, P, P, P, None, 4, 2, 4, 0, 8, 12, cap, P, P, P, P,
                                    P, P, wsf, None) == L.MOE_ERR_UNSUPPORTED
    # expert backward: a missing row buffer (the gathered dY rows)
    wse = lib.moe_expert_bwd_workspace_size(cap, 16)
    assert wse >= cap * 2 * 4                  # at least one n-tile's two partials per row
    assert lib.moe_expert_bwd_workspace_size(0, 16) == 0
    ebwd = lambda dyg, ws, nb: lib.moe_expert_bwd(  # noqa: E731
        P, P, P, P, P, None, 4, 2, 4, 0, 8, 16, cap, P, P, P, P, P, P, P,
        dyg, P, P, P, P, P, P, P, P, ws, nb, None)
    assert ebwd(None, P, wse) == L.MOE_ERR_ARG
    # expert backward: workspace missing or too small
    assert ebwd(P, None, wse) == L.MOE_ERR_ARG
    assert ebwd(P, P, wse - 1) == L.MOE_ERR_ARG
    # combine: k above the slot limit
    assert lib.moe_combine(P, P, None, 4, 33, 0, 8, P, None) == L.MOE_ERR_UNSUPPORTED
    assert lib.moe_combine(P, P, None, 4, 30, 3, 8, P, None) == L.MOE_ERR_UNSUPPORTED   # k + S > 32
    # route backward: workspace missing
    assert lib.moe_route_bwd(P, P, P, P, P, P, P, 4, 8, 4, 2, 0, 16, P, None, None, P, None, None, 0, None) == L.MOE_ERR_ARG
    # route backward: dxp without dst_row
    wsb = lib.moe_workspace_size(2, 4, 8, 4, 2, 16)
    assert lib.moe_route_bwd(P, P, P, P, P, P, P, 4, 8, 4, 2, 0, 16, P, P, None, P, None, P, wsb, None) == L.MOE_ERR_ARG
    # decode: T above 8, d not a multiple of 64, k > E, null x, workspace too small
    wd = lib.moe_decode_workspace_size(2, 128, 64, 4, 2)
    assert wd >= 256 + 2 * 2 * 64 * 4          # at least the barrier word and A
    assert lib.moe_decode_workspace_size(9, 128, 64, 4, 2) == 0
    dec = lambda T, d, f, E, k, x=P, ws=wd: lib.moe_decode_fwd(  # noqa: E731
        x, P, None, None, T, d, f, E, k, P, P, P, P, P, P, P, P, ws, None)
    assert dec(9, 128, 64, 4, 2) == L.MOE_ERR_UNSUPPORTED
    assert dec(2, 96, 64, 4, 2) == L.MOE_ERR_UNSUPPORTED
    assert dec(2, 128, 72, 4, 2) == L.MOE_ERR_UNSUPPORTED
    assert dec(2, 8256, 64, 4, 2) == L.MOE_ERR_UNSUPPORTED   # d above 8192
    assert dec(2, 128, 8320, 4, 2) == L.MOE_ERR_UNSUPPORTED  # f not cut into equal 8-column blocks
    assert dec(2, 128, 64, 4, 5) == L.MOE_ERR_ARG
    assert dec(2, 128, 64, 4, 2, x=None) == L.MOE_ERR_ARG
    assert dec(2, 128, 64, 4, 2, ws=wd - 1) == L.MOE_ERR_ARG
    assert dec(0, 128, 64, 4, 2, x=None) == L.MOE_OK      # nothing to do
    # timer: bad kernel id
    assert lib.moe_timer_start(0, 4) == L.MOE_ERR_ARG
    assert lib.moe_timer_start(max(L.KERNELS.values()) + 1, 4) == L.MOE_ERR_ARG
