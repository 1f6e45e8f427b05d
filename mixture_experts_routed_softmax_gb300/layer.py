"""The routed MoE expert layer on one GPU, driven through the C ABI.

PyTorch supplies device memory and the stream; every step of the layer runs
in the library's kernels. Forward: moe_route -> moe_permute -> moe_expert_fwd
-> moe_combine. Backward: moe_expert_bwd -> moe_route_bwd (which also applies
the permute's transpose to dXp while it writes dx).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib

BF16 = torch.bfloat16


def _p(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


@dataclass
class Buffers:
    """Every device buffer one forward + backward of T tokens needs."""
    T: int
    R_cap: int
    logits: torch.Tensor
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    counts: torch.Tensor
    offsets: torch.Tensor
    dst_row: torch.Tensor
    src_pair: torch.Tensor
    xp: torch.Tensor
    g: torch.Tensor
    u: torch.Tensor
    a: torch.Tensor
    yp: torch.Tensor
    y: torch.Tensor
    ws_permute: torch.Tensor
    ws_route: torch.Tensor
    # backward
    dyg: Optional[torch.Tensor] = None
    dyp: Optional[torch.Tensor] = None
    dg: Optional[torch.Tensor] = None
    du: Optional[torch.Tensor] = None
    dxp: Optional[torch.Tensor] = None
    d_topk_w: Optional[torch.Tensor] = None
    dx: Optional[torch.Tensor] = None
    dw_gate: Optional[torch.Tensor] = None
    dw_up: Optional[torch.Tensor] = None
    dw_down: Optional[torch.Tensor] = None
    dw_router: Optional[torch.Tensor] = None
    dbias: Optional[torch.Tensor] = None
    # the one-launch decode forward's workspace (decode_buffers)
    ws_decode: Optional[torch.Tensor] = None
    # the fused forward's counts (fused_buffers)
    ws_fused: Optional[torch.Tensor] = None
    ws_route_bwd: Optional[torch.Tensor] = None
    ws_expert_bwd: Optional[torch.Tensor] = None
    # the input of the last forward (the router backward reads it)
    x: Optional[torch.Tensor] = None


class MoELayer:
    """Weights of one layer (device tensors) and the calls that run it.

    w_router [d, E] fp32, bias [E] fp32 or None, w_gate / w_up [E+S, d, f]
    bf16, w_down [E+S, f, d] bf16 (the E routed experts, then the S shared
    experts every token goes through with weight 1); top-k routing; ``align``
    pads each expert's rows; ``act`` = (limit, alpha, up_offset) of the
    clamped SwiGLU, or None for the plain SwiGLU.
    """

    def __init__(self, w_router, bias, w_gate, w_up, w_down, k: int, align: int = 128,
                 act=None):
        self.lib = _lib.load()
        self.w_router = w_router.contiguous()
        self.bias = None if bias is None else bias.contiguous()
        self.w_gate = w_gate.contiguous()
        self.w_up = w_up.contiguous()
        self.w_down = w_down.contiguous()
        self.E = int(w_router.shape[1])
        EE, self.d, self.f = w_gate.shape
        self.S = int(EE) - self.E
        if self.S < 0:
            raise ValueError("w_gate holds fewer experts than the router")
        self.k = k
        self.align = align
        self.act = None if act is None else _lib.Swiglu(*[float(v) for v in act])
        dev = w_gate.device
        if dev.type != "cuda":
            raise RuntimeError("MoELayer runs on a CUDA device only")
        self.device = dev

    @classmethod
    def from_inputs(cls, inp: dict, k: int, align: int = 128, device="cuda", act=None):
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return cls(mv(inp["w_router"]), mv(inp.get("bias")), mv(inp["w_gate"]),
                   mv(inp["w_up"]), mv(inp["w_down"]), k, align, act)

    def _act(self):
        return None if self.act is None else _lib.ctypes.addressof(self.act)

    def row_capacity(self, T: int) -> int:
        return int(self.lib.moe_row_capacity(T, self.k + self.S, self.E + self.S, self.align))

    def buffers(self, T: int, backward: bool = True) -> Buffers:
        E, d, f, k, S = self.E, self.d, self.f, self.k, self.S
        R = self.row_capacity(T)
        kw = dict(device=self.device)
        ws_p = int(self.lib.moe_workspace_size(_lib.MOE_WS_PERMUTE, T, d, E, k, self.align))
        b = Buffers(
            T=T, R_cap=R,
            logits=torch.empty(T, E, dtype=torch.float32, **kw),
            topk_idx=torch.empty(T, k, dtype=torch.int32, **kw),
            topk_w=torch.empty(T, k, dtype=torch.float32, **kw),
            counts=torch.empty(E + S, dtype=torch.int32, **kw),
            offsets=torch.empty(E + S + 1, dtype=torch.int64, **kw),
            dst_row=torch.empty(T * (k + S), dtype=torch.int32, **kw),
            src_pair=torch.empty(R, dtype=torch.int32, **kw),
            xp=torch.empty(R, d, dtype=BF16, **kw),
            g=torch.empty(R, f, dtype=torch.float32, **kw),
            u=torch.empty(R, f, dtype=torch.float32, **kw),
            a=torch.empty(R, f, dtype=BF16, **kw),
            yp=torch.empty(R, d, dtype=torch.float32, **kw),
            y=torch.empty(T, d, dtype=BF16, **kw),
            ws_permute=torch.empty(max(ws_p, 256), dtype=torch.uint8, **kw),
            ws_route=torch.empty(
                int(self.lib.moe_workspace_size(_lib.MOE_WS_ROUTE, T, d, E, k, self.align)),
                dtype=torch.uint8, **kw),
        )
        if backward:
            ws_r = int(self.lib.moe_workspace_size(_lib.MOE_WS_ROUTE_BWD, T, d, E, k, self.align))
            b.dyg = torch.empty(R, d, dtype=BF16, **kw)
            b.dyp = torch.empty(R, d, dtype=BF16, **kw)
            b.dg = torch.empty(R, f, dtype=BF16, **kw)
            b.du = torch.empty(R, f, dtype=BF16, **kw)
            b.dxp = torch.empty(R, d, dtype=torch.float32, **kw)
            b.d_topk_w = torch.empty(T, k, dtype=torch.float32, **kw)
            b.dx = torch.empty(T, d, dtype=BF16, **kw)
            b.dw_gate = torch.empty(E + S, d, f, dtype=BF16, **kw)
            b.dw_up = torch.empty(E + S, d, f, dtype=BF16, **kw)
            b.dw_down = torch.empty(E + S, f, d, dtype=BF16, **kw)
            b.dw_router = torch.empty(d, E, dtype=torch.float32, **kw)
            b.dbias = torch.empty(E, dtype=torch.float32, **kw)
            b.ws_route_bwd = torch.empty(max(ws_r, 256), dtype=torch.uint8, **kw)
            ws_e = int(self.lib.moe_expert_bwd_workspace_size(R, f))
            b.ws_expert_bwd = torch.empty(max(ws_e, 256), dtype=torch.uint8, **kw)
        return b

    # ------------------------------------------------------------- calls --
    def route(self, x, b: Buffers, forced_idx=None, stream=None):
        _lib.call("moe_route", _p(x), _p(self.w_router), _p(self.bias), _p(forced_idx),
                  b.T, self.d, self.E, self.k, _p(b.logits), _p(b.topk_idx), _p(b.topk_w),
                  _p(b.ws_route), b.ws_route.numel(), _stream(stream))

    def permute(self, x, b: Buffers, topk_idx=None, stream=None):
        idx = b.topk_idx if topk_idx is None else topk_idx
        _lib.call("moe_permute", _p(idx), b.T, self.k, self.E, self.S, self.align, _p(x), self.d,
                  b.R_cap, _p(b.counts), _p(b.offsets), _p(b.dst_row), _p(b.src_pair),
                  _p(b.xp), _p(b.ws_permute), b.ws_permute.numel(), _stream(stream))

    def expert_fwd(self, b: Buffers, row_w=None, stream=None):
        _lib.call("moe_expert_fwd", _p(b.xp), _p(b.offsets), _p(row_w), self._act(), b.T, self.k,
                  self.E, self.S, self.d, self.f, b.R_cap, _p(self.w_gate), _p(self.w_up),
                  _p(self.w_down), _p(b.g), _p(b.u), _p(b.a), _p(b.yp), _stream(stream))

    def combine(self, rows, b: Buffers, out, weights=True, stream=None):
        _lib.call("moe_combine", _p(rows), _p(b.dst_row), _p(b.topk_w) if weights else None,
                  b.T, self.k, self.S, self.d, _p(out), _stream(stream))

    def expert_bwd(self, dy, b: Buffers, stream=None):
        _lib.call("moe_expert_bwd", _p(dy), _p(b.src_pair), _p(b.dst_row), _p(b.topk_w),
                  _p(b.offsets), self._act(), b.T, self.k, self.E, self.S, self.d, self.f, b.R_cap,
                  _p(b.xp), _p(b.g), _p(b.u), _p(b.a),
                  _p(self.w_gate), _p(self.w_up), _p(self.w_down),
                  _p(b.dyg), _p(b.dyp), _p(b.dg), _p(b.du), _p(b.dxp), _p(b.d_topk_w),
                  _p(b.dw_gate), _p(b.dw_up), _p(b.dw_down), _p(b.ws_expert_bwd),
                  b.ws_expert_bwd.numel(), _stream(stream))

    def route_bwd(self, b: Buffers, fused=True, stream=None, x=None):
        """Router backward. fused: dx = permute transpose of dXp + the router's
        term in one pass; else dx (already holding the permute transpose) += it.
        x: the layer input (default: the one the last forward recorded in b)."""
        x = b.x if x is None else x
        _lib.call("moe_route_bwd", _p(b.d_topk_w), _p(b.topk_w), _p(b.topk_idx),
                  _p(self.w_router), _p(b.offsets), _p(b.src_pair), _p(x), b.T, self.d,
                  self.E, self.k, self.S, self.align, _p(b.dx), _p(b.dxp) if fused else None,
                  _p(b.dst_row) if fused else None, _p(b.dw_router), _p(b.dbias),
                  _p(b.ws_route_bwd), b.ws_route_bwd.numel(), _stream(stream))

    # ------------------------------------------------------ whole layer --
    def forward(self, x, b: Buffers, forced_idx=None, stream=None):
        """y = layer(x) into b.y; every intermediate stays in ``b`` (x by reference)."""
        b.x = x
        self.route(x, b, forced_idx, stream)
        self.permute(x, b, None, stream)
        self.expert_fwd(b, None, stream)
        self.combine(b.yp, b, b.y, True, stream)
        return b.y

    def backward(self, dy, b: Buffers, stream=None):
        """Gradients of sum(y * dy) into b.dx, b.dw_*, b.dbias, b.d_topk_w.
        The permute's transpose runs inside the router backward's dx pass."""
        self.expert_bwd(dy, b, stream)
        self.route_bwd(b, fused=True, stream=stream)
        return b.dx

    # ------------------------------------------------------ fused forward --
    def fused_buffers(self, T: int) -> Buffers:
        """Buffers for forward_fused: routing, the layout, A, the scored Yp, y
        and the fused forward's counts (no G or U: nothing is kept for a backward)."""
        E, d, f, k, S = self.E, self.d, self.f, self.k, self.S
        R = self.row_capacity(T)
        kw = dict(device=self.device)
        ws_p = int(self.lib.moe_workspace_size(_lib.MOE_WS_PERMUTE, T, d, E, k, self.align))
        ws_f = int(self.lib.moe_expert_fwd_fused_workspace_size(R, E, S))
        return Buffers(
            T=T, R_cap=R,
            logits=torch.empty(T, E, dtype=torch.float32, **kw),
            topk_idx=torch.empty(T, k, dtype=torch.int32, **kw),
            topk_w=torch.empty(T, k, dtype=torch.float32, **kw),
            counts=torch.empty(E + S, dtype=torch.int32, **kw),
            offsets=torch.empty(E + S + 1, dtype=torch.int64, **kw),
            dst_row=torch.empty(T * (k + S), dtype=torch.int32, **kw),
            src_pair=torch.empty(R, dtype=torch.int32, **kw),
            xp=torch.empty(R, d, dtype=BF16, **kw), g=None, u=None,
            a=torch.empty(R, f, dtype=BF16, **kw),
            yp=torch.empty(R, d, dtype=torch.float32, **kw),
            y=torch.empty(T, d, dtype=BF16, **kw),
            ws_permute=torch.empty(max(ws_p, 256), dtype=torch.uint8, **kw),
            ws_route=torch.empty(
                int(self.lib.moe_workspace_size(_lib.MOE_WS_ROUTE, T, d, E, k, self.align)),
                dtype=torch.uint8, **kw),
            ws_fused=torch.empty(max(ws_f, 256), dtype=torch.uint8, **kw),
        )

    def expert_fwd_fused(self, b: Buffers, stream=None):
        """The expert GEMMs of the forward in one launch (moe_expert_fwd_fused):
        A into b.a and the scored rows into b.yp."""
        _lib.call("moe_expert_fwd_fused", _p(b.xp), _p(b.src_pair), _p(b.offsets), _p(b.topk_w),
                  self._act(), b.T, self.k, self.E, self.S, self.d, self.f, b.R_cap,
                  _p(self.w_gate), _p(self.w_up), _p(self.w_down), _p(b.a), _p(b.yp),
                  _p(b.ws_fused), b.ws_fused.numel(), _stream(stream))

    def forward_fused(self, x, b: Buffers, forced_idx=None, stream=None):
        """y = layer(x) for inference, b from fused_buffers(T): route, permute,
        the fused expert GEMMs, and the gather-sum of the already scored rows."""
        b.x = x
        self.route(x, b, forced_idx, stream)
        self.permute(x, b, None, stream)
        self.expert_fwd_fused(b, stream)
        self.combine(b.yp, b, b.y, False, stream)
        return b.y

    # ------------------------------------------------------------ decode --
    def decode_buffers(self, T: int) -> Buffers:
        """Buffers for decode_fwd: logits, top-k, y and the decode workspace."""
        E, d, k = self.E, self.d, self.k
        kw = dict(device=self.device)
        ws = int(self.lib.moe_decode_workspace_size(T, d, self.f, self.E, k))
        none = torch.empty(0, **kw)
        return Buffers(
            T=T, R_cap=0,
            logits=torch.empty(T, E, dtype=torch.float32, **kw),
            topk_idx=torch.empty(T, k, dtype=torch.int32, **kw),
            topk_w=torch.empty(T, k, dtype=torch.float32, **kw),
            counts=none, offsets=none, dst_row=none, src_pair=none, xp=none, g=none,
            u=none, a=none, yp=none,
            y=torch.empty(T, d, dtype=BF16, **kw),
            ws_permute=none, ws_route=none,
            ws_decode=torch.empty(max(ws, 256), dtype=torch.uint8, **kw),
        )

    def decode_fwd(self, x, b: Buffers, forced_idx=None, stream=None):
        """The whole forward of T <= 8 tokens in one launch (moe_decode_fwd);
        b from decode_buffers(T). Fills b.logits, b.topk_idx, b.topk_w, b.y.
        Routed experts with the plain SwiGLU only."""
        if self.S or self.act is not None:
            raise ValueError("the one-launch decode forward takes routed experts with the plain "
                             "SwiGLU only")
        b.x = x
        _lib.call("moe_decode_fwd", _p(x), _p(self.w_router), _p(self.bias), _p(forced_idx),
                  b.T, self.d, self.f, self.E, self.k, _p(self.w_gate), _p(self.w_up),
                  _p(self.w_down), _p(b.logits), _p(b.topk_idx), _p(b.topk_w), _p(b.y),
                  _p(b.ws_decode), b.ws_decode.numel(), _stream(stream))
        return b.y

    def status(self, stream=None) -> int:
        """Synchronise and read (and clear) the device status word."""
        return int(self.lib.moe_status(_stream(stream)))
