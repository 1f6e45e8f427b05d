"""Algorithmic FLOPs and HBM bytes of the routed MoE layer, per kernel.

Counting rules (real rows only; padding rows are overhead, not work):
  * one multiply-add = 2 FLOPs; the expert GEMMs of a pair cost 2*d*f each
    (gate, up, down), so the forward is 6*P*d*f + 2*T*d*E (router), the
    backward twice the expert GEMMs (dgrad + wgrad) plus the router's;
  * bytes are the minimum each kernel must move between HBM and the chip:
    each tensor it reads once, each tensor it writes once, expert weights only
    for experts that received rows (E_active), bf16 = 2 B, fp32 = 4 B.
The expert weight size matches PocketLLM "Qwen4-Exp Heterogeneous TP4
Performance", §Runtime architecture: one bf16 expert of hidden size 2560 and
ffn size 640 is 3 * 2560 * 640 * 2 B = 9.375 MiB. The expected number of
distinct experts a batch touches, E (1 - (1 - k/E)^T), gives 74.7 for 8
tokens of top-10 over 512 experts, as the same page's §Decode ceiling states.
"""
from __future__ import annotations

from dataclasses import dataclass


def expert_bytes(d: int, f: int, elem: int = 2) -> int:
    """Bytes of one expert's three weight matrices (gate, up, down)."""
    return 3 * d * f * elem


def expected_active_experts(E: int, k: int, T: int) -> float:
    """Expected distinct experts touched by T tokens each routed to k of E."""
    return E * (1.0 - (1.0 - k / E) ** T)


@dataclass(frozen=True)
class Shape:
    T: int
    d: int
    f: int
    E: int
    k: int
    E_active: int     # experts with at least one row

    @property
    def P(self) -> int:
        return self.T * self.k


def kernel_costs(s: Shape, backward: bool = True) -> dict:
    """{kernel: (flops, bytes)} for one pass of the layer, per kernel group
    (the groups match the library's timer ids)."""
    P, T, d, f, E, k = s.P, s.T, s.d, s.f, s.E, s.k
    W1 = s.E_active * d * f * 2          # one weight matrix set (bf16) over active experts
    c = {}
    c["router_logits"] = (2 * T * d * E, T * d * 2 + d * E * 4 + T * E * 4)
    c["topk"] = (0, T * E * 4 + T * k * 8)
    c["permute"] = (0, T * k * 4 + P * d * 2 + P * d * 2)          # idx, gathered x, Xp
    c["gateup_fwd"] = (4 * P * d * f, P * d * 2 + 2 * W1 + 3 * P * f * 2)
    c["down_fwd"] = (2 * P * f * d, P * f * 2 + W1 + P * d * 2)
    c["combine"] = (0, P * d * 2 + T * k * 8 + T * d * 2)
    if not backward:
        return c
    c["combine_bwd"] = (0, P * d * 2 + P * d * 2 + P * d * 2 + P * 4)   # dY gather, Yp, dYp, dw
    c["down_dgrad"] = (2 * P * d * f, P * d * 2 + W1 + 2 * P * f * 2 + 2 * P * f * 2)
    c["gateup_dgrad"] = (4 * P * f * d, 2 * P * f * 2 + 2 * W1 + P * d * 2)
    c["wgrad_down"] = (2 * P * f * d, P * f * 2 + P * d * 2 + W1)
    c["wgrad_gateup"] = (4 * P * d * f, P * d * 2 + 2 * P * f * 2 + 2 * W1)
    # the router backward includes the permute's transpose: dXp read once, x
    # read, dx written once, W_r read and dW_r written, the per-pair scalars
    c["route_bwd"] = (2 * P * d + 2 * P * d,
                      2 * T * d * 2 + P * d * 2 + 2 * d * E * 4 + T * k * 12)
    return c


def fused_forward_costs(s: Shape) -> dict:
    """{kernel: (flops, bytes)} of the inference forward with the fused
    expert GEMMs (moe_expert_fwd_fused): the router, top-k and permute as in
    kernel_costs, one fused launch (Xp read, the three weight matrices of
    each active expert, A written and read back, the scored Yp written; G
    and U stay in tensor memory), and the combine of the scored rows."""
    P, d, f = s.P, s.d, s.f
    W1 = s.E_active * d * f * 2
    c = kernel_costs(s, backward=False)
    del c["gateup_fwd"], c["down_fwd"]
    c["fused_fwd"] = (6 * P * d * f, P * d * 2 + 3 * W1 + 2 * P * f * 2 + P * d * 2)
    return c


def decode_costs(s: Shape) -> tuple[int, int]:
    """(flops, bytes) of the one-launch decode forward: the router and every
    pair's three expert products; x, W_r, logits, top-k, y and the three
    weight matrices of each selected expert, each moved once (the per-pair
    fp32 intermediates stay on chip or in L2)."""
    P, T, d, f, E, k = s.P, s.T, s.d, s.f, s.E, s.k
    fl = 2 * T * d * E + 6 * P * d * f
    by = T * d * 2 + d * E * 4 + T * E * 4 + T * k * 8 + 3 * s.E_active * d * f * 2 + T * d * 2
    return fl, by


def totals(s: Shape, backward: bool = True) -> tuple[int, int]:
    fl = by = 0
    for f_, b_ in kernel_costs(s, backward).values():
        fl += f_
        by += b_
    return fl, by


def roofline_seconds(flops: float, nbytes: float, tflops: float, gbs: float) -> float:
    """The slower of the tensor-core bound and the HBM bound."""
    return max(flops / (tflops * 1e12), nbytes / (gbs * 1e9))
