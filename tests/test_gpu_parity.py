"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Complete comparisons at sizes the oracle finishes in seconds: several tiles
in every GEMM dimension, ragged tails (d and f not multiples of the tile
widths), skewed loads with empty experts, k = 1 and k = E, one token, one
expert, every padding multiple, exactly tied logits. Integers bit-exact,
values within the bar of tests/harness.py (2e-2 x RMS; bf16 outputs plus
the format's own half-ulp).
"""
import numpy as np
import pytest
import torch

import workloads
from harness import check_routing_on_own_logits, compare_full, gpu_forward_backward, to_np

pytestmark = pytest.mark.gpu


def _layer(inp, k, align):
    from mixture_experts_routed_softmax_gb300.layer import MoELayer
    return MoELayer.from_inputs(inp, k, align)


def _case(name, T, d, f, E, k, align, zipf=None, tau=None):
    wl = workloads.Workload(name, T=T, d=d, f=f, E=E, k=k, zipf_s=zipf, align=align)
    inp = workloads.generate(wl, tau=tau)
    return wl, inp


CASES = {
    # name: (T, d, f, E, k, align, zipf_s, tau)
    "tiny": (256, 128, 256, 8, 2, 128, None, None),
    "ragged_a16": (300, 200, 136, 6, 2, 16, None, None),
    "multi_tile": (520, 392, 520, 8, 3, 128, None, None),
    "skewed_empty": (700, 264, 384, 16, 4, 32, 1.2, 1.5),
    "one_expert_k1": (333, 128, 256, 1, 1, 64, None, None),
    "k_equals_E": (64, 64, 64, 4, 4, 16, None, None),
    "one_token": (1, 128, 128, 8, 2, 16, None, None),
    "seven_tokens": (7, 96, 160, 8, 3, 256, None, None),
    # three groups of eight tokens in the few-token router, E not a multiple of 4
    "twentyfour_tokens": (24, 160, 192, 12, 3, 16, None, None),
    "wide_E": (256, 128, 64, 160, 6, 16, 1.1, 0.8),
    # the largest routing the ABI takes: 1024 experts, top-32 (most experts empty)
    "max_E_and_k": (96, 64, 64, 1024, 32, 16, None, None),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_layer_parity(name):
    T, d, f, E, k, align, zipf, tau = CASES[name]
    wl, inp = _case(name, T, d, f, E, k, align, zipf, tau)
    layer = _layer(inp, k, align)
    out, _ = compare_full(layer, inp, k, align)
    print(name, {k_: (round(v, 5) if isinstance(v, float) else v) for k_, v in out.items()})


def test_all_tokens_to_one_expert():
    T, d, f, E, k, align = 200, 128, 192, 8, 1, 16
    wl, inp = _case("one_hot", T, d, f, E, k, align)
    layer = _layer(inp, k, align)
    forced = torch.full((T, k), 3, dtype=torch.int32)
    b, _, _ = gpu_forward_backward(layer, inp, forced)
    counts = to_np(b.counts)
    assert counts[3] == T and counts.sum() == T
    for e in range(E):
        if e != 3:
            assert torch.count_nonzero(b.dw_gate[e]).item() == 0
            assert torch.count_nonzero(b.dw_down[e]).item() == 0
    # k = 1: every weight is exactly 1
    assert torch.all(b.topk_w == 1.0)


def test_two_runs_bitwise_equal():
    T, d, f, E, k, align = 512, 256, 384, 16, 4, 32
    wl, inp = _case("det", T, d, f, E, k, align, 1.1, 1.0)
    layer = _layer(inp, k, align)
    b1, _, _ = gpu_forward_backward(layer, inp)
    b2, _, _ = gpu_forward_backward(layer, inp)
    for name in ("logits", "topk_idx", "topk_w", "offsets", "dst_row", "src_pair", "y", "dx",
                 "dw_gate", "dw_up", "dw_down", "dw_router", "dbias", "d_topk_w"):
        assert torch.equal(getattr(b1, name), getattr(b2, name)), name
    R = int(b1.offsets[-1])
    for name in ("xp", "g", "u", "a", "yp", "dyg", "dyp", "dg", "du", "dxp"):
        assert torch.equal(getattr(b1, name)[:R], getattr(b2, name)[:R]), name


def test_epilogue_row_scaling_matches_unscaled_times_weight():
    """moe_expert_fwd with row_w scales each output row in the fp32 epilogue."""
    T, d, f, E, k, align = 256, 128, 256, 8, 2, 16
    wl, inp = _case("roww", T, d, f, E, k, align)
    layer = _layer(inp, k, align)
    b, _, _ = gpu_forward_backward(layer, inp, backward=False)
    R = b.R_cap
    rng = np.random.default_rng(0)
    row_w = torch.tensor(rng.random(R), dtype=torch.float32, device="cuda")
    unscaled = b.yp.clone()
    layer.expert_fwd(b, row_w=row_w)
    torch.cuda.synchronize()
    Rp = int(b.offsets[-1])
    ref = unscaled[:Rp].float() * row_w[:Rp, None]
    got = b.yp[:Rp].float()
    # the epilogue multiplies the same fp32 accumulator by the fp32 weight
    assert torch.equal(got, ref)


def test_bad_forced_index_raises_device_status():
    from mixture_experts_routed_softmax_gb300 import _lib
    T, d, f, E, k, align = 64, 64, 64, 4, 2, 16
    wl, inp = _case("badidx", T, d, f, E, k, align)
    layer = _layer(inp, k, align)
    b = layer.buffers(T, backward=False)
    forced = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    forced[:, 1] = 1
    forced[5, 1] = E + 3          # out of range: reported, never dereferenced
    layer.route(inp["x"].cuda(), b, forced_idx=forced)
    assert layer.status() == _lib.MOE_ERR_DEVICE_INDEX
    assert float(b.topk_w[5, 1]) == 0.0
    layer.permute(inp["x"].cuda(), b, topk_idx=forced)   # the bad pair is dropped from the layout
    assert layer.status() == _lib.MOE_ERR_DEVICE_INDEX
    assert int(b.dst_row[5 * k + 1]) == -1
    assert int(b.counts.sum()) == T * k - 1
    assert layer.status() == 0           # the status word was cleared by the read


def test_router_backward_fused_and_separate_dx_agree():
    """moe_route_bwd writes dx = permute-transpose(dXp) + router term in one
    pass (fused), or adds the router term to a dx that moe_combine already
    holds; the two differ only by the second bf16 rounding."""
    T, d, f, E, k, align = 300, 200, 136, 6, 2, 16
    wl, inp = _case("dxfuse", T, d, f, E, k, align)
    layer = _layer(inp, k, align)
    b, x, dy = gpu_forward_backward(layer, inp)          # fused path (the layer's default)
    dx_fused = b.dx.float().clone()
    dw_r = b.dw_router.clone()
    layer.combine(b.dxp, b, b.dx, weights=False)          # permute transpose into dx
    torch.cuda.synchronize()
    dx_expert = b.dx.float().clone()
    layer.route_bwd(b, fused=False)                        # then dx += router term
    assert layer.status() == 0
    dx_sep = b.dx.float()
    # the separate path rounds the expert part to bf16 before adding the router term
    bound = 2 ** -7 * (torch.abs(dx_expert) + torch.abs(dx_fused)) + 1e-6
    assert torch.all(torch.abs(dx_sep - dx_fused) <= bound)
    assert torch.equal(b.dw_router, dw_r)


def test_empty_batch():
    """T = 0: every call succeeds (the T-sized arrays are empty), the layout
    is all padding-free zeros, and every gradient of the empty batch is 0."""
    T, d, f, E, k, align = 0, 128, 256, 8, 2, 16
    wl, inp = _case("tiny", 64, d, f, E, k, align)     # weights only; the batch is empty
    layer = _layer(inp, k, align)
    b = layer.buffers(T)
    x = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    dy = torch.empty(0, d, dtype=torch.bfloat16, device="cuda")
    for buf in (b.dw_gate, b.dw_up, b.dw_down, b.dw_router, b.dbias):
        buf.fill_(7.0)                                 # must be overwritten with zeros
    layer.forward(x, b)
    layer.backward(dy, b)
    assert layer.status() == 0
    assert b.y.shape == (0, d) and b.dx.shape == (0, d)
    assert int(b.counts.abs().sum()) == 0 and int(b.offsets.abs().sum()) == 0
    assert torch.all(b.src_pair == -1)
    for name in ("dw_gate", "dw_up", "dw_down", "dw_router", "dbias"):
        assert torch.count_nonzero(getattr(b, name)).item() == 0, name


@pytest.mark.parametrize("T", [24, 300])
def test_exact_ties_pick_the_lower_index(T):
    """Two pairs of identical router columns (bias 0) give bitwise-equal fp32
    logits; the selection must put the lower expert index first, and the
    equal logits get equal weights. T = 24 runs the few-token CUDA-core
    router, T = 300 the tensor-core router."""
    d, f, E, k, align = 128, 64, 8, 3, 16
    wl, inp = _case("ties", T, d, f, E, k, align)
    wr = inp["w_router"].clone()
    wr[:, 2] = 4.0 * wr[:, 2]          # favoured, so the tied pairs reach the top-k
    wr[:, 5] = wr[:, 2]
    wr[:, 1] = 3.0 * wr[:, 1]
    wr[:, 6] = wr[:, 1]
    inp["w_router"] = wr
    layer = _layer(inp, k, align)
    b, _, _ = gpu_forward_backward(layer, inp, backward=False)
    lg = b.logits
    assert torch.equal(lg[:, 2], lg[:, 5]) and torch.equal(lg[:, 1], lg[:, 6])
    idx = to_np(b.topk_idx)
    w = to_np(b.topk_w)
    check_routing_on_own_logits(idx, w, to_np(lg), k)
    both = 0
    for t in range(T):
        sel = idx[t].tolist()
        for lo, hi in ((2, 5), (1, 6)):
            if hi in sel:
                assert lo in sel and sel.index(lo) < sel.index(hi), (t, sel)
                assert w[t, sel.index(lo)] == w[t, sel.index(hi)], (t, sel)
                both += 1
    assert both >= T // 4          # the ties were exercised
    # the float64 oracle breaks the same ties the same way: exact agreement
    from oracle import moe_oracle as mo
    ref = mo.select_topk(mo.router_logits(mo.as_f64(inp["x"]), mo.as_f64(wr)), k)
    tied = [t for t in range(T) if ({5, 6} & set(idx[t].tolist()))]
    np.testing.assert_array_equal(idx[tied], ref[tied])



# -------------------------------------------- clamped SwiGLU and shared experts
# (prime-rl PR #3885, §Changes, "FP8 routed experts" and "Fused FP8 shared
# expert"; the clamp constants are GPT-OSS-20B's, the others are a limit that
# binds at these scales)
F2_CASES = {
    # name: (T, d, f, E, k, S, align, act)
    "clamp_gptoss": (256, 128, 256, 8, 2, 0, 16, (7.0, 1.702, 1.0)),
    "clamp_binding": (300, 200, 136, 6, 2, 0, 16, (0.75, 1.702, 1.0)),
    "shared1": (300, 200, 136, 6, 2, 1, 16, None),
    "shared2_clamped": (520, 392, 520, 8, 3, 2, 128, (1.0, 1.702, 1.0)),
    "shared1_wide_E": (256, 128, 64, 160, 6, 1, 16, (1.5, 1.702, 1.0)),
    "qwen_like_shared": (1024, 2048, 768, 128, 8, 1, 16, (7.0, 1.702, 1.0)),
}


def _f2_case(name, T, d, f, E, k, S, align):
    """Inputs with E + S experts' weights; the router sees the first E."""
    wl = workloads.Workload(name, T=T, d=d, f=f, E=E + S, k=k, align=align)
    inp = workloads.generate(wl)
    inp["w_router"] = inp["w_router"][:, :E].contiguous()
    return inp


@pytest.mark.parametrize("name", sorted(F2_CASES))
def test_clamped_swiglu_and_shared_experts(name):
    from mixture_experts_routed_softmax_gb300.layer import MoELayer
    T, d, f, E, k, S, align, act = F2_CASES[name]
    inp = _f2_case(name, T, d, f, E, k, S, align)
    layer = MoELayer.from_inputs(inp, k, align, act=act)
    assert layer.S == S and layer.E == E
    out, b = compare_full(layer, inp, k, align)
    if act is not None and act[0] < 2:
        # the clamps bind somewhere, in both directions of U
        G, U = b.g[:int(b.offsets[-1])], b.u[:int(b.offsets[-1])]
        assert (G > act[0]).any() and (U > act[0]).any() and (U < -act[0]).any()
    print(name, {k_: (round(v, 5) if isinstance(v, float) else v) for k_, v in out.items()})
