"""Parity of the one-launch decode forward (moe_decode_fwd) with the float64
oracle.

Free routing: logits within tolerance, top-k indices exact up to near-ties.
Then the oracle's selection forced on the GPU: indices exact, weights and y
within the bar (y, a bf16 output: 2e-2 RMS plus half an ulp of bf16; the
exact top-k of the kernel's own fp32 logits). Cases span one to eight tokens, ragged expert counts
(E not a multiple of 32), k = 1 and k = 32 (256 pairs), E = 1024, narrow rows
(several warp groups per row lane set), rows wider than 4096 columns (two
column blocks), and the decode workloads' full layer shape.
Caller-chosen ids that repeat an expert, an id out of range, two runs
bitwise equal and T = 0 are covered separately.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import (assert_bf16_out_close, assert_close, check_routing,
                     check_routing_on_own_logits, tie_band, to_np)
from oracle import moe_oracle as mo

pytestmark = pytest.mark.gpu

CASES = {
    # name: (T, d, f, E, k)
    "one_token": (1, 128, 64, 8, 2),
    "three_tokens": (3, 192, 128, 20, 4),
    "eight_tokens_k1": (8, 256, 192, 7, 1),
    "eight_wide_E": (8, 320, 256, 160, 6),
    "k32_E1024": (8, 64, 128, 1024, 32),
    "layer_shape_T8": (8, 2048, 768, 16, 8),
    # rows wider than 4096 columns: each phase cuts them into two column blocks
    "two_column_blocks": (2, 4160, 4224, 4, 2),
}


def _inputs(name, T, d, f, E, k, bias=True):
    wl = workloads.Workload(name, T=T, d=d, f=f, E=E, k=k, align=16, backward=False)
    inp = workloads.generate(wl, with_dy=False)
    if not bias:
        inp["bias"] = None
    return inp


def _layer(inp, k):
    from mixture_experts_routed_softmax_gb300.layer import MoELayer
    return MoELayer.from_inputs(inp, k, 16)


def _run(layer, x, forced=None):
    b = layer.decode_buffers(x.shape[0])
    fi = None if forced is None else torch.as_tensor(forced, dtype=torch.int32).cuda()
    layer.decode_fwd(x, b, forced_idx=fi)
    return b


def _oracle(inp, k, idx=None):
    return mo.forward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                      inp["w_down"], k, idx=idx)


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_parity(name):
    T, d, f, E, k = CASES[name]
    inp = _inputs(name, T, d, f, E, k, bias=(name != "three_tokens"))
    layer = _layer(inp, k)
    x = inp["x"].cuda()
    fw = _oracle(inp, k)
    # free routing
    b = _run(layer, x)
    assert layer.status() == 0
    lg = to_np(b.logits)
    assert_close("logits", lg, fw["logits"])
    check_routing_on_own_logits(to_np(b.topk_idx), to_np(b.topk_w), lg, k)
    check_routing(to_np(b.topk_idx), fw["idx"], fw["logits"], tie_band(lg, fw["logits"]))
    # the oracle's selection forced
    b = _run(layer, x, fw["idx"])
    assert layer.status() == 0
    np.testing.assert_array_equal(to_np(b.topk_idx), fw["idx"])
    assert_close("topk_w", to_np(b.topk_w), fw["w"])
    err = assert_bf16_out_close("y", to_np(b.y), fw["y"])
    print(name, "y max|diff|/RMS", round(err, 5))


def test_decode_full_workload_shape():
    """The decode workload itself (2048 x 768, 128 experts, top-8), eight tokens."""
    wl = workloads.CONFIGS["decode_T8"]
    inp = workloads.generate(wl, with_dy=False)
    layer = _layer(inp, wl.k)
    x = inp["x"].cuda()
    fw = _oracle(inp, wl.k)
    b = _run(layer, x)
    assert layer.status() == 0
    lg = to_np(b.logits)
    assert_close("logits", lg, fw["logits"])
    check_routing(to_np(b.topk_idx), fw["idx"], fw["logits"], tie_band(lg, fw["logits"]))
    check_routing_on_own_logits(to_np(b.topk_idx), to_np(b.topk_w), lg, wl.k)
    b = _run(layer, x, fw["idx"])
    assert layer.status() == 0
    assert_bf16_out_close("y", to_np(b.y), fw["y"])


def test_decode_repeated_expert():
    """Every slot of every token on one expert: 16 pairs, more than one segment."""
    T, d, f, E, k = 8, 128, 128, 8, 2
    inp = _inputs("repeat", T, d, f, E, k)
    layer = _layer(inp, k)
    forced = np.full((T, k), 5, dtype=np.int64)
    forced[3, 1] = 2
    fw = _oracle(inp, k, idx=forced)
    b = _run(layer, inp["x"].cuda(), forced)
    assert layer.status() == 0
    np.testing.assert_array_equal(to_np(b.topk_idx), forced)
    assert_close("topk_w", to_np(b.topk_w), fw["w"])
    assert_bf16_out_close("y", to_np(b.y), fw["y"])


def test_decode_bad_forced_index():
    """An id outside [0, E) is reported and its pair dropped: that token's y
    is the oracle's over its remaining slots, the other tokens are unaffected."""
    from mixture_experts_routed_softmax_gb300 import _lib
    T, d, f, E, k = 4, 128, 64, 8, 3
    inp = _inputs("bad", T, d, f, E, k)
    layer = _layer(inp, k)
    forced = np.array([[0, 1, 2], [3, 4, 5], [6, E + 3, 1], [7, 0, 2]], dtype=np.int64)
    b = _run(layer, inp["x"].cuda(), forced)
    assert layer.status() == _lib.MOE_ERR_DEVICE_INDEX
    assert int(b.topk_idx[2, 1]) == E + 3 and float(b.topk_w[2, 1]) == 0.0
    good = [0, 1, 3]
    sub = {key: (v[good] if key == "x" else v) for key, v in inp.items()}
    fw_good = _oracle(sub, k, idx=forced[good])
    y = to_np(b.y)
    assert_bf16_out_close("y (valid tokens)", y[good], fw_good["y"])
    one = {key: (v[2:3] if key == "x" else v) for key, v in inp.items()}
    fw_one = _oracle(one, k - 1, idx=np.array([[6, 1]]))
    assert_bf16_out_close("y (token with a dropped slot)", y[2:3], fw_one["y"])


def test_decode_two_runs_bitwise_equal():
    T, d, f, E, k = 8, 256, 256, 32, 4
    inp = _inputs("det", T, d, f, E, k)
    layer = _layer(inp, k)
    x = inp["x"].cuda()
    b1 = _run(layer, x)
    y1, l1, w1 = b1.y.clone(), b1.logits.clone(), b1.topk_w.clone()
    b2 = _run(layer, x)
    assert layer.status() == 0
    assert torch.equal(y1, b2.y) and torch.equal(l1, b2.logits) and torch.equal(w1, b2.topk_w)


def test_decode_agrees_with_general_path_routing():
    """Same selection as moe_route on the same input (both decide in fp32 on
    logits that agree to within rounding; near-ties may differ)."""
    T, d, f, E, k = 8, 512, 128, 64, 4
    inp = _inputs("agree", T, d, f, E, k)
    layer = _layer(inp, k)
    x = inp["x"].cuda()
    b = _run(layer, x)
    g = layer.buffers(T, backward=False)
    layer.route(x, g)
    assert layer.status() == 0
    lg = to_np(g.logits)
    assert_close("logits vs moe_route", to_np(b.logits), lg)
    check_routing(to_np(b.topk_idx), to_np(g.topk_idx), lg, tie_band(to_np(b.logits), lg))


def test_decode_empty():
    inp = _inputs("empty", 1, 64, 64, 4, 2)
    layer = _layer(inp, 2)
    b = layer.decode_buffers(0)
    layer.decode_fwd(inp["x"][:0].cuda(), b)
    assert layer.status() == 0
