"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (MoELayer, each workload's own padding multiple).

Routing: the GPU's indices equal the oracle's selection on the GPU's own fp32
logits bit for bit, and the float64 oracle's up to near-ties; logits within
the bar. Layout: counts, offsets, dst_row, src_pair exact against the
oracle's stable-sort layout; every gathered Xp and dY row an exact copy;
every padding row zero. Values, against the float64 oracle evaluated expert
by expert (oracle/streamed.py), with the rules of tests/harness.py:
  * every element of y and dx (bf16 outputs) and of d_topk_w, dW_r, db;
  * every row of G, U, A, Yp, dYp, dG, dU, dXp and every element of dW_gate,
    dW_up, dW_down of three whole experts: the largest, a middle and the
    smallest non-empty one;
  * empty experts' weight gradients exactly zero, and the router gradients
    summing to zero over the experts (the softmax gradient of each token
    does).
"""
import numpy as np
import pytest
import torch

import workloads
from harness import (assert_bf16_out_close, assert_close, assert_mag_close, bf16_floor,
                     check_routing, check_routing_on_own_logits, tie_band, to_np)
from oracle import moe_oracle as mo
from oracle.streamed import stream_layer
from sampled_check import SampledChecker

pytestmark = pytest.mark.gpu

NAMES = ["gptoss20b", "qwen3_30b", "fine512", "smallm_T128", "smallm_T512", "smallm_T1024",
         "smallm_T2048"]


@pytest.mark.parametrize("name", NAMES)
def test_fullsize_parity(name):
    from mixture_experts_routed_softmax_gb300.layer import MoELayer
    wl = workloads.CONFIGS[name]
    inp = workloads.generate(wl, with_dy=wl.backward)
    T, k, E = wl.T, wl.k, wl.E
    x64 = mo.as_f64(inp["x"])
    bias = None if inp["bias"] is None else mo.as_f64(inp["bias"])
    logits = mo.router_logits(x64, mo.as_f64(inp["w_router"]), bias)
    idx = mo.select_topk(logits, k)
    layer = MoELayer.from_inputs(inp, k, wl.align)
    b = layer.buffers(T, backward=wl.backward)
    x = inp["x"].cuda()
    # free routing
    layer.forward(x, b)
    assert layer.status() == 0
    lg = to_np(b.logits)
    assert_close("logits", lg, logits)
    check_routing_on_own_logits(to_np(b.topk_idx), to_np(b.topk_w), lg, k)
    flips = check_routing(to_np(b.topk_idx), idx, logits, tie_band(lg, logits))
    # the oracle's routing on both sides from here on
    fi = torch.as_tensor(idx, dtype=torch.int32).cuda()
    layer.forward(x, b, forced_idx=fi)
    if wl.backward:
        dy = inp["dy"].cuda()
        layer.backward(dy, b)
    assert layer.status() == 0
    maps = mo.permute_maps(idx, E, wl.align, b.R_cap)
    np.testing.assert_array_equal(to_np(b.counts), maps["counts"])
    np.testing.assert_array_equal(to_np(b.offsets), maps["offsets"])
    np.testing.assert_array_equal(to_np(b.dst_row), maps["dst_row"])
    np.testing.assert_array_equal(to_np(b.src_pair), maps["src_pair"])
    R_pad = maps["R_pad"]
    dst = torch.as_tensor(maps["dst_row"]).cuda()
    tok_of_pair = torch.arange(T * k, device="cuda") // k
    assert torch.equal(b.xp[dst], x[tok_of_pair])
    if wl.backward:
        assert torch.equal(b.dyg[dst], dy[tok_of_pair])
    real = torch.zeros(R_pad, dtype=torch.bool, device="cuda")
    real[dst] = True
    pad = ~real
    for nm in ("xp", "g", "u", "a", "yp") + (("dyg", "dyp", "dg", "du", "dxp")
                                             if wl.backward else ()):
        assert torch.count_nonzero(getattr(b, nm)[:R_pad][pad]).item() == 0, f"{nm} padding"

    # ------------------------------------------------------- oracle values
    counts = maps["counts"]
    nonempty = np.flatnonzero(counts > 0)
    big = int(nonempty[np.argmax(counts[nonempty])])
    small = int(nonempty[np.argmin(counts[nonempty])])
    mid = int(nonempty[np.argsort(counts[nonempty])[len(nonempty) // 2]])
    keep = sorted({big, mid, small})
    ref = stream_layer(inp, logits, idx, k, keep=keep, backward=wl.backward)
    report = {"near_tie_tokens": flips}
    report["y"] = assert_bf16_out_close("y", to_np(b.y), ref["y"])
    report["y_bf16_floor"] = bf16_floor(ref["y"])
    if wl.backward:
        report["dx"] = assert_bf16_out_close("dx", to_np(b.dx), ref["dx"])
        report["dx_bf16_floor"] = bf16_floor(ref["dx"])
        report["d_topk_w"] = assert_close("d_topk_w", to_np(b.d_topk_w), ref["d_topk_w"])
        report["dw_router"] = assert_close("dw_router", to_np(b.dw_router), ref["dw_router"])
        report["dbias"] = assert_close("dbias", to_np(b.dbias), ref["dbias"])
    sc = SampledChecker(inp, logits, idx, k)
    dst_np = maps["dst_row"]
    for e in keep:
        rec = ref["experts"][e]
        em = sc.expert_mags(e)
        rows = torch.as_tensor(dst_np[rec["pairs"]]).cuda()
        bufs = [("G", b.g), ("U", b.u), ("A", b.a), ("Yu", b.yp)]
        if wl.backward:
            bufs += [("dYu", b.dyp), ("dG", b.dg), ("dU", b.du), ("dXp", b.dxp)]
        for key, buf in bufs:
            report[f"{key}[{e}]"] = assert_mag_close(f"{key}[{e}]", to_np(buf[rows]), rec[key],
                                                     em["M" + key])
        if wl.backward:
            for key, buf, mk in (("dw_gate", b.dw_gate, "Mdwg"), ("dw_up", b.dw_up, "Mdwu"),
                                 ("dw_down", b.dw_down, "Mdwd")):
                report[f"{key}[{e}]"] = assert_mag_close(f"{key}[{e}]", to_np(buf[e]), rec[key],
                                                         em[mk])
    if wl.backward:
        for e in np.flatnonzero(counts == 0)[:4]:
            for buf in (b.dw_gate, b.dw_up, b.dw_down):
                assert torch.count_nonzero(buf[int(e)]).item() == 0
            assert float(b.dbias[int(e)]) == 0.0
        # the softmax gradient sums to zero over the experts of each token
        db = to_np(b.dbias)
        assert abs(db.sum()) <= 1e-3 * np.abs(db).sum() + 1e-6
        dwr_all = to_np(b.dw_router)
        assert np.max(np.abs(dwr_all.sum(1))) <= 1e-3 * np.max(np.abs(dwr_all).sum(1)) + 1e-6
    print(name, {k_: (round(v, 4) if isinstance(v, float) else v) for k_, v in report.items()})
