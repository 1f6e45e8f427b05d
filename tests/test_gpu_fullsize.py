"""Parity at the workloads' full sizes, in the launch configuration bench.py
times (MoELayer, each workload's own padding multiple).

Checked in full: logits (tolerance), routing indices (exact up to near-ties),
counts, offsets, dst_row, src_pair (exact, against the oracle's stable-sort
layout), every gathered Xp row (an exact copy) and every padding row (zero).
Checked at sampled positions against the float64 oracle (oracle/sampled.py):
y, dx and the top-k weight gradients of sampled tokens; G, U, A, Yp, dYp,
dXp rows of their pairs; dW_gate / dW_up columns and dW_down rows of the
largest, a middle and the smallest non-empty expert; dW_r and db of the
smallest expert. Checked by properties at any size: empty experts' weight
gradients are exactly zero, and the router gradients sum to zero over the
experts (the softmax gradient of each token does).
"""
import numpy as np
import pytest
import torch

import workloads
from harness import MAG_C, RMS_REL_TOL, TOL, U_BF16, check_routing, tie_band, to_np
from oracle import moe_oracle as mo
from sampled_check import SampledChecker

pytestmark = pytest.mark.gpu

NAMES = ["gptoss20b", "qwen3_30b", "fine512", "smallm_T128", "smallm_T512", "smallm_T1024",
         "smallm_T2048"]


def _check(name, got, ref, mag):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    diff = np.abs(got - ref)
    norm = np.sqrt(np.sum(ref * ref))
    rms = norm / np.sqrt(ref.size)
    dn = np.sqrt(np.sum(diff * diff))
    assert dn <= RMS_REL_TOL * norm or dn <= U_BF16 * np.sqrt(np.sum(np.asarray(mag) ** 2)), \
        f"{name}: ||diff||/||ref|| = {dn / max(norm, 1e-300):.3e}"
    bound = np.maximum(TOL * rms, MAG_C * U_BF16 * np.asarray(mag)) + 1e-30
    worst = float(np.max(diff / bound))
    assert worst <= 1.0, f"{name}: worst |diff| / bound = {worst:.3f}"
    return float(np.max(diff) / max(rms, 1e-300))


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
    assert float(np.max(np.abs(lg - logits))) <= TOL * float(np.sqrt(np.mean(logits ** 2)))
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
    real = torch.zeros(R_pad, dtype=torch.bool, device="cuda")
    real[dst] = True
    pad = ~real
    for nm in ("xp", "g", "u", "a", "yp") + (("dyp", "dg", "du", "dxp") if wl.backward else ()):
        assert torch.count_nonzero(getattr(b, nm)[:R_pad][pad]).item() == 0, f"{nm} padding"

    # ---------------------------------------------------------- sampled values
    sc = SampledChecker(inp, logits, idx, k)
    counts = maps["counts"]
    nonempty = np.flatnonzero(counts > 0)
    big = int(nonempty[np.argmax(counts[nonempty])])
    small = int(nonempty[np.argmin(counts[nonempty])])
    mid = int(nonempty[np.argsort(counts[nonempty])[len(nonempty) // 2]])
    rng = np.random.default_rng(0)
    toks = set(rng.choice(T, size=min(T, 12), replace=False).tolist())
    for e in (big, small, mid):
        toks.add(int(sc.pairs_of[e][0] // k))
    toks = sorted(toks)
    ref = sc.tokens(toks)
    report = {"near_tie_tokens": flips}
    for key, buf, mkey in (("y", b.y, "My"),) + ((("dx", b.dx, "Mdx"),) if wl.backward else ()):
        got = to_np(buf[toks])
        report[key] = _check(key, got, np.stack([ref[t][key] for t in toks]),
                             np.stack([ref[t][mkey] for t in toks]))
    pairs = [t * k + j for t in toks for j in range(k)]
    rows = maps["dst_row"][pairs]
    flat = [ref[p // k]["pairs"][p % k] for p in pairs]
    for key, buf in (("G", b.g), ("U", b.u), ("A", b.a), ("Yu", b.yp)) + (
            (("dYu", b.dyp), ("dXp", b.dxp)) if wl.backward else ()):
        report[key] = _check(key, to_np(buf[torch.as_tensor(rows).cuda()]),
                             np.stack([q[key] for q in flat]), np.stack([q["M" + key] for q in flat]))
    if wl.backward:
        report["d_topk_w"] = _check("d_topk_w", to_np(b.d_topk_w[toks]),
                                    np.stack([ref[t]["dtw"] for t in toks]),
                                    np.stack([ref[t]["Mdtw"] for t in toks]))
        cols = sorted({0, wl.f - 1, int(rng.integers(wl.f))})
        for e in (big, mid, small):
            for c in cols:
                wc = sc.wgrad_cols(e, c)
                report[f"dw_gate[{e}]"] = _check("dw_gate", to_np(b.dw_gate[e][:, c]), wc["dwg"], wc["Mdwg"])
                report[f"dw_up[{e}]"] = _check("dw_up", to_np(b.dw_up[e][:, c]), wc["dwu"], wc["Mdwu"])
                report[f"dw_down[{e}]"] = _check("dw_down", to_np(b.dw_down[e][c, :]), wc["dwd"], wc["Mdwd"])
        for e in np.flatnonzero(counts == 0)[:4]:
            for buf in (b.dw_gate, b.dw_up, b.dw_down):
                assert torch.count_nonzero(buf[int(e)]).item() == 0
            assert float(b.dbias[int(e)]) == 0.0
        # router gradients of the smallest expert, from every token routed to it
        toks_e = sorted({int(p // k) for p in sc.pairs_of[small]})
        re_ = sc.tokens(toks_e)
        dwr_ref = sum(re_[t]["dl"][small] * x64[t] for t in toks_e)
        db_ref = sum(re_[t]["dl"][small] for t in toks_e)
        dwr = to_np(b.dw_router[:, small])
        scale = sum(abs(re_[t]["dl"][small]) * np.abs(x64[t]) for t in toks_e)
        assert np.max(np.abs(dwr - dwr_ref)) <= 2e-2 * np.sqrt(np.mean(dwr_ref ** 2)) + 4 * U_BF16 * np.max(scale)
        assert abs(float(b.dbias[small]) - db_ref) <= 4 * U_BF16 * sum(abs(re_[t]["dl"][small]) for t in toks_e) + 1e-6
        # the softmax gradient sums to zero over the experts of each token
        db = to_np(b.dbias)
        assert abs(db.sum()) <= 1e-3 * np.abs(db).sum() + 1e-6
        dwr_all = to_np(b.dw_router)
        assert np.max(np.abs(dwr_all.sum(1))) <= 1e-3 * np.max(np.abs(dwr_all).sum(1)) + 1e-6
    print(name, {k_: (round(v, 4) if isinstance(v, float) else v) for k_, v in report.items()})
