"""Shared helpers of the GPU parity tests: run the layer through the C ABI,
run the oracle on the same seeded inputs, and compare.

Comparison rules:
  * integers (routing indices, counts, offsets, dst_row, src_pair): exact;
  * values: max |gpu - oracle| <= TOL * RMS(oracle), per tensor, TOL = 2e-2;
  * routing indices are decided on fp32 logits on the GPU and on float64
    logits in the oracle. Where the float64 logits of two experts lie within
    the fp32 error band of each other the two may legitimately order them
    differently; there the GPU's choice is checked for validity (it is a
    top-k of the float64 logits up to the band) instead of equality, and the
    downstream parity runs with the oracle's indices passed in as
    forced_idx so both sides compute the same routing.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as mo

TOL = 2e-2


def to_np(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.numpy().astype(np.float64) if t.is_floating_point() else t.numpy()


def rel_err(got, ref) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    if rms == 0.0:
        return 0.0 if err == 0.0 else float("inf")
    return err / rms


def assert_close(name, got, ref, tol=TOL):
    e = rel_err(got, ref)
    assert e <= tol, f"{name}: max|diff| / RMS = {e:.3e} > {tol}"
    return e


def tie_band(logits_gpu, logits_ref) -> float:
    return 8.0 * float(np.max(np.abs(logits_gpu - logits_ref))) + 1e-6


def check_routing(idx_gpu, idx_ref, logits_ref, band):
    """Exact where the float64 order is clear; valid top-k within the band elsewhere.
    Returns the number of tokens that differ."""
    idx_gpu = np.asarray(idx_gpu, dtype=np.int64)
    diff = np.flatnonzero(np.any(idx_gpu != idx_ref, axis=1))
    for t in diff:
        lg = logits_ref[t]
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == len(sel), f"token {t}: repeated expert"
        rest = np.setdiff1d(np.arange(lg.size), sel)
        # every selected logit is at least every unselected one, up to the band
        if rest.size:
            assert lg[sel].min() >= lg[rest].max() - band, f"token {t}: not a top-k"
        # slots in descending order up to the band
        assert np.all(np.diff(lg[sel]) <= band), f"token {t}: slots out of order"
        # and the disagreement is a near-tie in float64
        ref_sel = idx_ref[t]
        assert abs(lg[sel].sum() - lg[ref_sel].sum()) <= len(sel) * band, f"token {t}: real flip"
    return int(diff.size)


def gpu_forward_backward(layer, inp, forced_idx=None, backward=True, dev="cuda"):
    """Run the layer through the C ABI. Returns (buffers, x_dev, dy_dev)."""
    x = inp["x"].to(dev)
    T = x.shape[0]
    b = layer.buffers(T, backward=backward)
    fi = None if forced_idx is None else torch.as_tensor(forced_idx, dtype=torch.int32).to(dev)
    layer.forward(x, b, forced_idx=fi)
    dy = None
    if backward:
        dy = inp["dy"].to(dev)
        layer.backward(dy, b)
    status = layer.status()
    assert status == 0, f"device status {status}"
    return b, x, dy


def compare_full(layer, inp, k, align, backward=True, report=None):
    """Complete parity of every output against the float64 oracle."""
    x64 = mo.as_f64(inp["x"])
    fw = mo.forward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                    inp["w_down"], k)
    # 1) free routing on the GPU: logits within tolerance, indices exact up to near-ties
    b, _, _ = gpu_forward_backward(layer, inp, None, backward=False)
    lg_gpu = to_np(b.logits)
    assert_close("logits", lg_gpu, fw["logits"])
    band = tie_band(lg_gpu, fw["logits"])
    flips = check_routing(to_np(b.topk_idx), fw["idx"], fw["logits"], band)
    # 2) everything downstream, with the oracle's routing forced on both sides
    b, _, _ = gpu_forward_backward(layer, inp, fw["idx"], backward=backward)
    out = {"near_tie_tokens": flips}
    np.testing.assert_array_equal(to_np(b.topk_idx), fw["idx"])
    assert_close("topk_w", to_np(b.topk_w), fw["w"])
    T = x64.shape[0]
    E = layer.E
    maps = mo.permute_maps(fw["idx"], E, align, b.R_cap)
    np.testing.assert_array_equal(to_np(b.counts), maps["counts"])
    np.testing.assert_array_equal(to_np(b.offsets), maps["offsets"])
    np.testing.assert_array_equal(to_np(b.dst_row), maps["dst_row"])
    np.testing.assert_array_equal(to_np(b.src_pair), maps["src_pair"])
    R_pad = maps["R_pad"]
    dst = maps["dst_row"]
    pad = np.setdiff1d(np.arange(R_pad), dst)

    def rows(buf):
        return to_np(buf[:R_pad])

    xp = rows(b.xp)
    np.testing.assert_array_equal(xp[dst], x64[np.arange(T * k) // k])   # a copy: exact
    assert np.all(xp[pad] == 0)
    for name, buf in (("G", b.g), ("U", b.u), ("A", b.a), ("Yu", b.yp)):
        r = rows(buf)
        out[name] = assert_close(name, r[dst], fw[name])
        assert np.all(r[pad] == 0), f"{name}: padding rows not zero"
    out["y"] = assert_close("y", to_np(b.y), fw["y"])
    if not backward:
        return out, b
    bw = mo.backward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                     inp["w_down"], k, inp["dy"], fwd=fw)
    for name, buf, key in (("dYp", b.dyp, "dYu"), ("dG", b.dg, "dG"), ("dU", b.du, "dU"),
                           ("dXp", b.dxp, "dXp")):
        r = rows(buf)
        out[name] = assert_close(name, r[dst], bw[key])
        assert np.all(r[pad] == 0), f"{name}: padding rows not zero"
    out["d_topk_w"] = assert_close("d_topk_w", to_np(b.d_topk_w), bw["d_topk_w"])
    for name, buf, key in (("dx", b.dx, "dx"), ("dw_gate", b.dw_gate, "dw_gate"),
                           ("dw_up", b.dw_up, "dw_up"), ("dw_down", b.dw_down, "dw_down"),
                           ("dw_router", b.dw_router, "dw_router")):
        out[name] = assert_close(name, to_np(buf), bw[key])
    out["dbias"] = assert_close("dbias", to_np(b.dbias), bw["dbias"])
    # experts with no rows get exactly zero weight gradients
    empty = np.flatnonzero(maps["counts"] == 0)
    for e in empty:
        for buf in (b.dw_gate, b.dw_up, b.dw_down):
            assert torch.count_nonzero(buf[e]).item() == 0
        assert float(b.dbias[e]) == 0.0
    if report is not None:
        report.update(out)
    return out, b
