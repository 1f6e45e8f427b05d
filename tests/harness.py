"""Shared helpers of the GPU parity tests: run the layer through the C ABI,
run the oracle on the same seeded inputs, and compare.

Comparison rules:
  * integers (routing indices, counts, offsets, dst_row, src_pair): exact;
  * routing: the GPU's top-k must equal, bit for bit, the oracle's selection
    run on the GPU's own fp32 logits (both take the decision in fp32 — the
    exact upcast keeps fp32 order — with ties to the lower expert index);
    against the float64 logits the indices must agree except where two
    float64 logits lie within the fp32 error band of each other, and there
    every differing slot must be such a near-tie (PocketLLM "Qwen4-Exp
    Heterogeneous TP4 Performance", §Numerical gates: exact ties vs real
    flips). Downstream parity runs with the oracle's indices passed to both
    sides (forced_idx), so no GPU output feeds the oracle;
  * the stated bar, max |gpu - oracle| <= 2e-2 RMS(oracle), holds plainly
    for the fp32 results: logits, topk_w, d_topk_w and the router gradients
    dW_r, db;
  * for the layer's bf16 outputs y and dx the same bar holds for the error
    the computation adds to the rounding of the output format itself:
    element-wise |gpu - oracle| <= 2e-2 RMS(oracle) + half an ulp of bf16 at
    the element. The rounding alone is up to 2^-8 of an element's magnitude
    (an element just above a power of two), so wherever a tensor holds an
    element of more than 5.12 RMS the correctly rounded oracle itself can
    miss the plain bar; the plain max|diff|/RMS is reported all the same;
  * every other tensor — the bf16 operands A, dYp, dG, dU, the fp32 rows G,
    U (fp32 accumulations: far inside the bar), Yp and dXp, and the bf16
    weight gradients — is held to
      - RMS-relative error ||gpu - oracle||_2 / ||oracle||_2 <= 1e-2, and
      - element-wise |gpu - oracle| <= max(2e-2 RMS(oracle), MAG_C u M),
    u = 2^-8 (bf16), M the element's magnitude from a first-order forward
    error analysis of the kernel chain: the same computation in float64 with
    every input and product taken in absolute value, each stored bf16
    value's own rounding and the rounding it inherits from its inputs
    propagated through each GEMM (|A| |B| sums) and each element-wise step
    (|f'| terms). These tensors are heavy-tailed (a weight gradient of a few
    rows is an outer product; A = silu(G) U is a product of Gaussians; a
    bf16 operand near a zero of silu' moves dG by more than its own ulp), so
    the bf16 operands the tensor cores take put their largest elements past
    2e-2 RMS whatever the kernels do. MAG_C = 1: an fp32 emulation of exactly
    the kernels' rounding points (tests/emulation.py) reaches 0.5 of this
    bound at its worst element (a bf16 value's own rounding, dYp).
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
    """The plain stated bar: max|diff| <= tol * RMS(ref)."""
    e = rel_err(got, ref)
    assert e <= tol, f"{name}: max|diff| / RMS = {e:.3e} > {tol}"
    return e


def half_ulp_bf16(v) -> np.ndarray:
    """Half a unit in the last place of bf16 (8 significant bits) at |v|:
    2^(floor(log2 |v|) - 8); 0 at v = 0."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    out = np.zeros_like(a)
    nz = a > 0
    out[nz] = np.exp2(np.floor(np.log2(a[nz])) - 8.0)
    return out


def assert_bf16_out_close(name, got, ref, tol=TOL):
    """A bf16 output: |got - ref| <= tol RMS(ref) + half an ulp of bf16 at the
    element (the larger of |got| and |ref|, in case the rounding crossed a
    power of two). Returns the plain metric max|diff| / RMS(ref)."""
    ref = np.asarray(ref, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    diff = np.abs(got - ref)
    bound = tol * rms + half_ulp_bf16(np.maximum(np.abs(got), np.abs(ref))) + 1e-30
    ratio = float(np.max(diff / bound))
    plain = float(np.max(diff)) / rms if rms > 0 else 0.0
    assert ratio <= 1.0, (f"{name}: worst |diff| / (2e-2 RMS + ulp/2) = {ratio:.3f} > 1 "
                          f"(max|diff|/RMS = {plain:.3e})")
    return plain


def bf16_floor(ref) -> float:
    """max|bf16(ref) - ref| / RMS(ref): what the output format's rounding of the
    exact answer alone makes of the plain metric."""
    r = np.asarray(ref, dtype=np.float64)
    if r.size == 0:
        return 0.0
    rb = torch.from_numpy(r).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    rms = float(np.sqrt(np.mean(r * r)))
    return float(np.max(np.abs(rb - r))) / rms if rms > 0 else 0.0


MAG_C = 1.0
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


def act_derivs(G, U, act=None):
    """The activation A(G, U) of act = (L, alpha, c) (None: the plain SwiGLU)
    and its first and second partial derivatives, element-wise:
    A, A_g, A_u, A_gg, A_gu (A_uu = 0). Zero past the clamps."""
    L, al, c = mo.PLAIN_SWIGLU if act is None else act
    gc = np.minimum(G, L)
    uc = np.clip(U, -L, L)
    s = 1.0 / (1.0 + np.exp(-al * gc))
    h = gc * s
    h1 = s + al * gc * s * (1 - s)
    h2 = al * s * (1 - s) * (2 + al * gc * (1 - 2 * s))
    ing = (G <= L).astype(np.float64)
    inu = ((U >= -L) & (U <= L)).astype(np.float64)
    return h * (uc + c), h1 * (uc + c) * ing, h * inu, h2 * (uc + c) * ing, h1 * ing * inu


def magnitudes(inp, fw, bw, k, act=None, shared=0):
    """Per-element first-order error magnitudes (see the module docstring).
    Keys follow the oracle's: G, U, A, Yu, y, dYu, dA, dG, dU, dXp, dx,
    d_topk_w, dw_gate, dw_up, dw_down, dw_router, dbias, logits."""
    x = mo.as_f64(inp["x"])
    ax = np.abs(x)
    T, d = x.shape
    idx = fw["idx"]
    E = int(np.asarray(mo.as_f64(inp["w_router"])).shape[1])
    EE = E + shared
    P = T * (k + shared)
    e_of_p = mo.pair_experts(idx, E, shared)
    tok = np.concatenate([np.arange(T * k) // k] + [np.arange(T)] * shared)
    w = np.concatenate([fw["w"].reshape(-1)] + [np.ones(T)] * shared)
    G, U, A = fw["G"], fw["U"], fw["A"]
    _, Ag, Au, Agg, Agu = act_derivs(G, U, act)
    f = G.shape[1]
    MG = np.zeros((P, f)); MU = np.zeros((P, f)); MYu = np.zeros((P, d))
    have_bw = bw is not None
    if have_bw:
        dy = mo.as_f64(inp["dy"])
        ady = np.abs(dy)
        dA, dG, dU = bw["dA"], bw["dG"], bw["dU"]
        MdYu = np.abs(w)[:, None] * ady[tok] + np.abs(bw["dYu"])
        MdA = np.zeros((P, f)); MdXp = np.zeros((P, d))
        MdG = np.zeros((P, f)); MdU = np.zeros((P, f))
        Mdwg = np.zeros((EE, d, f)); Mdwu = np.zeros((EE, d, f)); Mdwd = np.zeros((EE, f, d))
    for e in range(EE):
        pairs = np.flatnonzero(e_of_p == e)
        if pairs.size == 0:
            continue
        awg = np.abs(mo.as_f64(inp["w_gate"][e]))
        awu = np.abs(mo.as_f64(inp["w_up"][e]))
        xe = ax[tok[pairs]]
        MG[pairs] = xe @ awg + np.abs(G[pairs])
        MU[pairs] = xe @ awu + np.abs(U[pairs])
    MA = np.abs(Ag) * MG + np.abs(Au) * MU + np.abs(A)
    for e in range(EE):
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
            MdG[p_] = (MdA[p_] * np.abs(Ag[p_])
                       + np.abs(dA[p_]) * (np.abs(Agg[p_]) * MG[p_] + np.abs(Agu[p_]) * MU[p_])
                       + np.abs(dG[p_]))
            MdU[p_] = MdA[p_] * np.abs(Au[p_]) + np.abs(dA[p_] * Agu[p_]) * MG[p_] + np.abs(dU[p_])
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
        Mdtw = np.einsum("pd,pd->p", ady[tok[:T * k]], MYu[:T * k]).reshape(T, k)
        out["d_topk_w"] = Mdtw
        aw = np.abs(fw["w"])
        Mdl_sel = aw * (Mdtw + (aw * Mdtw).sum(1, keepdims=True)) + np.abs(
            np.take_along_axis(bw["dl"], idx, 1))
        Mdl = np.zeros((T, E))
        np.put_along_axis(Mdl, idx, Mdl_sel, axis=1)
        Mdx = np.zeros((T, d))
        np.add.at(Mdx, tok, MdXp)
        Mdx = Mdx + Mdl @ awr.T + np.abs(bw["dx"])
        out["dx"] = Mdx
        out["dw_router"] = ax.T @ Mdl
        out["dbias"] = Mdl.sum(0)
    return out


def tie_band(logits_gpu, logits_ref) -> float:
    return 8.0 * float(np.max(np.abs(logits_gpu - logits_ref))) + 1e-6


def check_routing(idx_gpu, idx_ref, logits_ref, band):
    """Exact where the float64 order is clear. At a token whose selection
    differs, every slot whose expert differs must hold an expert whose
    float64 logit is within the band of the oracle's expert in that slot (a
    near-tie: an order swap or a swap at the k-th place), and the selection
    must still be a valid top-k of the float64 logits up to the band.
    Returns the number of tokens that differ."""
    idx_gpu = np.asarray(idx_gpu, dtype=np.int64)
    idx_ref = np.asarray(idx_ref, dtype=np.int64)
    diff = np.flatnonzero(np.any(idx_gpu != idx_ref, axis=1))
    for t in diff:
        lg = logits_ref[t]
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == len(sel), f"token {t}: repeated expert"
        rest = np.setdiff1d(np.arange(lg.size), sel)
        if rest.size:
            assert lg[sel].min() >= lg[rest].max() - band, f"token {t}: not a top-k"
        for j in np.flatnonzero(sel != idx_ref[t]):
            a, r = int(sel[j]), int(idx_ref[t, j])
            assert abs(lg[a] - lg[r]) <= band, (
                f"token {t} slot {j}: expert {a} vs {r}, float64 logits "
                f"{lg[a]:.9g} vs {lg[r]:.9g} differ by more than the band {band:.3g}")
    return int(diff.size)


def check_routing_on_own_logits(idx_gpu, w_gpu, logits_gpu, k):
    """The GPU's indices equal, bit for bit, the oracle's selection run on
    the GPU's own fp32 logits; its weights equal the oracle's renormalised
    softmax of those logits within the stated bar."""
    lg = np.asarray(logits_gpu, dtype=np.float64)
    ref = mo.select_topk(lg, k)
    np.testing.assert_array_equal(np.asarray(idx_gpu, dtype=np.int64), ref)
    assert_close("topk_w (own logits)", w_gpu, mo.topk_weights(lg, ref))


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


def layer_act(layer):
    """The layer's activation as the oracle's (L, alpha, c) tuple, or None."""
    a = layer.act
    return None if a is None else (float(a.limit), float(a.alpha), float(a.up_offset))


def compare_full(layer, inp, k, align, backward=True, report=None):
    """Complete parity of every output against the float64 oracle. Returns
    ({tensor: max|diff| / RMS}, buffers). The layer's activation and shared
    experts (layer.act, layer.S) are the oracle's act and shared."""
    act, S = layer_act(layer), layer.S
    x64 = mo.as_f64(inp["x"])
    fw = mo.forward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                    inp["w_down"], k, act=act, shared=S)
    # 1) free routing on the GPU: indices exactly the oracle's selection on the
    #    GPU's fp32 logits; logits within the bar; against the float64 logits
    #    exact up to near-ties
    b, _, _ = gpu_forward_backward(layer, inp, None, backward=False)
    lg_gpu = to_np(b.logits)
    check_routing_on_own_logits(to_np(b.topk_idx), to_np(b.topk_w), lg_gpu, k)
    assert_close("logits", lg_gpu, fw["logits"])
    band = tie_band(lg_gpu, fw["logits"])
    flips = check_routing(to_np(b.topk_idx), fw["idx"], fw["logits"], band)
    # 2) everything downstream, with the oracle's routing forced on both sides
    b, _, dy = gpu_forward_backward(layer, inp, fw["idx"], backward=backward)
    bw = None
    if backward:
        bw = mo.backward(inp["x"], inp["w_router"], inp.get("bias"), inp["w_gate"], inp["w_up"],
                         inp["w_down"], k, inp["dy"], fwd=fw, act=act, shared=S)
    mag = magnitudes(inp, fw, bw, k, act=act, shared=S)

    out = {"near_tie_tokens": flips}
    np.testing.assert_array_equal(to_np(b.topk_idx), fw["idx"])
    out["topk_w"] = assert_close("topk_w", to_np(b.topk_w), fw["w"])
    T = x64.shape[0]
    E = layer.E
    maps = mo.permute_maps(fw["idx"], E, align, b.R_cap, shared=S)
    np.testing.assert_array_equal(to_np(b.counts), maps["counts"])
    np.testing.assert_array_equal(to_np(b.offsets), maps["offsets"])
    np.testing.assert_array_equal(to_np(b.dst_row), maps["dst_row"])
    np.testing.assert_array_equal(to_np(b.src_pair), maps["src_pair"])
    R_pad = maps["R_pad"]
    dst = maps["dst_row"]
    pad = np.setdiff1d(np.arange(R_pad), dst)
    tok = np.concatenate([np.arange(T * k) // k] + [np.arange(T)] * S)

    def rows(buf):
        return to_np(buf[:R_pad])

    xp = rows(b.xp)
    np.testing.assert_array_equal(xp[dst], x64[tok])   # a copy: exact
    assert np.all(xp[pad] == 0)
    for name, buf in (("G", b.g), ("U", b.u), ("A", b.a), ("Yu", b.yp)):
        r = rows(buf)
        out[name] = assert_mag_close(name, r[dst], fw[name], mag[name])
        assert np.all(r[pad] == 0), f"{name}: padding rows not zero"
    out["y"] = assert_bf16_out_close("y", to_np(b.y), fw["y"])
    out["y_bf16_floor"] = bf16_floor(fw["y"])
    if not backward:
        return out, b
    dyg = rows(b.dyg)
    np.testing.assert_array_equal(dyg[dst], mo.as_f64(inp["dy"])[tok])   # a copy: exact
    assert np.all(dyg[pad] == 0)
    for name, buf, key in (("dYp", b.dyp, "dYu"), ("dG", b.dg, "dG"), ("dU", b.du, "dU"),
                           ("dXp", b.dxp, "dXp")):
        r = rows(buf)
        out[name] = assert_mag_close(name, r[dst], bw[key], mag[key])
        assert np.all(r[pad] == 0), f"{name}: padding rows not zero"
    out["d_topk_w"] = assert_close("d_topk_w", to_np(b.d_topk_w), bw["d_topk_w"])
    out["dx"] = assert_bf16_out_close("dx", to_np(b.dx), bw["dx"])
    out["dx_bf16_floor"] = bf16_floor(bw["dx"])
    for name, buf in (("dw_gate", b.dw_gate), ("dw_up", b.dw_up), ("dw_down", b.dw_down)):
        out[name] = assert_mag_close(name, to_np(buf), bw[name], mag[name])
    for name, buf in (("dw_router", b.dw_router), ("dbias", b.dbias)):
        out[name] = assert_close(name, to_np(buf), bw[name])
    # experts with no rows get exactly zero weight gradients
    empty = np.flatnonzero(maps["counts"] == 0)
    for e in empty:
        for buf in (b.dw_gate, b.dw_up, b.dw_down):
            assert torch.count_nonzero(buf[e]).item() == 0
        if e < E:
            assert float(b.dbias[e]) == 0.0
    if report is not None:
        report.update(out)
    return out, b
