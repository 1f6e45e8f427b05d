"""The sampled evaluation (oracle/sampled.py + tests/sampled_check.py) and the
expert-by-expert evaluation (oracle/streamed.py) agree with the whole-layer
oracle and with the whole-tensor error magnitudes."""
import numpy as np

import workloads
from harness import magnitudes
from oracle import moe_oracle as mo
from oracle.streamed import stream_layer
from sampled_check import SampledChecker


def test_sampled_matches_full_oracle_and_magnitudes():
    wl = workloads.Workload("s", T=40, d=24, f=16, E=6, k=2, zipf_s=1.2)
    inp = workloads.generate(wl, tau=1.0)
    fw = mo.forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                    inp["w_down"], wl.k)
    bw = mo.backward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                     inp["w_down"], wl.k, inp["dy"], fwd=fw)
    mag = magnitudes(inp, fw, bw, wl.k)
    sc = SampledChecker(inp, fw["logits"], fw["idx"], wl.k)
    toks = sc.tokens(range(wl.T))
    for t, r in toks.items():
        np.testing.assert_allclose(r["y"], fw["y"][t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["dx"], bw["dx"][t], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(r["dtw"], bw["d_topk_w"][t], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["My"], mag["y"][t], rtol=1e-10)
        np.testing.assert_allclose(r["Mdx"], mag["dx"][t], rtol=1e-10)
        for j in range(wl.k):
            p = t * wl.k + j
            for key in ("G", "U", "A", "Yu", "dXp"):
                np.testing.assert_allclose(r["pairs"][j][key], fw[key][p] if key in fw else bw[key][p],
                                           rtol=1e-10, atol=1e-12)
            for key in ("G", "U", "A", "Yu", "dXp"):
                np.testing.assert_allclose(r["pairs"][j]["M" + key], mag[key][p], rtol=1e-10)
    counts = np.bincount(fw["idx"].reshape(-1), minlength=wl.E)
    for e in range(wl.E):
        for c in (0, wl.f - 1, 5):
            w = sc.wgrad_cols(e, c)
            np.testing.assert_allclose(w["dwg"], bw["dw_gate"][e][:, c], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(w["dwu"], bw["dw_up"][e][:, c], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(w["dwd"], bw["dw_down"][e][c, :], rtol=1e-10, atol=1e-12)
            if counts[e]:
                np.testing.assert_allclose(w["Mdwg"], mag["dw_gate"][e][:, c], rtol=1e-10)
                np.testing.assert_allclose(w["Mdwu"], mag["dw_up"][e][:, c], rtol=1e-10)
                np.testing.assert_allclose(w["Mdwd"], mag["dw_down"][e][c, :], rtol=1e-10)


def test_streamed_layer_matches_full_oracle():
    """Skewed routing with empty experts; kept experts' rows and weight
    gradients, and every token's y, dx, d_topk_w, dW_r, db."""
    wl = workloads.Workload("st", T=64, d=40, f=24, E=12, k=3, zipf_s=1.2)
    inp = workloads.generate(wl, tau=1.5)
    fw = mo.forward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                    inp["w_down"], wl.k)
    bw = mo.backward(inp["x"], inp["w_router"], inp["bias"], inp["w_gate"], inp["w_up"],
                     inp["w_down"], wl.k, inp["dy"], fwd=fw)
    counts = np.bincount(fw["idx"].reshape(-1), minlength=wl.E)
    assert (counts == 0).any()
    keep = [int(e) for e in np.flatnonzero(counts > 0)[:3]]
    st = stream_layer(inp, fw["logits"], fw["idx"], wl.k, keep=keep)
    for key, ref in (("y", fw["y"]), ("dx", bw["dx"]), ("d_topk_w", bw["d_topk_w"]),
                     ("dl", bw["dl"]), ("dw_router", bw["dw_router"]), ("dbias", bw["dbias"])):
        np.testing.assert_allclose(st[key], ref, rtol=1e-10, atol=1e-12, err_msg=key)
    mag = magnitudes(inp, fw, bw, wl.k)
    sc = SampledChecker(inp, fw["logits"], fw["idx"], wl.k)
    for e in keep:
        rec = st["experts"][e]
        pairs = rec["pairs"]
        np.testing.assert_array_equal(pairs, np.flatnonzero(fw["idx"].reshape(-1) == e))
        for key, src in (("G", fw), ("U", fw), ("A", fw), ("Yu", fw), ("dYu", bw), ("dG", bw),
                         ("dU", bw), ("dXp", bw)):
            np.testing.assert_allclose(rec[key], src[key][pairs], rtol=1e-10, atol=1e-12)
        for key in ("dw_gate", "dw_up", "dw_down"):
            np.testing.assert_allclose(rec[key], bw[key][e], rtol=1e-10, atol=1e-12)
        em = sc.expert_mags(e)
        for key in ("G", "U", "A", "Yu", "dYu", "dG", "dU", "dXp"):
            np.testing.assert_allclose(em["M" + key], mag[key][pairs], rtol=1e-10)
        np.testing.assert_allclose(em["Mdwg"], mag["dw_gate"][e], rtol=1e-10)
        np.testing.assert_allclose(em["Mdwu"], mag["dw_up"][e], rtol=1e-10)
        np.testing.assert_allclose(em["Mdwd"], mag["dw_down"][e], rtol=1e-10)
