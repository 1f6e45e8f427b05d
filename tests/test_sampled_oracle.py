"""The sampled evaluation (oracle/sampled.py + tests/sampled_check.py) agrees
with the whole-layer oracle and with the whole-tensor error magnitudes."""
import numpy as np

import workloads
from harness import magnitudes
from oracle import moe_oracle as mo
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
