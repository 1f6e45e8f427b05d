"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, by monkeypatching a
function of ``oracle.moe_oracle``) and checks that the brute-force twin or the
finite differences then disagree with it.
"""
import numpy as np
import pytest

from oracle import bruteforce, moe_oracle as mo


def _layer(seed=4, T=5, d=4, f=3, E=4):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((d, E))
    b = rng.standard_normal(E)
    wg = rng.standard_normal((E, d, f))
    wu = rng.standard_normal((E, d, f))
    wd = rng.standard_normal((E, f, d))
    dy = rng.standard_normal((T, d))
    return x, wr, b, wg, wu, wd, dy


def _agrees_with_bruteforce(k=2):
    x, wr, b, wg, wu, wd, dy = _layer()
    L = lambda a: a.tolist()  # noqa: E731
    bf = bruteforce.layer(L(x), L(wr), L(b), L(wg), L(wu), L(wd), k, L(dy))
    fw = mo.forward(x, wr, b, wg, wu, wd, k)
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy, fwd=fw)
    pairs = [(fw["y"], bf["y"]), (bw["dx"], bf["dx"]), (bw["dw_router"], bf["dwr"]),
             (bw["dw_gate"], bf["dwg"]), (bw["dw_up"], bf["dwu"]), (bw["dw_down"], bf["dwd"]),
             (bw["dbias"], bf["db"])]
    ok = np.array_equal(fw["idx"], np.array(bf["idx"]))
    return ok and all(np.allclose(a, np.array(b_), rtol=1e-9, atol=1e-10) for a, b_ in pairs)


def _sep_layer():
    rng = np.random.default_rng(21)
    while True:
        x = rng.standard_normal((3, 3)); wr = rng.standard_normal((3, 4)); b = rng.standard_normal(4)
        lg = np.sort(x @ wr + b, axis=1)[:, ::-1]
        if np.min(lg[:, 1] - lg[:, 2]) > 0.05:
            break
    wg = rng.standard_normal((4, 3, 2)); wu = rng.standard_normal((4, 3, 2)); wd = rng.standard_normal((4, 2, 3))
    return x, wr, b, wg, wu, wd, rng.standard_normal((3, 3))


def _agrees_with_fd(k=2):
    x, wr, b, wg, wu, wd, dy = _sep_layer()
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy)
    eps = 1e-6
    for name, arr in {"dx": x, "dw_router": wr, "dw_gate": wg, "dw_up": wu, "dw_down": wd}.items():
        flat = arr.reshape(-1)
        num = np.zeros(flat.size)
        for i in range(flat.size):
            o = flat[i]
            flat[i] = o + eps; lp = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy)
            flat[i] = o - eps; lm = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy)
            flat[i] = o
            num[i] = (lp - lm) / (2 * eps)
        if not np.allclose(bw[name].reshape(-1), num, rtol=1e-5, atol=1e-7):
            return False
    return True


def _agrees_on_ties():
    logits = np.array([[1.0, 3.0, 3.0, 0.5, 3.0], [0.0, 0.0, 0.0, 0.0, 0.0], [-1.0, 2.0, -1.0, 2.0, -0.0]])
    return all(list(mo.select_topk(logits, k)[t]) == bruteforce.topk_enumerate(list(logits[t]), k)
               for k in range(1, 6) for t in range(3))


def test_unmutated_oracle_passes():
    assert _agrees_with_bruteforce()
    assert _agrees_with_fd()
    assert _agrees_on_ties()


MUTANTS = {
    "dsilu drops the g*(1-s) term": ("dsilu", lambda g: 1.0 / (1.0 + np.exp(-g))),
    "silu with the wrong sign": ("silu", lambda g: g / (1.0 + np.exp(g))),
    "router backward sign flipped": (
        "router_backward",
        lambda w, dw, idx, E, _o=mo.router_backward: -_o(w, dw, idx, E)),
    "ties to the higher index": (
        "select_topk",
        lambda lg, k: (lg.shape[1] - 1 - np.argsort(-np.asarray(lg)[:, ::-1], axis=1, kind="stable"))[:, :k]),
    "weights not renormalised": (
        "topk_weights",
        lambda lg, idx: np.exp(np.take_along_axis(lg, idx, 1) - lg.max(1, keepdims=True))
        / np.exp(lg - lg.max(1, keepdims=True)).sum(1, keepdims=True)),
    "expert down weight transposed": (
        "expert_forward",
        lambda xe, wg, wu, wd: (lambda G, U: (G, U, mo.silu(G) * U, (mo.silu(G) * U) @ wd[:, ::-1]))(xe @ wg, xe @ wu)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(mo, attr, fn)
    caught_bf = not _agrees_with_bruteforce()
    caught_fd = not _agrees_with_fd()
    caught_ties = not _agrees_on_ties()
    assert caught_bf or caught_fd or caught_ties, name
