"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in the oracle (on the CPU, by monkeypatching a
function of ``oracle.moe_oracle``) and checks that the brute-force twin or the
finite differences then disagree with it.
"""
import numpy as np
import pytest

from oracle import bruteforce, moe_oracle as mo


# a clamp that binds at these scales (the pins of the clamped form run with it)
CLAMP = (1.0, 1.702, 1.0)


def _layer(seed=4, T=5, d=4, f=3, E=4, S=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((d, E))
    b = rng.standard_normal(E)
    wg = rng.standard_normal((E + S, d, f))
    wu = rng.standard_normal((E + S, d, f))
    wd = rng.standard_normal((E + S, f, d))
    dy = rng.standard_normal((T, d))
    return x, wr, b, wg, wu, wd, dy


def _agrees_with_bruteforce(k=2, act=None, S=0):
    x, wr, b, wg, wu, wd, dy = _layer(S=S)
    L = lambda a: a.tolist()  # noqa: E731
    bf = bruteforce.layer(L(x), L(wr), L(b), L(wg), L(wu), L(wd), k, L(dy), act=act, shared=S)
    fw = mo.forward(x, wr, b, wg, wu, wd, k, act=act, shared=S)
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy, fwd=fw, act=act, shared=S)
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


def _agrees_with_fd(k=2, act=None):
    x, wr, b, wg, wu, wd, dy = _sep_layer()
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy, act=act)
    eps = 1e-6
    for name, arr in {"dx": x, "dw_router": wr, "dw_gate": wg, "dw_up": wu, "dw_down": wd}.items():
        flat = arr.reshape(-1)
        num = np.zeros(flat.size)
        for i in range(flat.size):
            o = flat[i]
            flat[i] = o + eps; lp = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy, act=act)
            flat[i] = o - eps; lm = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy, act=act)
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
    assert _agrees_with_bruteforce(act=CLAMP, S=1)
    assert _agrees_with_fd()
    assert _agrees_with_fd(act=CLAMP)
    assert _agrees_on_ties()


def _swiglu_grad_no_g_term(G, U, act=None):
    L, al, c = mo.PLAIN_SWIGLU if act is None else act
    gc = np.minimum(G, L)
    s = 1.0 / (1.0 + np.exp(-al * gc))
    return s * (np.clip(U, -L, L) + c) * (G <= L), gc * s * ((U >= -L) & (U <= L))


_orig_swiglu = mo.swiglu
_orig_swiglu_grad = mo.swiglu_grad
_orig_forward = mo.forward


def _forward_shared_weight_2(*a, shared=0, **kw):
    """the shared experts' output added twice (weight 2 instead of 1)"""
    out = _orig_forward(*a, shared=shared, **kw)
    if shared:
        x, wg, wu, wd = a[0], a[3], a[4], a[5]
        E = np.asarray(a[1]).shape[1]
        for s_ in range(shared):
            _, _, _, yu = mo.expert_forward(mo.as_f64(x), wg[E + s_], wu[E + s_], wd[E + s_],
                                            kw.get("act"))
            out["y"] = out["y"] + yu
    return out


MUTANTS = {
    "dsilu drops the g*(1-s) term": ("swiglu_grad", _swiglu_grad_no_g_term),
    "silu with the wrong sign": (
        "swiglu", lambda G, U, act=None: -_orig_swiglu(-G, U, act) if act is None
        else _orig_swiglu(G, U, act)),
    "clamp of U dropped": (
        "swiglu", lambda G, U, act=None: _orig_swiglu(G, U, act) if act is None
        else _orig_swiglu(G, U, (act[0], act[1], act[2])) + (
            np.minimum(G, act[0]) / (1 + np.exp(-act[1] * np.minimum(G, act[0])))
            * (U - np.clip(U, -act[0], act[0])))),
    "clamp gradient kept past the limit": (
        "swiglu_grad", lambda G, U, act=None: _orig_swiglu_grad(G, U, act) if act is None
        else (_orig_swiglu_grad(np.minimum(G, act[0]), U, act)[0],
              _orig_swiglu_grad(G, np.clip(U, -act[0], act[0]), act)[1])),
    "shared expert weighted twice": ("forward", _forward_shared_weight_2),
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
        lambda xe, wg, wu, wd, act=None: (lambda G, U: (
            G, U, mo.swiglu(G, U, act), mo.swiglu(G, U, act) @ wd[:, ::-1]))(xe @ wg, xe @ wu)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(mo, attr, fn)
    caught_bf = not (_agrees_with_bruteforce() and _agrees_with_bruteforce(act=CLAMP, S=1))
    caught_fd = not (_agrees_with_fd() and _agrees_with_fd(act=CLAMP))
    caught_ties = not _agrees_on_ties()
    assert caught_bf or caught_fd or caught_ties, name
