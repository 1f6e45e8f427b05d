"""Pins of the CPU oracle against things other than itself.

Brute force (a separately written scalar-loop twin, with top-k by subset
enumeration), closed forms, the dense-MLP special case, finite differences.
All CPU, all float64.
"""
import itertools

import numpy as np
import pytest

from oracle import bruteforce, moe_oracle as mo


def _rand_layer(rng, T, d, f, E, bias=True, scale_r=1.0):
    x = rng.standard_normal((T, d))
    wr = rng.standard_normal((d, E)) * scale_r
    b = rng.standard_normal(E) if bias else None
    wg = rng.standard_normal((E, d, f)) / np.sqrt(d)
    wu = rng.standard_normal((E, d, f)) / np.sqrt(d)
    wd = rng.standard_normal((E, f, d)) / np.sqrt(f)
    dy = rng.standard_normal((T, d))
    return x, wr, b, wg, wu, wd, dy


def _lists(a):
    return None if a is None else np.asarray(a).tolist()


CASES = [(T, d, f, E, k) for (T, d, f, E) in [(1, 1, 1, 1), (3, 2, 3, 2), (5, 4, 3, 3), (8, 8, 8, 4), (7, 3, 5, 4)]
         for k in range(1, E + 1)]


@pytest.mark.parametrize("T,d,f,E,k", CASES)
def test_oracle_matches_bruteforce(T, d, f, E, k):
    rng = np.random.default_rng(1000 + 97 * T + 13 * d + 7 * f + 3 * E + k)
    x, wr, b, wg, wu, wd, dy = _rand_layer(rng, T, d, f, E)
    bf = bruteforce.layer(_lists(x), _lists(wr), _lists(b), _lists(wg), _lists(wu), _lists(wd), k, _lists(dy))
    fw = mo.forward(x, wr, b, wg, wu, wd, k)
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy, fwd=fw)
    np.testing.assert_array_equal(fw["idx"], np.array(bf["idx"]))
    np.testing.assert_allclose(fw["logits"], bf["logits"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(fw["w"], bf["w"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fw["y"], bf["y"], rtol=1e-11, atol=1e-12)
    for key_o, key_b in [("dx", "dx"), ("dw_router", "dwr"), ("dbias", "db"), ("dw_gate", "dwg"),
                         ("dw_up", "dwu"), ("dw_down", "dwd"), ("d_topk_w", "dtw"), ("dl", "dl")]:
        np.testing.assert_allclose(bw[key_o], np.array(bf[key_b]), rtol=1e-10, atol=1e-11, err_msg=key_o)


def test_topk_ties_lower_index_first():
    # exact ties: the lower expert index ranks first, both in the oracle and by enumeration
    logits = np.array([[1.0, 3.0, 3.0, 0.5, 3.0],
                       [0.0, 0.0, 0.0, 0.0, 0.0],
                       [-1.0, 2.0, -1.0, 2.0, -0.0]])
    for k in range(1, 6):
        idx = mo.select_topk(logits, k)
        for t in range(logits.shape[0]):
            assert list(idx[t]) == bruteforce.topk_enumerate(list(logits[t]), k)
    assert list(mo.select_topk(logits, 3)[0]) == [1, 2, 4]
    assert list(mo.select_topk(logits, 5)[1]) == [0, 1, 2, 3, 4]
    assert list(mo.select_topk(logits, 3)[2]) == [1, 3, 4]   # -0.0 == 0.0 > -1


def test_weights_closed_forms():
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((64, 16)) * 3
    for k in (1, 2, 5, 16):
        idx = mo.select_topk(logits, k)
        w = mo.topk_weights(logits, idx)
        assert np.all(np.abs(w.sum(1) - 1.0) < 1e-12)
        assert np.all(np.diff(w, axis=1) <= 0)             # slots ordered by descending weight
        if k == 1:
            assert np.all(w == 1.0)
        # renormalised weights equal the full softmax restricted to S and renormalised
        p = np.exp(logits - logits.max(1, keepdims=True))
        p /= p.sum(1, keepdims=True)
        ps = np.take_along_axis(p, idx, 1)
        np.testing.assert_allclose(w, ps / ps.sum(1, keepdims=True), rtol=1e-12)
        dw = rng.standard_normal(w.shape)
        dl = mo.router_backward(w, dw, idx, 16)
        assert np.all(np.abs(dl.sum(1)) < 1e-12)           # softmax gradient sums to zero


def _dense_mlp(x, wg, wu, wd, dy):
    """A dense SwiGLU MLP and its gradients, written out for this test."""
    g = x @ wg
    u = x @ wu
    sig = 1 / (1 + np.exp(-g))
    a = g * sig * u
    y = a @ wd
    da = dy @ wd.T
    dg = da * u * (sig + g * sig * (1 - sig))
    du = da * g * sig
    dx = dg @ wg.T + du @ wu.T
    return y, dx, x.T @ dg, x.T @ du, a.T @ dy


@pytest.mark.parametrize("E", [1, 2, 5])
def test_k_equals_E_identical_experts_is_dense_mlp(E):
    rng = np.random.default_rng(11 + E)
    T, d, f = 9, 6, 7
    x, wr, b, wg, wu, wd, dy = _rand_layer(rng, T, d, f, E)
    wg[:] = wg[0]
    wu[:] = wu[0]
    wd[:] = wd[0]
    fw = mo.forward(x, wr, b, wg, wu, wd, E)
    bw = mo.backward(x, wr, b, wg, wu, wd, E, dy, fwd=fw)
    y, dx, dwg, dwu, dwd = _dense_mlp(x, wg[0], wu[0], wd[0], dy)
    np.testing.assert_allclose(fw["y"], y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bw["dx"], dx, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bw["dw_gate"].sum(0), dwg, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bw["dw_up"].sum(0), dwu, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(bw["dw_down"].sum(0), dwd, rtol=1e-10, atol=1e-12)
    assert np.abs(bw["dw_router"]).max() < 1e-12       # identical experts: routing has no gradient
    assert np.abs(bw["dbias"]).max() < 1e-12


def _separated_layer(seed, T, d, f, E, k, gap=2e-2):
    rng = np.random.default_rng(seed)
    for _ in range(1000):
        lay = _rand_layer(rng, T, d, f, E)
        x, wr, b = lay[:3]
        lg = np.sort(mo.router_logits(x, wr, b), axis=1)[:, ::-1]
        if k == E or np.min(lg[:, k - 1] - lg[:, k]) > gap:
            return lay
    raise RuntimeError("no separated draw")


@pytest.mark.parametrize("T,d,f,E,k", [(3, 4, 5, 4, 2), (4, 3, 6, 3, 1), (2, 5, 4, 4, 4), (5, 6, 3, 6, 3)])
def test_backward_matches_finite_differences(T, d, f, E, k):
    x, wr, b, wg, wu, wd, dy = _separated_layer(7 * T + d, T, d, f, E, k)
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy)
    eps = 1e-6
    params = {"dx": x, "dw_router": wr, "dbias": b, "dw_gate": wg, "dw_up": wu, "dw_down": wd}
    for gname, arr in params.items():
        num = np.zeros_like(arr)
        for pos in itertools.product(*[range(s) for s in arr.shape]):
            old = arr[pos]
            arr[pos] = old + eps
            lp = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy)
            arr[pos] = old - eps
            lm = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy)
            arr[pos] = old
            num[pos] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(bw[gname], num, rtol=1e-6, atol=1e-8, err_msg=gname)


# ----------------------------------------------------- clamped SwiGLU, shared experts
# (prime-rl PR #3885, §Changes, "FP8 routed experts" and "Fused FP8 shared
# expert": a clamped SwiGLU, and shared experts whose output is added to the
# routed one in the write-back; the clamp's constants are the GPT-OSS-20B
# model's, the pages do not print them)

def test_clamped_swiglu_closed_forms():
    rng = np.random.default_rng(3)
    G = rng.standard_normal(4000) * 8
    U = rng.standard_normal(4000) * 8
    L, al, c = mo.CLAMPED_SWIGLU_GPT_OSS
    A = mo.swiglu(G, U, mo.CLAMPED_SWIGLU_GPT_OSS)
    # where neither clamp binds: g * sigmoid(alpha g) * (u + 1), written out here
    free = (G < L) & (np.abs(U) < L)
    assert free.sum() > 1000 and (~free).sum() > 500
    np.testing.assert_allclose(A[free], G[free] / (1 + np.exp(-al * G[free])) * (U[free] + c),
                               rtol=1e-14)
    # G above the limit: A no longer depends on G; U past the limit: nor on U
    big = G > L
    np.testing.assert_allclose(A[big], L / (1 + np.exp(-al * L)) * (np.clip(U[big], -L, L) + c),
                               rtol=1e-14)
    # the plain activation is the special case (inf, 1, 0), bitwise
    assert np.array_equal(mo.swiglu(G, U, (np.inf, 1.0, 0.0)), mo.silu(G) * U)
    # and the derivatives match central differences away from the kinks
    ok = (np.abs(G - L) > 1e-3) & (np.abs(np.abs(U) - L) > 1e-3)
    eps = 1e-6
    dg, du = mo.swiglu_grad(G, U, mo.CLAMPED_SWIGLU_GPT_OSS)
    ng = (mo.swiglu(G + eps, U, mo.CLAMPED_SWIGLU_GPT_OSS)
          - mo.swiglu(G - eps, U, mo.CLAMPED_SWIGLU_GPT_OSS)) / (2 * eps)
    nu = (mo.swiglu(G, U + eps, mo.CLAMPED_SWIGLU_GPT_OSS)
          - mo.swiglu(G, U - eps, mo.CLAMPED_SWIGLU_GPT_OSS)) / (2 * eps)
    np.testing.assert_allclose(dg[ok], ng[ok], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(du[ok], nu[ok], rtol=1e-6, atol=1e-7)
    assert np.all(dg[G > L] == 0) and np.all(du[np.abs(U) > L] == 0)


@pytest.mark.parametrize("S", [1, 2])
def test_shared_experts_add_a_dense_mlp(S):
    """With S shared experts the layer is the routed layer plus, per shared
    expert, a dense SwiGLU MLP of every token; the gradients add the same
    way, and the routing gradients do not see the shared experts."""
    rng = np.random.default_rng(40 + S)
    T, d, f, E, k = 7, 5, 6, 4, 2
    x, wr, b, wg, wu, wd, dy = _rand_layer(rng, T, d, f, E + S)
    fw0 = mo.forward(x, wr[:, :E], b[:E], wg[:E], wu[:E], wd[:E], k)
    bw0 = mo.backward(x, wr[:, :E], b[:E], wg[:E], wu[:E], wd[:E], k, dy, fwd=fw0)
    fw = mo.forward(x, wr[:, :E], b[:E], wg, wu, wd, k, shared=S)
    bw = mo.backward(x, wr[:, :E], b[:E], wg, wu, wd, k, dy, fwd=fw, shared=S)
    y, dx = fw0["y"].copy(), bw0["dx"].copy()
    for s in range(S):
        ys, dxs, dwg, dwu, dwd = _dense_mlp(x, wg[E + s], wu[E + s], wd[E + s], dy)
        y += ys
        dx += dxs
        np.testing.assert_allclose(bw["dw_gate"][E + s], dwg, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(bw["dw_up"][E + s], dwu, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(bw["dw_down"][E + s], dwd, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(fw["y"], y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(bw["dx"], dx, rtol=1e-10, atol=1e-12)
    for key in ("d_topk_w", "dl", "dw_router", "dbias"):
        np.testing.assert_allclose(bw[key], bw0[key], rtol=1e-12, atol=1e-14, err_msg=key)
    for key in ("dw_gate", "dw_up", "dw_down"):
        np.testing.assert_allclose(bw[key][:E], bw0[key], rtol=1e-12, atol=1e-14, err_msg=key)
    # the layout: each shared expert holds every token once, in token order
    maps = mo.permute_maps(fw["idx"], E, 4, shared=S)
    for s in range(S):
        g0 = maps["offsets"][E + s]
        assert maps["counts"][E + s] == T
        np.testing.assert_array_equal(maps["src_pair"][g0:g0 + T], T * k + s * T + np.arange(T))


@pytest.mark.parametrize("S", [0, 1])
def test_clamped_and_shared_backward_matches_finite_differences(S):
    T, d, f, E, k = 4, 3, 4, 4, 2
    act = (0.8, 1.702, 1.0)          # a limit that binds at these scales
    x, wr, b, wg, wu, wd, dy = _separated_layer(91 + S, T, d, f, E + S, k)
    wr, b = wr[:, :E], b[:E]
    lg = np.sort(mo.router_logits(x, wr, b), axis=1)[:, ::-1]
    assert np.min(lg[:, k - 1] - lg[:, k]) > 1e-3
    fw = mo.forward(x, wr, b, wg, wu, wd, k, act=act, shared=S)
    G, U = fw["G"], fw["U"]
    assert (G > act[0]).any() and (np.abs(U) > act[0]).any()          # the clamps bind
    assert np.min(np.abs(G - act[0])) > 1e-4 and np.min(np.abs(np.abs(U) - act[0])) > 1e-4
    bw = mo.backward(x, wr, b, wg, wu, wd, k, dy, fwd=fw, act=act, shared=S)
    eps = 1e-6
    for gname, arr in {"dx": x, "dw_router": wr, "dw_gate": wg, "dw_up": wu,
                       "dw_down": wd}.items():
        num = np.zeros_like(arr)
        for pos in itertools.product(*[range(s_) for s_ in arr.shape]):
            old = arr[pos]
            arr[pos] = old + eps
            lp = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy, act=act, shared=S)
            arr[pos] = old - eps
            lm = mo.layer_loss(x, wr, b, wg, wu, wd, k, dy, act=act, shared=S)
            arr[pos] = old
            num[pos] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(bw[gname], num, rtol=1e-6, atol=1e-8, err_msg=gname)
