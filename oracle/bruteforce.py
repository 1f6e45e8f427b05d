"""Scalar-loop twin of the routed MoE layer, for tiny shapes only.

TEST INFRASTRUCTURE ONLY (see ``oracle/moe_oracle.py``). Written separately
from the numpy oracle so that each pins the other: plain Python floats and
``math.exp``, nested loops, no numpy arithmetic. The top-k set is found by
enumerating every k-subset of the experts and keeping the one that beats every
expert outside it (higher logit, or equal logit and lower index), which is a
different procedure from the oracle's stable sort.

Definition followed: the layer as stated in ``oracle/moe_oracle.py`` (router
softmax, top-k, renormalise; SwiGLU experts; score-weighted sum), whose
sources are prime-rl PR #3885 (DeepSeek-V4.1 Flash perf work), §Changes, and
PocketLLM "Qwen4-Exp Heterogeneous TP4 Performance", §Runtime architecture.
"""
from __future__ import annotations

import itertools
import math


def _beats(li, i, lj, j):
    """Does expert i rank above expert j?"""
    return li > lj or (li == lj and i < j)


def topk_enumerate(logit_row, k):
    """Top-k of one row by enumeration of all subsets; ordered by rank."""
    E = len(logit_row)
    found = None
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all(_beats(logit_row[i], i, logit_row[j], j) for i in S for j in rest):
            assert found is None, "two subsets qualify"
            found = S
    assert found is not None
    # position of i inside S = number of members that rank above it
    ordered = [None] * k
    for i in found:
        pos = sum(1 for j in found if j != i and _beats(logit_row[j], j, logit_row[i], i))
        ordered[pos] = i
    return ordered


def _sigmoid(g):
    return 1.0 / (1.0 + math.exp(-g))


def _act(g, u, act):
    """The gated activation and its two partial derivatives at one element:
    A = gc * sigmoid(alpha gc) * (uc + c), gc = g clamped above at L, uc = u
    clamped to [-L, L]; act = (L, alpha, c), or None for silu(g) * u."""
    if act is None:
        s = _sigmoid(g)
        return g * s * u, u * (s + g * s * (1.0 - s)), g * s
    L, al, c = act
    gc = g if g <= L else L
    uc = u if -L <= u <= L else (L if u > L else -L)
    s = _sigmoid(al * gc)
    a = gc * s * (uc + c)
    da_dg = (s + al * gc * s * (1.0 - s)) * (uc + c) if g <= L else 0.0
    da_du = gc * s if -L <= u <= L else 0.0
    return a, da_dg, da_du


def layer(x, wr, b, wg, wu, wd, k, dy, act=None, shared=0):
    """Forward and backward with nested lists of Python floats.

    x [T][d], wr [d][E], b [E] or None, wg/wu [E+S][d][f], wd [E+S][f][d] (the
    last S = ``shared`` experts are shared: every token goes through them with
    weight 1), dy [T][d], act as in ``_act``. Returns a dict of nested lists:
    logits, idx, w, y, dx, dwr, db, dwg, dwu, dwd, dtw (gradient of the top-k
    weights).
    """
    T, d, E, f = len(x), len(x[0]), len(wr[0]), len(wg[0][0])
    EE = E + shared
    logits = [[sum(x[t][i] * wr[i][e] for i in range(d)) + (b[e] if b is not None else 0.0)
               for e in range(E)] for t in range(T)]
    idx = [topk_enumerate(logits[t], k) for t in range(T)]
    w = []
    for t in range(T):
        # softmax over all experts, then keep the selected ones and renormalise
        m = max(logits[t])
        p = [math.exp(logits[t][e] - m) for e in range(E)]
        z = sum(p)
        p = [v / z for v in p]
        s = sum(p[e] for e in idx[t])
        w.append([p[e] / s for e in idx[t]])

    y = [[0.0] * d for _ in range(T)]
    dx = [[0.0] * d for _ in range(T)]
    dwg = [[[0.0] * f for _ in range(d)] for _ in range(EE)]
    dwu = [[[0.0] * f for _ in range(d)] for _ in range(EE)]
    dwd = [[[0.0] * d for _ in range(f)] for _ in range(EE)]
    dtw = [[0.0] * k for _ in range(T)]
    for t in range(T):
        # slots j < k: the routed experts with their weights; then the shared
        # experts with weight 1
        for j in range(k + shared):
            e = idx[t][j] if j < k else E + (j - k)
            wj = w[t][j] if j < k else 1.0
            g = [sum(x[t][i] * wg[e][i][c] for i in range(d)) for c in range(f)]
            u = [sum(x[t][i] * wu[e][i][c] for i in range(d)) for c in range(f)]
            act_gu = [_act(g[c], u[c], act) for c in range(f)]
            a = [v[0] for v in act_gu]
            yu = [sum(a[c] * wd[e][c][o] for c in range(f)) for o in range(d)]
            for o in range(d):
                y[t][o] += wj * yu[o]
            if j < k:
                dtw[t][j] = sum(dy[t][o] * yu[o] for o in range(d))
            dyu = [wj * dy[t][o] for o in range(d)]
            da = [sum(dyu[o] * wd[e][c][o] for o in range(d)) for c in range(f)]
            dg = [da[c] * act_gu[c][1] for c in range(f)]
            du = [da[c] * act_gu[c][2] for c in range(f)]
            for i in range(d):
                dx[t][i] += sum(dg[c] * wg[e][i][c] + du[c] * wu[e][i][c] for c in range(f))
            for c in range(f):
                for o in range(d):
                    dwd[e][c][o] += a[c] * dyu[o]
            for i in range(d):
                for c in range(f):
                    dwg[e][i][c] += x[t][i] * dg[c]
                    dwu[e][i][c] += x[t][i] * du[c]
    # router: w_j = exp(l_j) / sum_{S} exp(l); dw_j/dl_i = w_j (delta_ij - w_i) on S
    dl = [[0.0] * E for _ in range(T)]
    for t in range(T):
        for jj in range(k):
            acc = 0.0
            for j in range(k):
                delta = 1.0 if j == jj else 0.0
                acc += dtw[t][j] * w[t][j] * (delta - w[t][jj])
            dl[t][idx[t][jj]] = acc
    for t in range(T):
        for i in range(d):
            dx[t][i] += sum(dl[t][e] * wr[i][e] for e in range(E))
    dwr = [[sum(x[t][i] * dl[t][e] for t in range(T)) for e in range(E)] for i in range(d)]
    db = [sum(dl[t][e] for t in range(T)) for e in range(E)]
    return {"logits": logits, "idx": idx, "w": w, "y": y, "dx": dx, "dwr": dwr, "db": db,
            "dwg": dwg, "dwu": dwu, "dwd": dwd, "dtw": dtw, "dl": dl}
