"""The whole float64 layer, one expert at a time, for layers too large to
hold every per-pair intermediate in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/moe_oracle.py``): only ``tests/`` use
it. It shares no code with the CUDA path.

The same definition and the same steps as ``moe_oracle.forward`` and
``moe_oracle.backward`` (routing softmax / top-k / renormalise; per expert
G = x W_gate, U = x W_up, A = silu(G) U, Yu = A W_down; y_t = sum_j w_tj Yu;
backward: dYu = w dy_t, d_topk_w = <dy_t, Yu>, dA = dYu W_down^T,
dG = dA U silu'(G), dU = dA silu(G), dXp = dG W_gate^T + dU W_up^T,
dW_down = A^T dYu, dW_gate = X^T dG, dW_up = X^T dU, dx_t = sum_j dXp +
dl W_r^T, dW_r = x^T dl, db = sum_t dl), evaluated expert by expert: each
expert's pairs are computed, their contributions added into the [T, d]
results, and the per-pair rows and weight gradients dropped — except for the
experts named in ``keep``, whose rows and weight gradients are returned. The
memory held is the [T, d] results plus one expert's rows.

Sources: as ``oracle/moe_oracle.py`` (prime-rl PR #3885, §Changes,
"Single-pass DeepEP local layout", "FP8 routed experts", "FP8 Mega MoE",
"dispatch.type = mega_moe"; Halo "Performance", §Levers that help).
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import as_f64, dsilu, router_backward, silu, topk_weights


def stream_layer(inputs: dict, logits: np.ndarray, idx: np.ndarray, k: int, keep=(),
                 backward: bool = True) -> dict:
    """Evaluate the layer under routing ``idx`` [T, k] with float64 ``logits``
    [T, E]. ``inputs`` holds torch CPU tensors x, w_router, w_gate, w_up,
    w_down and (for ``backward``) dy.

    Returns y [T, d]; with ``backward`` also dx [T, d], d_topk_w [T, k],
    dl [T, E], dw_router [d, E], dbias [E]; and ``experts``: {e: dict(pairs,
    G, U, A, Yu [, dYu, dG, dU, dXp, dw_gate, dw_up, dw_down])} for each e in
    ``keep`` (rows in ascending pair id)."""
    x = as_f64(inputs["x"])
    T, d = x.shape
    idx = np.asarray(idx, dtype=np.int64)
    w = topk_weights(logits, idx)
    w_flat = w.reshape(-1)
    E = logits.shape[1]
    e_of_p = idx.reshape(-1)
    order = np.argsort(e_of_p, kind="stable")
    bounds = np.zeros(E + 1, dtype=np.int64)
    bounds[1:] = np.cumsum(np.bincount(e_of_p, minlength=E))
    dy = as_f64(inputs["dy"]) if backward else None
    y = np.zeros((T, d))
    dx = np.zeros((T, d)) if backward else None
    d_topk_w = np.zeros(T * k) if backward else None
    kept = {}
    keep = set(int(e) for e in keep)
    for e in range(E):
        pairs = order[bounds[e]:bounds[e + 1]]
        if pairs.size == 0:
            continue
        toks = pairs // k
        xe = x[toks]
        wg, wu, wd = (as_f64(inputs["w_gate"][e]), as_f64(inputs["w_up"][e]),
                      as_f64(inputs["w_down"][e]))
        G = xe @ wg
        U = xe @ wu
        A = silu(G) * U
        Yu = A @ wd
        np.add.at(y, toks, w_flat[pairs, None] * Yu)
        rec = dict(pairs=pairs, G=G, U=U, A=A, Yu=Yu) if e in keep else None
        if backward:
            dYu = w_flat[pairs, None] * dy[toks]
            d_topk_w[pairs] = np.einsum("rd,rd->r", dy[toks], Yu)
            dA = dYu @ wd.T
            dG = dA * U * dsilu(G)
            dU = dA * silu(G)
            dXp = dG @ wg.T + dU @ wu.T
            np.add.at(dx, toks, dXp)
            if rec is not None:
                rec.update(dYu=dYu, dG=dG, dU=dU, dXp=dXp, dw_down=A.T @ dYu,
                           dw_gate=xe.T @ dG, dw_up=xe.T @ dU)
        if rec is not None:
            kept[e] = rec
    out = {"y": y, "w": w, "experts": kept}
    if backward:
        wr = as_f64(inputs["w_router"])
        dtw = d_topk_w.reshape(T, k)
        dl = router_backward(w, dtw, idx, E)
        dx = dx + dl @ wr.T
        out.update(dx=dx, d_topk_w=dtw, dl=dl, dw_router=x.T @ dl, dbias=dl.sum(axis=0))
    return out
