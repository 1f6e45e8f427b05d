"""Oracle values at sampled positions, for layers too large to run whole.

TEST INFRASTRUCTURE ONLY (see ``oracle/moe_oracle.py``). Each function here
evaluates one output element (or one row / column) of the float64 layer
straight from the definition in ``oracle/moe_oracle.py``, touching only the
rows it needs, so a 16k-token layer can be checked at chosen tokens, pairs
and weight columns in seconds.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import as_f64, dsilu, silu, topk_weights, router_backward


class SampledLayer:
    """Float64 evaluation of a layer at sampled positions.

    ``inputs`` holds torch CPU tensors (x, w_router, bias, w_gate, w_up,
    w_down, dy); ``idx`` is the routing [T, k] to evaluate under and
    ``logits`` the float64 logits [T, E] (both from ``moe_oracle.route``).
    """

    def __init__(self, inputs: dict, logits: np.ndarray, idx: np.ndarray, k: int):
        self.inp = inputs
        self.x = as_f64(inputs["x"])
        self.dy = as_f64(inputs["dy"]) if inputs.get("dy") is not None else None
        self.wr = as_f64(inputs["w_router"])
        self.logits = logits
        self.idx = np.asarray(idx, dtype=np.int64)
        self.k = k
        self.w = topk_weights(logits, self.idx)
        self.T, self.d = self.x.shape
        self.E = self.wr.shape[1]
        e_of_p = self.idx.reshape(-1)
        self.pairs_of = [np.flatnonzero(e_of_p == e) for e in range(self.E)]

    # per-pair quantities ---------------------------------------------------
    def pair_forward(self, p: int):
        """G, U, A [f] and Yu [d] of pair p = t*k + j."""
        t, j = divmod(p, self.k)
        e = int(self.idx[t, j])
        xt = self.x[t]
        G = xt @ as_f64(self.inp["w_gate"][e])
        U = xt @ as_f64(self.inp["w_up"][e])
        A = silu(G) * U
        Yu = A @ as_f64(self.inp["w_down"][e])
        return G, U, A, Yu

    def pair_backward(self, p: int):
        """dYu [d], dA, dG, dU [f], dXp [d] and dw (scalar) of pair p."""
        t, j = divmod(p, self.k)
        e = int(self.idx[t, j])
        G, U, A, Yu = self.pair_forward(p)
        dYu = self.w[t, j] * self.dy[t]
        dA = as_f64(self.inp["w_down"][e]) @ dYu
        dG = dA * U * dsilu(G)
        dU = dA * silu(G)
        dXp = as_f64(self.inp["w_gate"][e]) @ dG + as_f64(self.inp["w_up"][e]) @ dU
        dw = float(self.dy[t] @ Yu)
        return dYu, dA, dG, dU, dXp, dw

    # per-token quantities --------------------------------------------------
    def y(self, t: int) -> np.ndarray:
        out = np.zeros(self.d)
        for j in range(self.k):
            out += self.w[t, j] * self.pair_forward(t * self.k + j)[3]
        return out

    def dx_and_dtw(self, t: int):
        """dx_t (expert part plus router part) and the k top-k weight grads."""
        dx = np.zeros(self.d)
        dtw = np.zeros(self.k)
        for j in range(self.k):
            _, _, _, _, dXp, dw = self.pair_backward(t * self.k + j)
            dx += dXp
            dtw[j] = dw
        dl = router_backward(self.w[t:t + 1], dtw[None, :], self.idx[t:t + 1], self.E)[0]
        dx += self.wr @ dl
        return dx, dtw

    # weight-gradient columns / rows -----------------------------------------
    def _expert_rows(self, e: int, c: int):
        """For expert e and ffn column c: x rows, G[:,c], U[:,c], dA[:,c],
        and dYu [n_e, d] over all pairs routed to e."""
        pairs = self.pairs_of[e]
        toks = pairs // self.k
        xe = self.x[toks]
        wg_c = as_f64(self.inp["w_gate"][e][:, c])
        wu_c = as_f64(self.inp["w_up"][e][:, c])
        wd_c = as_f64(self.inp["w_down"][e][c, :])
        G = xe @ wg_c
        U = xe @ wu_c
        dYu = self.w.reshape(-1)[pairs, None] * self.dy[toks]
        dA = dYu @ wd_c
        return xe, G, U, dA, dYu

    def dw_gate_col(self, e: int, c: int) -> np.ndarray:
        """dW_gate[e][:, c] = sum over e's rows of x * dG[:, c]."""
        if self.pairs_of[e].size == 0:
            return np.zeros(self.d)
        xe, G, U, dA, _ = self._expert_rows(e, c)
        return xe.T @ (dA * U * dsilu(G))

    def dw_up_col(self, e: int, c: int) -> np.ndarray:
        """dW_up[e][:, c] = sum over e's rows of x * dU[:, c]."""
        if self.pairs_of[e].size == 0:
            return np.zeros(self.d)
        xe, G, U, dA, _ = self._expert_rows(e, c)
        return xe.T @ (dA * silu(G))

    def dw_down_row(self, e: int, c: int) -> np.ndarray:
        """dW_down[e][c, :] = sum over e's rows of A[:, c] * dYu."""
        if self.pairs_of[e].size == 0:
            return np.zeros(self.d)
        xe, G, U, _, dYu = self._expert_rows(e, c)
        return (silu(G) * U) @ dYu
