"""CPU oracle of the routed Mixture-of-Experts expert layer, forward and backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or runs
this module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg use it. It shares no code with the CUDA path.

Everything is plain numpy in float64. Inputs (bf16 / fp32) are upcast
exactly; nothing is rounded on the way. A library matmul and a stable sort are
the only library steps; there is no blocking, fusion or reordering beyond the
definition below.

The layer (per token t, with x_t its row of width d):

  routing      l_t = x_t . W_r + b                               (logits, [E])
               S_t = the k largest l_t,e, ordered by descending value,
                     equal values -> lower expert index first
               w_t,j = exp(l_t,S_j) / sum_{j'} exp(l_t,S_j')     (softmax over
                     all E experts, keep S_t, renormalise over S_t: the full
                     denominator cancels, so this is the same number)
  expert e     G = x_t . W_gate[e],  U = x_t . W_up[e]           ([f])
               A = silu(G) * U,  silu(g) = g * sigmoid(g)
               Yu = A . W_down[e]                                 ([d])
  combine      y_t = sum_j w_t,j * Yu(t, S_j)

Sources. The pages name top-k routing over many experts (PocketLLM
"Qwen4-Exp Heterogeneous TP4 Performance", §Runtime architecture: 512 routed
experts, top-10) but do not write the routing formula out; the reading above
(softmax, top-k, renormalise) is the plainest one. The padded expert-grouped
layout, the fp32 score-weighted gather-sum and gathers in backward are from
prime-rl PR #3885 (DeepSeek-V4.1 Flash perf work), §Changes, "Single-pass
DeepEP local layout". The fused SwiGLU (no clamp) is from Halo "Performance",
§Levers that help (fused GLU) and prime-rl PR #3885, §Changes (moe_experts with
SwiGLU). Gradients for x, the top-k weights and the expert weights are the ones
prime-rl PR #3885, §Changes, "dispatch.type = mega_moe" lists; forward, dgrad
and K-grouped wgrad passes are from prime-rl PR #3885, §Changes, "FP8 routed
experts" and "FP8 Mega MoE".

Pins (tests/test_oracle_*.py): a scalar-loop twin written separately
(``oracle/bruteforce.py``) on tiny shapes, with top-k by enumeration of all
subsets; closed forms (sum_j w = 1, k = 1 -> w = 1, sum_j dl = 0); the
special case k = E with identical experts, which reduces to one dense SwiGLU
MLP; permutation invariants and adjoint identities; central finite
differences of every gradient.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "as_f64", "router_logits", "select_topk", "topk_weights", "route",
    "permute_maps", "silu", "dsilu", "expert_forward", "forward",
    "backward", "router_backward", "layer_loss",
]


def as_f64(t) -> np.ndarray:
    """Exact upcast of a torch tensor (bf16 / fp32 / int) or array to float64."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().to("cpu")
            if t.dtype in (torch.bfloat16, torch.float16):
                t = t.to(torch.float32)
            return t.numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


# ----------------------------------------------------------------- routing --

def router_logits(x: np.ndarray, w_router: np.ndarray, bias=None) -> np.ndarray:
    """l = x . W_r (+ b): [T, d] x [d, E] -> [T, E]. The bias is added to the
    logits before any softmax, so it moves both the selection and the
    weights."""
    logits = x @ w_router
    if bias is not None:
        logits = logits + bias[None, :]
    return logits


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, by descending value; equal
    values keep the lower expert index first (a stable sort of -l).

    Works on fp32 logits too: the conversion to float64 is exact and
    monotone, so the order is the one fp32 comparisons give."""
    lg = np.asarray(logits, dtype=np.float64)
    order = np.argsort(-lg, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def topk_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Renormalised softmax weights of the selected experts:
    w_j = exp(l_j - m) / sum_j' exp(l_j' - m), m = the largest selected logit."""
    sel = np.take_along_axis(np.asarray(logits, dtype=np.float64), idx, axis=1)
    m = sel.max(axis=1, keepdims=True)
    ex = np.exp(sel - m)
    return ex / ex.sum(axis=1, keepdims=True)


def route(x, w_router, bias, k: int):
    """Router: returns (logits [T,E], idx [T,k], w [T,k]) in float64."""
    logits = router_logits(x, w_router, bias)
    idx = select_topk(logits, k)
    w = topk_weights(logits, idx)
    return logits, idx, w


# ----------------------------------------------------------------- permute --

def permute_maps(idx: np.ndarray, E: int, align: int, R_cap: int | None = None):
    """The padded expert-grouped layout, built by a stable sort of pair ids by
    expert (not by a histogram, so a histogram/scan builder is checked against
    a different method).

    Pair p = t*k + j goes to expert e = idx[t, j]. Expert e's rows start at
    offsets[e] = sum_{e'<e} ceil(n_e'/align)*align; inside a group, pairs keep
    ascending p. Returns dict: counts [E], offsets [E+1] (int64), dst_row [P]
    (row of pair p), src_pair [R_cap] (pair in row r, -1 for rows holding no
    pair), R_pad = offsets[E].
    """
    T, k = idx.shape
    P = T * k
    e_of_p = idx.reshape(-1).astype(np.int64)
    counts = np.bincount(e_of_p, minlength=E).astype(np.int64)
    padded = -(-counts // align) * align
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    order = np.argsort(e_of_p, kind="stable")          # pairs grouped by expert, p ascending
    group_start = np.zeros(E, dtype=np.int64)
    group_start[1:] = np.cumsum(counts)[:-1]
    sorted_e = e_of_p[order]
    rank = np.arange(P, dtype=np.int64) - group_start[sorted_e]
    dst_row = np.empty(P, dtype=np.int64)
    dst_row[order] = offsets[sorted_e] + rank
    if R_cap is None:
        R_cap = int(offsets[E])
    src_pair = np.full(R_cap, -1, dtype=np.int64)
    src_pair[dst_row] = np.arange(P, dtype=np.int64)
    return {"counts": counts, "offsets": offsets, "dst_row": dst_row,
            "src_pair": src_pair, "R_pad": int(offsets[E])}


# ------------------------------------------------------------------ expert --

def silu(g):
    """silu(g) = g * sigmoid(g)."""
    return g / (1.0 + np.exp(-g))


def dsilu(g):
    """d silu / d g = sigmoid(g) * (1 + g * (1 - sigmoid(g)))."""
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def expert_forward(xe, wg, wu, wd):
    """One expert on its rows xe [n, d]: returns G, U, A [n, f], Yu [n, d]."""
    G = xe @ wg
    U = xe @ wu
    A = silu(G) * U
    Yu = A @ wd
    return G, U, A, Yu


def _expert_slices(idx, E):
    """For each expert, the pair ids routed to it in ascending order."""
    e_of_p = idx.reshape(-1)
    order = np.argsort(e_of_p, kind="stable")
    counts = np.bincount(e_of_p, minlength=E)
    bounds = np.zeros(E + 1, dtype=np.int64)
    bounds[1:] = np.cumsum(counts)
    return [order[bounds[e]:bounds[e + 1]] for e in range(E)]


def forward(x, w_router, bias, w_gate, w_up, w_down, k: int, idx=None, keep=True):
    """Full layer forward in float64.

    ``x`` [T,d], ``w_router`` [d,E], ``bias`` [E] or None; expert weights as
    torch tensors or arrays, [E,d,f], [E,d,f], [E,f,d]; they are upcast one
    expert at a time so a large layer never holds all weights in float64.
    ``idx`` overrides the selection (the weights are still the renormalised
    softmax over the given set).

    Returns dict with logits, idx, w, y [T,d] and, when ``keep``, the per-pair
    intermediates G, U, A [P,f] and Yu [P,d] (pair p = t*k + j).
    """
    x = as_f64(x)
    T, d = x.shape
    logits = router_logits(x, as_f64(w_router), None if bias is None else as_f64(bias))
    if idx is None:
        idx = select_topk(logits, k)
    idx = np.asarray(idx, dtype=np.int64)
    w = topk_weights(logits, idx)
    E = logits.shape[1]
    P = T * k
    f = w_gate.shape[2]
    y = np.zeros((T, d))
    keep_G = np.zeros((P, f)) if keep else None
    keep_U = np.zeros((P, f)) if keep else None
    keep_A = np.zeros((P, f)) if keep else None
    keep_Yu = np.zeros((P, d)) if keep else None
    w_flat = w.reshape(-1)
    for e, pairs in enumerate(_expert_slices(idx, E)):
        if pairs.size == 0:
            continue
        toks = pairs // k
        G, U, A, Yu = expert_forward(x[toks], as_f64(w_gate[e]), as_f64(w_up[e]), as_f64(w_down[e]))
        np.add.at(y, toks, w_flat[pairs, None] * Yu)
        if keep:
            keep_G[pairs], keep_U[pairs], keep_A[pairs], keep_Yu[pairs] = G, U, A, Yu
    out = {"logits": logits, "idx": idx, "w": w, "y": y}
    if keep:
        out.update(G=keep_G, U=keep_U, A=keep_A, Yu=keep_Yu)
    return out


def router_backward(w: np.ndarray, dw: np.ndarray, idx: np.ndarray, E: int) -> np.ndarray:
    """Gradient of the renormalised softmax: dl_t,S_j = w_j (dw_j - sum_j' w_j' dw_j')
    on the selected experts, 0 elsewhere (the selection itself is piecewise
    constant). Returns dl [T, E]."""
    T, k = idx.shape
    inner = (w * dw).sum(axis=1, keepdims=True)
    dsel = w * (dw - inner)
    dl = np.zeros((T, E))
    np.put_along_axis(dl, idx, dsel, axis=1)
    return dl


def backward(x, w_router, bias, w_gate, w_up, w_down, k: int, dy, fwd=None, idx=None):
    """Full layer backward in float64 for upstream gradient ``dy`` [T, d].

    Returns dict: dx [T,d], dw_router [d,E], dbias [E], dw_gate [E,d,f],
    dw_up [E,d,f], dw_down [E,f,d], d_topk_w [T,k] (gradient of the weights
    w), dl [T,E], and the per-pair dYu [P,d] (= w * dy of the pair's token),
    dA, dG, dU [P,f], dXp [P,d].

    Steps: combine transpose (dYu = w * dy_t, dw = <dy_t, Yu>), down dgrad
    dA = dYu . W_down^T, SwiGLU gradient dG = dA * U * silu'(G),
    dU = dA * silu(G), gate/up dgrad dXp = dG . W_gate^T + dU . W_up^T,
    K-grouped wgrad per expert (dW_down = A^T dYu, dW_gate = X^T dG,
    dW_up = X^T dU; empty expert -> zeros), permute transpose
    dx_t = sum_j dXp(t, j), router backward (dl, dx += dl . W_r^T,
    dW_r = x^T dl, db = sum_t dl).
    """
    x = as_f64(x)
    dy = as_f64(dy)
    wr = as_f64(w_router)
    T, d = x.shape
    if fwd is None:
        fwd = forward(x, wr, bias, w_gate, w_up, w_down, k, idx=idx, keep=True)
    idx, w = fwd["idx"], fwd["w"]
    E = wr.shape[1]
    f = w_gate.shape[2]
    P = T * k
    w_flat = w.reshape(-1)
    tok = np.arange(P) // k
    dYu = w_flat[:, None] * dy[tok]
    d_topk_w = np.einsum("pd,pd->p", dy[tok], fwd["Yu"]).reshape(T, k)
    dA = np.zeros((P, f))
    dG = np.zeros((P, f))
    dU = np.zeros((P, f))
    dXp = np.zeros((P, d))
    dw_gate = np.zeros((E, d, f))
    dw_up = np.zeros((E, d, f))
    dw_down = np.zeros((E, f, d))
    for e, pairs in enumerate(_expert_slices(idx, E)):
        if pairs.size == 0:
            continue
        wg, wu, wd = as_f64(w_gate[e]), as_f64(w_up[e]), as_f64(w_down[e])
        G, U, A = fwd["G"][pairs], fwd["U"][pairs], fwd["A"][pairs]
        dA_e = dYu[pairs] @ wd.T
        dG_e = dA_e * U * dsilu(G)
        dU_e = dA_e * silu(G)
        dXp[pairs] = dG_e @ wg.T + dU_e @ wu.T
        dA[pairs], dG[pairs], dU[pairs] = dA_e, dG_e, dU_e
        xe = x[pairs // k]
        dw_down[e] = A.T @ dYu[pairs]
        dw_gate[e] = xe.T @ dG_e
        dw_up[e] = xe.T @ dU_e
    dx = dXp.reshape(T, k, d).sum(axis=1)
    dl = router_backward(w, d_topk_w, idx, E)
    dx = dx + dl @ wr.T
    dw_router = x.T @ dl
    dbias = dl.sum(axis=0)
    return {"dx": dx, "dw_router": dw_router, "dbias": dbias, "dw_gate": dw_gate,
            "dw_up": dw_up, "dw_down": dw_down, "d_topk_w": d_topk_w, "dl": dl,
            "dYu": dYu, "dA": dA, "dG": dG, "dU": dU, "dXp": dXp}


def layer_loss(x, w_router, bias, w_gate, w_up, w_down, k, dy, idx=None) -> float:
    """Scalar L = sum(y * dy); dL/dy = dy, so backward(dy) is its gradient.
    Used by the finite-difference pins."""
    y = forward(x, w_router, bias, w_gate, w_up, w_down, k, idx=idx, keep=False)["y"]
    return float((y * as_f64(dy)).sum())
