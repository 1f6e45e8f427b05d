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
    "permute_maps", "silu", "dsilu", "swiglu", "swiglu_grad", "PLAIN_SWIGLU",
    "CLAMPED_SWIGLU_GPT_OSS", "expert_forward", "forward", "backward",
    "router_backward", "layer_loss",
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

def pair_experts(idx: np.ndarray, E: int, shared: int = 0) -> np.ndarray:
    """The expert of every pair: routed pair p = t*k + j goes to idx[t, j];
    with S shared experts (every token's copy, weight 1: the shared expert
    of prime-rl PR #3885, §Changes, "Fused FP8 shared expert", whose output is
    added to the routed one in the write-back), pair T*k + s*T + t goes to
    expert E + s."""
    T, _ = idx.shape
    routed = idx.reshape(-1).astype(np.int64)
    extra = [np.full(T, E + s, dtype=np.int64) for s in range(shared)]
    return np.concatenate([routed] + extra) if extra else routed


def permute_maps(idx: np.ndarray, E: int, align: int, R_cap: int | None = None,
                 shared: int = 0):
    """The padded expert-grouped layout, built by a stable sort of pair ids by
    expert (not by a histogram, so a histogram/scan builder is checked against
    a different method).

    Pair p goes to expert pair_experts(idx, E, shared)[p] (routed pairs
    p = t*k + j first, then the shared experts' T pairs each). Expert e's rows
    start at offsets[e] = sum_{e'<e} ceil(n_e'/align)*align; inside a group,
    pairs keep ascending p. Returns dict: counts [E+S], offsets [E+S+1]
    (int64), dst_row [P] (row of pair p), src_pair [R_cap] (pair in row r, -1
    for rows holding no pair), R_pad = offsets[E+S].
    """
    e_of_p = pair_experts(idx, E, shared)
    P = e_of_p.size
    E = E + shared
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


# The experts' gated activation. The plain SwiGLU, A = silu(G) U, and the
# clamped form of GPT-OSS-style layers (prime-rl PR #3885, §Changes, "FP8
# routed experts" and "Fused FP8 shared expert" name a clamped SwiGLU without
# its constants; these are the GPT-OSS-20B model's own: limit 7, alpha 1.702,
# the up projection offset by 1):
#     A = h(min(G, L)) (clamp(U, -L, L) + c),   h(g) = g sigmoid(alpha g),
# with act = (L, alpha, c); the plain SwiGLU is act = (inf, 1, 0).
PLAIN_SWIGLU = (np.inf, 1.0, 0.0)
CLAMPED_SWIGLU_GPT_OSS = (7.0, 1.702, 1.0)


def swiglu(G, U, act=None):
    """A for act = (L, alpha, c) (None: the plain SwiGLU)."""
    L, al, c = PLAIN_SWIGLU if act is None else act
    gc = np.minimum(G, L)
    uc = np.clip(U, -L, L)
    return gc / (1.0 + np.exp(-al * gc)) * (uc + c)


def swiglu_grad(G, U, act=None):
    """(dA/dG, dA/dU) element-wise; zero where the clamp holds G or U at its
    limit (the derivative of the clamp, 1 inside [-L, L] and 0 outside)."""
    L, al, c = PLAIN_SWIGLU if act is None else act
    gc = np.minimum(G, L)
    uc = np.clip(U, -L, L)
    s = 1.0 / (1.0 + np.exp(-al * gc))
    dg = (s + al * gc * s * (1.0 - s)) * (uc + c) * (G <= L)
    du = gc * s * ((U >= -L) & (U <= L))
    return dg, du


def expert_forward(xe, wg, wu, wd, act=None):
    """One expert on its rows xe [n, d]: returns G, U, A [n, f], Yu [n, d]."""
    G = xe @ wg
    U = xe @ wu
    A = swiglu(G, U, act)
    Yu = A @ wd
    return G, U, A, Yu


def _expert_slices(idx, E, shared=0):
    """For each expert (routed, then shared), the pair ids routed to it in
    ascending order (pair numbering of ``pair_experts``)."""
    e_of_p = pair_experts(idx, E, shared)
    order = np.argsort(e_of_p, kind="stable")
    counts = np.bincount(e_of_p, minlength=E + shared)
    bounds = np.zeros(E + shared + 1, dtype=np.int64)
    bounds[1:] = np.cumsum(counts)
    return [order[bounds[e]:bounds[e + 1]] for e in range(E + shared)]


def _pair_tokens_weights(T, k, w, shared):
    """Token and combine weight of every pair: routed pairs their token and
    top-k weight, shared pairs their token and weight 1."""
    tok = np.concatenate([np.arange(T * k) // k] + [np.arange(T)] * shared)
    wt = np.concatenate([w.reshape(-1)] + [np.ones(T)] * shared)
    return tok, wt


def forward(x, w_router, bias, w_gate, w_up, w_down, k: int, idx=None, keep=True, act=None,
            shared: int = 0):
    """Full layer forward in float64.

    ``x`` [T,d], ``w_router`` [d,E], ``bias`` [E] or None; expert weights as
    torch tensors or arrays, [E+S,d,f], [E+S,d,f], [E+S,f,d] — the E routed
    experts, then the ``shared`` (S) shared experts every token goes through
    with weight 1; they are upcast one expert at a time so a large layer never
    holds all weights in float64. ``idx`` overrides the selection (the weights
    are still the renormalised softmax over the given set). ``act``: the
    activation's (L, alpha, c) (None: the plain SwiGLU).

    y_t = sum_j w_tj Yu(t, e_j) + sum_s Yu(t, E + s).

    Returns dict with logits, idx, w, y [T,d] and, when ``keep``, the per-pair
    intermediates G, U, A [P,f] and Yu [P,d] (pair numbering of
    ``pair_experts``: p = t*k + j, then T*k + s*T + t).
    """
    x = as_f64(x)
    T, d = x.shape
    logits = router_logits(x, as_f64(w_router), None if bias is None else as_f64(bias))
    if idx is None:
        idx = select_topk(logits, k)
    idx = np.asarray(idx, dtype=np.int64)
    w = topk_weights(logits, idx)
    E = logits.shape[1]
    P = T * (k + shared)
    f = w_gate.shape[2]
    assert w_gate.shape[0] == E + shared
    y = np.zeros((T, d))
    keep_G = np.zeros((P, f)) if keep else None
    keep_U = np.zeros((P, f)) if keep else None
    keep_A = np.zeros((P, f)) if keep else None
    keep_Yu = np.zeros((P, d)) if keep else None
    tok, wt = _pair_tokens_weights(T, k, w, shared)
    for e, pairs in enumerate(_expert_slices(idx, E, shared)):
        if pairs.size == 0:
            continue
        toks = tok[pairs]
        G, U, A, Yu = expert_forward(x[toks], as_f64(w_gate[e]), as_f64(w_up[e]),
                                     as_f64(w_down[e]), act)
        np.add.at(y, toks, wt[pairs, None] * Yu)
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


def backward(x, w_router, bias, w_gate, w_up, w_down, k: int, dy, fwd=None, idx=None, act=None,
             shared: int = 0):
    """Full layer backward in float64 for upstream gradient ``dy`` [T, d].

    Returns dict: dx [T,d], dw_router [d,E], dbias [E], dw_gate [E+S,d,f],
    dw_up [E+S,d,f], dw_down [E+S,f,d], d_topk_w [T,k] (gradient of the
    weights w), dl [T,E], and the per-pair dYu [P,d] (= the pair's combine
    weight * dy of its token), dA, dG, dU [P,f], dXp [P,d] (pair numbering of
    ``pair_experts``).

    Steps: combine transpose (dYu = w * dy_t, dw = <dy_t, Yu> for the routed
    pairs), down dgrad dA = dYu . W_down^T, activation gradient
    dG = dA * dA/dG, dU = dA * dA/dU (``swiglu_grad``), gate/up dgrad
    dXp = dG . W_gate^T + dU . W_up^T, K-grouped wgrad per expert
    (dW_down = A^T dYu, dW_gate = X^T dG, dW_up = X^T dU; empty expert ->
    zeros), permute transpose dx_t = sum of dXp over the token's pairs,
    router backward (dl, dx += dl . W_r^T, dW_r = x^T dl, db = sum_t dl).
    """
    x = as_f64(x)
    dy = as_f64(dy)
    wr = as_f64(w_router)
    T, d = x.shape
    if fwd is None:
        fwd = forward(x, wr, bias, w_gate, w_up, w_down, k, idx=idx, keep=True, act=act,
                      shared=shared)
    idx, w = fwd["idx"], fwd["w"]
    E = wr.shape[1]
    f = w_gate.shape[2]
    P = T * (k + shared)
    tok, wt = _pair_tokens_weights(T, k, w, shared)
    dYu = wt[:, None] * dy[tok]
    d_topk_w = np.einsum("pd,pd->p", dy[tok[:T * k]], fwd["Yu"][:T * k]).reshape(T, k)
    dA = np.zeros((P, f))
    dG = np.zeros((P, f))
    dU = np.zeros((P, f))
    dXp = np.zeros((P, d))
    dw_gate = np.zeros((E + shared, d, f))
    dw_up = np.zeros((E + shared, d, f))
    dw_down = np.zeros((E + shared, f, d))
    for e, pairs in enumerate(_expert_slices(idx, E, shared)):
        if pairs.size == 0:
            continue
        wg, wu, wd = as_f64(w_gate[e]), as_f64(w_up[e]), as_f64(w_down[e])
        G, U, A = fwd["G"][pairs], fwd["U"][pairs], fwd["A"][pairs]
        dA_e = dYu[pairs] @ wd.T
        gG, gU = swiglu_grad(G, U, act)
        dG_e = dA_e * gG
        dU_e = dA_e * gU
        dXp[pairs] = dG_e @ wg.T + dU_e @ wu.T
        dA[pairs], dG[pairs], dU[pairs] = dA_e, dG_e, dU_e
        xe = x[tok[pairs]]
        dw_down[e] = A.T @ dYu[pairs]
        dw_gate[e] = xe.T @ dG_e
        dw_up[e] = xe.T @ dU_e
    dx = np.zeros((T, d))
    np.add.at(dx, tok, dXp)
    dl = router_backward(w, d_topk_w, idx, E)
    dx = dx + dl @ wr.T
    dw_router = x.T @ dl
    dbias = dl.sum(axis=0)
    return {"dx": dx, "dw_router": dw_router, "dbias": dbias, "dw_gate": dw_gate,
            "dw_up": dw_up, "dw_down": dw_down, "d_topk_w": d_topk_w, "dl": dl,
            "dYu": dYu, "dA": dA, "dG": dG, "dU": dU, "dXp": dXp}


def layer_loss(x, w_router, bias, w_gate, w_up, w_down, k, dy, idx=None, act=None,
               shared: int = 0) -> float:
    """Scalar L = sum(y * dy); dL/dy = dy, so backward(dy) is its gradient.
    Used by the finite-difference pins."""
    y = forward(x, w_router, bias, w_gate, w_up, w_down, k, idx=idx, keep=False, act=act,
                shared=shared)["y"]
    return float((y * as_f64(dy)).sum())
