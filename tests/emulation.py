"""A plain PyTorch fp32 emulation of the layer with the kernels' bf16
rounding points, for kernel-level numerics tests.

Not the oracle (the oracle is float64 and never rounds): this restates the
same steps in torch fp32 on the device and rounds to bf16 exactly where the
kernels store bf16 (A, dYp, dG, dU, y, dx, the weight gradients; G, U, Yp
and dXp stay fp32, the down dgrad multiplies the unscaled rows of dY and
applies each pair's score to the fp32 product, and the top-k weight gradient
is <dY W_down^T, silu(G) U> from the fp32 G and U), so a kernel and this
emulation should differ only by fp32 summation order and the odd bf16
rounding it flips. The routing indices are inputs (the oracle's), so both
sides route identically.
"""
from __future__ import annotations

import torch


def bf(t):
    return t.to(torch.bfloat16).to(torch.float32)


def emulate(inp: dict, idx, k: int, device="cuda", backward=True) -> dict:
    f32 = dict(dtype=torch.float32, device=device)
    x = inp["x"].to(device).float()
    T, d = x.shape
    wr = inp["w_router"].to(**f32)
    E = wr.shape[1]
    idx = torch.as_tensor(idx, dtype=torch.int64, device=device)
    lg = x @ wr
    if inp.get("bias") is not None:
        lg = lg + inp["bias"].to(**f32)
    w = torch.softmax(torch.gather(lg, 1, idx), 1)
    P = T * k
    tok = torch.arange(P, device=device) // k
    e_of_p = idx.reshape(-1)
    f = inp["w_gate"].shape[2]
    out = {"logits": lg, "w": w}
    G = torch.zeros(P, f, **f32); U = torch.zeros(P, f, **f32); A = torch.zeros(P, f, **f32)
    Yu = torch.zeros(P, d, **f32)
    wf = w.reshape(-1)
    if backward:
        dy = inp["dy"].to(device).float()
        dYp = bf(wf[:, None] * dy[tok])
        dG = torch.zeros(P, f, **f32); dU = torch.zeros(P, f, **f32); dXp = torch.zeros(P, d, **f32)
        dwg = torch.zeros(E, d, f, **f32); dwu = torch.zeros(E, d, f, **f32)
        dwd = torch.zeros(E, f, d, **f32)
    for e in range(E):
        pp = (e_of_p == e).nonzero().flatten()
        if pp.numel() == 0:
            continue
        wg = inp["w_gate"][e].to(**f32)
        wu = inp["w_up"][e].to(**f32)
        wd = inp["w_down"][e].to(**f32)
        xe = x[tok[pp]]
        g32 = xe @ wg
        u32 = xe @ wu
        G[pp] = g32
        U[pp] = u32
        A[pp] = bf(g32 * torch.sigmoid(g32) * u32)
        Yu[pp] = A[pp] @ wd
        if backward:
            dA = (dy[tok[pp]] @ wd.T) * wf[pp][:, None]
            s = torch.sigmoid(G[pp])
            dG[pp] = bf(dA * U[pp] * (s * (1 + G[pp] * (1 - s))))
            dU[pp] = bf(dA * G[pp] * s)
            dXp[pp] = dG[pp] @ wg.T + dU[pp] @ wu.T
            dwg[e] = bf(xe.T @ dG[pp])
            dwu[e] = bf(xe.T @ dU[pp])
            dwd[e] = bf(A[pp].T @ dYp[pp])
    out.update(G=G, U=U, A=A, Yu=Yu, y=bf((wf[:, None] * Yu).reshape(T, k, d).sum(1)))
    if backward:
        # the top-k weight gradient from the unrounded A: <dy W_down^T, silu(G) U>
        A32 = torch.zeros(P, f, **f32)
        for e in range(E):
            pp = (e_of_p == e).nonzero().flatten()
            if pp.numel():
                A32[pp] = G[pp] * torch.sigmoid(G[pp]) * U[pp]
        dtw = torch.zeros(P, **f32)
        for e in range(E):
            pp = (e_of_p == e).nonzero().flatten()
            if pp.numel():
                dtw[pp] = ((dy[tok[pp]] @ inp["w_down"][e].to(**f32).T) * A32[pp]).sum(1)
        dtw = dtw.reshape(T, k)
        dl_sel = w * (dtw - (w * dtw).sum(1, keepdim=True))
        dl = torch.zeros(T, E, **f32).scatter_(1, idx, dl_sel)
        dx = bf(dXp.reshape(T, k, d).sum(1) + dl @ wr.T)     # one rounding (fused pass)
        out.update(dYu=dYp, dG=dG, dU=dU, dXp=dXp, dx=dx, dw_gate=dwg, dw_up=dwu, dw_down=dwd,
                   d_topk_w=dtw, dw_router=x.T @ dl, dbias=dl.sum(0))
    return out
