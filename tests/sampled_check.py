"""Full-size parity at sampled positions: oracle values (oracle/sampled.py)
and their first-order error magnitudes (the same analysis as
harness.magnitudes, evaluated only where sampled).

Magnitude rules (u = bf16 unit; see harness.py): a stored bf16 value
contributes its own |value|; a GEMM output inherits |A|.|B| sums of its
inputs' magnitudes; element-wise steps inherit |f'| times their inputs'.
"""
from __future__ import annotations

import numpy as np

from oracle.moe_oracle import as_f64, dsilu, router_backward, silu
from oracle.sampled import SampledLayer


def _sig(g):
    return 1.0 / (1.0 + np.exp(-g))


def _ddsilu(g):
    s = _sig(g)
    return s * (1 - s) * (2 + g * (1 - 2 * s))


class SampledChecker(SampledLayer):
    """SampledLayer plus magnitudes for the sampled outputs."""

    def _w(self, name, e):
        return as_f64(self.inp[name][e])

    def pairs_mag(self, pairs):
        """Forward and backward values and magnitudes of the given pairs, one
        expert at a time (each expert's weights are upcast once)."""
        pairs = np.asarray(sorted(set(int(p) for p in pairs)), dtype=np.int64)
        res = {}
        e_of = self.idx.reshape(-1)[pairs]
        for e in np.unique(e_of):
            ps = pairs[e_of == e]
            t = ps // self.k
            wg, wu, wd = self._w("w_gate", e), self._w("w_up", e), self._w("w_down", e)
            xe = self.x[t]
            ax = np.abs(xe)
            G, U = xe @ wg, xe @ wu
            A = silu(G) * U
            Yu = A @ wd
            MG = ax @ np.abs(wg) + np.abs(G)
            MU = ax @ np.abs(wu) + np.abs(U)
            MA = np.abs(dsilu(G) * U) * MG + np.abs(silu(G)) * MU + np.abs(A)
            MYu = MA @ np.abs(wd) + np.abs(Yu)
            cols = dict(G=G, U=U, A=A, Yu=Yu, MG=MG, MU=MU, MA=MA, MYu=MYu)
            if self.dy is not None:
                w = self.w.reshape(-1)[ps]
                dYu = w[:, None] * self.dy[t]
                MdYu = np.abs(w)[:, None] * np.abs(self.dy[t]) + np.abs(dYu)
                dA = dYu @ wd.T
                MdA = MdYu @ np.abs(wd).T
                ds = dsilu(G)
                dG = dA * U * ds
                dU = dA * silu(G)
                MdG = (MdA * np.abs(U * ds) + np.abs(dA) * MU * np.abs(ds)
                       + np.abs(dA * U * _ddsilu(G)) * MG + np.abs(dG))
                MdU = MdA * np.abs(silu(G)) + np.abs(dA * ds) * MG + np.abs(dU)
                dXp = dG @ wg.T + dU @ wu.T
                MdXp = MdG @ np.abs(wg).T + MdU @ np.abs(wu).T + np.abs(dXp)
                cols.update(dYu=dYu, MdYu=MdYu, dG=dG, MdG=MdG, dU=dU, MdU=MdU, dXp=dXp,
                            MdXp=MdXp, dtw=np.einsum("rd,rd->r", self.dy[t], Yu),
                            Mdtw=np.einsum("rd,rd->r", np.abs(self.dy[t]), MYu))
            for i, p in enumerate(ps):
                res[int(p)] = {k_: v[i] for k_, v in cols.items()}
        return res

    def tokens(self, toks):
        """{t: y_t, dx_t, d_topk_w[t] and their magnitudes, plus the pairs}."""
        toks = [int(t) for t in toks]
        pm = self.pairs_mag([t * self.k + j for t in toks for j in range(self.k)])
        out = {}
        for t in toks:
            ps = [pm[t * self.k + j] for j in range(self.k)]
            y = sum(self.w[t, j] * ps[j]["Yu"] for j in range(self.k))
            My = sum(abs(self.w[t, j]) * ps[j]["MYu"] for j in range(self.k)) + np.abs(y)
            r = dict(y=y, My=My, pairs=ps)
            if self.dy is not None:
                dtw = np.array([q["dtw"] for q in ps])
                Mdtw = np.array([q["Mdtw"] for q in ps])
                dl = router_backward(self.w[t:t + 1], dtw[None, :], self.idx[t:t + 1], self.E)[0]
                aw = np.abs(self.w[t])
                Mdl_sel = aw * (Mdtw + (aw * Mdtw).sum()) + np.abs(dl[self.idx[t]])
                Mdl = np.zeros(self.E)
                Mdl[self.idx[t]] = Mdl_sel
                dx = sum(q["dXp"] for q in ps) + self.wr @ dl
                Mdx = sum(q["MdXp"] for q in ps) + np.abs(self.wr) @ Mdl + np.abs(dx)
                r.update(dx=dx, Mdx=Mdx, dtw=dtw, Mdtw=Mdtw + np.abs(dtw), dl=dl)
            out[t] = r
        return out

    def wgrad_cols(self, e, c):
        """dW_gate[e][:, c], dW_up[e][:, c], dW_down[e][c, :] with magnitudes."""
        pairs = self.pairs_of[e]
        d = self.d
        if pairs.size == 0:
            z = np.zeros(d)
            return dict(dwg=z, dwu=z, dwd=z, Mdwg=z, Mdwu=z, Mdwd=z)
        toks = pairs // self.k
        xe = self.x[toks]
        ax = np.abs(xe)
        wd = self._w("w_down", e)
        cache = self.__dict__.setdefault("_expert_cache", {})
        if e not in cache:                   # full rows: MA needs every column
            wg, wu = self._w("w_gate", e), self._w("w_up", e)
            G = xe @ wg
            U = xe @ wu
            A = silu(G) * U
            MG = ax @ np.abs(wg) + np.abs(G)
            MU = ax @ np.abs(wu) + np.abs(U)
            MA = np.abs(dsilu(G) * U) * MG + np.abs(silu(G)) * MU + np.abs(A)
            cache.clear()
            cache[e] = (G, U, A, MG, MU, MA)
        G, U, A, MG, MU, MA = cache[e]
        w = self.w.reshape(-1)[pairs]
        dYu = w[:, None] * self.dy[toks]
        MdYu = np.abs(w)[:, None] * np.abs(self.dy[toks]) + np.abs(dYu)
        dA_c = dYu @ wd[c, :]
        MdA_c = MdYu @ np.abs(wd[c, :])
        g, u = G[:, c], U[:, c]
        ds = dsilu(g)
        dG_c = dA_c * u * ds
        dU_c = dA_c * silu(g)
        MdG_c = (MdA_c * np.abs(u * ds) + np.abs(dA_c) * MU[:, c] * np.abs(ds)
                 + np.abs(dA_c * u * _ddsilu(g)) * MG[:, c] + np.abs(dG_c))
        MdU_c = MdA_c * np.abs(silu(g)) + np.abs(dA_c * ds) * MG[:, c] + np.abs(dU_c)
        dwg = xe.T @ dG_c
        dwu = xe.T @ dU_c
        dwd = A[:, c] @ dYu
        return dict(dwg=dwg, dwu=dwu, dwd=dwd,
                    Mdwg=ax.T @ MdG_c + np.abs(dwg), Mdwu=ax.T @ MdU_c + np.abs(dwu),
                    Mdwd=MA[:, c] @ np.abs(dYu) + np.abs(A[:, c]) @ MdYu + np.abs(dwd))

    def expert_mags(self, e):
        """Magnitudes of every row of expert e (keys MG, MU, MA, MYu and, with
        dy, MdYu, MdG, MdU, MdXp; rows in ascending pair id) and of its whole
        weight gradients (Mdwg, Mdwu, Mdwd), by the rules above."""
        pairs = self.pairs_of[e]
        pm = self.pairs_mag(pairs)
        keys = ["G", "U", "A", "Yu"] + (["dYu", "dG", "dU", "dXp"] if self.dy is not None else [])
        out = {}
        for key in keys:
            out[key] = np.stack([pm[int(p)][key] for p in pairs])
            out["M" + key] = np.stack([pm[int(p)]["M" + key] for p in pairs])
        if self.dy is not None:
            ax = np.abs(self.x[pairs // self.k])
            dwg = self.x[pairs // self.k].T @ out["dG"]
            dwu = self.x[pairs // self.k].T @ out["dU"]
            dwd = out["A"].T @ out["dYu"]
            out.update(dwg=dwg, dwu=dwu, dwd=dwd,
                       Mdwg=ax.T @ out["MdG"] + np.abs(dwg), Mdwu=ax.T @ out["MdU"] + np.abs(dwu),
                       Mdwd=out["MA"].T @ np.abs(out["dYu"]) + np.abs(out["A"]).T @ out["MdYu"]
                       + np.abs(dwd))
        return out
