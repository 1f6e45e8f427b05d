"""Pins of the oracle's padded expert-grouped layout.

The invariants below determine the layout uniquely (each expert's group starts
at the sum of the earlier groups' padded sizes; inside a group pairs keep
ascending pair id), so a layout that passes them is the layout.
"""
import numpy as np
import pytest

from oracle import moe_oracle as mo


def _random_idx(rng, T, k, E, skew=0.0):
    p = np.exp(-skew * np.log(np.arange(1, E + 1)))
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])


@pytest.mark.parametrize("T,k,E,align,skew", [
    (1, 1, 1, 1, 0.0), (7, 2, 8, 16, 0.0), (64, 4, 32, 128, 0.0), (300, 8, 128, 16, 1.5),
    (129, 10, 512, 128, 2.0), (50, 3, 3, 4, 0.0), (33, 5, 5, 256, 0.0)])
def test_layout_invariants(T, k, E, align, skew):
    rng = np.random.default_rng(T * 31 + k)
    idx = _random_idx(rng, T, k, E, skew)
    P = T * k
    R_cap = P + E * (align - 1)
    m = mo.permute_maps(idx, E, align, R_cap)
    counts, offsets, dst_row, src_pair = m["counts"], m["offsets"], m["dst_row"], m["src_pair"]
    e_of_p = idx.reshape(-1)
    assert counts.sum() == P
    for e in range(E):
        assert counts[e] == np.count_nonzero(e_of_p == e)
    assert offsets[0] == 0 and np.all(offsets % align == 0)
    assert np.all(np.diff(offsets) == -(-counts // align) * align)
    assert m["R_pad"] == offsets[E] <= R_cap
    # dst_row is a bijection from the P pairs onto the real rows
    assert len(np.unique(dst_row)) == P
    real = src_pair >= 0
    assert real.sum() == P
    np.testing.assert_array_equal(src_pair[dst_row], np.arange(P))
    for p in range(P):
        e = e_of_p[p]
        assert offsets[e] <= dst_row[p] < offsets[e] + counts[e]
    # inside a group, pairs keep ascending pair id, and real rows come first
    for e in range(E):
        grp = src_pair[offsets[e]:offsets[e + 1]]
        assert np.all(grp[:counts[e]] >= 0) and np.all(grp[counts[e]:] == -1)
        assert np.all(np.diff(grp[:counts[e]]) > 0)
    assert np.all(src_pair[offsets[E]:] == -1)


def test_permute_and_combine_adjoints():
    rng = np.random.default_rng(9)
    T, k, E, d, align = 40, 3, 6, 5, 8
    idx = _random_idx(rng, T, k, E)
    m = mo.permute_maps(idx, E, align)
    R = m["R_pad"]
    w = rng.random((T, k))
    x = rng.standard_normal((T, d))
    z = rng.standard_normal((R, d))
    src = m["src_pair"]

    def permute(x):               # Xp[r] = x[token of row r], 0 on padding
        out = np.zeros((R, d))
        out[src >= 0] = x[src[src >= 0] // k]
        return out

    def permute_t(z):             # dx[t] = sum_j z[dst_row[t, j]]
        return z[m["dst_row"]].reshape(T, k, d).sum(1)

    def combine(z):               # y[t] = sum_j w[t, j] z[dst_row[t, j]]
        return (w[:, :, None] * z[m["dst_row"]].reshape(T, k, d)).sum(1)

    def combine_t(dy):            # dz[r] = w(pair of r) * dy[token of r], 0 on padding
        out = np.zeros((R, d))
        rows = src >= 0
        out[rows] = w.reshape(-1)[src[rows], None] * dy[src[rows] // k]
        return out

    dy = rng.standard_normal((T, d))
    assert abs((permute(x) * z).sum() - (x * permute_t(z)).sum()) < 1e-10
    assert abs((combine(z) * dy).sum() - (z * combine_t(dy)).sum()) < 1e-10


def test_expected_distinct_experts_matches_the_page():
    """8 tokens x top-10 of 512 experts touch 74.7 distinct experts on average
    (PocketLLM "Qwen4-Exp Heterogeneous TP4 Performance", §Decode ceiling):
    a Monte-Carlo run of uniform routing through the oracle's layout agrees."""
    rng = np.random.default_rng(0)
    E, k, T = 512, 10, 8
    closed = E * (1 - (1 - k / E) ** T)
    assert abs(closed - 74.7) < 0.05
    active = []
    for _ in range(4000):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)])
        active.append(np.count_nonzero(mo.permute_maps(idx, E, 1)["counts"]))
    assert abs(np.mean(active) - 74.7) < 0.2
