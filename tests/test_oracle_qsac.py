"""Pins of the oracle's QSAC centroid choice.

The score is checked against exact rational arithmetic (brute force over all
centroids), against the reduction to a plain nearest-residual-range choice
when every channel weighs the same, and against its symmetries.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import qwm_oracle as O


def _exact_scores(k, C, w):
    """sum_g w_g (range_g(k - C_j)/3)^2/12 over exact rationals (no rounding)."""
    d = k.shape[0]
    out = []
    for j in range(C.shape[0]):
        res = [Fraction(float(k[c])) - Fraction(float(C[j, c])) for c in range(d)]
        tot = Fraction(0)
        for g in range(d // 32):
            seg = res[32 * g:32 * g + 32]
            R = max(seg) - min(seg)
            tot += Fraction(float(w[g])) * (R / 3) ** 2 / 12
        out.append(tot)
    return out


def _tiny_case(seed, d=64, nC=12, n=200):
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.standard_normal(d))
    C = (rng.standard_normal((nC, d)) * sig).astype(np.float32)
    z = rng.integers(0, nC, n)
    k = ((C[z] + 0.3 * rng.standard_normal((n, d)) * sig)).astype(np.float32)
    s = (rng.standard_normal((256, d)) * sig) ** 2
    w = O.group_weights(s.mean(0).astype(np.float32))
    return k, C, w


@pytest.mark.parametrize("seed", [0, 1])
def test_brute_force_exact_argmin(seed):
    k, C, w = _tiny_case(seed)
    ties = 0
    for i in range(k.shape[0]):
        ex = _exact_scores(k[i], C, w)
        best = min(ex)
        j_exact = ex.index(best)                       # lowest index on a tie
        # the float64 score follows the exact one
        s64 = O.qsac_scores_exact(k[i], C, w)
        assert int(np.argmin(s64)) == j_exact
        for j in range(C.shape[0]):
            assert abs(s64[j] - float(ex[j])) <= 1e-12 * max(1.0, float(ex[j]))
        # the float32 decision agrees except on exact-score near-ties
        j32 = int(O.qsac_assign(k[i:i + 1], C, w)[0])
        if j32 != j_exact:
            gap = abs(float(ex[j32]) - float(best)) / float(best)
            assert gap < 1e-6
            ties += 1
    assert ties <= 2


def test_uniform_weights_reduce_to_nearest_residual_range():
    """With every channel equally sensitive the score is proportional to
    sum_g range_g^2: the plain range-aware choice of a 2-bit residual cache."""
    rng = np.random.default_rng(11)
    d, nC = 128, 16
    C = rng.standard_normal((nC, d)).astype(np.float32)
    k = (C[rng.integers(0, nC, 100)] + 0.4 * rng.standard_normal((100, d))).astype(np.float32)
    w = O.group_weights(np.full(d, 0.5, np.float32))
    got = O.qsac_assign(k, C, w)
    for i in range(k.shape[0]):
        best, bj = None, None
        for j in range(nC):
            tot = 0.0
            for g in range(d // 32):
                r = [float(k[i, c]) - float(C[j, c]) for c in range(32 * g, 32 * g + 32)]
                tot += (max(r) - min(r)) ** 2
            if best is None or tot < best - 1e-9 * best:
                best, bj = tot, j
        assert got[i] == bj


def test_permuting_centroids_permutes_indices():
    k, C, w = _tiny_case(2, n=80)
    perm = np.random.default_rng(3).permutation(C.shape[0])
    a = O.qsac_assign(k, C, w)
    b = O.qsac_assign(k, C[perm], w)
    assert (perm[b] == a).all()


def test_power_of_two_sensitivity_scale_leaves_choice_unchanged():
    k, C, w = _tiny_case(4, n=80)
    s = np.random.default_rng(5).uniform(0.1, 9.0, 64).astype(np.float32)
    a = O.qsac_assign(k, C, O.group_weights(s))
    b = O.qsac_assign(k, C, O.group_weights((s * np.float32(8.0)).astype(np.float32)))
    assert (a == b).all()


def test_group_weights_sum_each_group():
    s = np.arange(128, dtype=np.float32)
    w = O.group_weights(s)
    assert w.tolist() == [sum(range(32 * g, 32 * g + 32)) for g in range(4)]


def test_qsac_beats_nearest_centroid_on_weighted_int2_error():
    """The chosen centroid minimises the weighted INT2 error variance, so its
    total is never above that of the nearest centroid (the QVG choice)."""
    rng = np.random.default_rng(6)
    d, nC, n = 64, 12, 150
    sig = np.exp(rng.standard_normal(d))
    C = (rng.standard_normal((nC, d)) * sig).astype(np.float32)
    k = (rng.standard_normal((n, d)) * sig).astype(np.float32)     # keys between centroids
    w = O.group_weights((sig ** 2).astype(np.float32))
    j_q = O.qsac_assign(k, C, w)
    d2 = ((k[:, None, :].astype(np.float64) - C[None].astype(np.float64)) ** 2).sum(-1)
    j_n = d2.argmin(1)
    sq = np.array([O.qsac_scores_exact(k[i], C, w)[j_q[i]] for i in range(len(k))])
    sn = np.array([O.qsac_scores_exact(k[i], C, w)[j_n[i]] for i in range(len(k))])
    assert (sq <= sn * (1 + 1e-6)).all()
    assert (j_q != j_n).any() and sq.sum() < sn.sum()


def test_argmax_mistake_is_caught(monkeypatch):
    """Planting argmax for argmin in the oracle fails the brute-force pin."""
    k, C, w = _tiny_case(0, n=20)
    monkeypatch.setattr(O.np, "argmin", np.argmax)
    bad = O.qsac_assign(k, C, w)
    monkeypatch.undo()
    exact = [int(np.argmin([float(v) for v in _exact_scores(k[i], C, w)])) for i in range(20)]
    assert (bad != np.array(exact)).any()
