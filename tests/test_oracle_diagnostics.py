"""Pins of the oracle's nearest-centroid baseline and of the attention-shift
diagnostics.

The nearest-centroid decision is checked against exact rational squared
distances (brute force); the diagnostics against cases whose answer is known
without them: identical logits change no selection, a full-rank PSAC basis
with exact coefficients reproduces the exact logits, an exact cache has no
output error.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import qwm_oracle as O


def _tiny_case(seed, d=64, nC=12, n=150):
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.standard_normal(d))
    C = (rng.standard_normal((nC, d)) * sig).astype(np.float32)
    z = rng.integers(0, nC, n)
    k = (C[z] + 0.3 * rng.standard_normal((n, d)) * sig).astype(np.float32)
    v = rng.standard_normal((n, d)).astype(np.float32)
    qh = (rng.standard_normal((256, d)) * sig).astype(np.float32)
    q = (rng.standard_normal((40, d)) * sig).astype(np.float32)
    return k, v, C, qh, q


@pytest.mark.parametrize("seed", [0, 1])
def test_nearest_assign_brute_force(seed):
    k, _, C, _, _ = _tiny_case(seed)
    near_ties = 0
    for i in range(k.shape[0]):
        ex = [sum((Fraction(float(k[i, c])) - Fraction(float(C[j, c]))) ** 2 for c in range(k.shape[1]))
              for j in range(C.shape[0])]
        best = min(ex)
        j_exact = ex.index(best)
        j32 = int(O.nearest_assign(k[i:i + 1], C)[0])
        if j32 != j_exact:                             # float32 sums: only near-ties may differ
            assert abs(float(ex[j32]) - float(best)) / float(best) < 1e-6
            near_ties += 1
    assert near_ties <= 1


def test_nearest_scores_match_float64_distances():
    k, _, C, _, _ = _tiny_case(3)
    for i in range(10):
        s32 = O.nearest_scores_f32(k[i], C).astype(np.float64)
        s64 = ((k[i].astype(np.float64) - C.astype(np.float64)) ** 2).sum(axis=1)
        np.testing.assert_allclose(s32, s64, rtol=1e-5)


def test_nearest_and_qsac_differ_and_both_decode():
    """On keys without clean clusters the two assignments differ, and on every
    key QSAC's choice has a sensitivity-weighted residual-range score no larger
    than the nearest centroid's (QSAC minimises that score)."""
    k, v, C, qh, _ = _tiny_case(4)
    rng = np.random.default_rng(4)
    k = (k + 2.0 * rng.standard_normal(k.shape) * np.abs(k).mean(0)).astype(np.float32)   # no clean clusters
    s = O.sensitivity(qh).astype(np.float32)
    w = O.group_weights(s)
    U = np.zeros((0, k.shape[1]))
    a = O.append_head(k, v, C, w, U, assign="nearest")
    b = O.append_head(k, v, C, w, U, assign="qsac")
    assert (a.idx != b.idx).any()
    for i in range(k.shape[0]):
        sa = O.qsac_scores_exact(k[i], C, w)
        assert sa[b.idx[i]] <= sa[a.idx[i]] * (1 + 1e-6)
    with pytest.raises(ValueError):
        O.append_head(k, v, C, w, U, assign="farthest")


def test_top1_change_of_identical_and_swapped_logits():
    rng = np.random.default_rng(0)
    L = rng.standard_normal((50, 80))
    assert O.top1_change(L, L) == 0.0
    L2 = L.copy()
    am = np.argmax(L, axis=1)
    L2[np.arange(10), am[:10]] -= 100.0                 # move the top token of 10 rows
    assert O.top1_change(L, L2) == pytest.approx(10 / 50)


def test_full_rank_exact_compensation_reproduces_exact_attention():
    """r = d and exact coefficients: the compensated logits are q.k, so no
    selection changes and the key-only output error is zero."""
    k, v, C, qh, q = _tiny_case(5)
    d = k.shape[1]
    s = O.sensitivity(qh).astype(np.float32)
    w = O.group_weights(s)
    U, _, _ = O.psac_basis(qh, d)
    seg = O.append_head(k, v, C, w, U)
    ex = q.astype(np.float64) @ k.astype(np.float64).T
    comp = O.compensated_logits(q, [seg], {0: U}, e_exact=True)
    np.testing.assert_allclose(comp, ex, rtol=1e-9, atol=1e-9 * np.abs(ex).max())
    assert O.top1_change(ex, comp) == 0.0
    st = O.key_value_study(q, k, v, [seg], {0: U}, 1 / 8)
    assert st["output_rel_error_key_only"] < 1e-2      # fp16 coefficients only
    assert 0 < st["key_rel_error"] < st["value_rel_error"] < 1


def test_logit_error_is_zero_for_an_exact_cache_and_shrinks_with_psac():
    k, v, C, qh, q = _tiny_case(6)
    s = O.sensitivity(qh).astype(np.float32)
    w = O.group_weights(s)
    seg0 = O.append_head(k, v, C, w, np.zeros((0, k.shape[1])))
    U, _, _ = O.psac_basis(qh, 16)
    seg16 = O.append_head(k, v, C, w, U)
    e0 = O.logit_error(q, k, [seg0], {0: np.zeros((0, k.shape[1]))})
    e16 = O.logit_error(q, k, [seg16], {0: U})
    assert 0 < e16 < e0
    # a cache whose dequantised keys are the keys themselves has no logit error
    seg0.khat = k.astype(np.float64)
    assert O.logit_error(q, k, [seg0], {0: np.zeros((0, k.shape[1]))}) == 0.0
