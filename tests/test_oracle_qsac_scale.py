"""The float32 QSAC decision against the exact argmin at the sizes of the
benchmarked workloads (d = 128, 256 k-means centroids fitted on frame 0,
lognormal channel scales, 10x outlier channels in the 40-head workload).

The oracle decides the centroid in float32 (the precision the GPU decides
in), so a centroid whose exact score is within float32 rounding of the best
one can be chosen instead of the exact argmin.  The QSAC score is
sum_g w_g (range_g(k - C_j)/3)^2/12 (QuantWM Abstract, "historical Query
sensitivity and residual ranges"; roboind article, "Step 1").  Every
disagreement must be such a near-tie: the exact scores of the two choices
differ by less than 1e-6 relative.  The exact scores are rationals
(`fractions`), so the check does not rest on any floating-point order.
The counts are printed (pytest -s) and recorded in the design notes.
"""
from fractions import Fraction

import numpy as np
import pytest

from bit_kv_cache_qwm_gb300 import synth
from oracle import qwm_oracle as O

TIE_GAP = 1e-6


def _exact(k, Cj, w):
    tot = Fraction(0)
    for g in range(k.shape[0] // 32):
        res = [Fraction(float(k[c])) - Fraction(float(Cj[c])) for c in range(32 * g, 32 * g + 32)]
        tot += Fraction(float(w[g])) * ((max(res) - min(res)) / 3) ** 2 / 12
    return tot


def decision_vs_exact(name, head, n_tokens, chunk, kmeans_iters=25):
    """(disagreements, max relative gap, tokens) of the float32 decision
    against the exact argmin on `n_tokens` keys of append `chunk`."""
    wl = synth.workload(name)
    kf = synth.kmeans_keys(wl, [head])[0]
    rows = synth.kmeans_init_rows(wl, head, kf.shape[1], wl.n_centroids)
    C = synth.round_to_dtype(O.kmeans(kf, rows, kmeans_iters), wl.dtype)
    s = O.sensitivity(synth.hist_queries(wl, chunk, [head])[0]).astype(np.float32)
    w = O.group_weights(s)
    k = synth.keys(wl, chunk, [head], n=n_tokens)[0]
    j32 = O.qsac_assign(k, C, w)
    bad, worst = 0, 0.0
    for i in range(k.shape[0]):
        s64 = O.qsac_scores_exact(k[i], C, w)
        # exact argmin: the float64 candidates within 1e-9 of the best, decided exactly
        cand = np.flatnonzero(s64 <= s64.min() * (1 + 1e-9))
        ex = {int(j): _exact(k[i], C[j], w) for j in set(cand.tolist()) | {int(j32[i])}}
        best = min(ex[int(j)] for j in cand)
        j_exact = min(int(j) for j in cand if ex[int(j)] == best)
        if int(j32[i]) != j_exact:
            bad += 1
            worst = max(worst, float((ex[int(j32[i])] - best) / best))
    return bad, worst, k.shape[0]


@pytest.mark.parametrize("name,head,chunk", [
    ("bf16-h12-n32760", 0, 6),
    ("bf16-h40-n98280-outlier", 39, 20),
    ("bf16-h24-stream-n374400", 23, 79),
])
def test_float32_decision_is_exact_up_to_near_ties(name, head, chunk):
    bad, worst, n = decision_vs_exact(name, head, 300, chunk)
    print(f"\n{name} head {head}: {bad} of {n} float32 decisions differ from the exact argmin, "
          f"largest relative score gap {worst:.2e}")
    assert worst < TIE_GAP
    assert bad <= 3


@pytest.mark.parametrize("slip", ["range_not_squared", "weights_dropped"])
def test_planted_score_mistake_is_caught(monkeypatch, slip):
    """Two plausible slips in the float32 score -- the range entering
    linearly instead of squared, the sensitivity weights left out -- pick
    centroids whose exact score is clearly above the best one."""
    def wrong(k32, C32, w32):
        k = np.asarray(k32, dtype=np.float32)
        rho = (k[None, :] - np.asarray(C32, dtype=np.float32)).astype(np.float32)
        rg = rho.reshape(rho.shape[0], -1, 32)
        R = (rg.max(-1) - rg.min(-1)).astype(np.float32)
        if slip == "range_not_squared":
            t = np.asarray(w32, np.float32)[None, :] * R
        else:
            t = R * R
        return O._score_tree(t.astype(np.float32))
    monkeypatch.setattr(O, "qsac_scores_f32", wrong)
    bad, worst, _ = decision_vs_exact("bf16-h40-n98280-outlier", 39, 120, 20, kmeans_iters=5)
    monkeypatch.undo()
    assert bad > 0 and worst >= TIE_GAP
