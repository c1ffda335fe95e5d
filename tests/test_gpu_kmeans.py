"""qwm_kmeans (Lloyd on the GPU) against the oracle's k-means.

The centroids are an input of every other parity test, so k-means itself is
checked by properties: the starting rows are reproduced exactly; after one
iteration every key is assigned as the oracle assigns it unless its two best
centroids are tied within 1e-5 relative, and clusters with the same members
have the same mean to float32 rounding; after 25 iterations the inertia is
within 3% of the oracle's (k-means has many local optima, and one near-tie
can move the trajectory)."""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from oracle import qwm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    return q


def _setup(name, heads):
    wl = synth.workload(name)
    kf = synth.kmeans_keys(wl, heads)
    rows = np.stack([synth.kmeans_init_rows(wl, h, kf.shape[1], wl.n_centroids) for h in heads])
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    return wl, kf, rows, torch.from_numpy(kf).to("cuda", dt), torch.from_numpy(rows.astype(np.int32)).cuda()


def _inertia(X, C):
    X = X.astype(np.float64)
    C = C.astype(np.float64)
    d2 = (X * X).sum(1)[:, None] - 2 * X @ C.T + (C * C).sum(1)[None]
    return float(np.maximum(d2.min(1), 0).sum())


@pytest.mark.parametrize("name", ["bf16-h12-n32760", "tiny-f32-h1-n1024"])
def test_zero_iterations_returns_the_starting_rows(qwm, name):
    wl, kf, rows, kt, rt = _setup(name, [0])
    out = qwm.qwm_kmeans(kt, rt, wl.n_centroids, iters=0).float().cpu().numpy()
    assert np.array_equal(out[0], kf[0][rows[0]])


@pytest.mark.parametrize("name", ["bf16-h12-n32760", "tiny-f32-h1-n1024"])
def test_one_iteration_matches_the_oracle(qwm, name):
    wl, kf, rows, kt, rt = _setup(name, [0, 3] if name.startswith("bf16") else [0])
    got32 = qwm.qwm_kmeans(kt, rt, wl.n_centroids, iters=1)
    if wl.dtype == "f32":
        got = got32.cpu().numpy()
    else:
        got = got32.float().cpu().numpy()
    for i in range(kf.shape[0]):
        X = kf[i].astype(np.float64)
        C0 = X[rows[i]]
        d2 = ((X[:, None, :] - C0[None]) ** 2).sum(-1)
        a = d2.argmin(1)
        srt = np.sort(d2, 1)
        tie = (srt[:, 1] - srt[:, 0]) <= 1e-5 * srt[:, 1]
        ref = O.kmeans(X, rows[i], iters=1)
        ref_r = synth.round_to_dtype(ref, wl.dtype)
        # clusters without a tied member have the oracle's mean, rounded to the dtype
        clean = np.ones(wl.n_centroids, bool)
        clean[a[tie]] = False
        for j in np.flatnonzero(clean):
            np.testing.assert_allclose(got[i, j], ref_r[j], rtol=2 ** -7 if wl.dtype == "bf16" else 1e-6,
                                       atol=1e-6)


@pytest.mark.parametrize("name", ["bf16-h12-n32760", "tiny-f32-h1-n1024"])
def test_25_iterations_reach_the_oracles_inertia(qwm, name):
    wl, kf, rows, kt, rt = _setup(name, [0, 5] if name.startswith("bf16") else [0])
    got = qwm.qwm_kmeans(kt, rt, wl.n_centroids, iters=25).float().cpu().numpy()
    for i in range(kf.shape[0]):
        ref = synth.round_to_dtype(O.kmeans(kf[i], rows[i], iters=25), wl.dtype)
        a, b = _inertia(kf[i], got[i]), _inertia(kf[i], ref)
        assert a <= 1.03 * b and b <= 1.03 * a, (a, b)
        start = _inertia(kf[i], kf[i][rows[i]])
        assert a < start
