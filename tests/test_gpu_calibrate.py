"""qwm_calibrate on the GPU against the oracle.

s to 1e-5 relative; the basis: Ritz residual ||G u - lambda u|| / lambda_1
<= 1e-5 and U U^T = I to 1e-6 always.  When lambda_r / lambda_{r+1} >= 1.05
the projector distance to the oracle's (LAPACK) basis is bounded by what the
residual bound implies (Davis-Kahan sin-theta theorem):
    ||P - P_ref||_2 <= sqrt(r) * 1e-5 * lambda_1 / (lambda_r - lambda_{r+1}),
with a floor of 1e-4."""
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


def _tensor(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to("cuda", torch.bfloat16 if dtype == "bf16" else torch.float32)


def _check(qwm, qh, r, dtype, max_iter=64, oversample=16, expect_converged=True):
    H, n_h, d = qh.shape
    ctx = qwm.Qwm(H, d, r, 16, dtype=dtype, max_tokens=128, max_iter=max_iter, oversample=oversample,
                  max_hist=max(n_h, 1))
    ctx.calibrate(_tensor(qh, dtype))
    st = ctx.status()
    cal = ctx.get_calibration()
    for h in range(H):
        s_ref = O.sensitivity(qh[h])
        np.testing.assert_allclose(cal["s"][h], s_ref, rtol=1e-5, atol=1e-30)
        if r == 0:
            continue
        G = O.gram(qh[h])
        U_ref, lam_ref, en_ref = O.psac_basis(qh[h], r)
        lam_all = np.sort(np.linalg.eigvalsh(G))[::-1]
        U = cal["U"][h].astype(np.float64)
        lam = cal["lambda"][h].astype(np.float64)
        res = np.linalg.norm(G @ U.T - U.T * lam, axis=0) / lam_all[0]
        assert res.max() <= 1e-5, res.max()
        assert np.abs(U @ U.T - np.eye(r)).max() <= 1e-6
        np.testing.assert_allclose(lam, lam_ref, rtol=1e-5, atol=1e-6 * lam_all[0])
        assert abs(cal["energy"][h] - en_ref) <= 1e-5
        if r < d and lam_all[r - 1] / max(lam_all[r], 1e-300) >= 1.05:
            P = U.T @ U - U_ref.T @ U_ref
            bound = max(1e-4, 1.5 * np.sqrt(r) * 1e-5 * lam_all[0] / (lam_all[r - 1] - lam_all[r]))
            assert np.linalg.norm(P, 2) <= bound
        # sign rule
        for i in range(r):
            j = int(np.argmax(np.abs(U[i])))
            assert U[i, j] > 0
    if expect_converged:
        assert st == 0
    return st


def test_calibrate_tiny_f32(qwm):
    wl = synth.workload("tiny-f32-h1-n1024")
    _check(qwm, synth.hist_queries(wl, 0), wl.rank, "f32")


@pytest.mark.parametrize("r", [0, 1, 16, 32, 64])
def test_calibrate_bf16_ranks(qwm, r):
    wl = synth.workload("bf16-h12-n32760")
    _check(qwm, synth.hist_queries(wl, 0, heads=[0, 3, 6]), r, "bf16")


def test_calibrate_full_rank_jacobi_path(qwm):
    wl = synth.workload("tiny-f32-h1-n1024")
    _check(qwm, synth.hist_queries(wl, 0), 64, "f32")


def test_calibrate_outlier_heads_and_ring(qwm):
    wl = synth.workload("bf16-h40-n98280-outlier")
    _check(qwm, synth.hist_queries(wl, 0, heads=[0, 1, 2, 39]), 16, "bf16")
    ws = synth.workload("bf16-h24-stream-n374400")
    _check(qwm, synth.hist_queries(ws, 2, heads=[0, 23]), 16, "bf16")


def test_calibrate_degenerate_inputs(qwm):
    """One historical query (rank-1 Gram) and all-zero queries give finite,
    orthonormal bases and the exact sensitivity."""
    rng = np.random.default_rng(0)
    one = rng.standard_normal((1, 1, 64)).astype(np.float32)
    ctx = qwm.Qwm(1, 64, 4, 16, dtype="f32", max_tokens=128, max_hist=8)
    ctx.calibrate(_tensor(one, "f32"))
    cal = ctx.get_calibration()
    assert np.isfinite(cal["U"]).all()
    U = cal["U"][0].astype(np.float64)
    assert np.abs(U @ U.T - np.eye(4)).max() <= 1e-5
    u0 = one[0, 0] / np.linalg.norm(one[0, 0])
    assert abs(abs(U[0] @ u0) - 1) < 1e-5
    np.testing.assert_allclose(cal["s"][0], one[0, 0].astype(np.float64) ** 2, rtol=1e-6)
    zero = np.zeros((1, 8, 64), np.float32)
    ctx.calibrate(_tensor(zero, "f32"))
    cal = ctx.get_calibration()
    assert np.isfinite(cal["U"]).all() and (cal["s"] == 0).all()


def test_iteration_cap_reports_not_converged(qwm):
    """Equal channel scales give tiny eigen-gaps; one iteration cannot reach
    the residual tolerance, and the device status says so."""
    rng = np.random.default_rng(1)
    qh = rng.standard_normal((2, 1024, 128)).astype(np.float32)
    st = _check_status_only(qwm, qh, 16, max_iter=1)
    assert st == 5


def _check_status_only(qwm, qh, r, max_iter):
    H, n_h, d = qh.shape
    ctx = qwm.Qwm(H, d, r, 16, dtype="f32", max_tokens=128, max_iter=max_iter, max_hist=n_h)
    ctx.calibrate(_tensor(qh, "f32"))
    st = ctx.status()
    cal = ctx.get_calibration()
    assert np.isfinite(cal["U"]).all()
    return st
