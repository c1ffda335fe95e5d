"""Pins of the oracle's PSAC basis, coefficients and compensated logits."""
import numpy as np
import pytest

from oracle import qwm_oracle as O


def _qhist(seed, n=512, d=64):
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.standard_normal(d))
    return rng.standard_normal((n, d)) * sig


def test_basis_matches_svd_and_sign_rule():
    Q = _qhist(0)
    r = 8
    U, lam, energy = O.psac_basis(Q, r)
    _, sv, Vt = np.linalg.svd(Q, full_matrices=False)      # a different LAPACK path
    assert np.allclose(lam, sv[:r] ** 2, rtol=1e-10)
    P1 = U.T @ U
    P2 = Vt[:r].T @ Vt[:r]
    assert np.linalg.norm(P1 - P2, 2) < 1e-8
    assert np.allclose(U @ U.T, np.eye(r), atol=1e-12)
    for i in range(r):
        j = np.argmax(np.abs(U[i]))
        assert U[i, j] > 0
    assert abs(energy - (sv[:r] ** 2).sum() / (sv ** 2).sum()) < 1e-12


def test_basis_of_orthogonal_columns_is_unit_vectors():
    """Queries with orthogonal columns of distinct norms: G is diagonal, the
    eigenvectors are unit vectors ordered by column norm."""
    d = 64
    norms = np.random.default_rng(1).permutation(np.arange(1, d + 1)).astype(np.float64)
    Q = np.zeros((d, d))
    Q[np.arange(d), np.arange(d)] = norms
    Q = np.vstack([Q, np.zeros((5, d))])
    U, lam, _ = O.psac_basis(Q, 5)
    order = np.argsort(-norms)[:5]
    for i in range(5):
        e = np.zeros(d)
        e[order[i]] = 1.0
        assert np.allclose(U[i], e)
        assert lam[i] == pytest.approx(norms[order[i]] ** 2)


def _segment(seed, r, d=64, n=150, nC=8, e_basis=None):
    rng = np.random.default_rng(seed)
    sig = np.exp(rng.standard_normal(d))
    C = (rng.standard_normal((nC, d)) * sig).astype(np.float32)
    k = (C[rng.integers(0, nC, n)] + 0.3 * rng.standard_normal((n, d)) * sig).astype(np.float32)
    v = rng.standard_normal((n, d)).astype(np.float32)
    Qh = rng.standard_normal((400, d)) * sig
    U, _, _ = O.psac_basis(Qh, r)
    w = O.group_weights(O.sensitivity(Qh).astype(np.float32))
    seg = O.append_head(k, v, C, w, U, version=0)
    return k, seg, U, Qh, sig


def test_full_rank_compensation_restores_exact_logits():
    k, seg, U, _, sig = _segment(0, r=64)
    q = np.random.default_rng(9).standard_normal((20, 64)) * sig
    l_comp = q @ seg.khat.T + (q @ U.T) @ seg.e64.T
    l_true = q @ k.astype(np.float64).T
    assert np.max(np.abs(l_comp - l_true)) <= 1e-12 * np.max(np.abs(l_true))


def test_rank_zero_gives_quantised_logits():
    k, seg, U, _, sig = _segment(1, r=0)
    assert seg.e16.shape == (150, 0)
    q = np.random.default_rng(2).standard_normal((10, 64)) * sig
    P = O.attention_weights(q, [seg], {0: U}, 0.125)
    L = 0.125 * (q @ seg.khat.T)
    ref = np.exp(L - L.max(1, keepdims=True))
    assert np.allclose(P, ref / ref.sum(1, keepdims=True), rtol=1e-12)


def test_query_in_subspace_sees_exact_key():
    k, seg, U, _, _ = _segment(3, r=8)
    q = np.random.default_rng(4).standard_normal((10, 8)) @ U       # q in span(U_r)
    l_comp = q @ seg.khat.T + (q @ U.T) @ seg.e64.T
    l_true = q @ k.astype(np.float64).T
    assert np.max(np.abs(l_comp - l_true)) <= 1e-10 * np.max(np.abs(l_true))


def test_compensation_removes_the_captured_query_energy():
    """Over the historical queries themselves, the squared logit error left
    after compensation equals sum_{j>r} lambda_j (u_j . delta)^2 exactly."""
    k, seg, U, Qh, _ = _segment(5, r=8)
    delta = k.astype(np.float64) - seg.khat                       # [n, d]
    G = O.gram(Qh)
    lam, vec = np.linalg.eigh(G)
    lam, vec = lam[::-1], vec[:, ::-1]
    after = Qh @ (delta - seg.e64 @ U).T                           # logit errors left
    left = (after ** 2).sum(0)
    closed = ((delta @ vec[:, 8:]) ** 2 * lam[8:]).sum(1)
    assert np.allclose(left, closed, rtol=1e-8)
    before = ((Qh @ delta.T) ** 2).sum(0)
    assert (left <= before + 1e-9 * before).all()


def test_coefficients_are_stored_in_fp16():
    _, seg, _, _, _ = _segment(6, r=4)
    assert seg.e16.dtype == np.float16
    assert np.array_equal(seg.e16, seg.e64.astype(np.float16))
