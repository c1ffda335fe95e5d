"""Pins of the oracle's attention over the packed cache."""
import numpy as np
import pytest
import torch

from oracle import qwm_oracle as O


def _exact_cache(seed, n=256, d=64, nC=8):
    """Keys equal to centroids and values on exactly representable INT2 levels,
    so quantisation loses nothing."""
    rng = np.random.default_rng(seed)
    C = rng.standard_normal((nC, d)).astype(np.float32)
    idx = rng.integers(0, nC, n)
    k = C[idx].copy()
    # each group of values: zero + {0,1,2,3} * scale with min and max present
    G = d // 32
    zero = rng.integers(-64, 64, (n, G)).astype(np.float32) / 16      # f16-exact
    scale = rng.integers(1, 32, (n, G)).astype(np.float32) / 8        # f16-exact
    codes = rng.integers(0, 4, (n, G, 32))
    codes[:, :, 0] = 0
    codes[:, :, 1] = 3
    v = (zero[:, :, None] + codes * scale[:, :, None]).reshape(n, d).astype(np.float32)
    return C, k, v, idx


def test_reduces_to_textbook_attention():
    C, k, v, idx = _exact_cache(0)
    w = O.group_weights(np.ones(64, np.float32))
    U = np.zeros((0, 64))
    seg = O.append_head(k, v, C, w, U)
    assert (seg.idx == idx).all() or np.array_equal(C[seg.idx], C[idx])
    assert np.array_equal(seg.khat, k.astype(np.float64))
    assert np.array_equal(seg.vhat, v.astype(np.float64))
    q = np.random.default_rng(1).standard_normal((32, 64))
    out = O.attend_head(q, [seg], {0: U}, sigma=0.125)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None], torch.from_numpy(k.astype(np.float64))[None],
        torch.from_numpy(v.astype(np.float64))[None], scale=0.125)[0].numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_weights_are_a_distribution():
    C, k, v, _ = _exact_cache(2)
    k = k + np.float32(0.1) * np.random.default_rng(3).standard_normal(k.shape).astype(np.float32)
    Qh = np.random.default_rng(4).standard_normal((100, 64))
    U, _, _ = O.psac_basis(Qh, 4)
    seg = O.append_head(k.astype(np.float32), v, C, O.group_weights(np.ones(64, np.float32)), U)
    P = O.attention_weights(np.random.default_rng(5).standard_normal((16, 64)) * 5, [seg], {0: U}, 0.125)
    assert (P >= 0).all()
    assert np.allclose(P.sum(1), 1.0, atol=1e-14)


def test_segments_use_their_own_basis():
    """Two appends in two basis versions: each key's logit uses the basis its
    coefficients were stored in.  Checked against the equivalent folded key
    k_hat + U_t^T e computed per token."""
    rng = np.random.default_rng(6)
    d = 64
    C = rng.standard_normal((8, d)).astype(np.float32)
    w = O.group_weights(np.ones(d, np.float32))
    U0, _, _ = O.psac_basis(rng.standard_normal((100, d)), 4)
    U1, _, _ = O.psac_basis(rng.standard_normal((100, d)) * np.exp(rng.standard_normal(d)), 4)
    k0 = (C[rng.integers(0, 8, 50)] + 0.3 * rng.standard_normal((50, d))).astype(np.float32)
    k1 = (C[rng.integers(0, 8, 70)] + 0.3 * rng.standard_normal((70, d))).astype(np.float32)
    v0 = rng.standard_normal((50, d)).astype(np.float32)
    v1 = rng.standard_normal((70, d)).astype(np.float32)
    s0 = O.append_head(k0, v0, C, w, U0, version=0)
    s1 = O.append_head(k1, v1, C, w, U1, version=1)
    q = rng.standard_normal((9, d)) * 3
    out = O.attend_head(q, [s0, s1], {0: U0, 1: U1}, sigma=0.125)
    kf = np.vstack([s0.khat + s0.e16.astype(np.float64) @ U0, s1.khat + s1.e16.astype(np.float64) @ U1])
    L = 0.125 * q @ kf.T
    P = np.exp(L - L.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    assert np.allclose(out, P @ np.vstack([s0.vhat, s1.vhat]), rtol=1e-10, atol=1e-12)


def test_empty_cache_is_an_error():
    with pytest.raises(ValueError):
        O.attend_head(np.zeros((2, 64)), [], {}, 0.125)
