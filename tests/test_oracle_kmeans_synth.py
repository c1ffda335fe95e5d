"""Pins of the oracle's k-means and of the seeded input generator."""
import numpy as np
import torch

from bit_kv_cache_qwm_gb300 import synth
from oracle import qwm_oracle as O


def test_kmeans_recovers_separated_clusters_and_never_increases_inertia():
    rng = np.random.default_rng(0)
    centres = rng.standard_normal((6, 16)) * 20
    lab = rng.integers(0, 6, 600)
    X = centres[lab] + 0.1 * rng.standard_normal((600, 16))
    # start from one key of each cluster
    init = np.array([np.flatnonzero(lab == c)[0] for c in range(6)])
    prev = None
    for it in range(1, 8):
        Cm = O.kmeans(X, init, iters=it)
        inertia = ((X[:, None, :] - Cm[None]) ** 2).sum(-1).min(1).sum()
        if prev is not None:
            assert inertia <= prev + 1e-9
        prev = inertia
    # every true centre has a fitted centroid within the noise
    d = np.sqrt(((centres[:, None, :] - Cm[None]) ** 2).sum(-1)).min(1)
    assert (d < 0.05).all()


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(1).standard_normal(20000).astype(np.float32) * 37
    ours = synth.round_to_bf16(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ours, ref)


def test_generator_is_deterministic_and_prefix_stable():
    wl = synth.workload("bf16-h12-n32760")
    a = synth.keys(wl, 2, heads=[3], n=100)
    b = synth.keys(wl, 2, heads=[3])
    assert np.array_equal(a[0], b[0, :100])
    assert np.array_equal(synth.values(wl, 1, heads=[0, 5])[1], synth.values(wl, 1, heads=[5])[0])
    assert np.array_equal(synth.round_to_bf16(b), b)          # exactly bf16
    q = synth.queries(wl, 0, heads=[2], m=50)
    assert q.shape == (1, 50, 128)


def test_generator_distributions():
    wl = synth.workload("bf16-h40-n98280-outlier")
    sig = synth.channel_scale(wl, 0)
    out = synth.outlier_channels(wl, 0)
    assert len(out) == 4
    v = synth.values(wl, 0, heads=[0], n=2000)[0]
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1) < 0.02
    q = synth.queries(wl, 0, heads=[0], m=4000)[0]
    ratio = q.std(0) / sig
    assert np.all(np.abs(ratio - 1) < 0.1)


def test_stream_ring_is_last_queries_of_previous_chunk():
    wl = synth.workload("bf16-h24-stream-n374400")
    r = synth.hist_queries(wl, 3, heads=[1])
    q = synth.queries(wl, 2, heads=[1])
    assert np.array_equal(r[0], q[0, -4096:])
