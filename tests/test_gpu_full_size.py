"""Parity at the full sizes of the two largest workloads, in the launch
configuration the benchmark times (automatic kernel choice, all heads on the
GPU), on sampled outputs the oracle recomputes one by one:

* bf16-h40-n98280-outlier: 40 heads with 10x outlier channels, 20 appends of
  4,680 tokens (93,600 cached), then the timed append of 4,680 and attention
  of 4,680 query rows over 98,280 tokens.  The oracle re-encodes the last
  append of the first and last head (bit-exact bytes, e within its bound) and
  recomputes 16 seeded query rows of those heads over the GPU's cache bytes.
* bf16-h24-stream-n374400: 24 heads, 80 streaming steps, each with a new PSAC
  basis from the 4,096-query ring of the previous chunk (80 basis versions)
  and an append of 4,680 tokens, to 374,400 cached tokens; then attention of
  the last chunk's 4,680 query rows.  The oracle recomputes 16 seeded rows of
  the first and last head over all 80 segments.

The centroids are the seeded starting rows of the k-means on frame 0 (an input
both sides share; the parity does not depend on how the centroids were
fitted), the bases come from the oracle's calibration.  Tolerance as for the
other bf16 attention tests: max |O_gpu - O_oracle| <= 1e-2 * max|V_hat|.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import calibration, compare_segment_bytes, decode_gpu_segments
from oracle import qwm_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    return q


def _tensor(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)


def _start_centroids(wl):
    """The k-means starting rows of frame 0 for every head, rounded to bf16."""
    kf = synth.kmeans_keys(wl)
    rows = [kf[h][synth.kmeans_init_rows(wl, h, kf.shape[1], wl.n_centroids)] for h in range(wl.heads)]
    return synth.round_to_dtype(np.stack(rows), wl.dtype)


def _check_rows(ctx, cent, bases, q, got, heads, n_rows, seed):
    tiles = ctx.cache_tiles().cpu().numpy()
    table = ctx.tile_table().cpu().numpy()
    c = ctx.cfg
    rows = np.sort(np.random.default_rng(seed).choice(q.shape[1], n_rows, replace=False))
    for h in heads:
        segs = decode_gpu_segments(tiles[h], table, cent[h], c.head_dim, c.rank, c.n_centroids, ctx.n_tiles)
        b = {v: bases[v][h].astype(np.float64) for v in range(len(bases))}
        want = O.attend_head(q[h][rows], segs, b, 1 / np.sqrt(c.head_dim))
        vmax = max(np.abs(sg.vhat).max() for sg in segs)
        err = np.abs(got[h][rows] - want).max()
        assert err <= 1e-2 * vmax, (h, err, vmax)


def test_outlier_workload_full_size(qwm):
    name = "bf16-h40-n98280-outlier"
    wl = synth.workload(name)
    H, d, r, C = wl.heads, wl.head_dim, wl.rank, wl.n_centroids
    tiles_per_chunk = (wl.chunk + 127) // 128
    cent = _start_centroids(wl)
    s, U = calibration(name)
    ctx = qwm.Qwm(H, d, r, C, dtype="bf16", max_tokens=wl.n_chunks * tiles_per_chunk * 128)
    ctx.set_centroids(_tensor(cent))
    ctx.set_calibration(s, U)
    for ch in range(wl.n_chunks):
        ctx.append(_tensor(synth.keys(wl, ch)), _tensor(synth.values(wl, ch)))
    assert ctx.n_tokens == wl.n_tokens == 98280
    q = synth.queries(wl, 0)
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.resolved_attend_kernel == 6 and ctx.status() == 0
    assert np.isfinite(got).all()
    heads = [0, H - 1]
    _check_rows(ctx, cent, [U], q, got, heads, 16, 7)
    # the timed append: the last chunk's tiles of the checked heads
    last = wl.n_chunks - 1
    k, v = synth.keys(wl, last, heads), synth.values(wl, last, heads)
    gpu_tiles = ctx.cache_tiles().cpu().numpy()
    t0 = last * tiles_per_chunk
    for i, h in enumerate(heads):
        seg = O.append_head(k[i], v[i], cent[h], O.group_weights(s[h]), U[h].astype(np.float64))
        compare_segment_bytes(gpu_tiles[h, t0:t0 + tiles_per_chunk], seg, k[i], d, r, C)


def test_stream_workload_full_size(qwm):
    name = "bf16-h24-stream-n374400"
    wl = synth.workload(name)
    H, d, r, C = wl.heads, wl.head_dim, wl.rank, wl.n_centroids
    tiles_per_chunk = (wl.chunk + 127) // 128
    cent = _start_centroids(wl)
    ctx = qwm.Qwm(H, d, r, C, dtype="bf16", max_tokens=wl.n_chunks * tiles_per_chunk * 128,
                  max_versions=wl.n_chunks)
    ctx.set_centroids(_tensor(cent))
    bases = []
    for ch in range(wl.n_chunks):
        s, U = calibration(name, None, None, ch)   # the ring of the previous chunk's queries
        ctx.set_calibration(s, U)
        bases.append(U)
        ctx.append(_tensor(synth.keys(wl, ch)), _tensor(synth.values(wl, ch)))
    assert ctx.n_tokens == wl.n_tokens == 374400
    q = synth.queries(wl, wl.n_chunks - 1)
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.resolved_attend_kernel == 6 and ctx.status() == 0
    assert np.isfinite(got).all()
    _check_rows(ctx, cent, bases, q, got, [0, H - 1], 16, 11)
