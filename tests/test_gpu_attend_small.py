"""qwm_attend with few query rows (kernel 5: split over the cache tiles,
exact code products) on the GPU against the oracle.

Tolerance as for the other bf16 kernels: max |O_gpu - O_oracle| <= 1e-2 *
max|V_hat|; the oracle attends over the GPU's own cache bytes.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import calibration, centroids, decode_gpu_segments
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


def _oracle(ctx, cent, bases, q, heads_idx, scale):
    tiles = ctx.cache_tiles().cpu().numpy()
    table = ctx.tile_table().cpu().numpy()
    c = ctx.cfg
    out, vmax = [], 0.0
    for i in heads_idx:
        segs = decode_gpu_segments(tiles[i], table, cent[i], c.head_dim, c.rank, c.n_centroids, ctx.n_tiles)
        b = {v: bases[v][i].astype(np.float64) for v in range(len(bases))}
        out.append(O.attend_head(q[i], segs, b, scale))
        vmax = max(vmax, max(np.abs(sg.vhat).max() for sg in segs))
    return np.stack(out), vmax


def _ragged_context(qwm, name, C, r, sizes=(300, 1, 228, 129, 100, 64)):
    wl = synth.workload(name)
    heads = [0, 1]
    cent = centroids(name, tuple(heads), C, iters=25 if C <= 256 else 3)
    ctx = qwm.Qwm(2, 128, r, C, dtype="bf16", max_tokens=sum((n + 127) // 128 for n in sizes) * 128,
                  max_versions=3)
    ctx.set_centroids(_tensor(cent))
    bases = []
    for ch, n in enumerate(sizes):
        if ch % 2 == 0:
            s_, U = calibration(name, tuple(heads), r, step=len(bases))
            ctx.set_calibration(s_, U)
            bases.append(U)
        ctx.append(_tensor(synth.keys(wl, ch, heads, n)), _tensor(synth.values(wl, ch, heads, n)))
    return wl, ctx, cent, bases


@pytest.mark.parametrize("m", [1, 5, 16, 17, 64])
@pytest.mark.parametrize("name,C,r", [("bf16-h12-n32760", 256, 16), ("bf16-h24-append-sweep", 1024, 32),
                                      ("bf16-h24-append-sweep", 64, 8), ("bf16-h24-append-sweep", 256, 0),
                                      ("bf16-h24-append-sweep", 7, 3), ("bf16-h40-n98280-outlier", 256, 16)])
def test_small_m_variants(qwm, name, C, r, m):
    """Ragged appends (tails of 1 and 100 slots) under three basis versions,
    rank 0 / 3 / 8 / 16 / 32, 7 to 1024 centroids, outlier channels; M from 1
    to 64 rows (one to four row blocks, ragged)."""
    wl, ctx, cent, bases = _ragged_context(qwm, name, C, r)
    assert ctx.attend_kernel_for(m) == (7 if m > 16 and r <= 16 else 5)
    ctx.set_attend_kernel(5)
    q = synth.queries(wl, 3, [0, 1], m=m)
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.status() == 0
    want, vmax = _oracle(ctx, cent, bases, q, [0, 1], 1 / np.sqrt(128))
    err = np.abs(got - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)


@pytest.mark.parametrize("m", [1, 16, 17, 40, 64])
@pytest.mark.parametrize("name,C,r", [("bf16-h12-n32760", 256, 16), ("bf16-h24-append-sweep", 1024, 8),
                                      ("bf16-h24-append-sweep", 256, 0), ("bf16-h24-append-sweep", 7, 3),
                                      ("bf16-h40-n98280-outlier", 256, 16)])
def test_few_row_split_key_kernel(qwm, name, C, r, m):
    """Kernel 7 (kernel 6 with one 128-row query tile per CTA, the cache
    split over CTAs, partials merged by the few-row combine kernel): ragged
    appends under three basis versions, rank 0 / 3 / 8 / 16, 7 to 1024
    centroids, outlier channels, M from 1 to 64."""
    wl, ctx, cent, bases = _ragged_context(qwm, name, C, r)
    ctx.set_attend_kernel(7)
    q = synth.queries(wl, 3, [0, 1], m=m)
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.status() == 0
    want, vmax = _oracle(ctx, cent, bases, q, [0, 1], 1 / np.sqrt(128))
    err = np.abs(got - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)


def test_few_row_split_key_kernel_full_cache(qwm):
    """Kernel 7 over 12 heads x 32,760 cached tokens (259 tiles per head split
    over many CTAs), 48 rows; the oracle checks heads 0 and 11 completely; an
    explicit request for more than 64 rows is refused."""
    name = "bf16-h12-n32760"
    wl = synth.workload(name)
    heads = list(range(wl.heads))
    cent = centroids(name, tuple(heads))
    ctx = qwm.Qwm(wl.heads, 128, wl.rank, wl.n_centroids, dtype="bf16",
                  max_tokens=wl.n_chunks * ((wl.chunk + 127) // 128) * 128)
    ctx.set_centroids(_tensor(cent))
    s_, U = calibration(name, tuple(heads), wl.rank)
    ctx.set_calibration(s_, U)
    for ch in range(wl.n_chunks):
        ctx.append(_tensor(synth.keys(wl, ch)), _tensor(synth.values(wl, ch)))
    ctx.set_attend_kernel(7)
    q = synth.queries(wl, 0, m=48)
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.status() == 0 and np.isfinite(got).all()
    want, vmax = _oracle(ctx, cent, [U], q, [0, 11], 1 / np.sqrt(128))
    err = np.abs(got[[0, 11]] - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)
    with pytest.raises(qwm.QwmError) as e:
        ctx.attend(_tensor(synth.queries(wl, 0, m=65)))
    assert e.value.status == 2


def test_small_m_matches_large_m_kernel(qwm):
    """The same 64 rows through kernel 5 and through the tcgen05 kernel agree
    (both within the tolerance of the oracle, and of each other)."""
    wl, ctx, cent, bases = _ragged_context(qwm, "bf16-h12-n32760", 256, 16)
    q = _tensor(synth.queries(wl, 2, [0, 1], m=64))
    a = ctx.attend(q).float()
    ctx.set_attend_kernel(4)
    b = ctx.attend(q).float()
    vmax = max(np.abs(sg.vhat).max() for sg in
               decode_gpu_segments(ctx.cache_tiles().cpu().numpy()[0], ctx.tile_table().cpu().numpy(), cent[0],
                                   128, 16, 256, ctx.n_tiles))
    assert float((a - b).abs().max()) <= 2e-2 * vmax


def test_small_m_full_cache_sampled_heads(qwm):
    """12 heads, 7 appends of 4,680 tokens (32,760 cached, 259 tiles per head,
    the tiles split over many CTAs), 16 query rows; the oracle checks heads 0
    and 11 completely."""
    name = "bf16-h12-n32760"
    wl = synth.workload(name)
    heads = list(range(wl.heads))
    cent = centroids(name, tuple(heads))
    ctx = qwm.Qwm(wl.heads, 128, wl.rank, wl.n_centroids, dtype="bf16",
                  max_tokens=wl.n_chunks * ((wl.chunk + 127) // 128) * 128)
    ctx.set_centroids(_tensor(cent))
    s_, U = calibration(name, tuple(heads), wl.rank)
    ctx.set_calibration(s_, U)
    for ch in range(wl.n_chunks):
        ctx.append(_tensor(synth.keys(wl, ch)), _tensor(synth.values(wl, ch)))
    q = synth.queries(wl, 0, m=16)
    assert ctx.attend_kernel_for(16) == 5
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.status() == 0
    want, vmax = _oracle(ctx, cent, [U], q, [0, 11], 1 / np.sqrt(128))
    err = np.abs(got[[0, 11]] - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)
    assert np.isfinite(got).all()


def test_small_m_kernel_rejects_many_rows(qwm):
    wl, ctx, cent, bases = _ragged_context(qwm, "bf16-h12-n32760", 256, 16, sizes=(200,))
    ctx.set_attend_kernel(5)
    with pytest.raises(qwm.QwmError) as e:
        ctx.attend(_tensor(synth.queries(wl, 0, [0, 1], m=65)))
    assert e.value.status == 2
    assert ctx.attend_kernel_for(65) == 5          # the explicit choice stands
    ctx.set_attend_kernel(0)
    assert ctx.attend_kernel_for(65) == 6 and ctx.attend_kernel_for(64) == 7
    assert ctx.attend_kernel_for(17) == 7 and ctx.attend_kernel_for(16) == 5
