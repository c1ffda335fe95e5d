"""qwm_attend on the GPU against the oracle.

Tolerances (stated by the workload definitions): max |O_gpu - O_oracle| <=
1e-5 * max|V_hat| for float32 workloads and <= 1e-2 * max|V_hat| for bfloat16
ones.  The oracle attends over the GPU's own cache bytes (decoded from the
documented layout), so attention is checked apart from append; a second check
runs it over the oracle's own encoding.
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


def _tensor(x, dtype):
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to("cuda", torch.bfloat16 if dtype == "bf16" else torch.float32)


def _build(qwm, name, heads, chunk_sizes, versions=1, rank=None, max_tokens=None):
    """Context with the given appends; a new basis version every
    len(chunk_sizes)/versions appends."""
    wl = synth.workload(name)
    H = len(heads)
    r = wl.rank if rank is None else rank
    cent = centroids(name, tuple(heads))
    tiles = sum((n + 127) // 128 for n in chunk_sizes)
    ctx = qwm.Qwm(H, wl.head_dim, r, wl.n_centroids, dtype=wl.dtype,
                  max_tokens=max_tokens or tiles * 128, max_versions=max(versions, 1))
    ctx.set_centroids(_tensor(cent, wl.dtype))
    bases = []
    per = max(1, len(chunk_sizes) // versions)
    for ch, n in enumerate(chunk_sizes):
        if ch % per == 0 and len(bases) < versions:
            s, U = calibration(name, tuple(heads), r, step=len(bases))
            ctx.set_calibration(s, U)
            bases.append(U)
        ctx.append(_tensor(synth.keys(wl, ch, heads, n), wl.dtype),
                   _tensor(synth.values(wl, ch, heads, n), wl.dtype))
    return wl, ctx, cent, bases


def _oracle_on_gpu_bytes(ctx, cent, bases, q, heads_idx, scale):
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


@pytest.mark.parametrize("kernel", [1])
def test_attend_tiny_f32(qwm, kernel):
    wl, ctx, cent, bases = _build(qwm, "tiny-f32-h1-n1024", [0], [128] * 8)
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 0)
    got = ctx.attend(_tensor(q, "f32")).cpu().numpy()
    scale = 1 / np.sqrt(wl.head_dim)
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0], scale)
    assert np.abs(got - want).max() <= 1e-5 * vmax
    # the oracle's own encoding gives the same attention
    ref = O.OracleCache(1, wl.head_dim, wl.rank, cent)
    s, U = calibration(wl.name)
    ref.set_calibration(s, U.astype(np.float64))
    for ch in range(8):
        ref.append(synth.keys(wl, ch), synth.values(wl, ch))
    assert np.abs(got - ref.attend(q, scale)).max() <= 1e-5 * vmax


@pytest.mark.parametrize("kernel", [1])
def test_attend_ragged_versions_and_scale(qwm, kernel):
    """Ragged appends (tail tiles of 1 and 100 slots), three basis versions,
    an explicit softmax scale, M not a multiple of any tile size."""
    wl, ctx, cent, bases = _build(qwm, "tiny-f32-h1-n1024", [0], [300, 1, 228, 129, 100, 64], versions=3)
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 1, m=37)
    got = ctx.attend(_tensor(q, "f32"), scale=0.05).cpu().numpy()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0], 0.05)
    assert np.abs(got - want).max() <= 1e-5 * vmax


@pytest.mark.parametrize("kernel", [1])
def test_full_rank_compensation_on_gpu(qwm, kernel):
    """r = d: the compensated logits reproduce the exact keys up to the fp16
    storage of e, so attention is close to attention over the unquantised
    keys (and equal to the oracle's)."""
    name = "tiny-f32-h1-n1024"
    wl = synth.workload(name)
    cent = centroids(name)
    ctx = qwm.Qwm(1, 64, 64, 16, dtype="f32", max_tokens=512)
    ctx.set_centroids(_tensor(cent, "f32"))
    s, U = calibration(name, rank=64)
    ctx.set_calibration(s, U)
    for ch in range(4):
        ctx.append(_tensor(synth.keys(wl, ch), "f32"), _tensor(synth.values(wl, ch), "f32"))
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 0)
    got = ctx.attend(_tensor(q, "f32")).cpu().numpy()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, [U], q, [0], 1 / 8)
    assert np.abs(got - want).max() <= 1e-5 * vmax


@pytest.mark.parametrize("kernel", [1, 2, 3, 4, 6])
def test_attend_bf16_sampled_rows(qwm, kernel):
    """12 heads over 3 appends; the oracle checks every row of heads 0 and 9."""
    name = "bf16-h12-n32760"
    wl, ctx, cent, bases = _build(qwm, name, list(range(12)), [4680, 4680, 1000])
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 0, m=200)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0, 9], 1 / np.sqrt(128))
    assert np.abs(got[[0, 9]] - want).max() <= 1e-2 * vmax


@pytest.mark.parametrize("kernel", [1, 2, 3, 4, 6])
@pytest.mark.parametrize("name,C,r", [("bf16-h12-n32760", 256, 16), ("bf16-h24-append-sweep", 1024, 32),
                                      ("bf16-h24-append-sweep", 64, 8), ("bf16-h24-append-sweep", 256, 0),
                                      ("bf16-h40-n98280-outlier", 256, 16)])
def test_attend_bf16_variants(qwm, kernel, name, C, r):
    """Ragged appends (tails of 1 and 100 slots), three basis versions, rank
    0 / 8 / 16 / 32, centroids staged in shared memory (C <= 256) or read
    from global memory (C = 1024), outlier channels, M = 200 (two row blocks,
    ragged)."""
    wl = synth.workload(name)
    heads = [0, 1]
    cent = centroids(name, tuple(heads), C, iters=25 if C <= 256 else 3)
    sizes = [300, 1, 228, 129, 100, 64]
    ctx = qwm.Qwm(2, 128, r, C, dtype="bf16", max_tokens=sum((n + 127) // 128 for n in sizes) * 128,
                  max_versions=3)
    ctx.set_centroids(_tensor(cent, "bf16"))
    bases = []
    for ch, n in enumerate(sizes):
        if ch % 2 == 0:
            s_, U = calibration(name, tuple(heads), r, step=len(bases))
            ctx.set_calibration(s_, U)
            bases.append(U)
        ctx.append(_tensor(synth.keys(wl, ch, heads, n), "bf16"), _tensor(synth.values(wl, ch, heads, n), "bf16"))
    if kernel in (4, 6) and r > 16:
        ctx.set_attend_kernel(kernel)
        with pytest.raises(qwm.QwmError) as e:
            ctx.attend(_tensor(synth.queries(wl, 3, heads, m=8), "bf16"))
        assert e.value.status == 2                 # unsupported: r > 16
        return
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 3, heads, m=200)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0, 1], 1 / np.sqrt(128))
    err = np.abs(got - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)


def test_attend_full_size_bench_configuration(qwm):
    """The benchmarked workload at full size in the launch configuration the
    benchmark times (automatic kernel choice): 12 heads, 7 appends of 4,680
    tokens (32,760 cached), 4,680 query rows.  The oracle recomputes 48 seeded
    rows of heads 0 and 11 over the GPU's cache bytes."""
    name = "bf16-h12-n32760"
    wl, ctx, cent, bases = _build(qwm, name, list(range(12)), [wl_chunk for wl_chunk in [4680] * 7])
    q = synth.queries(wl, 0)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    assert ctx.resolved_attend_kernel == 6
    rows = np.sort(np.random.default_rng(5).choice(wl.n_query, 48, replace=False))
    qs = q[:, rows]
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, qs, [0, 11], 1 / np.sqrt(128))
    err = np.abs(got[[0, 11]][:, rows] - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)
    assert np.isfinite(got).all()


@pytest.mark.parametrize("kernel", [4, 6])
@pytest.mark.parametrize("sizes", [[100], [128, 5], [300, 1, 228], [64, 65, 1]])
def test_attend_two_tile_kernel_split_boundaries(qwm, sizes, kernel):
    """Kernels 4 and 6 (256 query rows per CTA) on a cache of one tile (no
    KV split), two tiles (one tile per split), five tiles (an odd count split
    2 + 3) and tiles whose second 64-key half is empty or holds one key, with
    M = 300 (two row blocks, the second ragged)."""
    name = "bf16-h12-n32760"
    wl, ctx, cent, bases = _build(qwm, name, [0, 1], sizes)
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 1, [0, 1], m=300)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    assert ctx.status() == 0
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0, 1], 1 / np.sqrt(128))
    err = np.abs(got - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)


def test_attend_f16_split_kernel_large_queries(qwm):
    """Kernel 6 scales each query row by a power of two into the float16
    range: rows with entries up to ~2^20 (beyond float16) give the same
    attention as the oracle (which sees the unscaled bf16 queries)."""
    name = "bf16-h12-n32760"
    wl, ctx, cent, bases = _build(qwm, name, [0, 1], [4680, 700])
    ctx.set_attend_kernel(6)
    q = synth.queries(wl, 2, [0, 1], m=260)
    boost = np.ones((1, 260, 1), np.float32)
    boost[:, ::3] = 2.0 ** 14                       # every third row far beyond float16
    q = synth.round_to_bf16(q * boost)
    scale = 1.0 / (np.sqrt(128) * 2.0 ** 13)        # keeps the logits of the boosted rows moderate
    got = ctx.attend(_tensor(q, "bf16"), scale=scale).float().cpu().numpy()
    assert ctx.status() == 0 and np.isfinite(got).all()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0, 1], scale)
    err = np.abs(got - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)


def test_attend_centroids_beyond_f16_fall_back(qwm):
    """Centroids outside the float16 range make kernel 6 unavailable: the
    automatic choice falls back to kernel 4 (an explicit kernel 6 is refused)
    and the attention still matches the oracle."""
    name = "bf16-h12-n32760"
    wl = synth.workload(name)
    heads = [0, 1]
    cent = centroids(name, tuple(heads)).copy()
    cent[1, 7, 3] = 2.0 ** 17                        # exactly representable in bf16, not in float16
    ctx = qwm.Qwm(2, 128, wl.rank, wl.n_centroids, dtype="bf16", max_tokens=2 * 128)
    ctx.set_centroids(_tensor(cent, "bf16"))
    assert ctx.resolved_attend_kernel == 4
    s_, U = calibration(name, tuple(heads))
    ctx.set_calibration(s_, U)
    ctx.append(_tensor(synth.keys(wl, 0, heads, 200), "bf16"), _tensor(synth.values(wl, 0, heads, 200), "bf16"))
    q = synth.queries(wl, 0, heads, m=100)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, [U], q, [0, 1], 1 / np.sqrt(128))
    assert np.abs(got - want).max() <= 1e-2 * vmax
    ctx.set_attend_kernel(6)
    with pytest.raises(qwm.QwmError) as e:
        ctx.attend(_tensor(q, "bf16"))
    assert e.value.status == 2


@pytest.mark.parametrize("kernel,m", [(1, 200), (2, 200), (3, 200), (4, 200), (6, 200), (6, 300), (5, 40), (7, 40)])
def test_attend_basis_change_every_tile(qwm, kernel, m):
    """A new basis version before every append of one tile or less (eight
    versions, tails of 100, 1 and 128 slots): the PSAC term of every tile uses
    another basis, so the tensor-core kernels switch their Z = q U_t^T buffer
    on every tile."""
    name = "bf16-h12-n32760"
    sizes = [100, 128, 1, 77, 128, 64, 120, 128]
    wl, ctx, cent, bases = _build(qwm, name, [0, 1], sizes, versions=len(sizes))
    assert len(bases) == len(sizes)
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 2, [0, 1], m=m)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    assert ctx.status() == 0 and np.isfinite(got).all()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0, 1], 1 / np.sqrt(128))
    err = np.abs(got - want).max()
    assert err <= 1e-2 * vmax, (err, vmax)
