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


@pytest.mark.parametrize("kernel", [1])
def test_attend_bf16_sampled_rows(qwm, kernel):
    """12 heads over 3 appends; the oracle checks every row of heads 0 and 9."""
    name = "bf16-h12-n32760"
    wl, ctx, cent, bases = _build(qwm, name, list(range(12)), [4680, 4680, 1000])
    ctx.set_attend_kernel(kernel)
    q = synth.queries(wl, 0, m=200)
    got = ctx.attend(_tensor(q, "bf16")).float().cpu().numpy()
    want, vmax = _oracle_on_gpu_bytes(ctx, cent, bases, q, [0, 9], 1 / np.sqrt(128))
    assert np.abs(got[[0, 9]] - want).max() <= 1e-2 * vmax
