"""Online-softmax rescaling of every attention kernel, against the oracle.

Attention over the packed cache with PSAC compensation (QuantWM Abstract;
roboind article, "Step 2") is a softmax over every cached token; the kernels
take it tile by tile with a running maximum, and the tensor-core kernels move
their reference maximum (and rescale the partial output) only when a tile's
maximum exceeds it by more than 2^8 in the exp2 domain.  Here the logits of
some query rows jump by far more than that in later tiles (tile 2 by ~20, tile
5 by ~60 in log2 units), drop back in tile 7 and never rise for other rows
(whose later tiles then underflow), so every kernel takes the rescale path
once or twice per row and the underflow path too.  Each kernel's output is
compared with the oracle over the GPU's own cache bytes (1e-2 of max|v_hat|,
the tolerance of the other attention tests).
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import decode_gpu_segments
from oracle import qwm_oracle as O

pytestmark = pytest.mark.gpu

H, D, R, C = 2, 128, 16, 32
N = 8 * 128   # eight full tiles


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    return q


def _bf(x):
    return synth.round_to_bf16(np.asarray(x, np.float64))


def _tensor(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda", torch.bfloat16)


@pytest.fixture(scope="module")
def cache(qwm):
    rng = np.random.default_rng(2024)
    u = rng.standard_normal((H, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    k = 0.05 * rng.standard_normal((H, N, D))
    for tile, amp in ((2, 20.0), (5, 60.0), (7, 5.0)):
        k[:, 128 * tile:128 * (tile + 1)] += amp * u[:, None, :]
    k = _bf(k)
    v = _bf(rng.standard_normal((H, N, D)))
    # centroids: keys of every tile, so the big ones have a near centroid
    cent = _bf(k[:, ::32][:, :C])
    qh = rng.standard_normal((H, 512, D))
    s = np.stack([O.sensitivity(qh[h]) for h in range(H)]).astype(np.float32)
    U = np.stack([O.psac_basis(qh[h], R)[0] for h in range(H)]).astype(np.float32)
    ctx = qwm.Qwm(H, D, R, C, dtype="bf16", max_tokens=N)
    ctx.set_centroids(_tensor(cent))
    ctx.set_calibration(s, U)
    ctx.append(_tensor(k), _tensor(v))
    assert ctx.status() == 0
    tiles = ctx.cache_tiles().cpu().numpy()
    table = ctx.tile_table().cpu().numpy()
    dec = [decode_gpu_segments(tiles[h], table, cent[h], D, R, C, ctx.n_tiles) for h in range(H)]
    # queries: half along +u (their logits jump in tiles 2 and 5), half along
    # -u (their first tiles hold the maximum; tiles 2 and 5 underflow)
    q = np.empty((H, 150, D))
    for h in range(H):
        sign = np.where(np.arange(150) % 2 == 0, 1.0, -1.0)[:, None]
        q[h] = sign * 8.0 * u[h][None, :] + 0.05 * rng.standard_normal((150, D))
    q = _bf(q)
    return ctx, dec, U, q


def _check(ctx, dec, U, q, m):
    got = ctx.attend(_tensor(q[:, :m])).float().cpu().numpy()
    assert ctx.status() == 0 and np.isfinite(got).all()
    for h in range(H):
        want = O.attend_head(q[h, :m], dec[h], {0: U[h].astype(np.float64)}, 1 / np.sqrt(D))
        vmax = max(np.abs(sg.vhat).max() for sg in dec[h])
        err = np.abs(got[h] - want).max()
        assert err <= 1e-2 * vmax, (err, vmax)


def test_logit_jumps_rescale_the_partial_output(cache):
    ctx, dec, U, q = cache
    # the jump really is far beyond the lazy threshold in the exp2 domain
    l2 = (q[0, 0] @ dec[0][5].khat[0]) / np.sqrt(D) * np.log2(np.e)   # a key of tile 5
    assert l2 > 40.0
    for kernel in (1, 2, 3, 4, 6):
        ctx.set_attend_kernel(kernel)
        _check(ctx, dec, U, q, 150)
    ctx.set_attend_kernel(0)


@pytest.mark.parametrize("kernel", [5, 7])
def test_logit_jumps_few_rows(cache, kernel):
    ctx, dec, U, q = cache
    ctx.set_attend_kernel(kernel)
    for m in (1, 16, 48):
        _check(ctx, dec, U, q, m)
    ctx.set_attend_kernel(0)
