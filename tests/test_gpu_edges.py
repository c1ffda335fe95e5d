"""The method's exact-tie and degenerate cases on the bf16 path, bit-exact
against the oracle (QuantWM Abstract; roboind article, "Step 1"):

* duplicate centroids: keys equal to (or next to) a centroid that appears
  three times; every copy has the same score, so the lowest index must win;
* constant groups: keys equal to a centroid (a residual of zero in every
  group) and values with whole 32-channel groups at one value give scale 0,
  so every code is 0 and the group decodes to its zero exactly;
* float16-subnormal parameters: residual and value groups whose ranges are
  far below 2^-14, so zero and scale land in the float16 subnormal range.

Each case also runs attention over the resulting cache (kernel 6 and the
float32 kernel are not involved in the encoding; the large-M default reads
these bytes) and checks it against the oracle over the same bytes.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import compare_segment_bytes, decode_gpu_segments
from oracle import qwm_oracle as O

pytestmark = pytest.mark.gpu

H, D, R, C = 2, 128, 16, 32


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


def _calibration(rng):
    qh = rng.standard_normal((H, 512, D)) * np.exp(rng.standard_normal((H, 1, D)))
    s = np.stack([O.sensitivity(qh[h]) for h in range(H)]).astype(np.float32)
    U = np.stack([O.psac_basis(qh[h], R)[0] for h in range(H)]).astype(np.float32)
    return s, U


def _check(qwm, cent, k, v, s, U):
    """Append k, v (float32 holding bf16 values) on the GPU, compare every
    byte with the oracle's encoding, then attend 150 rows over the cache."""
    n = k.shape[1]
    ctx = qwm.Qwm(H, D, R, C, dtype="bf16", max_tokens=((n + 127) // 128) * 128)
    ctx.set_centroids(_tensor(cent))
    ctx.set_calibration(s, U)
    ctx.append(_tensor(k), _tensor(v))
    assert ctx.status() == 0
    tiles = ctx.cache_tiles().cpu().numpy()
    segs = []
    for h in range(H):
        seg = O.append_head(k[h], v[h], cent[h], O.group_weights(s[h]), U[h].astype(np.float64))
        compare_segment_bytes(tiles[h, :(n + 127) // 128], seg, k[h], D, R, C)
        segs.append(seg)
    q = _bf(np.random.default_rng(9).standard_normal((H, 150, D)))
    got = ctx.attend(_tensor(q)).float().cpu().numpy()
    assert ctx.status() == 0 and np.isfinite(got).all()
    table = ctx.tile_table().cpu().numpy()
    for h in range(H):
        dec = decode_gpu_segments(tiles[h], table, cent[h], D, R, C, ctx.n_tiles)
        want = O.attend_head(q[h], dec, {0: U[h].astype(np.float64)}, 1 / np.sqrt(D))
        vmax = max(np.abs(sg.vhat).max() for sg in dec)
        assert np.abs(got[h] - want).max() <= 1e-2 * max(vmax, 1e-30)
    return segs


def test_duplicate_centroids_lowest_index_wins(qwm):
    rng = np.random.default_rng(1)
    cent = _bf(rng.standard_normal((H, C, D)) * 2.0)
    cent[:, 20] = cent[:, 5]
    cent[:, 31] = cent[:, 5]
    n = 300
    pick = rng.choice([5, 20, 31, 8], n)
    k = cent[:, pick].astype(np.float64)
    k[:, ::2] += 0.05 * rng.standard_normal((H, (n + 1) // 2, D))        # every other key exactly on a centroid
    k = _bf(k)
    v = _bf(rng.standard_normal((H, n, D)))
    s, U = _calibration(rng)
    segs = _check(qwm, cent, k, v, s, U)
    for seg in segs:
        assert not np.isin(seg.idx, [20, 31]).any()                    # the copies never win
        assert (seg.idx == 5).sum() > 0


def test_constant_groups_scale_zero(qwm):
    rng = np.random.default_rng(2)
    cent = _bf(rng.standard_normal((H, C, D)))
    n = 260
    k = cent[:, rng.integers(0, C, n)].copy()                          # residual 0 in every group
    v = _bf(rng.standard_normal((H, n, D)))
    v[:, :, 32:64] = 1.5                                               # a constant value group
    v[:, 100:, :32] = -0.75
    s, U = _calibration(rng)
    segs = _check(qwm, cent, k, v, s, U)
    for seg in segs:
        assert (seg.kscale == 0).all() and (seg.kcodes == 0).all()
        assert (seg.vscale[:, 1] == 0).all() and (seg.vzero[:, 1] == np.float16(1.5)).all()
        assert (seg.vhat[:, 32:64] == 1.5).all()


def test_float16_subnormal_parameters(qwm):
    rng = np.random.default_rng(3)
    cent = _bf(rng.standard_normal((H, C, D)))
    cent[:, :, 64:96] = 0.0                                            # group 2 of every centroid at zero
    n = 200
    k = cent[:, rng.integers(0, C, n)].copy()
    k[:, :, 64:96] = _bf(2e-6 * rng.standard_normal((H, n, 32)))       # residual range far below 2^-14
    v = _bf(rng.standard_normal((H, n, D)))
    v[:, :, :32] = _bf(3e-7 * rng.standard_normal((H, n, 32)))
    s, U = _calibration(rng)
    segs = _check(qwm, cent, k, v, s, U)
    tiny = 2.0 ** -14
    for seg in segs:
        ks = seg.kscale[:, 2].astype(np.float64)
        assert ((ks > 0) & (ks < tiny)).any() and (ks < tiny).all()
        vs = seg.vscale[:, 0].astype(np.float64)
        assert (vs < tiny).all() and (np.abs(seg.vzero[:, 0].astype(np.float64)) < tiny).all()
