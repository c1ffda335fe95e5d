"""qwm_append on the GPU against the oracle: bit-exact indices, codes and
float16 parameters; PSAC coefficients within one float16 ulp."""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import calibration, centroids, compare_segment_bytes
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


def _run_append(qwm, name, heads, chunk_sizes, n_centroids=None, rank=None, check_heads=None):
    wl = synth.workload(name)
    H = len(heads)
    C = wl.n_centroids if n_centroids is None else n_centroids
    r = wl.rank if rank is None else rank
    cent = centroids(name, tuple(heads), C, iters=25 if C <= 256 else 5)
    s, U = calibration(name, tuple(heads), r)
    total_tiles = sum((n + 127) // 128 for n in chunk_sizes)
    ctx = qwm.Qwm(H, wl.head_dim, r, C, dtype=wl.dtype, max_tokens=total_tiles * 128)
    ctx.set_centroids(_tensor(cent, wl.dtype))
    ctx.set_calibration(s, U)
    ref = O.OracleCache(H, wl.head_dim, r, cent)
    ref.set_calibration(s, U.astype(np.float64))
    ks = []
    for ch, n in enumerate(chunk_sizes):
        k = synth.keys(wl, ch, heads, n)
        v = synth.values(wl, ch, heads, n)
        ctx.append(_tensor(k, wl.dtype), _tensor(v, wl.dtype))
        ks.append(k)
    hs_check = range(H) if check_heads is None else check_heads
    for ch, n in enumerate(chunk_sizes):
        ref.append(ks[ch][list(hs_check)], synth.values(wl, ch, [heads[i] for i in hs_check], n),
                   heads=list(hs_check))
    torch.cuda.synchronize()
    tiles = ctx.cache_tiles().cpu().numpy()
    table = ctx.tile_table().cpu().numpy()
    assert ctx.status() == 0
    t0 = 0
    worst = 0.0
    for ch, n in enumerate(chunk_sizes):
        nt = (n + 127) // 128
        for h in hs_check:
            res = compare_segment_bytes(tiles[h, t0:t0 + nt], ref.segments[h][ch], ks[ch][h],
                                        wl.head_dim, r, C)
            worst = max(worst, res["worst_e_over_tol"])
        assert (table[t0:t0 + nt, 0] == 0).all()
        assert table[t0:t0 + nt, 1].sum() == n
        t0 += nt
    assert ctx.n_tokens == sum(chunk_sizes) and ctx.n_tiles == total_tiles
    return worst


def test_append_tiny_f32(qwm):
    # 8 appends of 128 plus ragged chunks: tail tiles of 1, 127 and 77 slots
    _run_append(qwm, "tiny-f32-h1-n1024", [0], [128] * 8 + [1, 127, 333])


def test_append_bf16_small_chunks(qwm):
    _run_append(qwm, "bf16-h12-n32760", [0, 5, 11], [300, 129, 1000])


@pytest.mark.parametrize("C,r", [(64, 8), (1024, 32), (256, 0), (7, 3)])
def test_append_sweep_shapes(qwm, C, r):
    _run_append(qwm, "bf16-h24-append-sweep", [0, 23], [260, 515], n_centroids=C, rank=r)


def test_append_full_size_sampled_heads(qwm):
    """The 12-head workload at full size (7 appends of 4,680 tokens, 259
    tiles); the oracle checks heads 0 and 7 completely."""
    wl = synth.workload("bf16-h12-n32760")
    _run_append(qwm, wl.name, list(range(wl.heads)), [wl.chunk] * wl.n_chunks, check_heads=[0, 7])


def test_saturated_parameters_set_status(qwm):
    """Residual ranges beyond 3 * 65504 saturate the float16 scale; the kernel
    flags it and the oracle agrees on the saturated bytes."""
    H, d, r, C = 1, 64, 0, 4
    rng = np.random.default_rng(0)
    cent = np.zeros((H, C, d), np.float32)
    k = (rng.standard_normal((H, 128, d)) * 1e5).astype(np.float32)
    v = rng.standard_normal((H, 128, d)).astype(np.float32)
    ctx = qwm.Qwm(H, d, r, C, dtype="f32", max_tokens=128)
    ctx.set_centroids(_tensor(cent, "f32"))
    s = np.ones((H, d), np.float32)
    ctx.set_calibration(s, np.zeros((H, 0, d), np.float32))
    ctx.append(_tensor(k, "f32"), _tensor(v, "f32"))
    bits = ctx.status_bits()
    assert bits & qwm.DEV_SATURATED
    seg = O.append_head(k[0], v[0], cent[0], O.group_weights(s[0]), np.zeros((0, d)))
    assert seg.saturated > 0
    tiles = ctx.cache_tiles().cpu().numpy()
    compare_segment_bytes(tiles[0, :1], seg, k[0], d, r, C)


def test_host_side_errors(qwm):
    wl = synth.workload("tiny-f32-h1-n1024")
    ctx = qwm.Qwm(1, 64, 4, 16, dtype="f32", max_tokens=256, max_versions=2)
    k = _tensor(synth.keys(wl, 0), "f32")
    with pytest.raises(qwm.QwmError) as e:
        ctx.append(k, k)
    assert e.value.status == 4                     # not calibrated
    ctx.set_centroids(_tensor(centroids(wl.name), "f32"))
    s, U = calibration(wl.name)
    ctx.set_calibration(s, U)                      # version 0 in slot 0
    ctx.set_calibration(s, U)                      # version 1 reuses slot 0 (no segment uses it)
    ctx.append(k, k)
    ctx.set_calibration(s, U)                      # version 2 in slot 1
    ctx.append(k, k)
    with pytest.raises(qwm.QwmError) as e:
        ctx.append(k, k)                           # a third tile does not fit in 256 slots
    assert e.value.status == 3
    assert ctx.n_tokens == 256 and ctx.n_segments == 2
    with pytest.raises(qwm.QwmError) as e:
        ctx.set_calibration(s, U)                  # both slots hold live segments
    assert e.value.status == 3
    assert ctx.version == 2
    table = ctx.tile_table().cpu().numpy()
    assert table[:2, 0].tolist() == [0, 1]
    ctx.rewind(1)                                  # drops the version-2 segment
    ctx.set_calibration(s, U)                      # version 3 takes slot 1
    assert ctx.version == 3 and ctx.n_tokens == 128
    ctx.rewind(0)
    with pytest.raises(qwm.QwmError) as e:
        ctx.attend(_tensor(synth.queries(wl, 0), "f32"))
    assert e.value.status == 1                     # empty cache
