"""The attention-shift diagnostics on the GPU: the nearest-centroid append mode
against the oracle's (bit-exact bytes), qwm_dequantize against the oracle's
decoding of the same bytes, and the diagnostics module against the oracle's
diagnostics computed from the GPU's cache bytes."""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import calibration, centroids, compare_segment_bytes, decode_gpu_segments
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


@pytest.mark.parametrize("name,heads,sizes", [("tiny-f32-h1-n1024", [0], [128, 300, 1]),
                                              ("bf16-h12-n32760", [0, 7], [300, 129])])
def test_nearest_assignment_bytes_match_oracle(qwm, name, heads, sizes):
    wl = synth.workload(name)
    H, d, r, C = len(heads), wl.head_dim, wl.rank, wl.n_centroids
    cent = centroids(name, tuple(heads))
    s, U = calibration(name, tuple(heads))
    ctx = qwm.Qwm(H, d, r, C, dtype=wl.dtype, max_tokens=sum((n + 127) // 128 for n in sizes) * 128)
    ctx.set_centroids(_tensor(cent, wl.dtype))
    ctx.set_calibration(s, U)
    ctx.set_assignment("nearest")
    ref = O.OracleCache(H, d, r, cent, assign="nearest")
    ref.set_calibration(s, U.astype(np.float64))
    ks = []
    for ch, n in enumerate(sizes):
        k, v = synth.keys(wl, ch, heads, n), synth.values(wl, ch, heads, n)
        ctx.append(_tensor(k, wl.dtype), _tensor(v, wl.dtype))
        ref.append(k, v)
        ks.append(k)
    tiles = ctx.cache_tiles().cpu().numpy()
    assert ctx.status() == 0
    t0 = 0
    for ch, n in enumerate(sizes):
        nt = (n + 127) // 128
        for h in range(H):
            compare_segment_bytes(tiles[h, t0:t0 + nt], ref.segments[h][ch], ks[ch][h], d, r, C)
        t0 += nt
    # QSAC and nearest choose differently on this data (else the mode is untested)
    qs = O.OracleCache(H, d, r, cent)
    qs.set_calibration(s, U.astype(np.float64))
    qs.append(ks[0], synth.values(wl, 0, heads, sizes[0]))
    assert any((qs.segments[h][0].idx != ref.segments[h][0].idx).any() for h in range(H))


def test_dequantize_matches_oracle_decoding(qwm):
    name = "bf16-h24-append-sweep"
    wl = synth.workload(name)
    heads, sizes = [0, 5], [300, 1, 100]
    cent = centroids(name, tuple(heads))
    s, U = calibration(name, tuple(heads))
    ctx = qwm.Qwm(2, 128, wl.rank, wl.n_centroids, dtype="bf16", max_tokens=5 * 128)
    ctx.set_centroids(_tensor(cent, "bf16"))
    ctx.set_calibration(s, U)
    for ch, n in enumerate(sizes):
        ctx.append(_tensor(synth.keys(wl, ch, heads, n), "bf16"), _tensor(synth.values(wl, ch, heads, n), "bf16"))
    kh, vh, e, valid = ctx.dequantize()
    kh, vh, e, valid = kh.cpu().numpy(), vh.cpu().numpy(), e.cpu().numpy(), valid.cpu().numpy()
    assert valid.sum() == sum(sizes) and valid.shape[0] == ctx.n_tiles * 128
    tiles, table = ctx.cache_tiles().cpu().numpy(), ctx.tile_table().cpu().numpy()
    for i in range(2):
        segs = decode_gpu_segments(tiles[i], table, cent[i], 128, wl.rank, wl.n_centroids, ctx.n_tiles)
        np.testing.assert_allclose(kh[i][valid], np.concatenate([g.khat for g in segs]), rtol=2e-7, atol=1e-30)
        np.testing.assert_allclose(vh[i][valid], np.concatenate([g.vhat for g in segs]), rtol=2e-7, atol=1e-30)
        assert np.array_equal(e[i][valid], np.concatenate([g.e16 for g in segs]).astype(np.float32))
        assert (kh[i][~valid] == 0).all() and (vh[i][~valid] == 0).all()


def test_diagnostics_run_reports_every_encoding(qwm):
    from bit_kv_cache_qwm_gb300 import diagnostics
    res = diagnostics.run("bf16-h12-n32760", [0, 3], rows=32, n_chunks=1)
    assert set(res["encodings"]) == {"nearest", "qsac", "qsac+psac"}
    for v in res["encodings"].values():
        for key, x in v.items():
            assert np.isfinite(x) and x >= 0, (key, x)


def test_diagnostics_agree_with_oracle(qwm):
    """diagnostics.measure on one cache (2 heads, 2 appends, QSAC + PSAC, 64
    query rows) against the oracle's diagnostics over the same cache bytes
    (float32 vs float64 argmax may differ on near-ties: one row per head at
    most)."""
    from bit_kv_cache_qwm_gb300 import diagnostics
    name = "bf16-h12-n32760"
    wl = synth.workload(name)
    heads, rows = [0, 3], 64
    dev = torch.device("cuda", 0)
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev, torch.bfloat16)
    ks = [synth.keys(wl, ch, heads) for ch in range(2)]
    vs = [synth.values(wl, ch, heads) for ch in range(2)]
    cent = centroids(name, tuple(heads))
    ctx = qwm.Qwm(2, 128, wl.rank, wl.n_centroids, dtype="bf16", max_tokens=2 * 37 * 128, max_hist=wl.n_hist)
    ctx.set_centroids(T(cent))
    s_, U = calibration(name, tuple(heads))      # the oracle's sensitivity and basis
    ctx.set_calibration(s_, U)
    for ch in range(2):
        ctx.append(T(ks[ch]), T(vs[ch]))
    K = torch.from_numpy(np.concatenate(ks, axis=1)).to(dev).float()
    V = torch.from_numpy(np.concatenate(vs, axis=1)).to(dev).float()
    qn = synth.queries(wl, 0, heads, m=rows)
    got = diagnostics.measure(ctx, K, V, torch.from_numpy(qn).to(dev).float(), 1 / np.sqrt(128))
    U = U.astype(np.float64)
    tiles, table = ctx.cache_tiles().cpu().numpy(), ctx.tile_table().cpu().numpy()
    q64, K64, V64 = qn.astype(np.float64), K.double().cpu().numpy(), V.double().cpu().numpy()
    changes, num, den = [], 0.0, 0.0
    # the module's reduction: Frobenius norms over all heads together
    sq = {k: [0.0, 0.0] for k in ("key", "value", "key_only", "value_only", "both")}
    sig = 1 / np.sqrt(128)
    for i in range(2):
        segs = decode_gpu_segments(tiles[i], table, cent[i], 128, wl.rank, wl.n_centroids, ctx.n_tiles)
        lq = O.compensated_logits(q64[i], segs, {0: U[i]})
        ex = q64[i] @ K64[i].T
        changes.append(np.argmax(ex, axis=1) != np.argmax(lq, axis=1))
        num += ((ex - lq) ** 2).sum()
        den += (ex ** 2).sum()
        khat = np.concatenate([g.khat for g in segs])
        vhat = np.concatenate([g.vhat for g in segs])
        o = O.softmax_rows(ex, sig) @ V64[i]
        pairs = {"key": (khat, K64[i]), "value": (vhat, V64[i]),
                 "key_only": (O.softmax_rows(lq, sig) @ V64[i], o),
                 "value_only": (O.softmax_rows(ex, sig) @ vhat, o),
                 "both": (O.softmax_rows(lq, sig) @ vhat, o)}
        for k, (a, b) in pairs.items():
            sq[k][0] += ((a - b) ** 2).sum()
            sq[k][1] += (b ** 2).sum()
    want = float(np.mean(np.concatenate(changes)))
    assert abs(got["top1_change"] - want) <= 2.0 / (2 * rows), (got["top1_change"], want)
    assert got["logit_rel_error"] == pytest.approx(np.sqrt(num / den), rel=1e-3)
    names = {"key": "key_rel_error", "value": "value_rel_error", "key_only": "output_rel_error_key_only",
             "value_only": "output_rel_error_value_only", "both": "output_rel_error"}
    for k, key in names.items():
        assert got[key] == pytest.approx(np.sqrt(sq[k][0] / sq[k][1]), rel=1e-3), key
