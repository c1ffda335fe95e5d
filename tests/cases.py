"""Shared set-up of parity cases: seeded inputs (synth), oracle-side
calibration and centroids, and the comparison helpers.

Only tests import this file.  Everything the oracle computes here comes from
the oracle; nothing is read back from the CUDA path except the outputs that
are compared.
"""
from __future__ import annotations

import functools

import numpy as np

from bit_kv_cache_qwm_gb300 import synth
from oracle import qwm_oracle as O


@functools.lru_cache(maxsize=8)
def centroids(name: str, heads: tuple | None = None, n_centroids: int | None = None, iters: int = 25):
    """Oracle k-means (Lloyd, float64) on the frame-0 keys, rounded to the
    workload dtype: float32 [heads, C, d]."""
    wl = synth.workload(name)
    hs = list(range(wl.heads)) if heads is None else list(heads)
    C = wl.n_centroids if n_centroids is None else n_centroids
    kf = synth.kmeans_keys(wl, hs)
    out = [O.kmeans(kf[i], synth.kmeans_init_rows(wl, h, kf.shape[1], C), iters)
           for i, h in enumerate(hs)]
    return synth.round_to_dtype(np.stack(out), wl.dtype)


@functools.lru_cache(maxsize=8)
def calibration(name: str, heads: tuple | None = None, rank: int | None = None, step: int = 0):
    """Oracle sensitivity (rounded to float32) and basis (rounded to float32)
    from the historical queries of `step`."""
    wl = synth.workload(name)
    hs = list(range(wl.heads)) if heads is None else list(heads)
    r = wl.rank if rank is None else rank
    qh = synth.hist_queries(wl, step, hs)
    s = np.stack([O.sensitivity(qh[i]) for i in range(len(hs))]).astype(np.float32)
    U = np.stack([O.psac_basis(qh[i], r)[0] for i in range(len(hs))]).astype(np.float32)
    return s, U


def f16_ulp(x) -> np.ndarray:
    """Spacing of float16 at |x| (2^-24 in the subnormal range)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -14)))
    return 2.0 ** (e - 10)


def split_tile(raw: np.ndarray, d: int, r: int, C: int) -> dict:
    """Sections of one tile's bytes."""
    L = O.tile_layout(d, r, C)
    names = ["idx", "kcode", "kqp", "e", "vcode", "vqp"]
    ends = [L[n] for n in names[1:]] + [L["tile_bytes"]]
    return {n: raw[L[n]:e] for n, e in zip(names, ends)}


def compare_segment_bytes(gpu_tiles: np.ndarray, seg: O.Segment, k32: np.ndarray, d: int, r: int,
                          C: int) -> dict:
    """Compare the GPU tiles of one append (one head) with the oracle's
    encoding: bit-exact sections except e, which must agree within one
    float16 ulp plus 1e-5 * ||k - k_hat||_2.  Returns counts; raises
    AssertionError with the first mismatch."""
    n = seg.idx.shape[0]
    ntile = (n + 127) // 128
    worst_e = 0.0
    for t in range(ntile):
        cnt = min(128, n - 128 * t)
        want = np.frombuffer(O.encode_tile(seg, 128 * t, cnt, d, r, C), np.uint8)
        got = gpu_tiles[t]
        gs, ws = split_tile(got, d, r, C), split_tile(want, d, r, C)
        for sec in ["idx", "kcode", "kqp", "vcode", "vqp"]:
            if not np.array_equal(gs[sec], ws[sec]):
                bad = np.flatnonzero(gs[sec] != ws[sec])
                raise AssertionError(f"tile {t} section {sec}: {bad.size} bytes differ, first at {bad[0]}")
        if r:
            eg = gs["e"].view(np.float16).reshape(128, r).astype(np.float64)
            ew = seg.e64[128 * t:128 * t + cnt]
            nrm = np.linalg.norm(k32[128 * t:128 * t + cnt].astype(np.float64) - seg.khat[128 * t:128 * t + cnt], axis=1)
            tol = np.maximum(f16_ulp(eg[:cnt]), f16_ulp(ew)) + 1e-5 * nrm[:, None]
            diff = np.abs(eg[:cnt] - ew.astype(np.float16).astype(np.float64))
            if not (diff <= tol).all():
                i = np.unravel_index(np.argmax(diff - tol), diff.shape)
                raise AssertionError(f"tile {t} e mismatch at {i}: gpu {eg[i]} oracle {ew[i]} tol {tol[i]}")
            worst_e = max(worst_e, float((diff / tol).max()))
            if cnt < 128:
                assert not eg[cnt:].any()
    return {"tiles": ntile, "worst_e_over_tol": worst_e}


def decode_gpu_segments(gpu_tiles_head: np.ndarray, table: np.ndarray, centroids32: np.ndarray,
                        d: int, r: int, C: int, n_tiles: int) -> list:
    """Oracle decoding of the GPU's cache bytes of one head (one Segment per tile)."""
    segs = []
    for t in range(n_tiles):
        ver, cnt = int(table[t, 0]), int(table[t, 1])
        segs.append(O.decode_tile(gpu_tiles_head[t].tobytes(), cnt, d, r, C, centroids32, ver))
    return segs
