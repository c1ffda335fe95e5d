"""Seeded synthetic inputs for the QuantWM 2-bit KV-cache hot path.

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the method's arithmetic (no assignment, quantisation,
compensation or attention) and imports neither the CUDA library nor the
oracle, so both sides of every parity test can read the same inputs from it.

Shapes follow the video world-model workloads described on the QuantWM pages
(roboind article, introduction and "Five types of model validation"): one
latent frame is 1,560 tokens, a causal chunk is 3 frames (4,680 tokens),
480p video of 93 frames.

Distributions (identical for every workload):
  channel scale  sigma_c = exp(N(0, 1)) per head; optional outlier channels
                 whose sigma is multiplied by a fixed factor;
  keys           K = (C_true[z] + 0.3 * eps) * sigma, C_true ~ N(0,1)^{16 x d},
                 z ~ U{0..15}, eps ~ N(0, 1);
  values         V ~ N(0, 1);
  queries        Q, Q_hist ~ N(0, 1) * sigma.
Values are drawn in float64 and rounded once to the workload dtype (float32,
or bfloat16 by round-to-nearest-even of the float32 bits); arrays come back as
float32 holding exactly representable values.

Every array is drawn from its own PCG64 stream keyed by
(workload seed, kind, head, index), so any head or chunk can be regenerated
alone, in any order, on any machine.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Sequence

import numpy as np

FRAME_TOKENS = 1560          # tokens per latent frame (480p)
CHUNK_FRAMES = 3             # frames per causal chunk
CHUNK_TOKENS = FRAME_TOKENS * CHUNK_FRAMES
N_TRUE_CENTRES = 16          # clusters the synthetic keys are drawn around
KEY_NOISE = 0.3              # standard deviation of eps around a true centre

# stream kinds
_SIGMA, _CTRUE, _KEYS, _VALS, _QUERY, _QHIST, _OUTL, _KMINIT, _ZSEL = range(9)


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: sizes of the cache, the chunks and the queries."""
    name: str
    seed: int
    heads: int
    head_dim: int
    dtype: str                    # "f32" or "bf16"
    n_centroids: int
    rank: int
    n_hist: int                   # historical queries per calibration
    n_query: int                  # query rows per attend call
    chunk: int                    # tokens per append call
    n_chunks: int                 # append calls that build the full cache
    kmeans_tokens: int            # keys of chunk 0 the centroids are fitted on
    outlier_channels: int = 0
    outlier_factor: float = 1.0
    steps: int = 0                # streaming workloads: calibrate/append/attend steps
    sweep: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return 32

    @property
    def n_tokens(self) -> int:
        return self.chunk * self.n_chunks


WORKLOADS = {
    # tiny float32 case the oracle finishes in seconds
    "tiny-f32-h1-n1024": Workload(
        name="tiny-f32-h1-n1024", seed=1001, heads=1, head_dim=64, dtype="f32",
        n_centroids=16, rank=4, n_hist=256, n_query=64, chunk=128, n_chunks=8,
        kmeans_tokens=1024),
    # 12 heads, 21-frame history (32,760 tokens), 3-frame query chunk
    "bf16-h12-n32760": Workload(
        name="bf16-h12-n32760", seed=1002, heads=12, head_dim=128, dtype="bf16",
        n_centroids=256, rank=16, n_hist=1024, n_query=CHUNK_TOKENS,
        chunk=CHUNK_TOKENS, n_chunks=7, kmeans_tokens=FRAME_TOKENS),
    # 40 heads, 60-frame history + one appended chunk, 4 outlier channels x10
    "bf16-h40-n98280-outlier": Workload(
        name="bf16-h40-n98280-outlier", seed=1003, heads=40, head_dim=128, dtype="bf16",
        n_centroids=256, rank=16, n_hist=1024, n_query=CHUNK_TOKENS,
        chunk=CHUNK_TOKENS, n_chunks=21, kmeans_tokens=FRAME_TOKENS,
        outlier_channels=4, outlier_factor=10.0),
    # append-only sweep: chunk length x centroids x rank
    "bf16-h24-append-sweep": Workload(
        name="bf16-h24-append-sweep", seed=1004, heads=24, head_dim=128, dtype="bf16",
        n_centroids=256, rank=16, n_hist=1024, n_query=0,
        chunk=CHUNK_TOKENS, n_chunks=1, kmeans_tokens=FRAME_TOKENS,
        sweep={"chunk": [1560, 3120, 4680, 6240, 7800],
               "n_centroids": [64, 256, 1024], "rank": [8, 16, 32]}),
    # 80 streaming steps to 240 frames (374,400 tokens), 4,096-query ring
    "bf16-h24-stream-n374400": Workload(
        name="bf16-h24-stream-n374400", seed=1005, heads=24, head_dim=128, dtype="bf16",
        n_centroids=256, rank=16, n_hist=4096, n_query=CHUNK_TOKENS,
        chunk=CHUNK_TOKENS, n_chunks=80, kmeans_tokens=FRAME_TOKENS, steps=80),
}


def _rng(wl: Workload, kind: int, head: int, index: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=wl.seed, spawn_key=(kind, head, index))
    return np.random.Generator(np.random.PCG64(ss))


def round_to_bf16(x) -> np.ndarray:
    """Round float64/float32 values to bfloat16 (via float32, nearest-even on the
    dropped 16 bits); returned as float32 holding bf16-representable values."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def round_to_dtype(x, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_to_bf16(x)
    raise ValueError(f"unknown dtype {dtype!r}")


def channel_scale(wl: Workload, head: int) -> np.ndarray:
    """sigma_c for one head, float64 [d]."""
    sig = np.exp(_rng(wl, _SIGMA, head).standard_normal(wl.head_dim))
    if wl.outlier_channels:
        ch = _rng(wl, _OUTL, head).choice(wl.head_dim, wl.outlier_channels, replace=False)
        sig[ch] *= wl.outlier_factor
    return sig


def outlier_channels(wl: Workload, head: int) -> np.ndarray:
    if not wl.outlier_channels:
        return np.zeros(0, dtype=np.int64)
    return np.sort(_rng(wl, _OUTL, head).choice(wl.head_dim, wl.outlier_channels, replace=False))


def true_centres(wl: Workload, head: int) -> np.ndarray:
    return _rng(wl, _CTRUE, head).standard_normal((N_TRUE_CENTRES, wl.head_dim))


def _stack(fn, heads: Sequence[int] | None, wl: Workload, *args) -> np.ndarray:
    hs = range(wl.heads) if heads is None else heads
    return np.stack([fn(wl, h, *args) for h in hs])


def _keys1(wl: Workload, head: int, chunk: int, n: int) -> np.ndarray:
    sig = channel_scale(wl, head)
    ct = true_centres(wl, head)
    rz = _rng(wl, _ZSEL, head, chunk)
    z = rz.integers(0, N_TRUE_CENTRES, size=n)
    eps = _rng(wl, _KEYS, head, chunk).standard_normal((n, wl.head_dim))
    return round_to_dtype((ct[z] + KEY_NOISE * eps) * sig, wl.dtype)


def keys(wl: Workload, chunk: int, heads: Sequence[int] | None = None, n: int | None = None) -> np.ndarray:
    """Keys of append call `chunk`: float32 [heads, n, d]."""
    return _stack(_keys1, heads, wl, chunk, wl.chunk if n is None else n)


def _vals1(wl: Workload, head: int, chunk: int, n: int) -> np.ndarray:
    return round_to_dtype(_rng(wl, _VALS, head, chunk).standard_normal((n, wl.head_dim)), wl.dtype)


def values(wl: Workload, chunk: int, heads: Sequence[int] | None = None, n: int | None = None) -> np.ndarray:
    """Values of append call `chunk`: float32 [heads, n, d]."""
    return _stack(_vals1, heads, wl, chunk, wl.chunk if n is None else n)


def _query1(wl: Workload, head: int, step: int, m: int) -> np.ndarray:
    sig = channel_scale(wl, head)
    return round_to_dtype(_rng(wl, _QUERY, head, step).standard_normal((m, wl.head_dim)) * sig, wl.dtype)


def queries(wl: Workload, step: int = 0, heads: Sequence[int] | None = None, m: int | None = None) -> np.ndarray:
    """Query chunk of attend call `step`: float32 [heads, M, d]."""
    return _stack(_query1, heads, wl, step, wl.n_query if m is None else m)


def _qhist1(wl: Workload, head: int, step: int, n: int) -> np.ndarray:
    sig = channel_scale(wl, head)
    return round_to_dtype(_rng(wl, _QHIST, head, step).standard_normal((n, wl.head_dim)) * sig, wl.dtype)


def hist_queries(wl: Workload, step: int = 0, heads: Sequence[int] | None = None) -> np.ndarray:
    """Historical queries used to calibrate before step `step`: float32 [heads, n_h, d].

    Streaming workloads keep a ring of the most recent n_h queries of earlier
    chunks; before the first step the ring is a seeded draw of its own.  Other
    workloads draw a fresh seeded set for every `step`.
    """
    if wl.steps and step > 0:
        q = queries(wl, step - 1, heads)
        return np.ascontiguousarray(q[:, -wl.n_hist:, :])
    return _stack(_qhist1, heads, wl, step, wl.n_hist)


def kmeans_init_rows(wl: Workload, head: int, n_frame: int, n_centroids: int) -> np.ndarray:
    """Seeded choice of distinct rows of frame 0 that start Lloyd's iteration."""
    return _rng(wl, _KMINIT, head).permutation(n_frame)[:n_centroids].astype(np.int64)


def kmeans_keys(wl: Workload, heads: Sequence[int] | None = None) -> np.ndarray:
    """The keys of frame 0 that the centroids are fitted on: the first
    `kmeans_tokens` keys appended, float32 [heads, kmeans_tokens, d]."""
    parts, got, ch = [], 0, 0
    while got < wl.kmeans_tokens:
        n = min(wl.chunk, wl.kmeans_tokens - got)
        parts.append(keys(wl, ch, heads, n))
        got += n
        ch += 1
    return np.concatenate(parts, axis=1)


def workload(name: str) -> Workload:
    return WORKLOADS[name]
