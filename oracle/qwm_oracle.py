"""Plain CPU oracle of the QuantWM 2-bit KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of the package entry
file and the CPU-baseline / reference leg of the benchmark may import or run
this module.  It shares no code with the CUDA library and imports nothing from
it; the CUDA path never imports this file.

Sources (web pages on the method; cited by title and section):
  [A] "QuantWM: Temporally Consistent 2-Bit KV Cache Quantization for World
      Models and Video Generation", Abstract (arXiv 2609.26425v2).
  [B] roboind news article on QuantWM: sections "The key to a smaller error is
      to make a bigger impact", "Step 1: Select a more appropriate
      concentration center after quantification" (QSAC), "Step 2: Compensate
      the critical direction with a small amount of information" (PSAC),
      Table 1 and Fig. 4.
The pages describe QSAC and PSAC in prose only.  The formulas below are the
reading this project fixes (listed with the reasons in the design notes):

  sensitivity   s_c = mean_i q_ic^2 over the historical queries            [A], [B Step 1]
  group weight  w_g = sum_{c in g} s_c, groups of 32 channels
  QSAC score    S_j = sum_g w_g (range_g(k - C_j) / 3)^2 / 12, j* = argmin [A], [B Step 1]
  INT2          per token and group: zero = f16(min), scale = f16(range/3),
                code = clamp(rne((x - zero)/scale), 0, 3), 4 codes a byte  [A], [B Step 1]
  PSAC          U_r = top-r eigenvectors of Q_hist^T Q_hist,
                e = U_r (k - k_hat) stored in fp16,
                logit = q.k_hat + (q U_r^T).e                              [A], [B Step 2]
  attention     O = softmax(sigma * logit) V_hat over every cached token

Precision.  Every floating-point result is float64.  The two places where a
floating-point value decides an integer -- the centroid argmin and the INT2
code -- are taken in float32, one IEEE operation at a time in a fixed order
(no fused multiply-add), because the pages fix no precision and float32 is the
precision the GPU kernel decides in.  `qsac_scores_exact` keeps the float64
score for diagnostics (how often the float32 decision differs from the exact
argmin).  float16 parameters are rounded to nearest-even by numpy's float16
conversion, saturated at +-65504.

Nothing here is blocked, fused or reordered: each function is the formula
written out with numpy primitives.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GROUP = 32
TILE = 128
F16_MAX = 65504.0
f32 = np.float32


# --------------------------------------------------------------------------
# calibration: sensitivity and the principal query subspace
# --------------------------------------------------------------------------

def sensitivity(q_hist) -> np.ndarray:
    """s_c = (1/n_h) sum_i q_ic^2 (float64), per row of [..., n_h, d].

    Historical-query sensitivity [A]; "which channels ... affect attention"
    [B Step 1].
    """
    q = np.asarray(q_hist, dtype=np.float64)
    return (q * q).mean(axis=-2)


def group_weights(s32) -> np.ndarray:
    """w_g = s_{32g} + s_{32g+1} + ... + s_{32g+31}, float32, summed left to right.

    The weight is an input to the centroid decision, so it is formed in the
    decision precision, one float32 addition at a time.
    """
    s = np.asarray(s32, dtype=f32)
    d = s.shape[-1]
    G = d // GROUP
    w = np.zeros(s.shape[:-1] + (G,), dtype=f32)
    for g in range(G):
        acc = s[..., GROUP * g].astype(f32)
        for c in range(GROUP * g + 1, GROUP * (g + 1)):
            acc = (acc + s[..., c]).astype(f32)
        w[..., g] = acc
    return w


def gram(q_hist) -> np.ndarray:
    """G = Q_hist^T Q_hist (float64), per head."""
    q = np.asarray(q_hist, dtype=np.float64)
    return np.swapaxes(q, -1, -2) @ q


def psac_basis(q_hist, r: int):
    """Top-r eigenvectors of Q_hist^T Q_hist, for one head [n_h, d].

    "the energy of historical queries tends to be concentrated in a few
    directions" [B Step 2].  Returns (U [r, d] with the eigenvectors as rows,
    in descending eigenvalue order; lam [r]; energy = sum(lam_1..r)/trace).
    Sign rule: the entry of largest magnitude of each vector is positive (on an
    exact tie of magnitudes the lowest channel decides).
    """
    G = gram(q_hist)
    lam, vec = np.linalg.eigh(G)              # ascending
    order = np.argsort(-lam, kind="stable")
    lam = lam[order]
    vec = vec[:, order]
    U = vec[:, :r].T.copy()
    for i in range(r):
        j = int(np.argmax(np.abs(U[i])))
        if U[i, j] < 0:
            U[i] = -U[i]
    tr = float(np.trace(G))
    energy = float(lam[:r].sum() / tr) if tr > 0 else 0.0
    return U, lam[:r].copy(), energy


# --------------------------------------------------------------------------
# QSAC: sensitivity-weighted, INT2-range-aware centroid choice  [A], [B Step 1]
# --------------------------------------------------------------------------

def _score_tree(t):
    """Fixed float32 summation order over groups: ((t0+t1)+(t2+t3)) or (t0+t1)."""
    G = t.shape[-1]
    if G == 1:
        return t[..., 0]
    if G == 2:
        return (t[..., 0] + t[..., 1]).astype(f32)
    if G == 4:
        a = (t[..., 0] + t[..., 1]).astype(f32)
        b = (t[..., 2] + t[..., 3]).astype(f32)
        return (a + b).astype(f32)
    raise ValueError("head_dim must give 1, 2 or 4 groups of 32")


def qsac_scores_f32(k32, C32, w32) -> np.ndarray:
    """Decision score of every centroid for one key, in float32.

    rho = f32(k - C_j); R_g = f32(max_g rho - min_g rho);
    t_g = f32(w_g * f32(R_g * R_g)); S_j = fixed tree sum of t_g.
    The positive constant 1/108 of sum_g w_g (R_g/3)^2/12 is left out: an
    exact positive factor does not move the argmin.
    k32 [d], C32 [C, d], w32 [G] -> S [C] float32.
    """
    k = np.asarray(k32, dtype=f32)
    C = np.asarray(C32, dtype=f32)
    w = np.asarray(w32, dtype=f32)
    rho = (k[None, :] - C).astype(f32)
    nC, d = rho.shape
    G = d // GROUP
    rg = rho.reshape(nC, G, GROUP)
    R = (rg.max(axis=-1) - rg.min(axis=-1)).astype(f32)
    t = (w[None, :] * (R * R).astype(f32)).astype(f32)
    return _score_tree(t)


def qsac_scores_exact(k, C, w) -> np.ndarray:
    """sum_g w_g (range_g(k - C_j)/3)^2 / 12 in float64 (diagnostics)."""
    k = np.asarray(k, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    rho = k[None, :] - C
    nC, d = rho.shape
    rg = rho.reshape(nC, d // GROUP, GROUP)
    R = rg.max(axis=-1) - rg.min(axis=-1)
    return ((R / 3.0) ** 2 / 12.0) @ w


def qsac_assign(k32, C32, w32) -> np.ndarray:
    """j* for every key row of k32 [n, d]; the lowest index wins a tie."""
    k = np.asarray(k32, dtype=f32)
    out = np.empty(k.shape[0], dtype=np.int64)
    for i in range(k.shape[0]):
        out[i] = int(np.argmin(qsac_scores_f32(k[i], C32, w32)))
    return out


def nearest_scores_f32(k32, C32) -> np.ndarray:
    """Squared distance of one key to every centroid, the decision of the
    nearest-centroid assignment that [B] Step 1 describes for QVG (each key is
    assigned to the centre it is closest to), in float32 with a fixed order:
    rho = f32(k - C_j); D_g = float32 sum over the 32 channels of group g, in
    channel order, of f32(rho * rho); S_j = the same tree sum over groups as
    the QSAC score.  k32 [d], C32 [C, d] -> S [C] float32."""
    k = np.asarray(k32, dtype=f32)
    C = np.asarray(C32, dtype=f32)
    rho = (k[None, :] - C).astype(f32)
    nC, d = rho.shape
    sq = (rho * rho).astype(f32).reshape(nC, d // GROUP, GROUP)
    acc = sq[..., 0].copy()
    for c in range(1, GROUP):
        acc = (acc + sq[..., c]).astype(f32)
    return _score_tree(acc)


def nearest_assign(k32, C32) -> np.ndarray:
    """Nearest centroid for every key row of k32 [n, d]; lowest index on a tie."""
    k = np.asarray(k32, dtype=f32)
    out = np.empty(k.shape[0], dtype=np.int64)
    for i in range(k.shape[0]):
        out[i] = int(np.argmin(nearest_scores_f32(k[i], C32)))
    return out


# --------------------------------------------------------------------------
# per-group asymmetric INT2 quantiser and 2-bit packing  [A], [B Step 1]
# --------------------------------------------------------------------------

def f16_saturate(x):
    """Round to float16 (nearest-even); values beyond the float16 range become
    +-65504.  Returns (float16 array, bool array of saturated entries)."""
    x = np.asarray(x)
    with np.errstate(over="ignore"):
        h = x.astype(np.float16)
    sat = np.isinf(h)
    h = np.where(sat, np.copysign(np.float16(F16_MAX), h), h).astype(np.float16)
    return h, sat


def quantize_int2(x32):
    """Quantise groups of 32 float32 values (last axis) to 2-bit codes.

    zero = f16(min); scale = f16(f32(range / 3)); range = f32(max - min);
    code = clamp(rint(f32(f32(x - zero) / scale)), 0, 3), all codes 0 when the
    scale is 0.  rint rounds halves to even.
    Returns (zero f16 [...], scale f16 [...], codes uint8 [..., 32], saturated bool [...]).
    """
    x = np.asarray(x32, dtype=f32)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    R = (mx - mn).astype(f32)
    zero, sat_z = f16_saturate(mn)
    scale, sat_s = f16_saturate((R / f32(3.0)).astype(f32))
    zf = zero.astype(f32)[..., None]
    sf = scale.astype(f32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = ((x - zf).astype(f32) / sf).astype(f32)
    code = np.clip(np.rint(t), 0, 3)
    code = np.where(sf == 0, 0, code)
    return zero, scale, code.astype(np.uint8), (sat_z | sat_s)


def dequantize(zero16, scale16, codes) -> np.ndarray:
    """x_hat = zero + code * scale in float64; zero/scale [...], codes [..., 32]."""
    z = np.asarray(zero16, dtype=np.float64)[..., None]
    s = np.asarray(scale16, dtype=np.float64)[..., None]
    return z + np.asarray(codes, dtype=np.float64) * s


def pack_codes(codes) -> np.ndarray:
    """Four 2-bit codes per byte: channel c -> byte c//4, bits 2*(c%4)..+1."""
    c = np.asarray(codes, dtype=np.uint8)
    c = c.reshape(c.shape[:-1] + (c.shape[-1] // 4, 4))
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def unpack_codes(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.stack([(p >> (2 * i)) & 3 for i in range(4)], axis=-1)
    return out.reshape(p.shape[:-1] + (p.shape[-1] * 4,)).astype(np.uint8)


def quantize_rows(x32):
    """Per token, per group of 32: rows [n, d] -> (zero [n,G], scale [n,G], codes [n,d], sat [n,G])."""
    x = np.asarray(x32, dtype=f32)
    n, d = x.shape
    z, s, c, sat = quantize_int2(x.reshape(n, d // GROUP, GROUP))
    return z, s, c.reshape(n, d), sat


def dequantize_rows(zero16, scale16, codes) -> np.ndarray:
    n, G = np.asarray(zero16).shape
    c = np.asarray(codes).reshape(n, G, GROUP)
    return dequantize(zero16, scale16, c).reshape(n, G * GROUP)


# --------------------------------------------------------------------------
# append: assign, quantise the key residual and the value, PSAC coefficients
# --------------------------------------------------------------------------

@dataclass
class Segment:
    """What one append call stores for one head (oracle form, unpacked)."""
    idx: np.ndarray          # [n] int64 centroid index
    kzero: np.ndarray        # [n, G] float16
    kscale: np.ndarray       # [n, G] float16
    kcodes: np.ndarray       # [n, d] uint8 0..3
    e16: np.ndarray          # [n, r] float16 stored PSAC coefficients
    vzero: np.ndarray        # [n, G] float16
    vscale: np.ndarray       # [n, G] float16
    vcodes: np.ndarray       # [n, d] uint8
    version: int             # basis version the coefficients are taken in
    khat: np.ndarray = field(default=None)   # [n, d] float64 dequantised key
    vhat: np.ndarray = field(default=None)   # [n, d] float64 dequantised value
    e64: np.ndarray = field(default=None)    # [n, r] float64 coefficients before fp16
    saturated: int = 0


def append_head(k32, v32, C32, w32, U, version: int = 0, assign: str = "qsac") -> Segment:
    """Encode one chunk of one head.  k32, v32 [n, d] float32; C32 [C, d]
    float32 (centroids already rounded to the cache dtype); w32 [G] float32;
    U [r, d] float64 (rows = basis vectors).  assign: "qsac" (QuantWM) or
    "nearest" (the nearest-centroid baseline)."""
    k = np.asarray(k32, dtype=f32)
    v = np.asarray(v32, dtype=f32)
    C = np.asarray(C32, dtype=f32)
    U = np.asarray(U, dtype=np.float64).reshape(-1, k.shape[1])
    if assign == "nearest":
        idx = nearest_assign(k, C)
    elif assign == "qsac":
        idx = qsac_assign(k, C, w32)
    else:
        raise ValueError(f"unknown assignment {assign!r}")
    rho = (k - C[idx]).astype(f32)                   # residual of the chosen centroid
    kz, ks, kc, ksat = quantize_rows(rho)
    khat = C[idx].astype(np.float64) + dequantize_rows(kz, ks, kc)
    e64 = (k.astype(np.float64) - khat) @ U.T        # PSAC: U_r (k - k_hat)
    e16 = e64.astype(np.float16)
    vz, vs, vc, vsat = quantize_rows(v)
    vhat = dequantize_rows(vz, vs, vc)
    return Segment(idx=idx, kzero=kz, kscale=ks, kcodes=kc, e16=e16, vzero=vz,
                   vscale=vs, vcodes=vc, version=version, khat=khat, vhat=vhat,
                   e64=e64, saturated=int(ksat.sum() + vsat.sum()))


# --------------------------------------------------------------------------
# attention over the packed cache with PSAC correction  [A], [B Step 2]
# --------------------------------------------------------------------------

def attend_head(q, segments, bases, sigma: float, e_exact: bool = False) -> np.ndarray:
    """O = softmax(sigma * l) V_hat for one head, float64.

    q [M, d]; segments: list of Segment (each with khat, vhat, e16, version);
    bases: {version: U [r, d]}.  For every key n of segment t:
        l_n = q . k_hat_n + (q U_t^T) . e_n
    with e_n the stored fp16 coefficients (float64 ones when e_exact).
    """
    q = np.asarray(q, dtype=np.float64)
    logits = []
    vhat = []
    for seg in segments:
        l = q @ seg.khat.T
        U = np.asarray(bases[seg.version], dtype=np.float64)
        if U.shape[0] > 0:
            z = q @ U.T
            e = seg.e64 if e_exact else seg.e16.astype(np.float64)
            l = l + z @ e.T
        logits.append(l)
        vhat.append(seg.vhat)
    if not logits:
        raise ValueError("attention over an empty cache")
    L = sigma * np.concatenate(logits, axis=1)
    L = L - L.max(axis=1, keepdims=True)
    P = np.exp(L)
    P /= P.sum(axis=1, keepdims=True)
    return P @ np.concatenate(vhat, axis=0)


def attention_weights(q, segments, bases, sigma: float, e_exact: bool = False) -> np.ndarray:
    """Softmax weights P [M, N] of `attend_head` (diagnostics and pins)."""
    q = np.asarray(q, dtype=np.float64)
    logits = []
    for seg in segments:
        l = q @ seg.khat.T
        U = np.asarray(bases[seg.version], dtype=np.float64)
        if U.shape[0] > 0:
            e = seg.e64 if e_exact else seg.e16.astype(np.float64)
            l = l + (q @ U.T) @ e.T
        logits.append(l)
    L = sigma * np.concatenate(logits, axis=1)
    L = L - L.max(axis=1, keepdims=True)
    P = np.exp(L)
    return P / P.sum(axis=1, keepdims=True)


# --------------------------------------------------------------------------
# byte layout of the packed cache (one 128-token tile per block)
# --------------------------------------------------------------------------

def index_bytes(n_centroids: int) -> int:
    return 1 if n_centroids <= 256 else 2


def bytes_per_token(d: int, r: int, n_centroids: int) -> int:
    """Cache bytes per token and head: index + K codes + V codes + (zero, scale)
    for K and V per group + r fp16 coefficients."""
    G = d // GROUP
    return index_bytes(n_centroids) + d // 4 + d // 4 + 2 * 2 * G + 2 * 2 * G + 2 * r


def tile_layout(d: int, r: int, n_centroids: int) -> dict:
    """Byte offsets of the sections of one 128-slot tile.

    [ idx | K codes | K (zero, scale) | e | V codes | V (zero, scale) ]
    idx: u8 (C <= 256) or u16 per slot; codes: d/4 bytes per slot; (zero, scale):
    one fp16 pair per slot and group, zero first; e: r fp16 per slot.
    """
    G = d // GROUP
    ib = index_bytes(n_centroids)
    sizes = [("idx", TILE * ib), ("kcode", TILE * d // 4), ("kqp", TILE * G * 4),
             ("e", TILE * r * 2), ("vcode", TILE * d // 4), ("vqp", TILE * G * 4)]
    off = {}
    o = 0
    for name, sz in sizes:
        off[name] = o
        o += sz
    off["tile_bytes"] = o
    return off


def encode_tile(seg: Segment, start: int, count: int, d: int, r: int, n_centroids: int) -> bytes:
    """Bytes of one tile holding tokens [start, start+count) of a segment; the
    unused slots are zero."""
    L = tile_layout(d, r, n_centroids)
    G = d // GROUP
    buf = np.zeros(L["tile_bytes"], dtype=np.uint8)
    sl = slice(start, start + count)
    ib = index_bytes(n_centroids)
    idx = seg.idx[sl].astype(np.uint8 if ib == 1 else np.uint16)
    buf[L["idx"]:L["idx"] + count * ib] = idx.view(np.uint8)
    kc = pack_codes(seg.kcodes[sl])
    buf[L["kcode"]:L["kcode"] + kc.size] = kc.reshape(-1)
    kqp = np.stack([seg.kzero[sl], seg.kscale[sl]], axis=-1).astype(np.float16)
    buf[L["kqp"]:L["kqp"] + count * G * 4] = kqp.reshape(-1).view(np.uint8)
    if r:
        buf[L["e"]:L["e"] + count * r * 2] = seg.e16[sl].astype(np.float16).reshape(-1).view(np.uint8)
    vc = pack_codes(seg.vcodes[sl])
    buf[L["vcode"]:L["vcode"] + vc.size] = vc.reshape(-1)
    vqp = np.stack([seg.vzero[sl], seg.vscale[sl]], axis=-1).astype(np.float16)
    buf[L["vqp"]:L["vqp"] + count * G * 4] = vqp.reshape(-1).view(np.uint8)
    return buf.tobytes()


def encode_segment(seg: Segment, d: int, r: int, n_centroids: int) -> bytes:
    n = seg.idx.shape[0]
    out = b""
    for t0 in range(0, n, TILE):
        out += encode_tile(seg, t0, min(TILE, n - t0), d, r, n_centroids)
    return out


def decode_tile(raw, count: int, d: int, r: int, n_centroids: int, centroids32, version: int) -> Segment:
    """Read the first `count` slots of one tile's bytes back into a Segment and
    dequantise it against the given centroids (float32 [C, d])."""
    L = tile_layout(d, r, n_centroids)
    G = d // GROUP
    b = np.frombuffer(bytes(raw), dtype=np.uint8)
    ib = index_bytes(n_centroids)
    idx = b[L["idx"]:L["idx"] + count * ib].view(np.uint8 if ib == 1 else np.uint16).astype(np.int64)
    kc = unpack_codes(b[L["kcode"]:L["kcode"] + count * d // 4].reshape(count, d // 4))
    kqp = b[L["kqp"]:L["kqp"] + count * G * 4].view(np.float16).reshape(count, G, 2)
    e16 = b[L["e"]:L["e"] + count * r * 2].view(np.float16).reshape(count, r)
    vc = unpack_codes(b[L["vcode"]:L["vcode"] + count * d // 4].reshape(count, d // 4))
    vqp = b[L["vqp"]:L["vqp"] + count * G * 4].view(np.float16).reshape(count, G, 2)
    C = np.asarray(centroids32, dtype=np.float64)
    kz, ks = kqp[..., 0].copy(), kqp[..., 1].copy()
    vz, vs = vqp[..., 0].copy(), vqp[..., 1].copy()
    khat = C[idx] + dequantize_rows(kz, ks, kc)
    vhat = dequantize_rows(vz, vs, vc)
    return Segment(idx=idx, kzero=kz, kscale=ks, kcodes=kc, e16=e16.copy(), vzero=vz,
                   vscale=vs, vcodes=vc, version=version, khat=khat, vhat=vhat,
                   e64=e16.astype(np.float64))


# --------------------------------------------------------------------------
# k-means (Lloyd) that builds the high-precision centroids  [B Step 1]
# --------------------------------------------------------------------------

def kmeans(keys, init_rows, iters: int = 25) -> np.ndarray:
    """Lloyd's iteration in float64 on keys [n, d], started from the rows
    `init_rows`.  Assignment to the nearest centroid in squared Euclidean
    distance (lowest index on a tie); a centroid left without keys keeps its
    previous position."""
    X = np.asarray(keys, dtype=np.float64)
    Cm = X[np.asarray(init_rows)].copy()
    for _ in range(iters):
        d2 = (X * X).sum(1)[:, None] - 2.0 * X @ Cm.T + (Cm * Cm).sum(1)[None, :]
        a = np.argmin(d2, axis=1)
        for j in range(Cm.shape[0]):
            m = a == j
            if m.any():
                Cm[j] = X[m].mean(axis=0)
    return Cm


# --------------------------------------------------------------------------
# a whole multi-head cache, as the library's three calls use it
# --------------------------------------------------------------------------

class OracleCache:
    """Mirror of the library's calibrate / append / attend sequence.

    Calibration is injected (float32 s per head and a float64 basis per head);
    each injection opens a new basis version, and every later append stores
    its coefficients in that version's basis.
    """

    def __init__(self, heads: int, d: int, r: int, centroids32, assign: str = "qsac"):
        self.H, self.d, self.r = heads, d, r
        self.assign = assign
        self.C = np.asarray(centroids32, dtype=f32)        # [H, C, d]
        self.version = -1
        self.w = None
        self.bases = [dict() for _ in range(heads)]
        self.segments = [[] for _ in range(heads)]

    def set_calibration(self, s32, U):
        self.version += 1
        self.w = group_weights(np.asarray(s32, dtype=f32))  # [H, G]
        U = np.asarray(U, dtype=np.float64).reshape(self.H, self.r, self.d)
        for h in range(self.H):
            self.bases[h][self.version] = U[h]

    def append(self, k32, v32, heads=None):
        hs = range(self.H) if heads is None else heads
        for i, h in enumerate(hs):
            self.segments[h].append(append_head(k32[i], v32[i], self.C[h], self.w[h],
                                                self.bases[h][self.version], self.version, self.assign))

    def attend(self, q, sigma: float, heads=None) -> np.ndarray:
        hs = range(self.H) if heads is None else heads
        return np.stack([attend_head(q[i], self.segments[h], self.bases[h], sigma)
                         for i, h in enumerate(hs)])


# --------------------------------------------------------------------------
# attention-shift diagnostics  [A] Abstract; [B] "The key to a smaller
# error ...", Figure 2, Table 1
# --------------------------------------------------------------------------

def compensated_logits(q, segments, bases, e_exact: bool = False) -> np.ndarray:
    """l [M, N] = q . k_hat_n + (q U_t^T) . e_n over all segments (float64)."""
    q = np.asarray(q, dtype=np.float64)
    out = []
    for seg in segments:
        l = q @ seg.khat.T
        U = np.asarray(bases[seg.version], dtype=np.float64)
        if U.shape[0] > 0:
            e = seg.e64 if e_exact else seg.e16.astype(np.float64)
            l = l + (q @ U.T) @ e.T
        out.append(l)
    return np.concatenate(out, axis=1)


def top1_change(logits_exact, logits_quant) -> float:
    """Fraction of query rows whose highest-scoring cached token differs
    between the exact and the quantised logits (the Table 1 measure)."""
    a = np.argmax(np.asarray(logits_exact), axis=1)
    b = np.argmax(np.asarray(logits_quant), axis=1)
    return float(np.mean(a != b))


def softmax_rows(logits, sigma: float) -> np.ndarray:
    L = sigma * np.asarray(logits, dtype=np.float64)
    L = L - L.max(axis=1, keepdims=True)
    P = np.exp(L)
    return P / P.sum(axis=1, keepdims=True)


def key_value_study(q, k, v, segments, bases, sigma: float) -> dict:
    """Key-only vs value-only quantisation of one head ([B], "The key to a
    smaller error ..."): relative reconstruction errors of K and V, and the
    relative output error when only K (PSAC included) or only V is taken from
    the cache, the other one exact.  q [M, d], k, v [N, d] (float, in cache
    order)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    khat = np.concatenate([s.khat for s in segments])
    vhat = np.concatenate([s.vhat for s in segments])
    o = softmax_rows(q @ k.T, sigma) @ v
    o_k = softmax_rows(compensated_logits(q, segments, bases), sigma) @ v
    o_v = softmax_rows(q @ k.T, sigma) @ vhat
    nrm = np.linalg.norm
    return {"key_rel_error": float(nrm(k - khat) / nrm(k)),
            "value_rel_error": float(nrm(v - vhat) / nrm(v)),
            "output_rel_error_key_only": float(nrm(o_k - o) / nrm(o)),
            "output_rel_error_value_only": float(nrm(o_v - o) / nrm(o))}


def logit_error(q, k, segments, bases) -> float:
    """Root mean square of q . k - l_quant over all (query, token) pairs,
    relative to the root mean square of q . k."""
    q = np.asarray(q, dtype=np.float64)
    exact = q @ np.asarray(k, dtype=np.float64).T
    d = exact - compensated_logits(q, segments, bases)
    return float(np.sqrt(np.mean(d * d) / np.mean(exact * exact)))
