"""Thin Python binding of libqwm (ctypes).

Argument marshalling only: every step of calibrate / append / attend runs in
the CUDA library.  PyTorch provides device memory and the current stream.
There is no fallback: if libqwm.so is missing or fails to load, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# QWM_DEBUG_BOUNDS=1 selects the checking build (build.build(debug_bounds=True))
LIB_PATH = os.path.join(_PKG, "libqwm_dbg.so" if os.environ.get("QWM_DEBUG_BOUNDS") == "1" else "libqwm.so")

QWM_F32, QWM_BF16 = 0, 1
DEV_NOT_CONVERGED, DEV_SATURATED, DEV_TIMEOUT, DEV_BOUNDS = 0x1, 0x2, 0x4, 0x8
# attention kernels (qwm_set_attend_kernel): automatic choice, float32 SIMT,
# bf16 mma.sync, tcgen05 with one query tile per CTA, tcgen05 with two query
# tiles per CTA, few-row split-KV (M <= 64), tcgen05 with the key split into
# its float16 centroid row and float16 residual, the same with one query tile
# per CTA and the cache split over CTAs for M <= 64
KERNEL_AUTO, KERNEL_SIMT, KERNEL_MMA, KERNEL_TC, KERNEL_TC2, KERNEL_SMALL, KERNEL_TC3, KERNEL_TC3_FEW = \
    0, 1, 2, 3, 4, 5, 6, 7

STATUS = {0: "QWM_OK", 1: "QWM_ERR_INVALID_ARG", 2: "QWM_ERR_UNSUPPORTED", 3: "QWM_ERR_CAPACITY",
          4: "QWM_ERR_NOT_CALIBRATED", 5: "QWM_ERR_NOT_CONVERGED", 6: "QWM_ERR_CUDA",
          7: "QWM_ERR_OOM", 8: "QWM_ERR_DEVICE"}


class qwm_config(ctypes.Structure):
    _fields_ = [("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("group", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("n_centroids", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("max_tokens", ctypes.c_int64), ("max_versions", ctypes.c_int32),
                ("max_iter", ctypes.c_int32), ("oversample", ctypes.c_int32),
                ("max_hist", ctypes.c_int32)]


class qwm_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("cache_bytes", "state_bytes", "workspace_bytes",
                                                "tile_bytes", "bytes_per_token")] + \
               [("max_tiles", ctypes.c_int64)] + \
               [(n, ctypes.c_size_t) for n in ("off_idx", "off_kcode", "off_kqp", "off_e", "off_vcode",
                                                "off_vqp", "st_status", "st_s", "st_w", "st_lambda",
                                                "st_energy", "st_centroids", "st_basis", "st_tiles",
                                                "st_iters", "st_centroids_f32", "st_centroids_f16")]


class QwmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


EXPORTS = ["qwm_status_string", "qwm_sizes", "qwm_create", "qwm_destroy", "qwm_set_centroids",
           "qwm_calibrate", "qwm_calibrate_static", "qwm_kmeans", "qwm_kmeans_workspace_bytes", "qwm_set_calibration", "qwm_get_calibration", "qwm_append",
           "qwm_attend", "qwm_rewind", "qwm_get_status", "qwm_peek_status_bits",
           "qwm_set_attend_kernel", "qwm_resolved_attend_kernel", "qwm_attend_kernel_for", "qwm_set_assignment",
           "qwm_dequantize", "qwm_selftest_wait_timeout", "qwm_num_tokens",
           "qwm_num_tiles", "qwm_num_segments", "qwm_version"]

_lib = None


def lib() -> ctypes.CDLL:
    """Load libqwm.so (built in-tree by build.py); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{os.path.basename(LIB_PATH)} not found at {LIB_PATH}: run bit_kv_cache_qwm_gb300/build.py")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
    L.qwm_status_string.restype = ctypes.c_char_p
    L.qwm_status_string.argtypes = [ctypes.c_int]
    sig = {
        "qwm_sizes": [P(qwm_config), P(qwm_layout)],
        "qwm_create": [P(qwm_config), VP, VP, VP, P(VP)],
        "qwm_destroy": [VP],
        "qwm_set_centroids": [VP, VP, VP],
        "qwm_calibrate": [VP, VP, I64, VP],
        "qwm_set_calibration": [VP, P(F), P(F), VP],
        "qwm_get_calibration": [VP, P(F), P(F), P(F), P(F), VP],
        "qwm_append": [VP, VP, VP, I64, VP],
        "qwm_attend": [VP, VP, I64, F, VP, VP],
        "qwm_rewind": [VP, I32],
        "qwm_get_status": [VP, VP],
        "qwm_peek_status_bits": [VP, P(ctypes.c_uint32), VP],
        "qwm_set_attend_kernel": [VP, I32],
        "qwm_set_assignment": [VP, I32],
        "qwm_dequantize": [VP, VP, VP, VP, VP],
        "qwm_selftest_wait_timeout": [I64, VP, VP],
        "qwm_calibrate_static": [I32, I32, I32, I32, I32, I32, VP, I64, VP, VP, VP, VP, VP, VP],
        "qwm_kmeans": [I32, I32, I32, I32, VP, I64, VP, I32, VP, VP, VP],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    L.qwm_kmeans_workspace_bytes.restype = ctypes.c_size_t
    L.qwm_kmeans_workspace_bytes.argtypes = [I32, I32, I32, I64]
    L.qwm_attend_kernel_for.restype = I32
    L.qwm_attend_kernel_for.argtypes = [VP, I64]
    for name, rt in [("qwm_resolved_attend_kernel", I32), ("qwm_num_tokens", I64), ("qwm_num_tiles", I64), ("qwm_num_segments", I32),
                     ("qwm_version", I32)]:
        fn = getattr(L, name)
        fn.argtypes = [VP]
        fn.restype = rt
    _lib = L
    return L


def _check(st: int, what: str):
    if st != 0:
        raise QwmError(st, what)


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _fptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _device_tensor(x, what: str, dtypes, ndim: int) -> torch.Tensor:
    """A contiguous CUDA tensor of one of `dtypes` with `ndim` dimensions, or ValueError."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError(f"{what}: a CUDA tensor is expected")
    if x.dtype not in dtypes or x.dim() != ndim or not x.is_contiguous():
        raise ValueError(f"{what}: a contiguous {ndim}-d tensor of {dtypes} is expected, got "
                         f"{x.dtype} {tuple(x.shape)}")
    return x


def _out_tensor(t, what: str, dtype, shape, device) -> torch.Tensor:
    if (not isinstance(t, torch.Tensor) or t.device != device or t.dtype != dtype
            or tuple(t.shape) != tuple(shape) or not t.is_contiguous()):
        raise ValueError(f"out[{what!r}]: a contiguous {dtype} tensor of shape {tuple(shape)} on {device} "
                         f"is expected")
    return t


def qwm_calibrate_static(q_hist: torch.Tensor, rank: int, max_iter: int = 64, oversample: int = 16,
                         out: Optional[dict] = None) -> dict:
    """Calibration that allocates nothing on the device inside the library
    (scratch in a fixed 8 MiB array of the library).  Output buffers are taken
    from `out` when given (contiguous float32 tensors on q_hist's device, and
    an int32 status word of one element), else allocated here by torch,
    outside the library.  Runs on q_hist's device and that device's current
    stream."""
    q_hist = _device_tensor(q_hist, "q_hist", (torch.bfloat16, torch.float32), 3)
    H, n_h, d = q_hist.shape
    dt = QWM_BF16 if q_hist.dtype == torch.bfloat16 else QWM_F32
    dev = q_hist.device
    rr = max(rank, 1)
    shapes = {"s": ((H, d), torch.float32), "U": ((H, rr, d), torch.float32),
              "lambda": ((H, rr), torch.float32), "energy": ((H,), torch.float32),
              "status": ((1,), torch.int32)}
    if out is None:
        out = {k: torch.empty(sh, dtype=dt_, device=dev) for k, (sh, dt_) in shapes.items()}
        out["status"].zero_()
    else:
        for k, (sh, dt_) in shapes.items():
            _out_tensor(out.get(k), k, dt_, sh, dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    with torch.cuda.device(dev):
        _check(lib().qwm_calibrate_static(H, d, rank, dt, max_iter, oversample, P(q_hist), n_h, P(out["s"]),
                                          P(out["U"]), P(out["lambda"]), P(out["energy"]), P(out["status"]),
                                          _stream()), "qwm_calibrate_static")
    return out


def selftest_wait_timeout(limit_cycles: int = 1 << 20) -> int:
    """Run the bounded-wait self-test on the current device and stream and
    return the status word it leaves (QWM_DEV_TIMEOUT when the wait ran out)."""
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(lib().qwm_selftest_wait_timeout(int(limit_cycles), ctypes.c_void_p(word.data_ptr()), _stream()),
           "qwm_selftest_wait_timeout")
    return int(word.item()) & 0xffffffff


def qwm_kmeans(keys: torch.Tensor, init_rows: torch.Tensor, n_centroids: int, iters: int = 25) -> torch.Tensor:
    """Lloyd's k-means on the GPU: keys [H][n][d] (bf16/f32, CUDA), init_rows
    [H][C] integer row indices (moved to the keys' device).  Returns centroids
    [H][C][d] in the keys' dtype, on the keys' device."""
    keys = _device_tensor(keys, "keys", (torch.bfloat16, torch.float32), 3)
    H, n, d = keys.shape
    dt = QWM_BF16 if keys.dtype == torch.bfloat16 else QWM_F32
    if not isinstance(init_rows, torch.Tensor) or init_rows.dtype.is_floating_point:
        raise ValueError("init_rows: an integer tensor is expected")
    if tuple(init_rows.shape) != (H, n_centroids):
        raise ValueError("init_rows: shape [H, C] expected")
    if not 1 <= n_centroids <= n:
        raise ValueError("n_centroids: between 1 and the number of keys")
    rows = init_rows.to(device=keys.device, dtype=torch.int32).contiguous()
    with torch.cuda.device(keys.device):
        ws = torch.empty(lib().qwm_kmeans_workspace_bytes(H, d, n_centroids, n) + 256, dtype=torch.uint8,
                         device=keys.device)
        out = torch.empty((H, n_centroids, d), dtype=keys.dtype, device=keys.device)
        _check(lib().qwm_kmeans(H, d, dt, n_centroids, ctypes.c_void_p(keys.data_ptr()), n,
                                ctypes.c_void_p(rows.data_ptr()), iters, ctypes.c_void_p(out.data_ptr()),
                                ctypes.c_void_p(ws.data_ptr()), _stream()), "qwm_kmeans")
    return out


def make_config(heads, head_dim, rank, n_centroids, dtype="bf16", max_tokens=4096, max_versions=4,
                max_iter=64, oversample=16, max_hist=4096) -> qwm_config:
    return qwm_config(heads=heads, head_dim=head_dim, group=32, rank=rank, n_centroids=n_centroids,
                      dtype=QWM_BF16 if dtype == "bf16" else QWM_F32, max_tokens=max_tokens,
                      max_versions=max_versions, max_iter=max_iter, oversample=oversample,
                      max_hist=max_hist)


def qwm_sizes(cfg: qwm_config) -> qwm_layout:
    out = qwm_layout()
    _check(lib().qwm_sizes(ctypes.byref(cfg), ctypes.byref(out)), "qwm_sizes")
    return out


class Qwm:
    """One libqwm context with its device buffers allocated through torch."""

    def __init__(self, heads, head_dim, rank, n_centroids, dtype="bf16", max_tokens=4096,
                 max_versions=4, max_iter=64, oversample=16, max_hist=4096, device=None):
        self.cfg = make_config(heads, head_dim, rank, n_centroids, dtype, max_tokens, max_versions,
                               max_iter, oversample, max_hist)
        self.layout = qwm_sizes(self.cfg)
        self.dtype = dtype
        self.tdtype = torch.bfloat16 if dtype == "bf16" else torch.float32
        self.device = (torch.device(device) if device is not None
                       else torch.device("cuda", torch.cuda.current_device()))
        L = self.layout
        with torch.cuda.device(self.device):
            self.cache = torch.empty(max(L.cache_bytes, 256), dtype=torch.uint8, device=self.device)
            self.state = torch.empty(max(L.state_bytes, 256), dtype=torch.uint8, device=self.device)
            self.workspace = torch.empty(max(L.workspace_bytes, 256), dtype=torch.uint8, device=self.device)
            torch.cuda.synchronize(self.device)
            h = ctypes.c_void_p()
            _check(lib().qwm_create(ctypes.byref(self.cfg), ctypes.c_void_p(self.cache.data_ptr()),
                                    ctypes.c_void_p(self.state.data_ptr()),
                                    ctypes.c_void_p(self.workspace.data_ptr()), ctypes.byref(h)),
                   "qwm_create")
        self._h = h

    # ---- helpers
    def _t(self, x: torch.Tensor, shape, what):
        if not isinstance(x, torch.Tensor) or x.device != self.device or x.dtype != self.tdtype:
            raise ValueError(f"{what}: expected a {self.tdtype} tensor on {self.device}")
        if tuple(x.shape) != tuple(shape) or not x.is_contiguous():
            raise ValueError(f"{what}: expected contiguous shape {tuple(shape)}, got {tuple(x.shape)}")
        return ctypes.c_void_p(x.data_ptr())

    @property
    def handle(self):
        return self._h

    # ---- the calls
    def set_centroids(self, cent: torch.Tensor):
        c = self.cfg
        _check(lib().qwm_set_centroids(self._h, self._t(cent, (c.heads, c.n_centroids, c.head_dim), "centroids"),
                                       _stream()), "qwm_set_centroids")

    def calibrate(self, q_hist: torch.Tensor):
        c = self.cfg
        n_h = q_hist.shape[1]
        _check(lib().qwm_calibrate(self._h, self._t(q_hist, (c.heads, n_h, c.head_dim), "q_hist"), n_h,
                                   _stream()), "qwm_calibrate")

    def set_calibration(self, s, U):
        c = self.cfg
        s = np.ascontiguousarray(np.asarray(s, dtype=np.float32).reshape(c.heads, c.head_dim))
        U = np.ascontiguousarray(np.asarray(U, dtype=np.float32).reshape(c.heads, c.rank, c.head_dim))
        _check(lib().qwm_set_calibration(self._h, _fptr(s), _fptr(U) if c.rank else None, _stream()),
               "qwm_set_calibration")

    def get_calibration(self) -> dict:
        c = self.cfg
        s = np.zeros((c.heads, c.head_dim), np.float32)
        U = np.zeros((c.heads, c.rank, c.head_dim), np.float32)
        lam = np.zeros((c.heads, c.rank), np.float32)
        en = np.zeros(c.heads, np.float32)
        _check(lib().qwm_get_calibration(self._h, _fptr(s), _fptr(U) if c.rank else None,
                                         _fptr(lam) if c.rank else None, _fptr(en), _stream()),
               "qwm_get_calibration")
        return {"s": s, "U": U, "lambda": lam, "energy": en}

    def append(self, k: torch.Tensor, v: torch.Tensor):
        c = self.cfg
        n = k.shape[1]
        shape = (c.heads, n, c.head_dim)
        _check(lib().qwm_append(self._h, self._t(k, shape, "k"), self._t(v, shape, "v"), n, _stream()),
               "qwm_append")

    def attend(self, q: torch.Tensor, out: Optional[torch.Tensor] = None, scale: float = 0.0) -> torch.Tensor:
        c = self.cfg
        M = q.shape[1]
        if out is None:
            out = torch.empty_like(q)
        _check(lib().qwm_attend(self._h, self._t(q, (c.heads, M, c.head_dim), "q"), M, float(scale),
                                self._t(out, (c.heads, M, c.head_dim), "out"), _stream()), "qwm_attend")
        return out

    def rewind(self, n_segments: int):
        _check(lib().qwm_rewind(self._h, int(n_segments)), "qwm_rewind")

    def status(self) -> int:
        return lib().qwm_get_status(self._h, _stream())

    def status_bits(self) -> int:
        b = ctypes.c_uint32(0)
        _check(lib().qwm_peek_status_bits(self._h, ctypes.byref(b), _stream()), "qwm_peek_status_bits")
        return int(b.value)

    def set_assignment(self, mode: str):
        """Centroid assignment of later appends: "qsac" or "nearest"."""
        _check(lib().qwm_set_assignment(self._h, {"qsac": 0, "nearest": 1}[mode]), "qwm_set_assignment")

    def dequantize(self):
        """(k_hat, v_hat, e) float32 [H, n_tiles*128, d / d / r] and the valid
        slot mask [n_tiles*128] (cache order)."""
        H, d, r = self.cfg.heads, self.cfg.head_dim, self.cfg.rank
        n = self.n_tiles * 128
        kh = torch.empty((H, n, d), dtype=torch.float32, device=self.device)
        vh = torch.empty((H, n, d), dtype=torch.float32, device=self.device)
        e = torch.empty((H, n, max(r, 1)), dtype=torch.float32, device=self.device)
        _check(lib().qwm_dequantize(self._h, ctypes.c_void_p(kh.data_ptr()), ctypes.c_void_p(vh.data_ptr()),
                                    ctypes.c_void_p(e.data_ptr()), _stream()), "qwm_dequantize")
        counts = self.tile_table()[: self.n_tiles, 1].to(torch.int64)
        valid = (torch.arange(128, device=counts.device)[None, :] < counts[:, None]).reshape(-1)
        return kh, vh, e[..., :r], valid

    def set_attend_kernel(self, k: int):
        _check(lib().qwm_set_attend_kernel(self._h, int(k)), "qwm_set_attend_kernel")

    @property
    def resolved_attend_kernel(self) -> int:
        """The attention kernel for more than 64 query rows."""
        return int(lib().qwm_resolved_attend_kernel(self._h))

    def attend_kernel_for(self, m: int) -> int:
        """The attention kernel qwm_attend runs for m query rows."""
        return int(lib().qwm_attend_kernel_for(self._h, int(m)))

    @property
    def n_tokens(self) -> int:
        return int(lib().qwm_num_tokens(self._h))

    @property
    def n_tiles(self) -> int:
        return int(lib().qwm_num_tiles(self._h))

    @property
    def n_segments(self) -> int:
        return int(lib().qwm_num_segments(self._h))

    @property
    def version(self) -> int:
        return int(lib().qwm_version(self._h))

    def cache_tiles(self) -> torch.Tensor:
        """View of the cache as [H, max_tiles, tile_bytes] uint8."""
        L = self.layout
        return self.cache[: L.cache_bytes].view(self.cfg.heads, L.max_tiles, L.tile_bytes)

    def tile_table(self) -> torch.Tensor:
        """View of the tile table as [max_tiles, 2] int32 (basis version, valid slots)."""
        L = self.layout
        return self.state[L.st_tiles: L.st_tiles + 8 * L.max_tiles].view(torch.int32).view(L.max_tiles, 2)

    def close(self):
        if getattr(self, "_h", None):
            lib().qwm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
