"""The C-ABI library loads, exports every declared entry point, and its host
logic (layout, argument checks) is right.  No CUDA call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

from oracle import qwm_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    q.lib()
    return q


def declared_functions():
    src = open(os.path.join(ROOT, "include", "qwm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qwm_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(qwm):
    names = declared_functions()
    assert len(names) >= 15
    L = qwm.lib()
    for n in names:
        assert hasattr(L, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", qwm.LIB_PATH], capture_output=True, text=True).stdout
    for n in names:
        assert re.search(rf"\bT {n}$", out, flags=re.M), n
    assert set(qwm.EXPORTS) <= set(names)


@pytest.mark.parametrize("d,r,C", [(128, 16, 256), (64, 4, 16), (128, 0, 64), (128, 32, 1024), (128, 8, 256)])
def test_layout_matches_definition(qwm, d, r, C):
    cfg = qwm.make_config(heads=3, head_dim=d, rank=r, n_centroids=C, dtype="bf16", max_tokens=1000)
    L = qwm.qwm_sizes(cfg)
    want = O.tile_layout(d, r, C)
    assert L.tile_bytes == want["tile_bytes"]
    assert L.bytes_per_token == O.bytes_per_token(d, r, C)
    for name in ["idx", "kcode", "kqp", "e", "vcode", "vqp"]:
        assert getattr(L, "off_" + name) == want[name]
    assert L.max_tiles == 8
    assert L.cache_bytes == 3 * 8 * want["tile_bytes"]
    for f in ["st_status", "st_s", "st_w", "st_lambda", "st_energy", "st_centroids", "st_basis", "st_tiles", "st_iters"]:
        assert getattr(L, f) % 256 == 0
    assert L.state_bytes >= L.st_iters + 3 * 4


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, 2), ("head_dim", 0, 2), ("group", 16, 1), ("rank", -1, 1), ("rank", 129, 1),
    ("n_centroids", 0, 1), ("n_centroids", 1025, 1), ("dtype", 5, 1), ("max_tokens", 0, 1),
    ("max_versions", 0, 1), ("max_iter", 0, 1), ("oversample", -1, 1), ("heads", 0, 1), ("max_hist", 0, 1)])
def test_bad_config_is_rejected(qwm, field, value, status):
    cfg = qwm.make_config(heads=2, head_dim=128, rank=16, n_centroids=256)
    setattr(cfg, field, value)
    out = qwm.qwm_layout()
    assert qwm.lib().qwm_sizes(ctypes.byref(cfg), ctypes.byref(out)) == status


def test_create_rejects_null_and_misaligned_buffers(qwm):
    cfg = qwm.make_config(heads=2, head_dim=128, rank=16, n_centroids=256)
    h = ctypes.c_void_p()
    L = qwm.lib()
    assert L.qwm_create(ctypes.byref(cfg), None, None, None, ctypes.byref(h)) == 1
    assert L.qwm_create(ctypes.byref(cfg), ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1008),
                        ctypes.c_void_p(0x2000), ctypes.byref(h)) == 1
    assert h.value is None


def test_fault_injection_oom_fails_create_before_any_cuda_call(qwm, monkeypatch):
    """QWM_FAULT_INJECT=oom: qwm_create returns QWM_ERR_OOM after its argument
    checks and before any CUDA call (so this runs without a GPU: the buffer
    addresses are never touched), and leaves no context; invalid arguments
    are still reported as such."""
    cfg = qwm.make_config(heads=2, head_dim=128, rank=16, n_centroids=256)
    L = qwm.lib()
    monkeypatch.setenv("QWM_FAULT_INJECT", "oom")
    h = ctypes.c_void_p()
    fake = [ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)]
    assert L.qwm_create(ctypes.byref(cfg), *fake, ctypes.byref(h)) == 7      # QWM_ERR_OOM
    assert h.value is None
    assert L.qwm_create(ctypes.byref(cfg), None, None, None, ctypes.byref(h)) == 1
    monkeypatch.setenv("QWM_FAULT_INJECT", "launch")                      # not a create fault
    assert L.qwm_create(ctypes.byref(cfg), None, None, None, ctypes.byref(h)) == 1


def test_null_context_calls_fail_cleanly(qwm):
    L = qwm.lib()
    assert L.qwm_append(None, None, None, 10, None) == 1
    assert L.qwm_attend(None, None, 10, 0.0, None, None) == 1
    assert L.qwm_rewind(None, 0) == 1
    assert L.qwm_num_tokens(None) == -1
    assert L.qwm_destroy(None) == 0
    for s in range(9):
        assert L.qwm_status_string(s)


def test_static_calibration_and_kmeans_reject_host_tensors():
    """Host (CPU) tensors, wrong shapes and wrong output buffers are refused
    before the library is called, so no host pointer reaches a kernel."""
    import torch
    from bit_kv_cache_qwm_gb300 import qwm
    with pytest.raises(ValueError):
        qwm.qwm_calibrate_static(torch.zeros(2, 64, 128, dtype=torch.bfloat16), 16)
    with pytest.raises(ValueError):
        qwm.qwm_kmeans(torch.zeros(2, 300, 128, dtype=torch.bfloat16), torch.zeros(2, 16, dtype=torch.int32), 16)
    # output dictionary checks run before any device work: a host tensor is refused
    with pytest.raises(ValueError):
        qwm._out_tensor(torch.zeros(2, 128), "s", torch.float32, (2, 128), torch.device("cuda", 0))
    with pytest.raises(ValueError):
        qwm._device_tensor(torch.zeros(3), "x", (torch.float32,), 1)
