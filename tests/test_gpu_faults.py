"""Failure paths on the GPU without a GPU fault.

* Host-side injection (QWM_FAULT_INJECT, read by the library at every call):
  `launch` makes every launching call return QWM_ERR_CUDA before it launches,
  with the context unchanged, so that after the variable is cleared the same
  calls produce exactly the cache of a context that never failed; `oom` makes
  context creation fail.
* The QWM_DEBUG_BOUNDS build (libqwm_dbg.so): a cache slot whose centroid
  index byte names a centroid beyond the table (planted in the cache bytes)
  is reported through the status bit QWM_DEV_BOUNDS and read as centroid 0 by
  every attention kernel and by qwm_dequantize.  This runs in a child process
  that loads only the checking build; the regular library never sees the
  planted byte.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import calibration, centroids

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    return q


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)


def _context(qwm, name, heads):
    wl = synth.workload(name)
    cent = centroids(name, tuple(heads))
    ctx = qwm.Qwm(len(heads), wl.head_dim, wl.rank, wl.n_centroids, dtype="bf16", max_tokens=8 * 128,
                  max_versions=2)
    ctx.set_centroids(_bf16(cent))
    s, U = calibration(name, tuple(heads))
    ctx.set_calibration(s, U)
    return wl, ctx


def test_launch_fault_leaves_the_context_unchanged(qwm, monkeypatch):
    name, heads = "bf16-h12-n32760", [0, 1]
    wl, ctx = _context(qwm, name, heads)
    _, ref = _context(qwm, name, heads)
    k0, v0 = _bf16(synth.keys(wl, 0, heads, 300)), _bf16(synth.values(wl, 0, heads, 300))
    k1, v1 = _bf16(synth.keys(wl, 1, heads, 200)), _bf16(synth.values(wl, 1, heads, 200))
    q = _bf16(synth.queries(wl, 0, heads, m=100))
    for c in (ctx, ref):
        c.append(k0, v0)
    n0, v_before = ctx.n_tokens, ctx.version
    monkeypatch.setenv("QWM_FAULT_INJECT", "launch")
    for call in (lambda: ctx.append(k1, v1), lambda: ctx.attend(q), lambda: ctx.calibrate(q),
                 lambda: ctx.dequantize()):
        with pytest.raises(qwm.QwmError) as e:
            call()
        assert e.value.status == 6                       # QWM_ERR_CUDA, nothing launched
    assert ctx.n_tokens == n0 and ctx.version == v_before
    monkeypatch.delenv("QWM_FAULT_INJECT")
    ctx.append(k1, v1)
    ref.append(k1, v1)
    torch.cuda.synchronize()
    assert ctx.n_tokens == ref.n_tokens == 500
    nt = ctx.n_tiles
    assert torch.equal(ctx.cache_tiles()[:, :nt], ref.cache_tiles()[:, :nt])
    assert torch.equal(ctx.tile_table()[:nt], ref.tile_table()[:nt])
    assert torch.equal(ctx.attend(q), ref.attend(q))
    assert ctx.status() == 0


def test_oom_fault_on_create(qwm, monkeypatch):
    monkeypatch.setenv("QWM_FAULT_INJECT", "oom")
    with pytest.raises(qwm.QwmError) as e:
        qwm.Qwm(2, 128, 16, 256, dtype="bf16", max_tokens=256)
    assert e.value.status == 7                           # QWM_ERR_OOM
    monkeypatch.delenv("QWM_FAULT_INJECT")
    ctx = qwm.Qwm(2, 128, 16, 256, dtype="bf16", max_tokens=256)
    assert ctx.n_tokens == 0


def test_bounded_wait_runs_out_and_the_context_stays_usable(qwm):
    """A wait on an mbarrier that nothing arrives at (the attention kernels'
    bounded wait, limited to ~2^20 SM cycles here) gives up, reports
    QWM_DEV_TIMEOUT in the status word it was handed, and the kernel returns:
    the CUDA context then runs a full calibrate / append / attend as usual."""
    assert qwm.selftest_wait_timeout(1 << 20) == qwm.DEV_TIMEOUT
    name, heads = "bf16-h12-n32760", [0, 1]
    wl, ctx = _context(qwm, name, heads)
    ctx.append(_bf16(synth.keys(wl, 0, heads, 300)), _bf16(synth.values(wl, 0, heads, 300)))
    out = ctx.attend(_bf16(synth.queries(wl, 0, heads, m=100)))
    assert torch.isfinite(out.float()).all() and ctx.status() == 0


_CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
from bit_kv_cache_qwm_gb300 import qwm, synth
from cases import calibration, centroids
assert qwm.LIB_PATH.endswith("libqwm_dbg.so"), qwm.LIB_PATH
name, heads = "bf16-h12-n32760", (0,)
wl = synth.workload(name)
C = 16
cent = centroids(name, heads, C, iters=5)
def t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)
ctx = qwm.Qwm(1, 128, 16, C, dtype="bf16", max_tokens=3 * 128)
ctx.set_centroids(t(cent))
s, U = calibration(name, heads)
ctx.set_calibration(s, U)
ctx.append(t(synth.keys(wl, 0, list(heads), 300)), t(synth.values(wl, 0, list(heads), 300)))
q_large = t(synth.queries(wl, 0, list(heads), m=130))
q_small = t(synth.queries(wl, 0, list(heads), m=16))
kernels = [(k, q_large) for k in (1, 2, 3, 4, 6)] + [(5, q_small)]
clean = {}
for k, q in kernels:
    ctx.set_attend_kernel(k)
    clean[k] = ctx.attend(q).float()
    assert ctx.status_bits() == 0, k
# plant an index beyond the table in slot 5 of tile 0 (the idx section starts the tile)
L = ctx.layout
ctx.cache.view(-1)[L.off_idx + 5] = 200
torch.cuda.synchronize()
for k, q in kernels:
    ctx.set_attend_kernel(k)
    got = ctx.attend(q).float()
    bits = ctx.status_bits()
    assert bits == qwm.DEV_BOUNDS, (k, bits)
    assert torch.isfinite(got).all(), k
    # the planted slot now reads centroid 0: the output moves, stays finite
khat, vhat, e, valid = ctx.dequantize()
assert ctx.status_bits() == 0       # qwm_dequantize clamps in every build
assert torch.isfinite(khat).all()
print("debug-bounds ok")
"""


def test_debug_bounds_build_flags_a_planted_index():
    from bit_kv_cache_qwm_gb300 import build
    build.build(debug_bounds=True)
    env = dict(os.environ, QWM_DEBUG_BOUNDS="1")
    env.pop("QWM_FAULT_INJECT", None)
    res = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True, text=True,
                         timeout=600)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
    assert "debug-bounds ok" in res.stdout
