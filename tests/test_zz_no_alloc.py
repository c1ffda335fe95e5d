"""qwm_calibrate_static: the calibration entry point for callers that cannot
allocate device memory (its scratch is an array compiled into the library).

It must give the same sensitivity, basis and eigenvalues as qwm_calibrate
(through a context with a caller workspace), within the calibration
tolerances used elsewhere, on two calls in a row (the second call reuses the
array the first one left behind).  This file runs last so that a failure here
does not hide the rest of the suite; it also passes on its own.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    return q


def _projector_distance(U1, U2):
    return np.linalg.norm(U1.T @ U1 - U2.T @ U2, 2)


@pytest.mark.parametrize("name,dtype,r", [("bf16-h12-n32760", "bf16", 16), ("tiny-f32-h1-n1024", "f32", 4)])
def test_static_calibration_matches_context_calibration(qwm, name, dtype, r):
    wl = synth.workload(name)
    qh_np = synth.hist_queries(wl, 0)
    qh = torch.from_numpy(qh_np).to("cuda", torch.bfloat16 if dtype == "bf16" else torch.float32)
    H, n_h, d = qh.shape
    ctx = qwm.Qwm(H, d, r, 16, dtype=dtype, max_tokens=128, max_hist=n_h)
    ctx.calibrate(qh)
    assert ctx.status() == 0
    ref = ctx.get_calibration()
    outs = []
    for _ in range(2):
        out = qwm.qwm_calibrate_static(qh, r)
        torch.cuda.synchronize()
        assert int(out["status"].item()) == 0
        outs.append({k: v.cpu().numpy() for k, v in out.items()})
    for o in outs:
        np.testing.assert_allclose(o["s"], ref["s"], rtol=1e-5, atol=1e-30)
        np.testing.assert_allclose(o["lambda"], ref["lambda"], rtol=1e-5, atol=1e-6 * ref["lambda"].max())
        np.testing.assert_allclose(o["energy"], ref["energy"], atol=1e-5)
        for h in range(H):
            assert _projector_distance(o["U"][h].astype(np.float64), ref["U"][h].astype(np.float64)) <= 1e-4
    # the second call, on the array the first one left behind, gives the same result
    for k in outs[0]:
        assert np.array_equal(outs[0][k], outs[1][k]), k


def test_static_calibration_rejects_oversized_requests(qwm):
    """At d = 128 one split of partial sums plus A^2 is 128 KiB per head: 63
    heads fit in the 8 MiB array, 64 do not (rejected before any launch)."""
    q = torch.zeros((64, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(qwm.QwmError) as e:
        qwm.qwm_calibrate_static(q, 16)
    assert e.value.status == 3
    out = qwm.qwm_calibrate_static(q[:63], 16)
    torch.cuda.synchronize()
    assert (out["s"] == 0).all() and torch.isfinite(out["U"]).all()
