"""qwm_calibrate's eigen-solver runs on the context's own stream, forked after
the Gram sums and group weights; qwm_append quantises at once and computes the
PSAC coefficients after the join, qwm_attend joins first.  The cache bytes and
the attention output of that path must equal those of the same appends after
qwm_set_calibration with the same sensitivity and basis (nothing pending).
The eigen-solver takes longer than the quantisation of these chunks, so a
missing join would leave coefficients computed from a basis slot not yet
written."""
import numpy as np
import pytest
import torch

from bit_kv_cache_qwm_gb300 import synth
from cases import centroids

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qwm():
    from bit_kv_cache_qwm_gb300 import build
    build.build()
    from bit_kv_cache_qwm_gb300 import qwm as q
    return q


def _t(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to("cuda", torch.bfloat16)


def test_overlapped_calibration_matches_host_calibration(qwm):
    name = "bf16-h12-n32760"
    wl = synth.workload(name)
    heads = [0, 1, 2, 3]
    H, d, r, C = len(heads), wl.head_dim, wl.rank, wl.n_centroids
    cent = _t(centroids(name, tuple(heads)))
    qh = [_t(synth.hist_queries(wl, step, heads)) for step in range(2)]
    ks = [_t(synth.keys(wl, ch, heads)) for ch in range(2)]
    vs = [_t(synth.values(wl, ch, heads)) for ch in range(2)]
    q = _t(synth.queries(wl, 0, heads, m=300))

    def make():
        ctx = qwm.Qwm(H, d, r, C, dtype="bf16", max_tokens=2 * 37 * 128, max_versions=2, max_hist=wl.n_hist)
        ctx.set_centroids(cent)
        return ctx

    # calibrations alone, read back (each read joins its own eigen-solver)
    cals = []
    for step in range(2):
        c = make()
        c.calibrate(qh[step])
        cals.append(c.get_calibration())
        c.close()
    # overlapped path: calibrate, append, calibrate, append, attend
    a = make()
    for step in range(2):
        a.calibrate(qh[step])
        a.append(ks[step], vs[step])
    out_a = a.attend(q)
    # host-calibrated path
    b = make()
    for step in range(2):
        b.set_calibration(cals[step]["s"], cals[step]["U"])
        b.append(ks[step], vs[step])
    out_b = b.attend(q)
    torch.cuda.synchronize()
    assert a.status() == 0 and b.status() == 0
    n = a.n_tiles
    assert n == b.n_tiles == 2 * 37
    assert torch.equal(a.cache_tiles()[:, :n], b.cache_tiles()[:, :n])
    assert torch.equal(out_a, out_b)
