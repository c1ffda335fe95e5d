"""Attention-shift diagnostics on synthetic data.

QuantWM Abstract: 2-bit keys have the smaller reconstruction error but the
larger output error, because small key perturbations change QK^T and shift
the tokens queries select.  roboind article: "The key to a smaller error ..."
(key-only vs value-only quantisation), Figure 2 (the highest-scoring
historical token moves) and Table 1 (the fraction of queries whose
highest-scoring historical token changes against BF16).

The caches are built by the library on the GPU (calibrate, append) for three
encodings of the same keys and values: nearest-centroid assignment without
compensation (the QVG-style baseline the pages compare with), QSAC without
compensation, and QSAC with PSAC (rank r); `qwm_dequantize` gives their
keys, values and coefficients in float32, and the comparisons against the
unquantised keys and values run here in torch (float32).  Measured per
encoding:
  top1_change        fraction of (head, query) pairs whose argmax token differs
  logit_rel_error    RMS(q.k - l_quant) / RMS(q.k) over all (query, token) pairs
  key_rel_error      ||K - K_hat|| / ||K||  (Frobenius, all heads)
  value_rel_error    ||V - V_hat|| / ||V||
  output_rel_error_key_only    O with quantised (compensated) keys, exact values
  output_rel_error_value_only  O with exact keys, quantised values
  output_rel_error             both quantised (what qwm_attend computes)

  python -m bit_kv_cache_qwm_gb300.diagnostics --workload bf16-h12-n32760 --heads 0,1,2,3 --rows 256

This module is a measurement tool, not part of the product path: its
comparisons run in eager torch on dequantised copies, and no library call
(calibrate, append, attend) uses it.
"""
import argparse
import json

import numpy as np
import torch

from . import synth

ENCODINGS = (("nearest", False), ("qsac", False), ("qsac", True))


def _rel(a, b):
    return float(torch.linalg.vector_norm(a - b) / torch.linalg.vector_norm(b))


def measure(ctx, K, V, q, sigma: float) -> dict:
    """The diagnostics of one cache (a qwm.Qwm context holding exactly the
    keys K and values V [H, N, d], in cache order) for query rows q [H, M, d]
    (float32 tensors on the context's device)."""
    L = q @ K.transpose(1, 2)                                   # exact logits [H, M, N]
    P = torch.softmax(sigma * L, dim=-1)
    O = P @ V
    kh, vh, e, valid = ctx.dequantize()
    kh, vh, e = kh[:, valid], vh[:, valid], e[:, valid]
    Lq = q @ kh.transpose(1, 2)
    if ctx.cfg.rank > 0:
        U = torch.from_numpy(ctx.get_calibration()["U"]).to(q.device).float()   # [H, r, d]
        Lq = Lq + (q @ U.transpose(1, 2)) @ e.transpose(1, 2)
    Pq = torch.softmax(sigma * Lq, dim=-1)
    return {
        "top1_change": float((Lq.argmax(dim=-1) != L.argmax(dim=-1)).float().mean()),
        "logit_rel_error": float(torch.sqrt(((L - Lq) ** 2).mean() / (L ** 2).mean())),
        "key_rel_error": _rel(kh, K),
        "value_rel_error": _rel(vh, V),
        "output_rel_error_key_only": _rel(Pq @ V, O),
        "output_rel_error_value_only": _rel(P @ vh, O),
        "output_rel_error": _rel(Pq @ vh, O),
    }


def run(workload: str, heads=None, rows: int = 256, n_chunks=None, device=None) -> dict:
    """The three encodings of the workload's keys and values (all appends, or
    the first n_chunks) for `rows` query rows of the given heads."""
    from . import qwm
    wl = synth.workload(workload)
    heads = list(range(wl.heads)) if heads is None else list(heads)
    H, d, C, r = len(heads), wl.head_dim, wl.n_centroids, wl.rank
    n_chunks = wl.n_chunks if n_chunks is None else n_chunks
    dev = torch.device("cuda", 0) if device is None else torch.device(device)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev, tdt)
    ks = [T(synth.keys(wl, ch, heads)) for ch in range(n_chunks)]
    vs = [T(synth.values(wl, ch, heads)) for ch in range(n_chunks)]
    K = torch.cat(ks, dim=1).float()
    V = torch.cat(vs, dim=1).float()
    q = T(synth.queries(wl, 0, heads, m=rows)).float()
    qh = T(synth.hist_queries(wl, 0, heads))
    kf = synth.kmeans_keys(wl, heads)
    init = np.stack([synth.kmeans_init_rows(wl, h, kf.shape[1], C) for h in heads]).astype(np.int32)
    cent = qwm.qwm_kmeans(T(kf), torch.from_numpy(init).to(dev), C, iters=25 if C <= 256 else 5)
    tiles = n_chunks * ((wl.chunk + 127) // 128)
    out = {"workload": wl.name, "heads": heads, "tokens": int(K.shape[1]), "query_rows": rows,
           "rank": r, "n_centroids": C, "encodings": {}}
    for assign, psac in ENCODINGS:
        rank = r if psac else 0
        ctx = qwm.Qwm(H, d, rank, C, dtype=wl.dtype, max_tokens=tiles * 128, max_hist=qh.shape[1], device=dev)
        ctx.set_centroids(cent)
        ctx.set_assignment(assign)
        ctx.calibrate(qh)
        for k, v in zip(ks, vs):
            ctx.append(k, v)
        res = measure(ctx, K, V, q, 1.0 / np.sqrt(d))
        assert ctx.status() == 0
        out["encodings"][f"{assign}{'+psac' if psac else ''}"] = res
        ctx.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="bf16-h12-n32760")
    ap.add_argument("--heads", default="", help="comma-separated head indices (default: all)")
    ap.add_argument("--rows", type=int, default=256)
    ap.add_argument("--chunks", type=int, default=0)
    a = ap.parse_args()
    heads = [int(x) for x in a.heads.split(",")] if a.heads else None
    print(json.dumps(run(a.workload, heads, a.rows, a.chunks or None)))


if __name__ == "__main__":
    main()
