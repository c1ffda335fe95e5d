"""bench.py's host-side helpers on CPU: the DRAM traffic it reports comes from
a committed ncu summary only while that summary's recorded source hash matches
the kernel source; the whole-job value scales with the number of replicas."""
import hashlib
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _summary(tmp_path, sha, nbytes):
    p = tmp_path / "summary.md"
    p.write_text(f"Captured on kernel source `x.cu`,\nsource sha256: {sha}\n\ndram bytes per launch: {nbytes}\n")
    return str(p)


def test_traffic_only_for_the_captured_source(tmp_path):
    src = tmp_path / "kernel.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    assert bench.profiled_traffic(_summary(tmp_path, sha, 123456), str(src)) == 123456.0
    src.write_bytes(b"__global__ void k() { }\n")              # source changed since the capture
    assert bench.profiled_traffic(_summary(tmp_path, sha, 123456), str(src)) is None
    assert bench.profiled_traffic(str(tmp_path / "missing.md"), str(src)) is None


def test_committed_summaries_name_their_sources():
    """Every committed kernel summary that records a source hash also records
    a per-launch DRAM byte count in the machine-readable form, and names a
    source file that exists."""
    prof = os.path.join(ROOT, "profiles")
    csrc = os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc")
    for name in sorted(os.listdir(prof)):
        text = open(os.path.join(prof, name)).read()
        if "source sha256: " not in text:
            continue
        assert "dram bytes per launch: " in text, name
        src = re.search(r"bit_kv_cache_qwm_gb300/csrc/([a-z_0-9]+\.cu)", text)
        assert src and os.path.exists(os.path.join(csrc, src.group(1))), name
        got = bench.profiled_traffic(os.path.join(prof, name), os.path.join(csrc, src.group(1)))
        assert got is None or got > 0


def test_append_bytes_and_oracle_extrapolation():
    """641 B per token-head at d = 128 (bf16 k and v in, 129 B out), and the
    oracle sample's extrapolation scales each part by what it left out."""
    assert bench.append_bytes_per_token_head(128, 129) == 641
    wl = bench.synth.workload("tiny-f32-h1-n1024")
    smp = bench.oracle_sample(wl)
    spent, full, parts = bench.oracle_step(wl, smp)
    assert spent > 0 and full >= spent * 0.5
    assert abs(sum(parts.values()) - full) < 1e-9 * max(full, 1.0)


def test_whole_job_value_scales_with_replicas():
    one = bench.whole_job_tflops(1e12, 1, 2.0)
    assert bench.whole_job_tflops(1e12, 4, 2.0) == 4 * one
    assert one == 1e12 / 2e-3 / 1e12


def test_alu_roofline_of_the_exhaustive_search():
    """3 C d operations per token-head against 128 lanes x SMs x clock."""
    r = bench.alu_roofline(1e9, 256, 128, 152, 2070.0)
    assert r["ops_per_token_head"] == 3 * 256 * 128
    assert abs(r["peak"] - 128 * 152 * 2070e6 / 1e12) < 1e-9
    assert abs(r["frac"] - 1e9 * 3 * 256 * 128 / (128 * 152 * 2070e6)) < 1e-12
