"""bench.py's host-side helpers on CPU: the DRAM traffic it reports comes from
a committed ncu summary only while that summary's recorded source hash matches
the kernel source; the whole-job value scales with the number of replicas."""
import hashlib
import os
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
    """Every committed kernel summary that bench.py reads records a source hash
    and a per-launch DRAM byte count in the machine-readable form."""
    prof = os.path.join(ROOT, "profiles")
    for name, src in (("attend_tc2_bf16-h12-n32760.md", "attend_tc.cu"),
                      ("attend_small_bf16-h40-n98280-outlier_m16.md", "attend_small.cu")):
        path = os.path.join(prof, name)
        text = open(path).read()
        assert "source sha256: " in text and "dram bytes per launch: " in text, name
        got = bench.profiled_traffic(path, os.path.join(ROOT, "bit_kv_cache_qwm_gb300", "csrc", src))
        assert got is None or got > 0


def test_whole_job_value_scales_with_replicas():
    one = bench.whole_job_tflops(1e12, 1, 2.0)
    assert bench.whole_job_tflops(1e12, 4, 2.0) == 4 * one
    assert one == 1e12 / 2e-3 / 1e12
