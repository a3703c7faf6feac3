"""bench.py quotes an ncu capture's DRAM traffic only while the kernel sources it was taken
from are unchanged (a hash of them is stored beside the figure). No GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(path, sha, traffic):
    with open(path, "w") as f:
        f.write("# a capture\n\nsome text = not a key\n")
        f.write(f"- kernel_source_sha256 = {sha}\n- dram_bytes_per_launch = {traffic}\n")


def test_traffic_is_quoted_only_for_the_sources_it_was_taken_from(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.source_sha(["k.cu"])
    _write(prof / "k.md", sha, 12345)
    assert bench.profile_traffic("k.md", ["k.cu"]) == 12345.0
    src.write_text("__global__ void k() { /* changed */ }\n")  # the source moved on
    assert bench.profile_traffic("k.md", ["k.cu"]) is None
    assert bench.profile_traffic("missing.md", ["k.cu"]) is None
    _write(prof / "bad.md", bench.source_sha(["k.cu"]), "n/a")
    assert bench.profile_traffic("bad.md", ["k.cu"]) is None


def test_committed_profiles_parse():
    """Every committed summary carries both machine-readable keys."""
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        if not name.endswith(".md") or name == "decode_step_m1.md":  # a launch list only
            continue
        text = open(os.path.join(ROOT, "profiles", name)).read()
        assert "- kernel_source_sha256 = " in text, name
        assert "- dram_bytes_per_launch = " in text, name


def test_the_headline_profile_matches_the_current_sources():
    """The default workload's roofline traffic comes from a capture of the current kernel
    sources, and that capture read the weights once (14 008 320 algorithmic bytes per launch,
    plus the tensor-copy row pad and x: well under 2 % more)."""
    t = bench.profile_traffic("gemv_tma_ffn.md")
    assert t is not None
    assert 14008320 <= t <= 1.02 * 14008320
