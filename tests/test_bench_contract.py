"""Host-side pieces of bench.py's contract: the recorded DRAM traffic is used
only while the kernel sources it was measured on are unchanged."""

import os
import shutil

import bench
from draft_sampling_lossless_gb300 import synth


def test_recorded_traffic_matches_the_committed_sources():
    wl = synth.WORKLOADS["qwen3_4b"]
    t = bench.recorded_traffic("draft_persistent_tc", wl)
    # the committed capture exists and is at least the algorithmic bytes
    # (z once per position and W once)
    if t is not None:
        alg = wl.R * wl.gamma * wl.V * 2 + wl.r * wl.V * 2
        assert t >= alg


def test_recorded_traffic_is_dropped_when_a_source_changes(tmp_path, monkeypatch):
    wl = synth.WORKLOADS["qwen3_4b"]
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    shutil.copytree(os.path.join(bench.ROOT, "draft_sampling_lossless_gb300", "csrc"),
                    root / "draft_sampling_lossless_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    before = bench.recorded_traffic("draft_persistent_tc", wl)
    src = root / "draft_sampling_lossless_gb300" / "csrc" / "draft_tc.cu"
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench.recorded_traffic("draft_persistent_tc", wl) is None
    assert bench.recorded_traffic("no_such_kernel", wl) is None
    if before is not None:
        src.write_text(src.read_text()[: -len("\n// edited\n")])
        assert bench.recorded_traffic("draft_persistent_tc", wl) == before
