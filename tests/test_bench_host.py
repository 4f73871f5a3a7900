"""Host-side logic of bench.py (no GPU): the recorded DRAM traffic is
reported only while the sources of the workload's kernel family are the ones
it was captured on, and each family's hash covers exactly its sources."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(tmp_path, lines):
    p = tmp_path / "traffic.txt"
    p.write_text("# header\n" + "\n".join(lines) + "\n")
    return str(p)


def test_traffic_reported_only_for_matching_family_hash(tmp_path, monkeypatch):
    g, v = bench.kernel_source_hash("gemm"), bench.kernel_source_hash("gemv")
    assert g != v
    path = _write(tmp_path, [f"c2 source={g} dram_bytes_per_launch=123",
                             f"c4 source={v} dram_bytes_per_launch=456",       # wrong family
                             f"v1 source={v} dram_bytes_per_launch=789",
                             f"c5 source=0000000000000000 dram_bytes_per_launch=1"])
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", path)
    assert bench.profiled_traffic("c2") == 123
    assert bench.profiled_traffic("c4") is None
    assert bench.profiled_traffic("v1") == 789
    assert bench.profiled_traffic("c5") is None
    assert bench.profiled_traffic("c3") is None                                # no line


def test_missing_traffic_file_gives_none(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.txt"))
    assert bench.profiled_traffic("c2") is None


def test_family_sources_exist_and_cover_the_kernels():
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_masked_gb300", "csrc")
    for fam, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), (fam, n)
    # every kernel source file belongs to at least one family
    listed = {n for names in bench.KERNEL_SOURCES.values() for n in names}
    for n in os.listdir(csrc):
        if n.endswith((".cu", ".cuh")):
            assert n in listed, n
