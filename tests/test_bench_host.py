"""Host-side logic of bench.py that needs no GPU: the kernel source hash and
the DRAM traffic it takes from a committed ncu summary, which counts only
while the summary was taken on the current source of the kernel."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_kernel_source_hash_is_stable_and_per_kernel():
    a = bench.kernel_source_hash("fwd_tc.cu")
    assert a == bench.kernel_source_hash("fwd_tc.cu")
    assert re.fullmatch(r"[0-9a-f]{16}", a)
    assert a != bench.kernel_source_hash("bwd_tc.cu")


def test_profiled_traffic_needs_workload_and_source_to_match(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k_w.md").write_text(
        "# summary\n\n"
        "traffic_per_launch: workload=w1 bytes=123456 source=aaaa\n"
        "traffic_per_launch: workload=w2 bytes=777 source=bbbb\n")
    (prof / "ignored.csv").write_text("traffic_per_launch: workload=w1 bytes=1 source=aaaa\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda name: "aaaa")
    assert bench.profiled_traffic("fwd_tc.cu", "w1") == 123456
    # taken on another source of the kernel, or for another workload: no figure
    assert bench.profiled_traffic("fwd_tc.cu", "w2") is None
    assert bench.profiled_traffic("fwd_tc.cu", "w3") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda name: "cccc")
    assert bench.profiled_traffic("fwd_tc.cu", "w1") is None


def test_committed_summaries_carry_a_traffic_line():
    prof = os.path.join(ROOT, "profiles")
    pat = re.compile(r"traffic_per_launch:\s*workload=(\S+)\s+bytes=(\d+)\s+source=([0-9a-f]{16})")
    found = 0
    for fn in sorted(os.listdir(prof)):
        if fn.startswith(("fwd_tc_", "bwd_tc_")) and fn.endswith(".md"):
            text = open(os.path.join(prof, fn)).read()
            m = pat.search(text)
            assert m, f"{fn} has no traffic_per_launch line"
            assert int(m.group(2)) > 0
            found += 1
    assert found >= 4
