"""Host logic of the benchmark's DRAM-traffic record: the recorded ncu counters
are reported only while the attention kernel's sources match the captured
version, compared without their comments (a comment edit does not change the
compiled kernel; any code edit does)."""
import json
import os
import shutil
import sys

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
import bench  # noqa: E402

SRC = ("vdit_attn.cu", "vdit_ptx.cuh")


def copy_tree(tmp_path):
    csrc = tmp_path / "block_sparse_video_frame_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in SRC:
        shutil.copy(os.path.join(bench.ROOT, "block_sparse_video_frame_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "attn_fwd_traffic.json"),
                tmp_path / "profiles" / "attn_fwd_traffic.json")
    return csrc


def test_committed_record_is_reported_only_for_its_sources():
    """While the record's source hash matches, the bench reports its counters;
    once the kernel's code has changed since the capture, it reports none."""
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "attn_fwd_traffic.json")))
    current = rec["source_sha256_16"] == bench.attn_kernel_source_hash()
    want = rec["dram_bytes_per_launch_captured"] if current else None
    assert bench.recorded_traffic(rec["captured_workload"]) == want
    for wl, v in rec["scaled_to"].items():
        assert bench.recorded_traffic(wl) == (v if current else None)
    assert bench.recorded_traffic("no_such_workload") is None


def test_comment_edit_keeps_and_code_edit_drops_the_record(tmp_path, monkeypatch):
    csrc = copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.attn_kernel_source_hash()
    # the copied record is made current for the copied sources
    rec_path = tmp_path / "profiles" / "attn_fwd_traffic.json"
    rec = json.loads(rec_path.read_text())
    rec["source_sha256_16"] = base
    rec_path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("sr720p") is not None
    f = csrc / "vdit_attn.cu"
    text = f.read_text()
    f.write_text("// a new comment line\n" + text.replace("\n", "   // trailing note\n", 3) + "\n\n")
    assert bench.attn_kernel_source_hash() == base
    assert bench.recorded_traffic("sr720p") is not None
    f.write_text(text.replace("constexpr int kStagesV = 3;", "constexpr int kStagesV = 4;"))
    assert bench.attn_kernel_source_hash() != base
    assert bench.recorded_traffic("sr720p") is None
