"""The committed ncu summaries and how the bench uses them.

Each summary under profiles/ names the hash of the kernel source it was taken on; the
bench reads DRAM traffic from a summary only while that hash matches, and reports null
traffic once the kernel has changed.  These CPU tests check the fields the bench reads
and that a summary names the command that made it.
"""
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tree_speculative_decoding_tv_gb300", "csrc")

# kernel name -> the source file that defines it
SOURCES = {
    "tree_attn_kernel": "tv_attn.cu",
    "tree_attn_merge_kernel": "tv_attn.cu",
    "argmax_span_kernel": "tv_accept.cu",
    "argmax_rows_kernel": "tv_accept.cu",
    "accept_kernel": "tv_accept.cu",
    "build_mask_kernel": "tv_mask.cu",
    "kv_commit_kernel": "tv_commit.cu",
    "gdn_tree_kernel": "tv_gdn.cu",
    "gdn_commit_kernel": "tv_gdn_commit.cu",
    "build_tree_kernel": "tv_tree.cu",
}

SUMMARIES = sorted(p for p in glob.glob(os.path.join(ROOT, "profiles", "*.md"))
                   if os.path.basename(p).split("_config")[0].split("_gdn")[0] in SOURCES)


def _fields(path):
    text = open(path).read()
    return text, dict(line.split(":", 1) for line in text.splitlines()
                      if re.match(r"^(source_sha256_16|traffic_bytes_per_launch|algorithmic_bytes_per_launch):", line))


def test_there_are_kernel_summaries():
    names = {os.path.basename(p) for p in SUMMARIES}
    # every kernel of the library has a summary on the workload it was captured on
    for kernel in SOURCES:
        assert any(n.startswith(kernel + "_") for n in names), kernel


@pytest.mark.parametrize("path", SUMMARIES, ids=[os.path.basename(p) for p in SUMMARIES])
def test_summary_fields(path):
    text, f = _fields(path)
    assert re.fullmatch(r"[0-9a-f]{16}", f.get("source_sha256_16", "").strip())
    assert float(f["traffic_bytes_per_launch"]) > 0
    assert "--clock-control none" in text  # the capture left the clocks alone
    assert "ncu " in text                  # and the summary names the command that made it


def test_launch_list_summary_names_its_command():
    text = open(os.path.join(ROOT, "profiles", "launches_bench_config5.md")).read()
    assert "--metrics gpu__time_duration.sum --clock-control none" in text
    assert "share of ours" in text


def test_bench_reads_traffic_only_from_a_matching_summary(tmp_path, monkeypatch):
    import bench
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda name: "0123456789abcdef" if name == "tv_attn.cu" else "x")
    (tmp_path / "profiles" / "tree_attn_kernel_config5.md").write_text(
        "ncu --clock-control none\nsource_sha256_16: 0123456789abcdef\ntraffic_bytes_per_launch: 123.5\n")
    assert bench.profiled_traffic("tree_attn_kernel", "tv_attn.cu", 5) == 123.5
    # the same summary against another source's hash does not match: no traffic
    assert bench.profiled_traffic("tree_attn_kernel", "tv_mask.cu", 5) is None
    # no summary for a workload: no traffic
    assert bench.profiled_traffic("tree_attn_kernel", "tv_attn.cu", 9) is None


def test_peaks_fall_back_when_the_measured_file_is_missing(monkeypatch, tmp_path):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, source = bench.load_peaks()
    assert source.startswith("fallback")
    assert peaks == bench.FALLBACK_PEAKS
