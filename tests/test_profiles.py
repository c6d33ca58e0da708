"""The committed ncu summaries describe the kernels as they are.

Each summary under profiles/ names the hash of the kernel source it was taken on; the
bench reads DRAM traffic from a summary only while that hash matches.  These CPU tests
keep every summary in step with its source and check the fields the bench reads.
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
    "argmax_rows_kernel": "tv_accept.cu",
    "gdn_tree_kernel": "tv_gdn.cu",
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
    for want in ("tree_attn_kernel_config2.md", "argmax_rows_kernel_config2.md", "gdn_tree_kernel_gdn128.md"):
        assert want in names


@pytest.mark.parametrize("path", SUMMARIES, ids=[os.path.basename(p) for p in SUMMARIES])
def test_summary_matches_its_source(path):
    import bench
    kernel = os.path.basename(path).split("_config")[0].split("_gdn")[0]
    text, f = _fields(path)
    assert f.get("source_sha256_16", "").strip() == bench.source_hash(SOURCES[kernel]), \
        f"{os.path.basename(path)} was taken on another version of {SOURCES[kernel]}"
    assert float(f["traffic_bytes_per_launch"]) > 0
    assert "--clock-control none" in text  # the capture left the clocks alone
    assert "ncu " in text                  # and the summary names the command that made it


def test_launch_list_summary_names_its_command():
    text = open(os.path.join(ROOT, "profiles", "launches_bench_config2.md")).read()
    assert "--metrics gpu__time_duration.sum --clock-control none" in text
    assert "share of ours" in text


def test_bench_reads_traffic_only_from_a_matching_summary(tmp_path, monkeypatch):
    import bench
    # the committed summary of the attention kernel matches its source: its traffic is read
    assert bench.profiled_traffic("tree_attn_kernel", "tv_attn.cu", 2) > 0
    # the same summary against another source file does not match: no traffic
    assert bench.profiled_traffic("tree_attn_kernel", "tv_mask.cu", 2) is None
    # no summary for a workload: no traffic
    assert bench.profiled_traffic("tree_attn_kernel", "tv_attn.cu", 9) is None


def test_peaks_fall_back_when_the_measured_file_is_missing(monkeypatch, tmp_path):
    import bench
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, source = bench.load_peaks()
    assert source.startswith("fallback")
    assert peaks == bench.FALLBACK_PEAKS
