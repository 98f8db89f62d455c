"""Host logic of bench.py without a GPU: the per-kernel source hash that ties a
committed ncu traffic figure to the sources it was taken on, the parsing of
that figure, and the single-rank timing helpers."""
import os
import shutil

import bench

CSRC = os.path.join(bench.ROOT, "linear_attention_recurrence_chunk_gb300", "csrc")
CHAIN_MARK = "// -------------------------------------------------------------- chain kernel"


def _copy(tmp_path):
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d)
    return str(d)


def test_prep_hash_ignores_the_chain_sections_only(tmp_path):
    d = _copy(tmp_path)
    base = bench._kernel_src_sha("chunk_prep_tc", d)
    assert base == bench._kernel_src_sha("chunk_prep_tc", CSRC)
    f = os.path.join(d, "kda_chunk_tc.cu")
    text = open(f, encoding="utf-8").read()
    i = text.index(CHAIN_MARK) + len(CHAIN_MARK)
    open(f, "w", encoding="utf-8").write(text[:i] + "\n// a change in the chain kernels" + text[i:])
    assert bench._kernel_src_sha("chunk_prep_tc", d) == base           # chain edits keep the figure
    assert bench._kernel_src_sha("", d) != bench._kernel_src_sha("", CSRC)   # the whole-library hash moves
    j = text.index("__global__ void __launch_bounds__(kPrepTcThreads, 1)")
    open(f, "w", encoding="utf-8").write(text[:j] + "// a change in the prep kernel\n" + text[j:])
    assert bench._kernel_src_sha("chunk_prep_tc", d) != base           # prep edits void it
    open(os.path.join(d, "tc_ptx.cuh"), "a").write("\n// shared header\n")
    open(f, "w", encoding="utf-8").write(text)
    assert bench._kernel_src_sha("chunk_prep_tc", d) != base           # so do shared-header edits


def test_traffic_line_parsing(tmp_path):
    d = _copy(tmp_path)
    sha = bench._kernel_src_sha("chunk_prep_tc", d)
    p = tmp_path / "profiles"
    p.mkdir()
    (p / "x.md").write_text(f"text\ntraffic: kernel=chunk_prep_tc dram_bytes_per_unit=2000.5 src_sha={sha}\n")
    assert bench._traffic_from_profiles("chunk_prep_tc", 10, str(p), d) == 20005.0
    (p / "x.md").write_text("traffic: kernel=chunk_prep_tc dram_bytes_per_unit=2000.5 src_sha=0123456789abcdef\n")
    assert bench._traffic_from_profiles("chunk_prep_tc", 10, str(p), d) is None   # stale: no figure
    assert bench._traffic_from_profiles("chunk_chain_tc", 10, str(p), d) is None


def test_single_rank_helpers():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.min_over_ranks(2.0, 1) == 2.0
    assert abs(bench.job_throughput(1000.0, 4, 2.0, 1) - 1000.0 * 4 / 0.002) < 1e-6
