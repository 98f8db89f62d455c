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
    d2 = _copy(tmp_path / "b")
    open(os.path.join(d2, "prep_split_body.cuh"), "a").write("\n// the two-stream prep body\n")
    assert bench._kernel_src_sha("chunk_prep_tc", d2) != base          # and edits of the prep body's header


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


def test_algorithmic_bytes_of_the_prefill_workloads():
    """The roofline numerators: q, k, g, v, o at 2 bytes and beta at 4 per
    head-token (1284 B at d = 128), plus 128 KiB per (sequence, head) for each
    state read or written; the prep kernel is charged its inputs (1028 B per
    head-token), the chain kernels o and the states."""
    import kda_synth as ks

    wl = ks.workloads()
    w1 = wl["prefill_b1_h32_t65536_d128"]            # S0 given: read and written
    ht = 65536 * 32
    assert bench.prefill_alg_bytes(w1, "path") == ht * 1284 + 2 * 32 * 128 * 128 * 4 == 2_696_937_472
    assert bench.prefill_alg_bytes(w1, "chunk_prep_tc") == ht * 1028
    assert bench.prefill_alg_bytes(w1, "chunk_chain_tc") == ht * 256 + 2 * 32 * 128 * 128 * 4
    w2 = wl["prefill_b8_h96_t8192_d128"]             # no S0: final states written only
    assert bench.prefill_alg_bytes(w2, "path") == 8 * 8192 * 96 * 1284 + 8 * 96 * 128 * 128 * 4
    w4 = wl["varlen_12seq_1m_h32_d128"]
    assert abs(bench.prefill_alg_bytes(w4, "path") - 4.31e10) / 4.31e10 < 0.01
