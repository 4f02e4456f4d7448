"""The benchmark's byte accounting and its ncu-summary lookup (CPU only)."""

import pytest

import bench
import kda_inputs


def test_algorithmic_bytes_of_the_headline_launch():
    # q, k 32,768; g 32,768; beta 256; ten lower 16x16 dA blocks x 2 = 20,480;
    # dq, dk, dg 98,304; db 256
    assert bench.algorithmic_bytes_per_unit() == 184832
    assert kda_inputs.CONFIGS[kda_inputs.HEADLINE].units * bench.algorithmic_bytes_per_unit() == 1514143744


def test_option_bytes():
    base = bench.algorithmic_bytes_per_unit()
    assert bench.algorithmic_bytes_per_unit(accumulate=True) - base == 3 * 64 * 128 * 4 + 64 * 4
    assert base - bench.algorithmic_bytes_per_unit(io_out=True) == 2 * 64 * 128 * 2
    assert base - bench.algorithmic_bytes_per_unit(group=4) == 2 * 64 * 128 * 2 * 3 / 4
    assert bench.FWD_BYTES_PER_UNIT == 98560


@pytest.mark.parametrize("lens", [[64], [128, 64], [320]])
def test_varlen_bytes_of_whole_chunks_equal_the_fixed_length_count(lens):
    chunks = sum(n // 64 for n in lens)
    for acc in (False, True):
        assert bench.varlen_algorithmic_bytes(lens, 3, accumulate=acc) == \
            3 * chunks * bench.algorithmic_bytes_per_unit(accumulate=acc)


def test_varlen_bytes_of_a_short_chunk():
    # 20 valid rows: per-row tensors for 20 rows, and the lower-block part of their dA
    # rows (rows 0..15 read one 16-wide block, rows 16..19 two)
    per_row = (2 * 128 * 2 + 128 * 4 + 4      # q, k (bf16), g, beta
               + 3 * 128 * 4 + 4)             # dq, dk, dg, db (fp32)
    da = 2 * 4 * (16 * 16 + 4 * 32)
    assert bench.varlen_algorithmic_bytes([20], 1) == 20 * per_row + da


def test_traffic_is_null_when_the_summary_is_for_other_sources(monkeypatch):
    name, workload = "kda_intra_bwd_tc_kernel", kda_inputs.CONFIGS[kda_inputs.HEADLINE].name
    current = bench.ncu_traffic(name, workload)
    if current is None:
        pytest.skip("the committed summary predates the current sources")
    assert current > 0.9 * kda_inputs.CONFIGS[kda_inputs.HEADLINE].units * bench.algorithmic_bytes_per_unit()
    monkeypatch.setattr(bench, "source_hash", lambda kernel: "0" * 16)
    assert bench.ncu_traffic(name, workload) is None


def test_option_launches_find_their_own_summaries():
    """The split-TF32, factor_diag and variable-length launches of the backward report
    the traffic of their own summaries; other options and combinations report none."""
    import argparse
    base = dict(gva=1, accumulate=False, fold_dg=False, io_dtype_out=False, varlen=False,
                factor_diag=False, split_tf32=False, path="kda_intra_bwd")
    a = lambda **kw: argparse.Namespace(**{**base, **kw})  # noqa: E731
    w = kda_inputs.CONFIGS[kda_inputs.HEADLINE].name
    assert bench.summary_name(a(), w) == w
    assert bench.summary_name(a(path="kda_intra_fwd"), w) == w
    assert bench.summary_name(a(split_tf32=True), w) == "split_tf32_" + w
    assert bench.summary_name(a(factor_diag=True), w) == "factor_diag_" + w
    assert bench.summary_name(a(varlen=True), "varlen_T32768_H16") == "varlen_T32768_H16"
    for kw in (dict(gva=4), dict(accumulate=True), dict(fold_dg=True), dict(io_dtype_out=True),
               dict(varlen=True, factor_diag=True), dict(varlen=True, path="kda_intra_fwd")):
        assert bench.summary_name(a(**kw), w) is None, kw
    # each named summary exists and is for the current sources
    for summary in (w, "split_tf32_" + w, "factor_diag_" + w, "varlen_T32768_H16"):
        traffic = bench.ncu_traffic("kda_intra_bwd_tc_kernel", summary)
        if traffic is None:
            pytest.skip("a committed summary predates the current sources")
        assert traffic > 0.9 * 1.5e9


def test_source_hash_sees_code_only():
    """A kernel's hash (which ties an ncu summary to its sources) ignores comments and
    blank lines, keeps literals, and changes with the code."""
    a = "int x = 1; // one\n/* two\n lines */\nint y;\n"
    b = "int x = 1;\n\n// another comment\n   \nint y;   \n"
    assert bench.code_only(a) == bench.code_only(b) == "int x = 1;\nint y;"
    assert bench.code_only("int x = 2;") != bench.code_only("int x = 1;")
    s = 'const char *s = "// kept /* too */"; char c = \'/\';'
    assert bench.code_only(s) == s
    for kernel in bench.KERNEL_SOURCES:
        assert len(bench.source_hash(kernel)) == 16


def test_config_selection():
    assert bench.parse_configs("2") == [kda_inputs.HEADLINE]
    assert bench.parse_configs("gate_stress") == [kda_inputs.GATE_STRESS]
    assert bench.parse_configs("long_B1_T32768_H32") == [kda_inputs.LONG]
    assert bench.parse_configs("all") == list(range(len(kda_inputs.CONFIGS)))
    for bad in ("9", "-1", "nope"):
        with pytest.raises(ValueError):
            bench.parse_configs(bad)


def test_small_workloads_are_timed_with_an_l2_flush():
    """The single-chunk and small workloads fit in the L2 and are flushed between calls;
    the others exceed twice the L2 and run back to back."""
    import types
    args = types.SimpleNamespace(gva=1, varlen=False, accumulate=False, io_dtype_out=False)
    fits = [bench.launch_bytes(args, c, 2, False) < 2 * bench.L2_BYTES for c in kda_inputs.CONFIGS]
    assert fits == [True, True, False, False, False]


def test_fallback_peak_is_the_nominal_hbm_rate():
    assert bench.FALLBACK_HBM_GBS == 8000.0
