"""CPU checks of the benchmark's host logic: the traffic line is taken from the profile summary
only while the kernel sources hash the same, the clock summary reads nvidia-smi's CSV rows
(median SM clock, throttle reasons), the default run keeps at least three warm-up steps, and the
parity summary of the bench line counts mismatches and near-ties."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_defaults_keep_three_warmup_steps():
    a = bench.parse_args([])
    assert a.warmup >= 3 and a.steps >= 1 and a.gpus == 1 and a.impl == "ours"
    assert a.workload == "single"


def _summary(path, digest, traffic):
    with open(path, "w") as f:
        f.write("# summary\n\n- kernel_source_sha256: `%s`\n- traffic_bytes_per_launch: %d\n" % (digest, traffic))


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    monkeypatch.setattr(bench, "KERNEL_SRCS", [str(src)])
    prof = tmp_path / "p.md"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(prof))
    digest = bench.kernel_source_hash()
    _summary(prof, digest, 135527765)
    assert bench.recorded_traffic() == 135527765
    src.write_text("kernel v2")                     # the kernel changed since the capture
    assert bench.recorded_traffic() is None
    prof.unlink()
    assert bench.recorded_traffic() is None


def test_committed_profile_has_the_machine_read_lines():
    text = open(bench.TRAFFIC_FILE).read()
    assert "kernel_source_sha256:" in text and "traffic_bytes_per_launch:" in text


def test_clock_summary_reads_samples_and_reasons():
    cs = bench.ClockSampler(0, log_path=os.devnull)
    cs.rows = [
        ["2026/12/02 20:00:00.000", "2032", "2032", "650.5", "0x0", "Not Active", "Not Active",
         "Not Active", "Not Active"],
        ["2026/12/02 20:00:00.200", "1552", "2032", "1090.9", "0x4", "Not Active", "Not Active",
         "Not Active", "Active"],
        ["2026/12/02 20:00:00.400", "1702", "2032", "1064.4", "0x4", "Not Active", "Not Active",
         "Not Active", "Active"],
    ]
    s = cs.summary()
    assert s["sm_mhz"] == pytest.approx(1702.0)
    assert s["sm_max_mhz"] == 2032.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3 and s["power_w_max"] == pytest.approx(1090.9)


def test_source_hash_ignores_comments(tmp_path, monkeypatch):
    src = tmp_path / "k.cuh"
    src.write_text("// kernel\nint f(int x) { return x + 1; }  // add one\n/* block */\n")
    monkeypatch.setattr(bench, "KERNEL_SRCS", [str(src)])
    h = bench.kernel_source_hash()
    src.write_text("// the kernel, described anew\n\nint f(int x) { return x + 1; }\n")
    assert bench.kernel_source_hash() == h
    src.write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_source_hash() != h


def test_parity_summary_counts_mismatches_and_near_ties():
    """The bench line's parity summary: a real sample mismatch, a near-tie mismatch (counted
    apart), an unmasked row's sample (ignored), an argmax mismatch and the selection test."""
    import types

    import bench
    L = 6
    res = types.SimpleNamespace(
        H=np.zeros((1, L)), A=np.arange(L)[None, :], Y=np.arange(L)[None, :] + 10,
        gap=np.array([[1.0, 1e-7, 1.0, 1.0, 1.0, 1.0]]),
        sum_margin=np.array([0.5]), order_margin=np.array([0.5]))
    H = np.full((1, L), 2e-6)
    A = res.A.copy()
    A[0, 5] = 0
    Y = res.Y.copy()
    Y[0, 0] += 1            # masked, clear gap: a mismatch
    Y[0, 1] += 1            # masked, gap below 1e-6: a near-tie
    Y[0, 2] += 1            # not masked: no sample is compared
    before = np.array([[1, 1, 0, 1, 1, 1]], np.uint8)
    after = np.array([[0, 1, 0, 1, 1, 1]], np.uint8)
    p = bench.parity_summary(H, A, Y, after, before, res, after.copy())
    assert p["rows"] == L and abs(p["max_abs_dH"] - 2e-6) < 1e-12
    assert p["argmax_mismatch"] == 1
    assert p["sample_mismatch"] == 1 and p["sample_ties"] == 1
    assert p["selection_equal"] and not p["canvas_tie"]
    other = after.copy()
    other[0, 3] = 0
    res.order_margin = np.array([1e-5])
    p = bench.parity_summary(H, A, Y, after, before, res, other)
    assert not p["selection_equal"] and p["canvas_tie"]
