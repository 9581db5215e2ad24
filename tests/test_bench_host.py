"""Host-side logic of the benchmark, on the CPU: planted proposals accept exactly
the planned counts (checked with the oracle's acceptance rule), the clock summary
reads nvidia-smi's CSV and flags throttle reasons, the profiler traffic is
reported only while the GEMM sources match the ones it was captured on, and the
roofline peaks fall back when no measured file exists."""
import json
import os

import numpy as np
import pytest

import bench
from oracle import spec


@pytest.mark.parametrize("B,taus", [(16, [6, 7]), (16, [1]), (16, [4]), (10, [6, 7]), (4, [6, 7]), (2, [1, 2])])
def test_planted_proposals_accept_the_planned_count(B, taus):
    rng = np.random.default_rng(3)
    vocab, rounds = 50, 9
    streams = [rng.integers(0, vocab, size=rounds * B + B + 2) for _ in range(3)]
    props, accs = bench.plan_proposals(streams, taus, rounds, B, vocab)
    assert props.shape == (rounds, 3, max(B - 1, 1))
    for s, st in enumerate(streams):
        g = 1  # st[0] is the first token (the prefill's); st[g] is the token after the anchor
        for r in range(rounds):
            posterior = st[g: g + B]           # the target's greedy tokens at the block positions
            a = spec.count_leading_matches(props[r, s, : B - 1], posterior[: B - 1])
            assert a == accs[r, s] == min(taus[r % len(taus)], B) - 1
            g += a + 1


def test_clock_summary_reads_samples_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [
        "0, 1980, 2070, 900.1, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1100.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 1995, 2070, 1000.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = c.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1995 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler(0).summary()["samples"] == 0


def _fake_root(tmp_path, kernel_text, recorded_hash):
    csrc = tmp_path / "block_diffusion_speculative_ctx_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "gemm_tc.cu").write_text(kernel_text)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"wl": {"gemm_gate_up": {"source_hash": recorded_hash, "sources": ["gemm_tc.cu"],
                                 "dram_bytes_per_launch": 123.0}}}))


def test_traffic_only_while_the_kernel_is_unchanged(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _fake_root(tmp_path, "kernel v1", "0" * 16)
    assert bench.ncu_traffic("gemm_gate_up", "wl") is None             # recorded on other sources
    h = bench.kernel_source_hash(["gemm_tc.cu"])
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"wl": {"gemm_gate_up": {"source_hash": h, "sources": ["gemm_tc.cu"], "dram_bytes_per_launch": 123.0}}}))
    assert bench.ncu_traffic("gemm_gate_up", "wl") == 123.0
    assert bench.ncu_traffic("gemm_head", "wl") is None and bench.ncu_traffic("gemm_gate_up", "other") is None
    (tmp_path / "block_diffusion_speculative_ctx_gb300" / "csrc" / "gemm_tc.cu").write_text("kernel v2")
    assert bench.ncu_traffic("gemm_gate_up", "wl") is None             # the kernel changed since


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks()[-1] == "fallback"
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6782.0, "bf16_tflops": 1895.0, "bf16_tflops_sustained": 1725.0}))
    assert bench.measured_peaks() == (6782.0, 1895.0, 1725.0, "measured")


def test_committed_traffic_record_names_existing_sources():
    with open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")) as f:
        d = json.load(f)
    csrc = os.path.join(os.path.dirname(bench.__file__), "block_diffusion_speculative_ctx_gb300", "csrc")
    for wl in d.values():
        for e in wl.values():
            assert all(os.path.exists(os.path.join(csrc, f)) for f in e["sources"])
            assert e["dram_bytes_per_launch"] > 0


def test_oracle_baseline_is_one_sequence_at_a_time(monkeypatch):
    """The CPU oracle handles a batch sequence by sequence: its tokens/s at planted tau is
    tau over the time of one sequence's round, whatever the batch, and the line carries the
    draft / verify split of the median sample."""
    from synth import configs
    times = iter([(0.5, 0.1, 0.4), (0.3, 0.1, 0.2), (0.4, 0.1, 0.3)])

    def fake(w, ctx, state=None):
        s, td, tv = next(times)
        st = state or [None, None, None, None, [0.0, 0.0]]
        st[4][0], st[4][1] = td, tv
        return s, st

    monkeypatch.setattr(bench, "cpu_sample_round_s", fake)
    for batch in (1, 8):
        times = iter([(0.5, 0.1, 0.4), (0.3, 0.1, 0.2), (0.4, 0.1, 0.3)] + [(0.4, 0.1, 0.3)] * 5)
        b = bench.cpu_baseline(configs.get("qwen3_8b_b1_p512").with_(batch=batch), budget_s=0.0)
        assert b["kind"] == "oracle" and abs(b["value"] - 6.5 / b["s_per_round"]) < 1e-12
        assert b["s_per_round"] in (0.5, 0.4, 0.3)
        assert abs(b["t_draft_ms"] + b["t_verify_ms"] - 1e3 * b["s_per_round"]) < 1e-9
