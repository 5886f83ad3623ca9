"""bench.py's measurement arithmetic on CPU: the HBM roofline of the dominant stage, the per-stage
record, and the oracle baseline's threaded runner (forward and backward timed separately)."""
import pytest

import bench
from bwd_ssm_conv_gb300.workloads import WORKLOADS, make_inputs, workload

PEAKS = {"hbm_gbs": 6000.0}


def test_roofline_is_hbm_bytes_over_time_against_the_measured_peak():
    w = workload(bench.DEFAULT_WORKLOAD)
    stage_ms = {"conv_fwd": 0.05, "scan_fwd": 0.2, "scan_bwd": 0.5, "conv_bwd": 0.1}
    r = bench.roofline_of(w, stage_ms, PEAKS, "measured", 152, 2000.0)
    tokens = w.n_seqs * w.n_tok
    D = w.channels
    # bf16, d_state 16, chunk 256: x dt z dy in, dx ddt dz out (14 D bytes), checkpoints
    # (0.25 D), B C in and dB dC out (4 x 16 x 2)
    per_tok = 14 * D + 0.25 * D + 4 * 16 * 2
    assert r["kernel"] == "ssm_scan_bwd" and r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_bytes_per_token"] == pytest.approx(per_tok)
    assert r["achieved"] == pytest.approx(per_tok * tokens / 0.5e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0)
    alu = r["alu"]
    assert alu["peak"] == pytest.approx(152 * 128 * 2 * 2000e6 / 1e12)
    assert alu["algorithmic_flops_per_launch"] == 20 * tokens * D * 16


def test_stage_record_fractions():
    w = workload(bench.DEFAULT_WORKLOAD)
    rec = bench.stage_record(w, {"scan_fwd": 0.1}, PEAKS)
    gbs = rec["stage_hbm_gbs"]["scan_fwd"]
    per_tok = (4 * w.channels) * 2 + 2 * 16 * 2 + 0.25 * w.channels
    assert gbs == pytest.approx(per_tok * w.n_seqs * w.n_tok / 0.1e-3 / 1e9, rel=1e-3)
    assert rec["stage_frac_of_measured"]["scan_fwd"] == pytest.approx(gbs / 6000.0, rel=1e-3)
    assert rec["stage_frac_of_8tbs"]["scan_fwd"] == pytest.approx(gbs / 8000.0, rel=1e-3)


def test_targets_are_the_two_long_bf16_configurations():
    assert bench.TARGET_WORKLOADS == (WORKLOADS[3].name, WORKLOADS[4].name)


@pytest.mark.parametrize("threads", [1, 3])
def test_oracle_runner_times_forward_and_backward(threads):
    w = WORKLOADS[0]  # 1 x 64 tokens, d_inner 16: milliseconds
    inp = make_inputs(w)
    slices = bench.oracle_slices(w, inp, w.n_seqs, 4)
    assert sum(s["H"] for s in slices) == w.n_head
    f, b = bench.oracle_run(w, slices, w.n_seqs, threads)
    assert f > 0 and b > 0
    rec = bench.oracle_baseline(w, inp, threads, budget_cpu_s=10.0)
    assert rec["cores"] == threads and rec["kind"] == "oracle"
    assert rec["value"] == pytest.approx(w.n_seqs * w.n_tok / (rec["fwd_s"] + rec["bwd_s"]))
    assert rec["fwd_tokens_s"] > rec["value"] and rec["bwd_tokens_s"] > rec["value"]


def test_forward_only_workload_has_no_backward_time():
    w = WORKLOADS[2].with_(n_seqs=1, n_tok=16, n_head=2)
    inp = make_inputs(w)
    f, b = bench.oracle_run(w, bench.oracle_slices(w, inp, 1, 2), 1, 2)
    assert f > 0 and b == 0.0


def test_oracle_sample_size_respects_the_budget():
    w = WORKLOADS[1]
    inp = make_inputs(w)
    seqs, per_seq = bench.oracle_seqs_for(w, inp, budget_cpu_s=1e-9)
    assert seqs == 1 and per_seq > 0
    seqs, _ = bench.oracle_seqs_for(w, inp, budget_cpu_s=1e9)
    assert seqs == w.n_seqs
