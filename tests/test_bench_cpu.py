"""bench.py's host arithmetic on CPU: the algorithmic bytes that the roofline
fractions divide by, the whole-job throughput, and the rule that a DRAM
traffic figure is reported only for the kernel sources it was measured on.

The byte counts are pinned to the per-element rule of the hot path (bf16:
u, delta, z read and y written, 8 B per B*L*D element forward; u, delta, z,
dy read as bf16 and du, ddelta, dz written as f32, 20 B backward) plus the
per-(b, t, n) and per-(d, n) terms, written out here for the headline sizes
as plain integers (rounded: 673.8 MB forward, 1681.6 MB backward).
"""

import pytest

import bench
from mamba_selective_scan_fwd_gb300 import build
from mamba_selective_scan_fwd_gb300.inputs import Workload


def test_headline_algorithmic_bytes():
    w = bench.pick_workload("mamba2.8b-layer-bf16")
    assert (w.Bsz, w.L, w.Dch, w.N, w.io) == (4, 4096, 5120, 16, "bf16")
    fwd, bwd = bench.algorithmic_bytes(w)
    # 83,886,080 elements; B, C rows 262,144 values each; A 81,920; D and bias 5,120 each; last_state 327,680
    assert fwd == 8 * 83_886_080 + 2 * 2 * 262_144 + 4 * (81_920 + 2 * 5_120) + 4 * 327_680 == 673_816_576
    # backward: B, C read (io) and dB, dC written (f32); A, D, bias read and dA, dD, dbias written (f32)
    assert bwd == 20 * 83_886_080 + 2 * 262_144 * (2 + 4) + 8 * (81_920 + 2 * 5_120) == 1_681_604_608
    assert round(fwd / 1e6, 1) == 673.8 and round(bwd / 1e6, 1) == 1681.6


@pytest.mark.parametrize("io,e", [("f32", 4), ("bf16", 2), ("f16", 2)])
def test_io_element_size(io, e):
    w = Workload("probe", 1, 10, 3, 2, io)
    fwd, bwd = bench.algorithmic_bytes(w)
    bld, bln, small = 30, 20, 2 * 3 + 3 * 2
    assert fwd == 4 * bld * e + 2 * bln * e + 4 * small + 4 * 1 * 3 * 2
    assert bwd == 4 * bld * e + 12 * bld + 2 * bln * (e + 4) + 8 * small


def test_job_throughput_is_all_ranks_over_the_slowest():
    # 3 ranks of 1e6 units each, the slowest took 2 ms
    assert bench.job_throughput(1e6, 3, 2.0) == pytest.approx(1.5e9)


def test_traffic_reported_only_for_its_sources(monkeypatch):
    w = bench.pick_workload("mamba2.8b-layer-bf16")
    monkeypatch.setattr(build, "source_digest", lambda: bench.TRAFFIC_SRC_DIGEST)
    assert bench.measured_traffic("k_bwd_main", w) == bench.TRAFFIC[("k_bwd_main", w.name)]
    assert bench.measured_traffic("k_fwd_y", w) == bench.TRAFFIC[("k_fwd_y", w.name)]
    assert bench.measured_traffic("k_bwd_main", bench.pick_workload("long-seq-bf16")) is None
    monkeypatch.setattr(build, "source_digest", lambda: "0" * 16)
    assert bench.measured_traffic("k_bwd_main", w) is None


def test_traffic_figures_are_plausible():
    """DRAM bytes of a main pass are at least its algorithmic bytes (the saved
    states and partials come on top) and within a few times of them."""
    w = bench.pick_workload("mamba2.8b-layer-bf16")
    fwd, bwd = bench.algorithmic_bytes(w)
    bwd_main = bwd - 2 * w.Bsz * w.L * w.N * 4 - 4 * (w.Dch * w.N + 2 * w.Dch)
    assert bwd_main <= bench.TRAFFIC[("k_bwd_main", w.name)] <= 3 * bwd_main
    assert fwd <= bench.TRAFFIC[("k_fwd_y", w.name)] <= 4 * fwd


def test_unknown_workload_exits():
    with pytest.raises(SystemExit):
        bench.pick_workload("no-such-workload")


def test_mufu_counts():
    w = bench.pick_workload("mamba2.8b-layer-bf16")
    m = bench.mufu_counts(w)
    # 83,886,080 (t, d) elements x 16 states: the 1.342 G exponentials of each direction's scan
    assert m["scan_ex2_per_direction"] == 1_342_177_280
    assert m["fwd_all"] == 83_886_080 * 20 and m["bwd_all"] == 83_886_080 * 21


def test_reference_arm_reports_the_same_config():
    w = bench.pick_workload("mamba2.8b-layer-bf16")
    c = bench.config_of(w, 1)
    assert c == bench.config_of(w, 1)
    assert (c["workload"], c["Bsz"], c["L"], c["Dch"], c["N"], c["io"]) == ("mamba2.8b-layer-bf16", 4, 4096, 5120, 16,
                                                                           "bf16")
    assert c["step"] == "ss_fwd_save + ss_bwd_saved"
    assert bench.config_of(bench.pick_workload("mamba130m-layer-bf16-fwd"), 1)["step"] == "ss_fwd"


def _peaks(**kw):
    p = {"hbm_gbs": 7000.0, "hbm_kind": "measured", "ex2_per_clk_per_sm": 30.0, "fma_per_clk_per_sm": 128.0,
         "sms": 152, "sm_mhz": 2000.0}
    p.update(kw)
    return p


def test_analyse_rooflines_of_a_training_step():
    w = bench.pick_workload("mamba2.8b-layer-bf16")
    plan = {"segments": [(608, 1), (32, 19)]}
    # launches: fwd = summary, main(seg0), main(seg1); bwd = summary, carry, main x2, reduce_bc, reduce_params
    k_fwd = [0.05, 0.4, 0.1]
    k_bwd = [0.06, 0.004, 0.9, 0.2, 0.05, 0.01]
    out = bench.analyse(w, plan, 2.0, sum(k_fwd), sum(k_bwd), k_fwd, k_bwd, _peaks())
    fwd_b, bwd_b = bench.algorithmic_bytes(w)
    exps = 1_342_177_280  # B L D N
    fp32_peak = 152 * 128 * 2000e6  # f32 results / s
    # backward main pass: FP32-bound, 11 operations per state update at 38.9 Top/s -> 0.379 ms, above its
    # bytes (which exclude dB / dC and the parameter gradients) at 7000 GB/s (0.240 ms) and its exponentials
    bwd_main = bwd_b - 2 * w.Bsz * w.L * w.N * 4 - 4 * (w.Dch * w.N + 2 * w.Dch)
    r = out["roofline"]
    assert r["bound"] == "alu" and r["unit"] == "Gop/s" and r["ms"] == pytest.approx(1.1)
    assert r["roofline_ms"] == pytest.approx(11 * exps / fp32_peak * 1e3, rel=1e-3)
    assert r["achieved"] == pytest.approx(11 * exps / 1.1e-3 / 1e9, rel=1e-3)
    assert r["frac"] == pytest.approx(11 * exps / 1.1e-3 / fp32_peak, rel=1e-3)
    assert r["floors_ms"]["hbm"] == pytest.approx(bwd_main / 7e12 * 1e3, rel=1e-3)
    assert r["hbm"]["achieved"] == pytest.approx(bwd_main / 1.1e-3 / 1e9, rel=1e-3)
    # forward: 1.342 G exponentials at 152 x 30 x 2000 MHz = 9120 Gexp2/s -> 0.147 ms, above its 4 FP32
    # operations per update (0.138 ms) and 673.8 MB / 7 TB/s
    rf = out["roofline_fwd"]
    assert rf["bound"] == "alu" and rf["unit"] == "Gexp2/s" and rf["peak"] == pytest.approx(9120.0)
    assert rf["roofline_ms"] == pytest.approx(exps / 9.12e12 * 1e3, rel=1e-3)
    assert rf["floors_ms"]["fp32"] == pytest.approx(4 * exps / fp32_peak * 1e3, rel=1e-3)
    t_roof = rf["roofline_ms"] + 11 * exps / fp32_peak * 1e3
    assert out["roofline_step_frac"] == pytest.approx(t_roof / 2.0, abs=1e-4)
    # a slow memory makes the same pass HBM-bound
    slow = bench.analyse(w, plan, 2.0, sum(k_fwd), sum(k_bwd), k_fwd, k_bwd, _peaks(hbm_gbs=1000.0))
    assert slow["roofline"]["bound"] == "hbm" and slow["roofline"]["unit"] == "GB/s"
    assert slow["roofline"]["achieved"] == pytest.approx(bwd_main / 1.1e-3 / 1e9, rel=1e-3)
    assert list(out["kernel_ms"]) == [
        "k_fwd chunk summary (32 units x 19 chunks)", "k_fwd y + saved states (608 units x 1 chunk)",
        "k_fwd y + saved states (32 units x 19 chunks)", "k_bwd reverse summary (32 units x 19 chunks)",
        "k_bwd_carry (32 units x 19 chunks)", "k_bwd main (608 units x 1 chunk)", "k_bwd main (32 units x 19 chunks)",
        "k_bwd_reduce_bc", "k_bwd_reduce_params"]


def test_analyse_forward_only_step():
    w = bench.pick_workload("mamba130m-layer-bf16-fwd")
    plan = {"segments": [(384, 2)]}
    out = bench.analyse(w, plan, 0.2, 0.2, 0.0, [0.05, 0.15], [], _peaks())
    assert "roofline_fwd" not in out and "bwd_ms" not in out
    assert out["roofline"]["ms"] == pytest.approx(0.15)
    assert list(out["kernel_ms"]) == ["k_fwd chunk summary (384 units x 2 chunks)", "k_fwd y (384 units x 2 chunks)"]
