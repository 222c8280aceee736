"""The algorithmic work behind bench.py's roofline figures, against closed
forms: expert FLOPs = T * top_k * 6 * H * I (T * 629,145,600 at the Beam
shapes), weight bytes = touched experts * 3 * H * I * bytes per weight
(78,643,200 per BF16 expert), plus the layer's BF16 input and output. No GPU
needed."""
import numpy as np
import pytest

import beam_synth as S


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def _counts(E, touched):
    c = np.zeros(E, dtype=np.int64)
    c[:touched] = 3
    return c


def test_decode_bf16_closed_forms(bench):
    wl = S.WORKLOADS["decode"]
    a = bench._algorithmic(wl, _counts(wl.E, 220), "bf16")
    assert a["touched"] == 220
    # gate and up of 220 experts once, plus x: the bench's decode figure
    assert a["gu_bytes"] == 220 * 2 * 2560 * 5120 * 2 + 64 * 5120 * 2 == 11_534_991_360
    assert a["dn_bytes"] == 220 * 5120 * 2560 * 2 + 64 * 5120 * 2
    assert a["gu_flops"] + a["dn_flops"] == 64 * 629_145_600
    # the whole layer: 78.64 MB per touched expert, x in and h out, the FP32 router
    assert a["layer_bytes"] == 220 * 78_643_200 + 2 * 64 * 5120 * 2 + 256 * 5120 * 4
    assert a["layer_flops"] == 64 * 629_145_600 + 2 * 64 * 5120 * 256


def test_prefill_flops_scale_with_tokens(bench):
    wl = S.WORKLOADS["prefill"]
    a = bench._algorithmic(wl, _counts(wl.E, wl.E), "bf16")
    assert a["gu_flops"] == 2 * (8192 * 8) * 2 * 2560 * 5120 == 3_435_973_836_800
    assert a["gu_flops"] + a["dn_flops"] == 8192 * 629_145_600


@pytest.mark.parametrize("kind,per_weight,per_row", [("fp8", 1.0, 4), ("nvfp4", 0.5 + 1 / 16, 0)])
def test_quantised_weight_bytes(bench, kind, per_weight, per_row):
    """E4M3: one byte per weight and an FP32 scale per output row; NVFP4: half
    a byte per weight and one E4M3 block scale per 16 weights."""
    wl = S.WORKLOADS["decode"]
    a = bench._algorithmic(wl, _counts(wl.E, 100), kind)
    want_gu = int(100 * 2 * 2560 * (5120 * per_weight + per_row)) + 64 * 5120 * 2
    assert a["gu_bytes"] == want_gu
    # FLOPs do not depend on the weight format
    b = bench._algorithmic(wl, _counts(wl.E, 100), "bf16")
    assert a["gu_flops"] == b["gu_flops"] and a["dn_flops"] == b["dn_flops"]


def test_peaks_come_from_the_measured_file(bench, tmp_path, monkeypatch):
    """The roofline denominators are MEASURED_PEAKS.json's figures when the
    file is there (source "measured") and the stated fallback otherwise."""
    import json
    import os
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            want = json.load(f)
        p = bench._peaks()
        assert p["source"] == "measured"
        assert p["hbm"] == float(want["hbm_gbs"]) and p["bf16"] == float(want["bf16_tflops"])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench._peaks()
    assert p["source"] == "fallback" and p["hbm"] == 6400.0 and p["bf16"] == 1800.0


def test_cpu_baseline_runs_for_its_minimum_time(bench):
    """The oracle sample is repeated until it has taken the minimum time (at
    least once, at most max_runs times), and the rate counts every run."""
    import time
    calls = []
    run = lambda: (calls.append(1), time.sleep(0.02))
    v, runs, dt = bench.time_oracle(run, 4, min_s=0.1, max_runs=50)
    assert runs == len(calls) and 4 <= runs <= 7 and dt >= 0.1
    assert abs(v - 4 * runs / dt) < 1e-9
    v, runs, dt = bench.time_oracle(run, 4, min_s=10.0, max_runs=3)
    assert runs == 3
    v, runs, dt = bench.time_oracle(run, 4, min_s=0.0)
    assert runs == 1


def _fake_peaks():
    return {"hbm": 6500.0, "bf16": 1800.0, "bf16_sustained": 1355.0, "source": "measured"}


@pytest.mark.parametrize("name,kind,touched,want", [
    ("decode", "bf16", 220, "hbm"),        # 11.5 GB of weights, 0.04 TFLOP
    ("prefill", "bf16", 256, "tensor"),    # 13.5 GB: 2.08 ms at the copy rate; 3.44 TFLOP: 2.54 ms
    ("skew", "bf16", 256, "hbm"),          # T = 4096: 13.5 GB (2.07 ms) against 1.72 TFLOP (1.27 ms)
    ("prefill", "fp8", 256, "tensor"),     # 6.7 GB (1.04 ms) against 3.44 TFLOP at 2 x 1355 (1.27 ms)
    ("prefill", "nvfp4", 256, "hbm"),      # 3.8 GB (0.58 ms) against 3.44 TFLOP at 6 x 1355 (0.42 ms)
])
def test_roofline_takes_the_binding_bound(bench, name, kind, touched, want):
    """The roofline of the gate/up launch is the bound with the larger least
    time (algorithmic bytes / copy rate against FLOPs / sustained tensor
    rate), whatever the launch takes; the other bound's fraction is kept."""
    wl = S.WORKLOADS[name]
    a = bench._algorithmic(wl, _counts(wl.E, touched), kind)
    peaks = _fake_peaks()
    if kind != "bf16":
        rt = bench.TENSOR_RATIO[kind]
        peaks = dict(peaks, bf16=rt * peaks["bf16"], bf16_sustained=rt * peaks["bf16_sustained"])
    t_bytes = a["gu_bytes"] / (peaks["hbm"] * 1e9)
    t_flops = a["gu_flops"] / (peaks["bf16_sustained"] * 1e12)
    for launch_s in (1.05 * max(t_bytes, t_flops), 3.0 * max(t_bytes, t_flops)):
        r = bench.gemm_roofline("k", a["gu_bytes"], a["gu_flops"], launch_s * 1e3, peaks, kind, None)
        assert r["bound"] == want
        assert r["other_bound"]["bound"] == ("tensor" if want == "hbm" else "hbm")
        # the binding bound's fraction is the larger one, and both follow from the time
        f_bytes = a["gu_bytes"] / launch_s / 1e9 / peaks["hbm"]
        f_flops = a["gu_flops"] / launch_s / 1e12 / peaks["bf16_sustained"]
        got = {r["bound"]: r["frac"], r["other_bound"]["bound"]: r["other_bound"]["frac"]}
        assert got["hbm"] == pytest.approx(f_bytes, abs=1e-4)
        assert got["tensor"] == pytest.approx(f_flops, abs=1e-4)
        assert r["frac"] >= r["other_bound"]["frac"]
