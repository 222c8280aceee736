"""The synthetic inputs follow their stated recipe: shapes and dtypes of the
layer, seeded and repeatable, N(0, std) values rounded once to BF16, the
skewed workload's bias b_e = 3 * rank_e^-1.1 over a permutation, and the
routing edge cases. No GPU needed."""
import numpy as np
import torch

import beam_synth as S


def test_workload_shapes_follow_the_layer():
    for name in ("decode", "prefill", "skew", "long_prefill"):
        wl = S.WORKLOADS[name]
        assert (wl.H, wl.E, wl.I, wl.n_group, wl.topk_group, wl.top_k, wl.routed_scale) == \
            (5120, 256, 2560, 8, 4, 8, 2.5)
    assert [S.WORKLOADS[n].T for n in ("decode", "prefill", "skew", "long_prefill")] == \
        [64, 8192, 4096, 16384]
    assert [S.WORKLOADS[n].seed for n in ("tiny", "decode", "prefill", "skew", "long_prefill")] \
        == [0, 1, 2, 3, 4]
    lp = S.WORKLOADS["long_prefill"]
    assert lp.pre_norm and lp.residual_k == 50


def test_tiny_inputs_dtypes_values_and_repeatability():
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl)
    assert d["x"].shape == (64, 256) and d["x"].dtype == torch.bfloat16
    assert d["w_router"].shape == (256, 256) and d["w_router"].dtype == torch.float32
    assert d["w_gate"].shape == d["w_up"].shape == (256, 128, 256)
    assert d["w_down"].shape == (256, 256, 128)
    assert all(d[k].dtype == torch.bfloat16 for k in ("w_gate", "w_up", "w_down"))
    assert d["bias"] is None
    # standard deviations of the stated normals (many samples: within 2%)
    for k, std in (("x", 1.0), ("w_router", 0.05), ("w_gate", 0.02), ("w_down", 0.02)):
        s = d[k].float().std().item()
        assert abs(s / std - 1.0) < 0.02, (k, s)
    assert abs(d["w_up"].float().mean().item()) < 1e-3
    again = S.make_inputs(wl)
    assert all(torch.equal(d[k], again[k]) for k in ("x", "w_router", "w_gate", "w_up", "w_down"))
    other = S.make_inputs(wl.replace(seed=1))
    assert not torch.equal(d["x"], other["x"])


def test_skew_bias_is_a_permuted_power_law():
    b = S.skew_bias(256, 3).double().numpy()
    want = np.sort(3.0 * np.arange(1, 257, dtype=np.float64) ** -1.1)[::-1]
    assert np.allclose(np.sort(b)[::-1], want, rtol=1e-7, atol=0)   # FP32 values of the ranks
    assert b.max() == 3.0
    assert np.array_equal(b, S.skew_bias(256, 3).double().numpy())
    assert not np.array_equal(b, S.skew_bias(256, 4).double().numpy())
    assert not np.all(np.diff(b) <= 0)          # spread over a permutation, not by index


def test_routing_edge_case_inputs():
    wl, d = S.make_custom(16, 256, 256, 128, 8, 4, 8, seed=5, router_mode="dup_rows")
    wr = d["w_router"]
    assert torch.equal(wr[1], wr[0]) and torch.equal(wr[33], wr[0])
    assert torch.equal(wr[200], wr[199])
    _, d = S.make_custom(16, 256, 256, 128, 8, 4, 8, seed=5, router_mode="hot_group")
    assert torch.equal(d["bias"][:8], torch.full((8,), 20.0))
    assert torch.count_nonzero(d["bias"][8:]) == 0
    _, d = S.make_custom(16, 256, 256, 128, 8, 4, 8, seed=5, router_mode="hot_expert")
    assert d["bias"][5] == 20.0 and torch.count_nonzero(d["bias"]) == 1
