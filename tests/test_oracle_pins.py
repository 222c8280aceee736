"""Pins for the CPU oracle: each check ties it to something other than itself.

Closed forms, hand-worked examples (tests/golden/), brute force on tiny
inputs and library routines. A plausible mistake in the oracle -- a dropped
term, a wrong sign or index, a transposed operand, top-1 instead of top-2 --
fails at least one of these. No GPU needed.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _tiny():
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl)
    return wl, d


def _getter(d):
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = (d["w_gate"][e].float().numpy(), d["w_up"][e].float().numpy(),
                        d["w_down"][e].float().numpy())
        return cache[e]
    return get


# --------------------------------------------------------------------------
# elementwise pieces
# --------------------------------------------------------------------------
def test_bf16_round_matches_torch():
    g = torch.Generator().manual_seed(7)
    v = torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 4)
    # exact halfway cases between two BF16 values: ties must go to even
    base = torch.tensor([1.0, 1.0078125, -3.0, 1000.0], dtype=torch.float32)
    half = base.view(torch.int32) + 0x8000
    v = torch.cat([v, half.view(torch.float32)])
    ref = v.to(torch.bfloat16).to(torch.float32).numpy()
    got = O.bf16_round(v.numpy())
    assert np.array_equal(ref.view(np.uint32), got.view(np.uint32))


def test_sigmoid_and_silu_closed_forms():
    assert O.sigmoid(np.array([0.0]))[0] == 0.5
    assert abs(O.sigmoid(np.array([math.log(3.0)]))[0] - 0.75) < 1e-15
    assert abs(O.silu(np.array([2.0]))[0] - 2.0 / (1.0 + math.exp(-2.0))) < 1e-15
    # sigmoid(-z) = 1 - sigmoid(z)
    z = np.linspace(-8, 8, 33)
    assert np.allclose(O.sigmoid(-z), 1.0 - O.sigmoid(z), atol=1e-15)


def test_rmsnorm_hand_vector():
    v = np.array([[3.0, 4.0]])
    # mean of squares 12.5 -> divide by sqrt(12.5)
    want = np.array([[3.0, 4.0]]) / math.sqrt(12.5)
    assert np.allclose(O.rms_norm(v, eps=0.0), want, atol=1e-15)
    g = np.array([2.0, -1.0])
    assert np.allclose(O.rms_norm(v, g, eps=0.0), want * g, atol=1e-15)
    # with eps: 3 / sqrt(12.5 + 0.5)
    assert abs(O.rms_norm(v, eps=0.5)[0, 0] - 3.0 / math.sqrt(13.0)) < 1e-15


def test_rmsnorm_unit_rms():
    x = np.random.default_rng(3).normal(size=(17, 512)) * 7.0
    n = O.rms_norm(x, eps=1e-6)
    rms = np.sqrt((n * n).mean(-1))
    assert np.allclose(rms, 1.0, atol=1e-6)


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------
def test_router_orientation_one_hot():
    """logit[e] for x = unit vector j equals w_router[e, j] (not w_router[j, e])."""
    rng = np.random.default_rng(1)
    E, H = 16, 16          # square on purpose: a transposed operand still runs
    w = rng.normal(size=(E, H))
    for j in (0, 5, 15):
        x = np.zeros((1, H))
        x[0, j] = 1.0
        s64, _ = O.router_scores(x, w)
        assert np.allclose(s64[0], 1.0 / (1.0 + np.exp(-w[:, j])), atol=1e-15)


def test_router_bias_before_sigmoid():
    x = np.zeros((1, 4))
    w = np.zeros((8, 4))
    b = np.array([0.0, math.log(3.0), -math.log(3.0), 0, 0, 0, 0, 0])
    s64, _ = O.router_scores(x, w, b)
    assert np.allclose(s64[0, :3], [0.5, 0.75, 0.25], atol=1e-15)


def test_hand_routing_golden():
    g = _gold("routing_hand_example.json")
    s = np.array([g["scores"]], dtype=np.float64)
    sel = O.group_limited_topk(s.astype(np.float32), g["n_group"], g["topk_group"],
                               g["top_k"])
    assert sorted(sel["kept"][0].tolist()) == g["expected_kept"]
    assert sel["idx"][0].tolist() == g["expected_idx"]
    w = O.combine_weights(s, sel["idx"], g["scale"])
    assert np.allclose(w[0], g["expected_weights"], atol=1e-12)


def test_all_zero_logits_equal_weights():
    """logit 0 everywhere: every score is 0.5, all ties -> lowest indices,
    weights 2.5/8 each."""
    T, E, H = 3, 256, 8
    sel = O.route(np.zeros((T, H)), np.zeros((E, H)), None, 8, 4, 8, 2.5)
    assert (sel["idx"] == np.arange(8)).all()   # groups 0..3 kept, experts 0..7
    assert np.allclose(sel["weights"], 2.5 / 8, atol=1e-15)


def test_weights_sum_to_scale():
    """(a) the selected weights of every token sum to 2.5."""
    wl, d = _tiny()
    sel = O.route(d["x"].float().numpy(), d["w_router"].numpy(), None,
                  wl.n_group, wl.topk_group, wl.top_k, wl.routed_scale)
    assert np.allclose(sel["weights"].sum(1), 2.5, atol=1e-12)
    assert (sel["weights"] > 0).all()


def _brute_force_select(s32, n_group, topk_group, top_k):
    """Enumerate every subset of topk_group groups; keep the one with the
    largest total group score (ties: lexicographically smallest subset), then
    fully sort its experts."""
    E = s32.shape[0]
    gsize = E // n_group
    gsc = []
    for g in range(n_group):
        vals = sorted(s32[g * gsize:(g + 1) * gsize].tolist(), reverse=True)
        gsc.append(float(np.float32(vals[0]) + np.float32(vals[1])))
    best, best_val = None, None
    for sub in itertools.combinations(range(n_group), topk_group):
        # largest total first; an exact tie on the total falls back to the
        # sorted score list; combinations() runs in lexicographic order and
        # only a strictly better subset replaces the best one
        val = (sum(gsc[g] for g in sub), sorted((gsc[g] for g in sub), reverse=True))
        if best is None or val > best_val:
            best, best_val = sub, val
    experts = [e for g in best for e in range(g * gsize, (g + 1) * gsize)]
    experts.sort(key=lambda e: (-float(s32[e]), e))
    return list(best), experts[:top_k]


def test_group_limit_brute_force():
    """(b) every selected expert lies in a kept group, and enumerating all
    C(8,4) = 70 group subsets gives the same groups and experts."""
    wl, d = _tiny()
    sel = O.route(d["x"].float().numpy(), d["w_router"].numpy(), None,
                  wl.n_group, wl.topk_group, wl.top_k, wl.routed_scale)
    for t in range(wl.T):
        kept = set(sel["kept"][t].tolist())
        assert all(e // 32 in kept for e in sel["idx"][t])
        groups, experts = _brute_force_select(sel["s32"][t], 8, 4, 8)
        assert set(groups) == kept
        assert sel["idx"][t].tolist() == experts


def test_plain_topk_when_all_groups_kept():
    """topk_group = n_group reduces to plain top-k (a stable library sort)."""
    rng = np.random.default_rng(5)
    s = rng.random((20, 256)).astype(np.float32)
    s[3, 17] = s[3, 200]                 # an exact tie: lower index first
    sel = O.group_limited_topk(s, 8, 8, 8)
    for t in range(20):
        ref = np.argsort(-s[t].astype(np.float64), kind="stable")[:8]
        assert sel["idx"][t].tolist() == ref.tolist()


def test_group_score_is_top2_sum():
    s = np.zeros((1, 8), dtype=np.float32)
    s[0, :4] = [0.1, 0.9, 0.3, 0.2]
    s[0, 4:] = [0.5, 0.5, 0.5, 0.0]
    gs = O.group_scores(s, 2)
    assert np.allclose(gs[0], [np.float32(0.9) + np.float32(0.3), 1.0])


def test_near_tie_margins():
    s = np.full((1, 16), 0.1, dtype=np.float32)
    s[0, [0, 1, 4, 5]] = [0.9, 0.8, 0.7, 0.6]
    s[0, 2] = np.float32(0.6) + np.float32(3e-6)    # 3rd best at 0.600003
    sel = O.group_limited_topk(s, 4, 2, 4)
    # kept g0 (1.7) and g1 (1.3); selected 0,1,4,2; next candidate 5 at 0.6
    assert sel["idx"][0].tolist() == [0, 1, 4, 2]
    assert 0 < sel["topk_margin"][0] < 1e-5
    assert O.near_ties(sel)[0]
    # group scores 1.7, 1.3, 0.2, 0.2: the kept pair ends at 1.3, the next is 0.2
    assert abs(sel["group_margin"][0] - 1.1) < 1e-6


# --------------------------------------------------------------------------
# experts and combine
# --------------------------------------------------------------------------
def test_swiglu_closed_form():
    """H=2, I=1, one token, computed by hand: g = 1*1 + 2*0.5 = 2,
    u = 0.25 + 0.5 = 0.75, a = silu(2) * 0.75, y = a * [1, -2]."""
    x = np.array([[1.0, 2.0]])
    wg = np.array([[1.0, 0.5]])
    wu = np.array([[0.25, 0.25]])
    wd = np.array([[1.0], [-2.0]])
    a = 2.0 / (1.0 + math.exp(-2.0)) * 0.75
    y = O.swiglu_expert(x, wg, wu, wd)
    assert np.allclose(y, [[a, -2.0 * a]], atol=1e-15)
    # swapping gate and up gives a different value (guards the convention)
    assert not np.allclose(O.swiglu_expert(x, wu, wg, wd), y)


def test_expert_orientation_one_hot():
    rng = np.random.default_rng(9)
    H, I = 6, 4
    wg, wu, wd = rng.normal(size=(I, H)), rng.normal(size=(I, H)), rng.normal(size=(H, I))
    x = np.zeros((1, H))
    x[0, 2] = 1.0
    g, u = wg[:, 2], wu[:, 2]
    a = g / (1 + np.exp(-g)) * u
    assert np.allclose(O.swiglu_expert(x, wg, wu, wd)[0], wd @ a, atol=1e-14)


def test_dense_reduction_when_all_experts_selected():
    """(e) one group, every expert kept: the layer is the dense weighted sum
    2.5 * sum_e s_e / (sum s) * f_e(x), written here as a separate loop."""
    wl, d = S.make_custom(T=5, H=32, E=16, I=8, n_group=1, topk_group=1,
                          top_k=16, seed=11)
    x = d["x"].float().numpy().astype(np.float64)
    wr = d["w_router"].numpy()
    get = _getter(d)
    res = O.moe_forward(x, wr, None, get, n_group=1, topk_group=1, top_k=16,
                        scale=2.5)
    want = np.zeros_like(x)
    for t in range(x.shape[0]):
        logits = [float(np.dot(x[t], wr[e].astype(np.float64))) for e in range(16)]
        s = [1.0 / (1.0 + math.exp(-v)) for v in logits]
        tot = sum(s)
        for e in range(16):
            wg, wu, wdn = (m.astype(np.float64) for m in get(e))
            gg = wg @ x[t]
            uu = wu @ x[t]
            aa = [gv / (1.0 + math.exp(-gv)) * uv for gv, uv in zip(gg, uu)]
            want[t] += 2.5 * s[e] / tot * (wdn @ np.array(aa))
    assert np.allclose(res["out"], want, rtol=1e-12, atol=1e-14)


def test_moe_forward_per_token_brute_force():
    """Expert-major combine equals a per-token loop over the 8 slots."""
    wl, d = _tiny()
    get = _getter(d)
    x = d["x"].float().numpy()
    res = O.moe_forward(x, d["w_router"].numpy(), None, get)
    sel = res["sel"]
    for t in range(0, wl.T, 7):
        want = np.zeros(wl.H)
        for j in range(8):
            e = int(sel["idx"][t, j])
            wg, wu, wdn = (m.astype(np.float64) for m in get(e))
            xt = x[t].astype(np.float64)
            g = wg @ xt
            u = wu @ xt
            want += sel["weights"][t, j] * (wdn @ (g / (1 + np.exp(-g)) * u))
        assert np.allclose(res["out"][t], want, rtol=1e-12, atol=1e-15)


def test_permutation_brute_force():
    rng = np.random.default_rng(2)
    T, k, E = 37, 8, 64
    idx = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    p = O.permutation(idx, E)
    rows = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    rows.append(t * k + j)
    assert p["row_pair"].tolist() == rows
    assert p["offsets"][-1] == T * k
    assert all(p["offsets"][e + 1] - p["offsets"][e] == (idx == e).sum() for e in range(E))


# --------------------------------------------------------------------------
# residual stream
# --------------------------------------------------------------------------
def test_residual_weights_square_sum():
    """(c) the two residual weights' squares sum to 1 for every k >= 2."""
    for k in range(2, 300):
        a, b = O.residual_coeffs(k)
        assert abs(a * a + b * b - 1.0) < 1e-15
    with pytest.raises(ValueError):
        O.residual_coeffs(1)


def test_residual_chain_equal_weights():
    """(d) embedding = step 1, then 104 additions of orthogonal sublayer
    outputs: every one of the 105 contributions ends with weight 1/sqrt(105)."""
    facts = _gold("beam_layer_facts.json")
    n_add = facts["residual_additions"]["value"]
    n = n_add + 1
    basis = np.eye(n)
    h = basis[0:1]
    for k in range(2, n + 1):
        h = O.residual_step(h, basis[k - 1:k], k, apply_norm=False)
    assert np.allclose(h[0], 1.0 / math.sqrt(105), atol=1e-12)
    assert n == 105


def test_residual_step_with_norm_matches_parts():
    rng = np.random.default_rng(4)
    h = rng.normal(size=(3, 64))
    o = rng.normal(size=(3, 64)) * 5.0
    got = O.residual_step(h, o, 50, eps=1e-6)
    n = o / np.sqrt((o * o).mean(-1, keepdims=True) + 1e-6)
    assert np.allclose(got, math.sqrt(49 / 50) * h + n / math.sqrt(50), atol=1e-14)


def test_prenorm_rounds_to_bf16():
    rng = np.random.default_rng(8)
    h = rng.normal(size=(4, 32)).astype(np.float32)
    r = O.moe_forward(h, np.zeros((8, 32), np.float32), None,
                      lambda e: (np.zeros((2, 32)), np.zeros((2, 32)), np.zeros((32, 2))),
                      n_group=1, topk_group=1, top_k=2, pre_norm=True)
    want = torch.from_numpy(O.rms_norm(h.astype(np.float64))).to(torch.bfloat16).double().numpy()
    assert np.array_equal(r["x"], want)


def test_forward_residual_keeps_the_layer_input():
    """With every expert weight zero the MoE output is exactly 0, RMSNorm(0)
    is 0, and the step leaves h_k = sqrt((k-1)/k) * h_{k-1}: the residual
    branch carries the layer input itself, not its pre-normed copy (the
    input's RMS is 7 here, so the two differ)."""
    rng = np.random.default_rng(13)
    T, H, E, I, k = 5, 32, 8, 4, 11
    h = rng.normal(size=(T, H)) * 7.0
    zero = (np.zeros((I, H)), np.zeros((I, H)), np.zeros((H, I)))
    r = O.moe_forward(h, rng.normal(size=(E, H)), None, lambda e: zero, n_group=2,
                      topk_group=1, top_k=2, pre_norm=True, residual_k=k)
    assert np.array_equal(r["out"], np.zeros((T, H)))
    assert np.allclose(r["h"], math.sqrt((k - 1) / k) * h, rtol=1e-15, atol=0)


def test_prenorm_gain_scales_each_channel():
    """A pre-norm gain of powers of two scales each channel of the BF16
    pre-norm output exactly (BF16 rounding commutes with a power-of-two
    factor), and the router then sees the scaled x."""
    rng = np.random.default_rng(14)
    T, H, E = 6, 32, 8
    h = rng.normal(size=(T, H)) * 3.0
    g = np.tile([0.5, 1.0, 2.0, 4.0], H // 4)
    zero = (np.zeros((2, H)), np.zeros((2, H)), np.zeros((H, 2)))
    kw = dict(n_group=1, topk_group=1, top_k=2, pre_norm=True)
    wr = rng.normal(size=(E, H))
    plain = O.moe_forward(h, wr, None, lambda e: zero, **kw)
    gained = O.moe_forward(h, wr, None, lambda e: zero, pre_gain=g, **kw)
    assert np.array_equal(gained["x"], plain["x"] * g[None, :])
    assert np.allclose(gained["sel"]["s64"], 1.0 / (1.0 + np.exp(-(plain["x"] * g) @ wr.T)),
                       rtol=1e-14, atol=0)


def test_residual_step_post_gain_hand_case():
    """h_{k-1} = 0, sub-layer output 3 in every channel: RMSNorm gives
    3 / sqrt(9 + eps) per channel, times the gain, times 1/sqrt(4)."""
    g = np.array([1.0, 2.0, 0.5, -1.0])
    h = O.residual_step(np.zeros((1, 4)), np.full((1, 4), 3.0), 4, gain=g)
    assert np.allclose(h[0], 0.5 * 3.0 / math.sqrt(9.0 + 1e-6) * g, rtol=1e-15, atol=0)


def _check_gains(run, h, k):
    """run(pre_gain, post_gain) -> result dict with x and h. With per-channel
    powers of two as gains, the BF16 pre-norm output scales exactly, channel
    by channel, and the post-norm branch h_k - sqrt((k-1)/k) h_{k-1} scales
    by the post-norm gain."""
    g = np.tile([0.5, 1.0, 2.0, 4.0], h.shape[1] // 4)
    base, pre, post = run(None, None), run(g, None), run(None, g)
    assert np.array_equal(pre["x"], base["x"] * g[None, :])
    keep = math.sqrt((k - 1) / k) * h
    assert np.allclose(post["h"] - keep, (base["h"] - keep) * g[None, :], rtol=1e-13, atol=1e-13)
    assert not np.allclose(post["h"], base["h"])


def test_gains_reach_the_moe_and_dense_sublayers():
    rng = np.random.default_rng(18)
    T, H, E, I = 5, 32, 8, 8
    h = rng.normal(size=(T, H)) * 2.0
    wr = rng.normal(size=(E, H))
    W = [tuple(rng.normal(size=s) * 0.2 for s in ((I, H), (I, H), (H, I))) for _ in range(E)]
    k = 6
    _check_gains(lambda pg, qg: O.moe_forward(
        h, wr, None, lambda e: W[e], n_group=2, topk_group=1, top_k=2, pre_norm=True,
        pre_gain=pg, residual_k=k, post_gain=qg), h, k)
    _check_gains(lambda pg, qg: O.dense_mlp_forward(
        h, *W[0], pre_norm=True, pre_gain=pg, residual_k=k, post_gain=qg), h, k)


# --------------------------------------------------------------------------
# page facts
# --------------------------------------------------------------------------
def test_layer_shape_facts():
    f = _gold("beam_layer_facts.json")
    H, I, E = f["hidden_size"]["value"], f["expert_intermediate"]["value"], \
        f["experts_per_layer"]["value"]
    wl = S.WORKLOADS["prefill"]
    assert (wl.H, wl.I, wl.E, wl.top_k, wl.n_group, wl.topk_group, wl.routed_scale) == \
        (H, I, E, f["experts_per_token"]["value"], f["n_group"]["value"],
         f["topk_group"]["value"], f["routed_scaling_factor"]["value"])
    per_expert = 3 * H * I
    assert per_expert == 39_321_600 and round(per_expert / 1e6) == \
        f["expert_params_approx_millions"]["value"]
    L = f["moe_layers"]["value"]
    experts_all = L * E * per_expert
    total = f["total_params"]["value"]
    assert f["bf16_params"]["value"] + f["f32_params"]["value"] == total
    assert round(100 * experts_all / total, 1) == f["expert_param_share_percent"]["value"]
    # FP32 router [E, H] per MoE layer plus one FP32 E-vector per layer
    assert L * E * H + L * E == f["f32_params"]["value"]
    # NVFP4 packs two values per byte: the U8 count is half of all expert params
    assert 2 * f["nvfp4_u8_bytes"]["value"] == experts_all
    k = f["experts_per_token"]["value"]
    active = k * L * per_expert + (total - experts_all)
    assert round(active / 1e9, 1) == f["active_params_billions"]["value"]
    assert f["dense_layers"]["value"] + L == f["num_layers"]["value"]


# --------------------------------------------------------------------------
# dense SwiGLU MLP of the first layers
# --------------------------------------------------------------------------
def test_dense_mlp_closed_form():
    """H=2, I=1 by hand (as the expert case): x=[1,2], g=2, u=0.75."""
    x = np.array([[1.0, 2.0]])
    r = O.dense_mlp_forward(x, np.array([[1.0, 0.5]]), np.array([[0.25, 0.25]]),
                            np.array([[1.0], [-2.0]]))
    a = 2.0 / (1.0 + math.exp(-2.0)) * 0.75
    assert np.allclose(r["out"], [[a, -2.0 * a]], atol=1e-15)
    assert r["h"] is None


def test_dense_mlp_is_one_expert_with_unit_weight():
    """The dense MLP equals the expert combine with a single expert that every
    token uses with weight 1 (a separate code path: moe_combine)."""
    rng = np.random.default_rng(12)
    T, H, I = 9, 32, 24
    x = rng.normal(size=(T, H))
    wg, wu, wd = rng.normal(size=(I, H)) * .1, rng.normal(size=(I, H)) * .1, rng.normal(size=(H, I)) * .1
    d = O.dense_mlp_forward(x, wg, wu, wd)
    m = O.moe_combine(x, np.zeros((T, 1), np.int64), np.ones((T, 1)), lambda e: (wg, wu, wd))
    assert np.allclose(d["out"], m, rtol=1e-13, atol=1e-15)
    h = O.dense_mlp_forward(x, wg, wu, wd, residual_k=7, pre_norm=True)
    xn = O.bf16_round(O.rms_norm(x)).astype(np.float64)
    want = math.sqrt(6 / 7) * x + O.rms_norm(O.swiglu_expert(xn, wg, wu, wd)) / math.sqrt(7)
    assert np.allclose(h["h"], want, atol=1e-12)
