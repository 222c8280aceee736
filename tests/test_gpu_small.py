"""GPU parity at sizes the oracle finishes in seconds: the tiny Beam layer,
shape sweeps with ragged token counts, routing edge cases, the residual step,
the pre-norm path and the bounded-wait failure path. All calls go through the
C ABI (the ctypes binding)."""
import math

import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O
from _helpers import (OUT_REL_TOL, bf16_ulp, compare_routing, expert_getter, host,
                      oracle_outputs, rel_err, validated_prenorm_x)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    return B


def _params(B, wl, flags=0, residual_k=0):
    return B.make_params(wl.T, wl.H, wl.E, wl.I, wl.n_group, wl.topk_group, wl.top_k,
                         wl.routed_scale, wl.rms_eps, residual_k, flags)


def _run_forward(B, wl, d, flags, residual_k=0):
    p = _params(B, wl, flags, residual_k)
    ws = B.alloc_workspace(p)
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device="cuda")
    out = B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"],
                    bias=d["bias"], topk_idx=idx, topk_w=w, workspace=ws)
    assert B.status() == 0, B.last_error()
    return out, idx, w, ws, p


def _workspace_x(B, ws, p, wl, h64, gain=None):
    """The GPU's BF16 pre-norm x from the workspace, validated element by
    element against the oracle (validated_prenorm_x)."""
    lay = B.workspace_layout(p)
    xg = ws[lay["xn"]:lay["xn"] + wl.T * wl.H * 2].view(torch.bfloat16).float().cpu().numpy()
    x64, _ = validated_prenorm_x(xg.reshape(wl.T, wl.H), h64, gain, wl.rms_eps)
    return x64


def _oracle_sel(wl, d):
    x = host(d["x"]).astype(np.float64)
    sel = O.route(x, host(d["w_router"]), host(d["bias"]), wl.n_group, wl.topk_group,
                  wl.top_k, wl.routed_scale)
    return x, sel


def _full_layer_check(B, wl, d, fp32_out=True, extra_flags=0):
    flags = (B.FLAG_FP32_OUT if fp32_out else 0) | extra_flags
    out, idx, w, ws, p = _run_forward(B, wl, d, flags)
    x, sel = _oracle_sel(wl, d)
    ties, chosen = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    toks = np.arange(wl.T)
    want = oracle_outputs(x, chosen, toks, expert_getter(d))
    got = host(out)
    err = rel_err(got, want)
    assert err <= OUT_REL_TOL, f"rel err {err}"
    return out, idx, w, ws, p, sel, ties


# ---------------------------------------------------------------- routing
def test_route_tiny_bitexact(B):
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    p = _params(B, wl, B.FLAG_RETURN_SCORES)
    idx, w, sc = B.route(p, d["x"], d["w_router"])
    assert B.status() == 0
    x, sel = _oracle_sel(wl, d)
    assert np.max(np.abs(host(sc) - sel["s64"])) < 2e-6
    ties, _ = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    assert ties.sum() == 0
    assert np.allclose(w.cpu().numpy().sum(1), 2.5, atol=1e-5)


@pytest.mark.parametrize("T,H,mode", [(512, 256, "random"), (700, 384, "random"),
                                      (1031, 256, "dup_rows")])
def test_route_tensor_core_path(B, T, H, mode):
    """T >= 512 with E = 256: logits on the tensor cores with the exact
    three-way BF16 split of the FP32 router weight."""
    wl, d = S.make_custom(T=T, H=H, E=256, I=128, n_group=8, topk_group=4, top_k=8,
                          seed=T, device="cuda", router_mode=mode)
    p = _params(B, wl, B.FLAG_RETURN_SCORES)
    idx, w, sc = B.route(p, d["x"], d["w_router"], bias=d["bias"])
    assert B.status() == 0
    x, sel = _oracle_sel(wl, d)
    assert np.max(np.abs(host(sc) - sel["s64"])) < 2e-6
    compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)


def test_route_deterministic(B):
    wl = S.WORKLOADS["tiny"].replace(T=300, seed=5)
    d = S.make_inputs(wl, "cuda")
    p = _params(B, wl)
    a = B.route(p, d["x"], d["w_router"])
    b = B.route(p, d["x"], d["w_router"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("mode", ["dup_rows", "hot_expert", "hot_group"])
def test_route_edge_cases(B, mode):
    wl, d = S.make_custom(T=77, H=256, E=256, I=128, n_group=8, topk_group=4, top_k=8,
                          seed=21, device="cuda", router_mode=mode)
    p = _params(B, wl)
    idx, w, _ = B.route(p, d["x"], d["w_router"], bias=d["bias"])
    x, sel = _oracle_sel(wl, d)
    compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    g = idx.cpu().numpy()
    if mode == "hot_expert":
        assert (g == 5).any(axis=1).all()
    if mode == "hot_group":
        assert (np.sort(g, axis=1) == np.arange(8)).all()
        assert np.allclose(w.cpu().numpy(), 2.5 / 8, atol=1e-6)
    if mode == "dup_rows":
        # experts 0, 1 and 33 have identical scores: 0 and 1 share group 0
        s = sel["s32"]
        assert np.array_equal(s[:, 0], s[:, 1]) and np.array_equal(s[:, 0], s[:, 33])


def test_route_bias_and_prenorm(B):
    wl, d = S.make_custom(T=33, H=384, E=256, I=128, n_group=8, topk_group=4, top_k=8,
                          seed=4, device="cuda", skew_bias=True)
    gain = (1.0 + 0.1 * torch.randn(wl.H, generator=torch.Generator().manual_seed(1))).cuda()
    p = _params(B, wl, B.FLAG_PRE_NORM | B.FLAG_RETURN_SCORES)
    ws = B.alloc_workspace(p)
    idx, w, sc = B.route(p, d["x"], d["w_router"], bias=d["bias"], pre_gain=gain, workspace=ws)
    assert B.status() == 0
    h = host(d["x"]).astype(np.float64)
    g64 = gain.double().cpu().numpy()
    xo = _workspace_x(B, ws, p, wl, h, g64)
    sel = O.route(xo, host(d["w_router"]), host(d["bias"]), 8, 4, 8, 2.5)
    compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)


# ---------------------------------------------------------------- layer
def test_forward_tiny(B):
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    _full_layer_check(B, wl, d, fp32_out=True)
    _full_layer_check(B, wl, d, fp32_out=False)


@pytest.mark.parametrize("T,H,I", [(1, 256, 128), (7, 256, 256), (64, 512, 128),
                                   (300, 256, 128), (129, 512, 256)])
def test_forward_shape_sweep(B, T, H, I):
    wl, d = S.make_custom(T=T, H=H, E=256, I=I, n_group=8, topk_group=4, top_k=8,
                          seed=T + H + I, device="cuda")
    _full_layer_check(B, wl, d)


@pytest.mark.parametrize("mode", ["hot_expert", "hot_group", "dup_rows"])
def test_forward_routing_edge_cases(B, mode):
    # hot_group: 248 empty experts, 8 experts with every token (several token tiles)
    wl, d = S.make_custom(T=300, H=256, E=256, I=128, n_group=8, topk_group=4, top_k=8,
                          seed=31, device="cuda", router_mode=mode)
    _full_layer_check(B, wl, d)


def test_forward_dense_all_experts(B):
    """(e) one group, every expert selected: the dense weighted sum."""
    wl, d = S.make_custom(T=20, H=128, E=32, I=128, n_group=1, topk_group=1, top_k=32,
                          seed=3, device="cuda")
    _full_layer_check(B, wl, d)


def test_forward_plain_topk(B):
    """topk_group = n_group: no group limit."""
    wl, d = S.make_custom(T=50, H=256, E=64, I=128, n_group=2, topk_group=2, top_k=6,
                          seed=8, device="cuda")
    _full_layer_check(B, wl, d)


def test_forward_permutation_stage(B):
    """Counts, offsets and the expert-ordered rows equal the oracle's stable
    permutation (no near ties on this input, checked)."""
    wl = S.WORKLOADS["tiny"].replace(T=200, seed=9)
    d = S.make_inputs(wl, "cuda")
    out, idx, w, ws, p, sel, ties = _full_layer_check(B, wl, d)
    assert ties.sum() == 0
    lay = B.workspace_layout(p)
    R = wl.T * wl.top_k
    raw = ws.cpu()

    def arr(name, n, dt):
        return raw[lay[name]:lay[name] + n * 4].view(dt).numpy()
    perm = O.permutation(sel["idx"], wl.E)
    assert np.array_equal(arr("counts", wl.E, torch.int32), perm["counts"])
    assert np.array_equal(arr("offsets", wl.E + 1, torch.int32), perm["offsets"])
    row_tok = arr("row_token", R, torch.int32)
    assert np.array_equal(row_tok, perm["row_pair"] // wl.top_k)
    row_w = arr("row_weight", R, torch.float32)
    want_w = sel["weights"].ravel()[perm["row_pair"]]
    assert np.max(np.abs(row_w - want_w)) <= 1e-5
    # permuted x rows and the SwiGLU intermediate of a few rows
    xp = raw[lay["xperm"]:lay["xperm"] + R * wl.H * 2].view(torch.bfloat16).float().numpy()
    xp = xp.reshape(R, wl.H)
    x = host(d["x"])
    assert np.array_equal(xp, x[perm["row_pair"] // wl.top_k])
    act = raw[lay["act"]:lay["act"] + R * wl.I * 2].view(torch.bfloat16).float().numpy()
    act = act.reshape(R, wl.I)
    get = expert_getter(d)
    for r in range(0, R, 97):
        pair = perm["row_pair"][r]
        e = sel["idx"].ravel()[pair]
        wg, wu, _ = get(int(e))
        xr = x[pair // wl.top_k].astype(np.float64)
        g = wg.astype(np.float64) @ xr
        u = wu.astype(np.float64) @ xr
        a = O.silu(g) * u
        # BF16 rounding of the FP32 product (half an ulp) plus accumulation-order slack
        assert np.all(np.abs(act[r] - a) <= bf16_ulp(a) + 1e-6)


def test_forward_empty_batch(B):
    wl = S.WORKLOADS["tiny"].replace(T=0)
    p = _params(B, wl)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    d = S.make_inputs(S.WORKLOADS["tiny"], "cuda")
    out = torch.empty((0, wl.H), dtype=torch.bfloat16, device="cuda")
    B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], out=out,
              workspace=dummy)
    assert B.status() == 0


@pytest.mark.parametrize("T,E,n_group", [(64, 256, 8), (1100, 32, 1)])
def test_forward_run_to_run(B, T, E, n_group):
    """Routing is bit-identical across runs. The down projection adds each
    token's expert outputs into its FP32 row with L2 reductions whose order
    varies, so the FP32 output agrees to the rounding of a reordered sum of
    top_k terms (bound 1e-5 of the largest output, far inside the 2e-2
    parity tolerance), and the BF16 output with the residual differs by at
    most one BF16 rounding step plus the FP32 rounding of its two O(1) terms
    (1e-6; it shows where the terms cancel). Weight-major (T=64) and wide
    (T=1100) paths."""
    wl, d = S.make_custom(T=T, H=256, E=E, I=256, n_group=n_group, topk_group=min(4, n_group),
                          top_k=8, seed=77, device="cuda")
    o1, i1, w1, *_ = _run_forward(B, wl, d, B.FLAG_FP32_OUT)
    o2, i2, w2, *_ = _run_forward(B, wl, d, B.FLAG_FP32_OUT)
    assert torch.equal(i1, i2) and torch.equal(w1, w2)
    a, b = host(o1), host(o2)
    assert np.max(np.abs(a - b)) <= 1e-5 * np.max(np.abs(a))
    h1, *_ = _run_forward(B, wl, d, 0, residual_k=9)
    h2, *_ = _run_forward(B, wl, d, 0, residual_k=9)
    a, b = host(h1), host(h2)
    excess = np.abs(a - b) - bf16_ulp(np.maximum(np.abs(a), np.abs(b)))
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess[i] <= 1e-6, f"element {i}: {a[i]} vs {b[i]}"


# Prefill paths (many tokens per expert): E small enough that the mean tokens
# per expert exceeds 24. Covers one and several 256-token groups per expert,
# groups rounded up to 16 tokens, several weight slices in both GEMMs (and a
# last half slice of the down projection when H % 512 == 256), and K loops
# longer than the shared-memory ring.
@pytest.fixture(params=["default", "weight_major"])
def prefill_gemm(request, B):
    """Extra forward flags selecting the prefill GEMM kernels: by default the
    wide 2-SM kernel for both GEMMs; BEAM_FLAG_PREFILL_WEIGHT_MAJOR runs both
    on the weight-major kernel with 128-token tiles."""
    return 0 if request.param == "default" else B.FLAG_PREFILL_WEIGHT_MAJOR


@pytest.mark.parametrize("T,H,I,E,n_group,topk_group,top_k", [
    (300, 256, 256, 32, 1, 1, 8),
    (1100, 512, 256, 32, 1, 1, 8),
    (700, 256, 256, 64, 2, 2, 6),
    (1537, 768, 256, 64, 2, 2, 8),
    (900, 1024, 512, 32, 1, 1, 8),
])
def test_forward_token_major_path(B, prefill_gemm, T, H, I, E, n_group, topk_group, top_k):
    wl, d = S.make_custom(T=T, H=H, E=E, I=I, n_group=n_group, topk_group=topk_group,
                          top_k=top_k, seed=T + E, device="cuda")
    _full_layer_check(B, wl, d, extra_flags=prefill_gemm)


@pytest.mark.parametrize("T,H", [(700, 384), (1500, 640)])
def test_forward_weight_major_wide_tiles(B, T, H):
    """Many tokens per expert with H not a multiple of 256: the weight-major
    GEMMs with 128-token tiles (several tiles per expert)."""
    wl, d = S.make_custom(T=T, H=H, E=32, I=128, n_group=1, topk_group=1, top_k=8,
                          seed=T, device="cuda")
    _full_layer_check(B, wl, d)


def test_forward_token_major_hot_group(B, prefill_gemm):
    """1000 tokens all routed to experts 0..7 (four groups of 250 each) and
    248 empty experts, on the prefill GEMM paths."""
    wl, d = S.make_custom(T=1000, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8,
                          seed=5, device="cuda", router_mode="hot_group")
    _full_layer_check(B, wl, d, extra_flags=prefill_gemm)


def test_forward_token_major_residual(B):
    """Token-major path with pre-norm, post-norm and the residual at k=9."""
    wl = S.Workload("tm_resid", T=900, H=512, E=32, I=256, n_group=1, topk_group=1, seed=6,
                    wr_std=0.05, pre_norm=True, residual_k=9)
    d = S.make_inputs(wl, "cuda")
    p = _params(B, wl, B.FLAG_PRE_NORM, 9)
    ws = B.alloc_workspace(p)
    idx = torch.empty((wl.T, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, 8), dtype=torch.float32, device="cuda")
    hk = B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"],
                   topk_idx=idx, topk_w=w, workspace=ws)
    assert B.status() == 0
    h = host(d["x"]).astype(np.float64)
    xo = _workspace_x(B, ws, p, wl, h)
    sel = O.route(xo, host(d["w_router"]), None, 1, 1, 8, 2.5)
    _, chosen = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    o = oracle_outputs(xo, chosen, np.arange(wl.T), expert_getter(d))
    want = O.residual_step(h, o, 9, None, wl.rms_eps, True)
    assert rel_err(host(hk), want) <= OUT_REL_TOL


# ---------------------------------------------------------------- residual
@pytest.mark.parametrize("fp32_in,norm", [(False, True), (True, True), (False, False)])
def test_residual_step(B, fp32_in, norm):
    h, o = S.residual_inputs(37, 5120, seed=12, device="cuda")
    if fp32_in:
        o = o.float() * 3.0
    gain = (1.0 + 0.1 * torch.randn(5120, generator=torch.Generator().manual_seed(2))).cuda()
    k = 50
    got = B.residual_step(h, o, k, post_gain=gain, eps=1e-6, apply_norm=norm)
    assert B.status() == 0
    want = O.residual_step(host(h), host(o), k, host(gain), 1e-6, norm)
    err = np.abs(host(got) - want)
    # within one BF16 ulp of the FP64 value (the output rounding) plus FP32 slack
    assert np.all(err <= bf16_ulp(want) * 1.0 + 1e-6)


def test_residual_step_in_place(B):
    h, o = S.residual_inputs(8, 256, seed=3, device="cuda")
    want = O.residual_step(host(h), host(o), 9)
    B.residual_step(h, o, 9, out=h)
    assert np.all(np.abs(host(h) - want) <= bf16_ulp(want) + 1e-6)


def test_forward_prenorm_residual_small(B):
    """The long-prefill pipeline at small size: pre-norm, MoE, post-norm,
    residual at k=50."""
    wl = S.Workload("small_long", T=96, H=256, E=256, I=128, seed=4, wr_std=0.05,
                    pre_norm=True, residual_k=50)
    d = S.make_inputs(wl, "cuda")
    p = _params(B, wl, B.FLAG_PRE_NORM, 50)
    ws = B.alloc_workspace(p)
    idx = torch.empty((wl.T, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, 8), dtype=torch.float32, device="cuda")
    hk = B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"],
                   topk_idx=idx, topk_w=w, workspace=ws)
    assert B.status() == 0
    h = host(d["x"]).astype(np.float64)
    # the kernel's BF16 x equals the oracle's except where both roundings are valid
    xo = _workspace_x(B, ws, p, wl, h)
    sel = O.route(xo, host(d["w_router"]), None, 8, 4, 8, 2.5)
    _, chosen = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    o = oracle_outputs(xo, chosen, np.arange(wl.T), expert_getter(d))
    want = O.residual_step(h, o, 50, None, wl.rms_eps, True)
    assert rel_err(host(hk), want) <= OUT_REL_TOL


# ---------------------------------------------------------------- failures
def test_bounded_wait_times_out_and_context_survives(B):
    B.debug_wait_timeout(50_000_000)   # 50 ms, nothing ever arrives
    assert B.status() == 5             # BEAM_ERR_TIMEOUT
    assert "timed out" in B.last_error()
    assert B.status() == 0             # flag cleared
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    idx, w, _ = B.route(_params(B, wl), d["x"], d["w_router"])
    assert B.status() == 0 and idx.shape == (64, 8)


def test_workspace_too_small_is_rejected(B):
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    p = _params(B, wl)
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.BeamError) as ei:
        B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"],
                  workspace=small)
    assert ei.value.code == 3


def test_misaligned_pointer_is_rejected(B):
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    p = _params(B, wl)
    flat = torch.empty(wl.T * wl.H + 1, dtype=torch.bfloat16, device="cuda")
    xs = flat[1:].view(wl.T, wl.H)
    with pytest.raises(B.BeamError) as ei:
        B.route(p, xs, d["w_router"])
    assert ei.value.code == 1


def test_empty_batch_every_entry_point(B):
    """T = 0 returns BEAM_OK without launching work for the quantised-expert
    layers, the dense MLP and the attention sublayer, with a workspace of a
    few bytes."""
    base, d = S.make_custom(T=1, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8,
                            seed=5, device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    fp8 = tuple(B.quantize_e4m3_rows(d[k]) for k in ("w_gate", "w_up", "w_down"))
    f4 = tuple(B.quantize_nvfp4(d[k]) for k in ("w_gate", "w_up", "w_down"))
    assert B.status() == 0, B.last_error()
    for flag, q, fwd in ((B.FLAG_FP8_EXPERTS, fp8, B.forward_fp8),
                         (B.FLAG_NVFP4_EXPERTS, f4, B.forward_nvfp4)):
        p = B.make_params(0, base.H, base.E, base.I, base.n_group, base.topk_group, base.top_k,
                          base.routed_scale, base.rms_eps, 0, flag)
        out = torch.empty((0, base.H), dtype=torch.bfloat16, device="cuda")
        fwd(p, d["x"], d["w_router"], *q, out=out, workspace=dummy)
        assert B.status() == 0, B.last_error()
    out = torch.empty((0, base.H), dtype=torch.bfloat16, device="cuda")
    B.dense_forward(0, base.H, base.I, d["x"], d["w_gate"][0], d["w_up"][0], d["w_down"][0],
                    out=out, workspace=dummy)
    assert B.status() == 0, B.last_error()
    a = S.attn_inputs(1, 256, 4, 2, 3, "cuda", head_dim=128)
    pa = B.make_attn_params(0, 256, 4, 2, 128, 512, 10000.0, 1e-6, 0, 0)
    out = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    B.attention_forward(pa, a["x"], a["w_qkvg"], a["w_o"], a["q_gain"], a["k_gain"], out=out,
                        workspace=dummy)
    assert B.status() == 0, B.last_error()
