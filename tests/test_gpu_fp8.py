"""GPU parity of the E4M3 (FP8) expert-weight path against the oracle's FP8
restatement: the row quantiser bit-exact (codes and scales), the quantised
expert input bit-exact, and the sublayer output within the output tolerance
on every GEMM path (weight-major decode tiles, 128-token tiles, the
token-major prefill kernels), with pre-norm and residual, and the dense MLP.
All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O
from _helpers import (OUT_REL_TOL, act_rows_reader, check_act_codes_fp8, compare_routing,
                      expert_getter_fp8, host, oracle_outputs_fp8_checked, validated_prenorm_x,
                      rel_err, weights_from_chosen)

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
                         wl.routed_scale, wl.rms_eps, residual_k, flags | B.FLAG_FP8_EXPERTS)


def _quantize_experts(B, d):
    q = tuple(B.quantize_e4m3_rows(d[k]) for k in ("w_gate", "w_up", "w_down"))
    assert B.status() == 0, B.last_error()
    return q


def _check_codes(B, w, q):
    """GPU codes and scales of a weight tensor equal the oracle quantiser's."""
    a = w.float().cpu().numpy().reshape(-1, w.shape[-1])
    want_c, want_s = O.quantize_rows_e4m3(a)
    assert np.array_equal(q[0].cpu().numpy().reshape(a.shape), want_c)
    assert np.array_equal(q[1].cpu().numpy().reshape(-1), want_s)


def _run(B, wl, d, q, flags=0, residual_k=0, pre_gain=None):
    p = _params(B, wl, flags, residual_k)
    ws = B.alloc_workspace(p)
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device="cuda")
    out = B.forward_fp8(p, d["x"], d["w_router"], *q, bias=d["bias"], pre_gain=pre_gain,
                        topk_idx=idx, topk_w=w, workspace=ws)
    assert B.status() == 0, B.last_error()
    return out, idx, w, ws, p


def _expected(x64, idx, chosen, q, ws, lay, wl):
    """Oracle FP8 output per token, with every pair row's SwiGLU codes and
    scale validated against the GPU's workspace."""
    want, ok = oracle_outputs_fp8_checked(x64, idx.cpu().numpy(), weights_from_chosen(chosen),
                                          expert_getter_fp8(*q), act_rows_reader(ws, lay, wl.I),
                                          wl.E)
    return want, ok


def _layer_check(B, wl, d, q=None, extra_flags=0):
    if q is None:
        q = _quantize_experts(B, d)
    out, idx, w, ws, p = _run(B, wl, d, q, B.FLAG_FP32_OUT | extra_flags)
    x = host(d["x"]).astype(np.float64)
    sel = O.route(x, host(d["w_router"]), host(d["bias"]), wl.n_group, wl.topk_group,
                  wl.top_k, wl.routed_scale)
    ties, chosen = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    want, ok = _expected(x, idx, chosen, q, ws, B.workspace_layout(p), wl)
    err = rel_err(host(out)[ok], want[ok])
    assert err <= OUT_REL_TOL, f"rel err {err}"
    return out, idx, w, ws, p, sel, ties, q


# ------------------------------------------------------------- quantiser
def test_quantizer_bitexact(B):
    g = torch.Generator().manual_seed(17)
    a = torch.randn(300, 640, generator=g) * torch.exp(torch.randn(300, 1, generator=g) * 4)
    a[3] = 0.0                                   # zero row: scale 1, codes 0
    a[5, :] = 1e-30                              # tiny but non-zero row: all codes 448
    a[7, ::2] = 3e-4                             # subnormal codes beside a large value
    a[7, 1] = 200.0
    a[9, 10] = -5e4                              # large magnitude
    w = a.to(torch.bfloat16).cuda()
    q = B.quantize_e4m3_rows(w)
    assert B.status() == 0
    _check_codes(B, w, q)
    # a 3-D expert tensor is quantised row by row over its last dimension
    w3 = (torch.randn(4, 128, 256, generator=g) * 0.02).to(torch.bfloat16).cuda()
    q3 = B.quantize_e4m3_rows(w3)
    assert q3[0].shape == (4, 128, 256) and q3[1].shape == (4, 128)
    _check_codes(B, w3, q3)


# ------------------------------------------------------------- the layer
def test_fp8_forward_tiny(B):
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    q = _quantize_experts(B, d)
    for name, k in (("w_gate", 0), ("w_up", 1), ("w_down", 2)):
        _check_codes(B, d[name], q[k])
    out, idx, w, ws, p, sel, ties, _ = _layer_check(B, wl, d, q)
    # the quantised expert input in expert order is bit-exact
    if ties.sum() == 0:
        lay = B.workspace_layout(p)
        R = wl.T * wl.top_k
        raw = ws.cpu()
        perm = O.permutation(sel["idx"], wl.E)
        xc = raw[lay["xperm"]:lay["xperm"] + R * wl.H].numpy().reshape(R, wl.H)
        xs = raw[lay["x_scale"]:lay["x_scale"] + R * 4].view(torch.float32).numpy()
        want_c, want_s = O.quantize_rows_e4m3(host(d["x"])[perm["row_pair"] // wl.top_k])
        assert np.array_equal(xc, want_c) and np.array_equal(xs, want_s)


@pytest.mark.parametrize("T,H,I", [(1, 256, 128), (7, 256, 256), (64, 512, 128),
                                   (300, 256, 128), (129, 512, 256)])
def test_fp8_forward_shape_sweep(B, T, H, I):
    wl, d = S.make_custom(T=T, H=H, E=256, I=I, n_group=8, topk_group=4, top_k=8,
                          seed=T + H + I + 1, device="cuda")
    _layer_check(B, wl, d)


@pytest.mark.parametrize("mode", ["hot_expert", "hot_group"])
def test_fp8_forward_routing_edge_cases(B, mode):
    wl, d = S.make_custom(T=300, H=256, E=256, I=128, n_group=8, topk_group=4, top_k=8,
                          seed=32, device="cuda", router_mode=mode)
    _layer_check(B, wl, d)


@pytest.fixture(params=["default", "weight_major"])
def prefill_gemm(request, B):
    """The prefill GEMM kernels (as in the BF16 tests): the wide 2-SM kernel,
    or the weight-major kernel with BEAM_FLAG_PREFILL_WEIGHT_MAJOR."""
    return 0 if request.param == "default" else B.FLAG_PREFILL_WEIGHT_MAJOR


@pytest.mark.parametrize("T,H,I,E,n_group,topk_group,top_k", [
    (300, 256, 256, 32, 1, 1, 8),
    (1100, 512, 256, 32, 1, 1, 8),
    (1537, 768, 256, 64, 2, 2, 8),
])
def test_fp8_forward_token_major(B, prefill_gemm, T, H, I, E, n_group, topk_group, top_k):
    wl, d = S.make_custom(T=T, H=H, E=E, I=I, n_group=n_group, topk_group=topk_group,
                          top_k=top_k, seed=T + E + 1, device="cuda")
    _layer_check(B, wl, d, extra_flags=prefill_gemm)


def test_fp8_forward_weight_major_wide_tiles(B):
    """Many tokens per expert, H not a multiple of 256: 128-token tiles."""
    wl, d = S.make_custom(T=700, H=384, E=32, I=128, n_group=1, topk_group=1, top_k=8,
                          seed=70, device="cuda")
    _layer_check(B, wl, d)


def test_fp8_forward_run_to_run(B):
    """Routing and the quantised activations are bit-identical across runs;
    the combined FP32 output agrees to the rounding of a reordered sum (the
    down projection's L2 reductions land in a varying order)."""
    wl, d = S.make_custom(T=1100, H=256, E=32, I=256, n_group=1, topk_group=1, top_k=8,
                          seed=78, device="cuda")
    q = _quantize_experts(B, d)
    o1, i1, w1, ws1, p = _run(B, wl, d, q, B.FLAG_FP32_OUT)
    o2, i2, w2, ws2, _ = _run(B, wl, d, q, B.FLAG_FP32_OUT)
    assert torch.equal(i1, i2) and torch.equal(w1, w2)
    lay = B.workspace_layout(p)
    R = wl.T * wl.top_k
    a = slice(lay["act_q"], lay["act_q"] + R * wl.I)
    assert torch.equal(ws1[a], ws2[a])
    x, y = host(o1), host(o2)
    assert np.max(np.abs(x - y)) <= 1e-5 * np.max(np.abs(x))


def test_fp8_prenorm_residual(B):
    """Pre-norm, FP8 experts, post-norm and the residual at k = 50."""
    wl = S.Workload("f8_long", T=96, H=256, E=256, I=128, seed=44, wr_std=0.05,
                    pre_norm=True, residual_k=50)
    d = S.make_inputs(wl, "cuda")
    q = _quantize_experts(B, d)
    hk, idx, w, ws, p = _run(B, wl, d, q, B.FLAG_PRE_NORM, 50)
    h = host(d["x"]).astype(np.float64)
    lay = B.workspace_layout(p)
    xg = ws[lay["xn"]:lay["xn"] + wl.T * wl.H * 2].view(torch.bfloat16).float().cpu().numpy()
    # the GPU's BF16 x, each element the oracle's rounding or (on a midpoint) the other one
    xo, _ = validated_prenorm_x(xg.reshape(wl.T, wl.H), h, None, wl.rms_eps)
    sel = O.route(xo, host(d["w_router"]), None, 8, 4, 8, 2.5)
    _, chosen = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    o, _ = _expected(xo, idx, chosen, q, ws, lay, wl)
    want = O.residual_step(h, o, 50, None, wl.rms_eps, True)
    assert rel_err(host(hk), want) <= OUT_REL_TOL


def test_fp8_rejects_missing_flag(B):
    wl = S.WORKLOADS["tiny"]
    d = S.make_inputs(wl, "cuda")
    q = _quantize_experts(B, d)
    p = B.make_params(wl.T, wl.H, wl.E, wl.I)        # no FLAG_FP8_EXPERTS
    with pytest.raises(B.BeamError) as ei:
        B.forward_fp8(p, d["x"], d["w_router"], *q)
    assert ei.value.code == 1


# ------------------------------------------------------------- dense MLP
@pytest.mark.parametrize("T,H,I,resid", [(5, 256, 384, 0), (300, 512, 768, 0),
                                         (1030, 256, 512, 0), (200, 256, 384, 3)])
def test_fp8_dense_mlp(B, T, H, I, resid):
    x, wg, wu, wd = S.dense_inputs(T, H, I, seed=T + I, device="cuda")
    q = tuple(B.quantize_e4m3_rows(w) for w in (wg, wu, wd))
    flags = B.FLAG_FP8_EXPERTS | (0 if resid else B.FLAG_FP32_OUT)
    dp = B.DenseParams(T, H, I, 1e-6, resid, flags)
    ws = torch.empty(B.dense_workspace_size(dp), dtype=torch.uint8, device="cuda")
    out = B.dense_forward_fp8(T, H, I, x, *q, residual_k=resid, flags=flags, workspace=ws)
    assert B.status() == 0, B.last_error()
    xh = host(x).astype(np.float64)
    qh = tuple((c.cpu().numpy(), s.cpu().numpy()) for c, s in q)
    a64 = O.swiglu_act_fp8(xh, qh[0], qh[1])
    lay = B.dense_workspace_layout(dp)
    raw = ws.cpu()
    act_q = raw[lay["act_q"]:lay["act_q"] + T * I].numpy().reshape(T, I)
    act_s = raw[lay["act_scale"]:lay["act_scale"] + T * 4].view(torch.float32).numpy()
    ok, codes, scale = check_act_codes_fp8(a64, act_q, act_s)
    assert ok.mean() >= 0.9
    y = O.dequantize_rows_e4m3(codes, scale) @ O.dequantize_rows_e4m3(*qh[2]).T
    want = O.residual_step(xh, y, resid) if resid else y
    assert rel_err(host(out)[ok], want[ok]) <= OUT_REL_TOL
