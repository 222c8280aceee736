"""GPU parity of the NVFP4 expert-weight path (E2M1 codes, E4M3 block
scales per 16 elements, FP32 group scales; the FP4 tensor cores with block
scaling) against the oracle's NVFP4 restatement: the quantiser (codes,
block scales, group scales) exact, the quantised expert input exact, every
SwiGLU row's quantisation validated, and the sublayer output within the
output tolerance on the decode (32-token) and 128-token tiles, with
pre-norm and residual, and the dense MLP. All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O
from _helpers import (OUT_REL_TOL, act_rows_reader_nvfp4, check_act_codes_nvfp4,
                      compare_routing, expert_getter_nvfp4, host, nvfp4_pad,
                      oracle_outputs_nvfp4_checked, rel_err, validated_prenorm_x,
                      sf_groups_to_plain, weights_from_chosen)

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
                         wl.routed_scale, wl.rms_eps, residual_k, flags | B.FLAG_NVFP4_EXPERTS)


def _quantize_experts(B, d):
    q = tuple(B.quantize_nvfp4(d[k]) for k in ("w_gate", "w_up", "w_down"))
    assert B.status() == 0, B.last_error()
    return q


def _check_quantiser(w, q, rows_per_group):
    """Library NVFP4 codes, block scales and group scales equal the oracle's
    (codes compared by value: a signed and an unsigned zero are both 0)."""
    a = w.float().cpu().numpy().reshape(-1, w.shape[-1])
    R, K = a.shape
    pk, sb, g = O.quantize_nvfp4(a, rows_per_group)
    got_codes = q[0].cpu().numpy().reshape(R, K // 2)
    assert np.array_equal(O.e2m1_decode(O.unpack_e2m1(got_codes)),
                          O.e2m1_decode(O.unpack_e2m1(pk)))
    assert np.array_equal(sf_groups_to_plain(q[1].cpu().numpy(), R, K), sb)
    assert np.array_equal(q[2].cpu().numpy(), g)


def _run(B, wl, d, q, flags=0, residual_k=0):
    p = _params(B, wl, flags, residual_k)
    ws = B.alloc_workspace(p)
    idx = torch.empty((wl.T, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((wl.T, wl.top_k), dtype=torch.float32, device="cuda")
    out = B.forward_nvfp4(p, d["x"], d["w_router"], *q, bias=d["bias"], topk_idx=idx, topk_w=w,
                          workspace=ws)
    assert B.status() == 0, B.last_error()
    return out, idx, w, ws, p


def _layer_check(B, wl, d, q=None, extra_flags=0):
    if q is None:
        q = _quantize_experts(B, d)
    out, idx, w, ws, p = _run(B, wl, d, q, B.FLAG_FP32_OUT | extra_flags)
    x = host(d["x"]).astype(np.float64)
    sel = O.route(x, host(d["w_router"]), host(d["bias"]), wl.n_group, wl.topk_group,
                  wl.top_k, wl.routed_scale)
    ties, chosen = compare_routing(sel, idx.cpu().numpy(), w.cpu().numpy(), wl)
    want = oracle_outputs_nvfp4_checked(
        x, idx.cpu().numpy(), weights_from_chosen(chosen), expert_getter_nvfp4(*q),
        act_rows_reader_nvfp4(ws, B.workspace_layout(p), wl.I, nvfp4_pad(wl.T, wl.top_k, wl.E)),
        wl.E, nvfp4_pad(wl.T, wl.top_k, wl.E))
    err = rel_err(host(out), want)
    assert err <= OUT_REL_TOL, f"rel err {err}"
    return out, idx, w, ws, p, sel, ties, q


# ------------------------------------------------------------- quantiser
def test_quantizer_exact(B):
    g = torch.Generator().manual_seed(23)
    w = torch.randn(4, 256, 512, generator=g) * 0.02
    w[1] *= 50.0                                  # a matrix with a different group scale
    w[2, 7, :] = 0.0                              # a zero row
    w[2, 9, 16:32] = 1e-6                         # a block whose scale rounds to zero
    w[3, 0, 5] = 3.0                              # one large element
    w = w.to(torch.bfloat16).cuda()
    q = B.quantize_nvfp4(w)
    assert B.status() == 0, B.last_error()
    assert q[0].shape == (4, 256, 256) and q[1].numel() == 4 * 256 * 512 // 16 and q[2].shape == (4,)
    _check_quantiser(w, q, 256)
    # one scale per row (the activations' grouping)
    w2 = (torch.randn(256, 320 * 2, generator=g) * torch.exp(torch.randn(256, 1, generator=g))).to(torch.bfloat16).cuda()
    q2 = B.quantize_nvfp4(w2, rows_per_group=1)
    _check_quantiser(w2, q2, 1)


# ------------------------------------------------------------- the layer
def test_nvfp4_forward_small(B):
    wl, d = S.make_custom(T=64, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8,
                          seed=91, device="cuda")
    q = _quantize_experts(B, d)
    for name, k in (("w_gate", 0), ("w_up", 1), ("w_down", 2)):
        _check_quantiser(d[name], q[k], d[name].shape[1])
    out, idx, w, ws, p, sel, ties, _ = _layer_check(B, wl, d, q)
    # the quantised expert input (padded expert order) equals the oracle's
    lay = B.workspace_layout(p)
    perm = O.permutation(idx.cpu().numpy(), wl.E)
    pad = nvfp4_pad(wl.T, wl.top_k, wl.E)
    poff = np.concatenate([[0], np.cumsum((perm["counts"] + pad - 1) // pad * pad)])
    nrows = int(poff[-1])
    raw = ws.cpu()
    xc = raw[lay["xperm"]:lay["xperm"] + nrows * wl.H // 2].numpy().reshape(nrows, wl.H // 2)
    xsf = sf_groups_to_plain(raw[lay["x_sf"]:lay["x_sf"] + (nrows // pad) * (wl.H // 64) * 512].numpy(),
                             nrows, wl.H, pad)
    xg = raw[lay["x_scale"]:lay["x_scale"] + nrows * 4].view(torch.float32).numpy()
    x = host(d["x"])
    for e in np.nonzero(perm["counts"])[0][:64]:
        pr = perm["row_pair"][perm["offsets"][e]:perm["offsets"][e + 1]]
        rows = poff[e] + np.arange(len(pr))
        pk, sb, g = O.quantize_nvfp4(x[pr // wl.top_k], 1)
        assert np.array_equal(O.e2m1_decode(O.unpack_e2m1(xc[rows])), O.e2m1_decode(O.unpack_e2m1(pk)))
        assert np.array_equal(xsf[rows], sb) and np.array_equal(xg[rows], g)
        pad_rows = np.arange(poff[e] + len(pr), poff[e + 1])
        assert np.all(xc[pad_rows] == 0) and np.all(xsf[pad_rows] == 0)


@pytest.mark.parametrize("T,H,I", [(1, 256, 256), (7, 256, 512), (64, 512, 256),
                                   (300, 256, 256), (129, 512, 512)])
def test_nvfp4_forward_shape_sweep(B, T, H, I):
    wl, d = S.make_custom(T=T, H=H, E=256, I=I, n_group=8, topk_group=4, top_k=8,
                          seed=T + H + I + 2, device="cuda")
    _layer_check(B, wl, d)


@pytest.mark.parametrize("T,H,I", [(90, 512, 512), (40, 768, 2560), (40, 512, 3840)])
def test_nvfp4_down_two_tile_units(B, T, H, I):
    """The decode-shaped NVFP4 down GEMM runs 256 hidden rows (two weight
    tiles into two accumulators) per unit: about 22 tokens per expert (some
    experts with two 32-token tiles), three units per expert (H = 768), and
    long rows (I = 3840, 15 K-blocks of 256)."""
    wl, d = S.make_custom(T=T, H=H, E=32, I=I, n_group=1, topk_group=1, top_k=8,
                          seed=T + H + I + 5, device="cuda")
    _layer_check(B, wl, d)


@pytest.mark.parametrize("mode", ["hot_expert", "hot_group"])
def test_nvfp4_forward_routing_edge_cases(B, mode):
    wl, d = S.make_custom(T=300, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8,
                          seed=33, device="cuda", router_mode=mode)
    _layer_check(B, wl, d)


@pytest.fixture(params=["tm", "weight_major"])
def nvfp4_prefill_gemm(request, B):
    """Many tokens per expert: the token-major two-CTA kernel (default) or,
    with BEAM_FLAG_PREFILL_WEIGHT_MAJOR, the weight-major kernel with
    128-token tiles."""
    return 0 if request.param == "tm" else B.FLAG_PREFILL_WEIGHT_MAJOR


@pytest.mark.parametrize("T,H,I", [(700, 256, 256), (1100, 512, 256), (1537, 768, 512)])
def test_nvfp4_forward_128_token_tiles(B, T, H, I, nvfp4_prefill_gemm):
    """Many tokens per expert: expert rows padded to 128, 128-row token tiles."""
    wl, d = S.make_custom(T=T, H=H, E=32, I=I, n_group=1, topk_group=1, top_k=8,
                          seed=T + 3, device="cuda")
    _layer_check(B, wl, d, extra_flags=nvfp4_prefill_gemm)


@pytest.mark.parametrize("mode", ["hot_expert", "hot_group"])
def test_nvfp4_prefill_routing_edge_cases(B, mode, nvfp4_prefill_gemm):
    """Token-major tiles under skewed routing: one expert with most rows
    (many 256-row groups and a tail) and experts with a handful of rows."""
    wl, d = S.make_custom(T=1200, H=256, E=32, I=256, n_group=1, topk_group=1, top_k=8,
                          seed=57, device="cuda", router_mode=mode)
    _layer_check(B, wl, d, extra_flags=nvfp4_prefill_gemm)


def test_nvfp4_forward_run_to_run(B):
    wl, d = S.make_custom(T=900, H=256, E=32, I=256, n_group=1, topk_group=1, top_k=8,
                          seed=79, device="cuda")
    q = _quantize_experts(B, d)
    o1, i1, *_ = _run(B, wl, d, q, B.FLAG_FP32_OUT)
    o2, i2, *_ = _run(B, wl, d, q, B.FLAG_FP32_OUT)
    # routing bit-identical; the combined FP32 output to the rounding of a
    # reordered sum (L2 reductions in the down projection's epilogue)
    assert torch.equal(i1, i2)
    x, y = host(o1), host(o2)
    assert np.max(np.abs(x - y)) <= 1e-5 * np.max(np.abs(x))


def test_nvfp4_prenorm_residual(B):
    wl = S.Workload("f4_long", T=96, H=256, E=256, I=256, seed=45, wr_std=0.05,
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
    o = oracle_outputs_nvfp4_checked(
        xo, idx.cpu().numpy(), weights_from_chosen(chosen), expert_getter_nvfp4(*q),
        act_rows_reader_nvfp4(ws, lay, wl.I, nvfp4_pad(wl.T, wl.top_k, wl.E)),
        wl.E, nvfp4_pad(wl.T, wl.top_k, wl.E))
    want = O.residual_step(h, o, 50, None, wl.rms_eps, True)
    assert rel_err(host(hk), want) <= OUT_REL_TOL


def test_nvfp4_rejects_wrong_flags(B):
    wl, d = S.make_custom(T=8, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8,
                          seed=1, device="cuda")
    q = _quantize_experts(B, d)
    p = B.make_params(wl.T, wl.H, wl.E, wl.I)
    with pytest.raises(B.BeamError) as ei:
        B.forward_nvfp4(p, d["x"], d["w_router"], *q)
    assert ei.value.code == 1
    p = B.make_params(8, 256, 256, 128, flags=B.FLAG_NVFP4_EXPERTS)   # I % 256 != 0
    dummy = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.BeamError) as ei:
        B.forward_nvfp4(p, d["x"], d["w_router"], *q, workspace=dummy)
    assert ei.value.code == 2


# ------------------------------------------------------------- dense MLP
@pytest.mark.parametrize("T,H,I,resid", [(5, 256, 512, 0), (300, 512, 768, 0),
                                         (1030, 256, 512, 0), (200, 256, 512, 3)])
def test_nvfp4_dense_mlp(B, T, H, I, resid):
    x, wg, wu, wd = S.dense_inputs(T, H, I, seed=T + I + 1, device="cuda")
    q = tuple(B.quantize_nvfp4(w[None]) for w in (wg, wu, wd))
    q = tuple((c[0], sf, g) for c, sf, g in q)
    flags = B.FLAG_NVFP4_EXPERTS | (0 if resid else B.FLAG_FP32_OUT)
    dp = B.DenseParams(T, H, I, 1e-6, resid, flags)
    ws = torch.empty(B.dense_workspace_size(dp), dtype=torch.uint8, device="cuda")
    out = B.dense_forward_nvfp4(T, H, I, x, *q, residual_k=resid, flags=flags, workspace=ws)
    assert B.status() == 0, B.last_error()
    xh = host(x).astype(np.float64)
    qh = tuple((c.cpu().numpy(), sf_groups_to_plain(sf.cpu().numpy(), c.shape[0], 2 * c.shape[1]),
                g.cpu().numpy()) for c, sf, g in q)
    a64 = O.swiglu_act_nvfp4(xh, qh[0], qh[1])
    lay = B.dense_workspace_layout(dp)
    rows = np.arange(T)
    codes, sf, g = act_rows_reader_nvfp4(ws, lay, I, 32 if T <= 24 else 128)(rows)
    codes, sf, g = check_act_codes_nvfp4(a64, codes, sf, g)
    y = O.dequantize_nvfp4(codes, sf, g, 1) @ O.dequantize_nvfp4(*qh[2], H).T
    want = O.residual_step(xh, y, resid) if resid else y
    assert rel_err(host(out), want) <= OUT_REL_TOL
