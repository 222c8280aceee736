"""The allocation-free router, beam_moe_route_static, against beam_moe_route.

beam_moe_route_static serves callers that cannot allocate device memory: it
keeps its scratch in a fixed array inside the library instead of a caller
workspace. Both entry points run the same kernels, so two calls in a row of
the static one (on different inputs, so stale scratch contents would show)
must give what the workspace entry point gives, within the routing
tolerances the other tests use. All calls go through the C ABI.

This file is collected last on purpose, and it also passes on its own in a
fresh process.
"""
import numpy as np
import pytest
import torch

import beam_synth as S

pytestmark = pytest.mark.gpu

W_TOL = 1e-5      # combine weights, absolute (the routing tolerance of the other tests)
S_TOL = 2e-6      # sigmoid scores, absolute


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    return B


def _case(B, wl, seed, flags):
    wl = wl.replace(seed=seed)
    d = S.make_inputs(wl, "cuda")
    gain = None
    if flags & B.FLAG_PRE_NORM:
        gain = (1.0 + 0.1 * torch.randn(wl.H, generator=torch.Generator().manual_seed(seed)))
        gain = gain.cuda()
    p = B.make_params(wl.T, wl.H, wl.E, wl.I, wl.n_group, wl.topk_group, wl.top_k,
                      wl.routed_scale, wl.rms_eps, 0, flags)
    return p, d, gain


def _compare(B, p, d, gain):
    ref_idx, ref_w, ref_s = B.route(p, d["x"], d["w_router"], bias=d["bias"], pre_gain=gain)
    idx, w, sc = B.route_static(p, d["x"], d["w_router"], bias=d["bias"], pre_gain=gain)
    assert B.status() == 0, B.last_error()
    assert torch.equal(idx, ref_idx)
    assert torch.max(torch.abs(w - ref_w)).item() <= W_TOL
    if ref_s is not None:
        assert torch.max(torch.abs(sc - ref_s)).item() <= S_TOL
    assert np.allclose(w.sum(1).cpu().numpy(), p.routed_scale, atol=W_TOL)


@pytest.mark.parametrize("name,flags", [
    ("tiny", "scores"),            # H=256: with the sigmoid scores returned
    ("decode", "prenorm"),         # Beam shapes, T=64, pre-norm + logit bias
])
def test_route_static_matches_route_on_two_calls(B, name, flags):
    wl = S.WORKLOADS[name]
    if name == "decode":
        # the router needs no expert weights: a small I keeps the inputs light
        wl = wl.replace(I=128, skew_bias=True)
    f = B.FLAG_RETURN_SCORES if flags == "scores" else B.FLAG_PRE_NORM
    for seed in (wl.seed, wl.seed + 17):       # two calls in a row, different inputs
        p, d, gain = _case(B, wl, seed, f)
        _compare(B, p, d, gain)


def test_route_static_tensor_core_router_on_two_calls(B):
    """T >= 512 with E = 256: the router runs on the tensor cores, so the
    static scratch also holds the three-way BF16 split of the router weight
    and the router GEMM's work list. Small H keeps it inside the limit."""
    wl = S.WORKLOADS["tiny"].replace(T=512)
    for seed in (3, 29):                       # two calls in a row, different inputs
        p, d, gain = _case(B, wl, seed, B.FLAG_RETURN_SCORES)
        _compare(B, p, d, gain)


def test_route_static_rejects_oversize_without_launching(B):
    wl = S.WORKLOADS["long_prefill"]
    p = B.make_params(wl.T, wl.H, wl.E, wl.I, flags=B.FLAG_PRE_NORM)
    x = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.BeamError) as ei:
        B.route_static(p, x, x, topk_idx=x, topk_w=x)
    assert ei.value.code == 2
    assert "static scratch holds 8388608 bytes" in str(ei.value)
    assert B.status() == 0
