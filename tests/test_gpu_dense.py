"""GPU parity of the dense SwiGLU MLP sublayer (the first layers of the model)
against the oracle, through the C ABI. It runs on the expert GEMM kernels as
one expert that every token uses, so these cases cover small and large T
(both GEMM paths), ragged sizes, pre-norm and the residual step."""
import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O
from _helpers import OUT_REL_TOL, host, rel_err, validated_prenorm_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    return B


def _check(B, T, H, I, seed, pre_norm=False, residual_k=0, fp32_out=False, sample=None):
    x, wg, wu, wd = S.dense_inputs(T, H, I, seed, "cuda")
    flags = (B.FLAG_PRE_NORM if pre_norm else 0) | (B.FLAG_FP32_OUT if fp32_out else 0)
    dp = B.DenseParams(T, H, I, 1e-6, residual_k, flags)
    ws = torch.empty(B.dense_workspace_size(dp), dtype=torch.uint8, device="cuda")
    out = B.dense_forward(T, H, I, x, wg, wu, wd, residual_k=residual_k, flags=flags, workspace=ws)
    assert B.status() == 0, B.last_error()
    toks = np.arange(T) if sample is None else sample
    h64 = host(x).astype(np.float64)[toks]
    if pre_norm:
        # the GPU's BF16 x, each element the oracle's rounding or (on a
        # midpoint) the other one; the oracle's MLP runs on it
        lay = B.dense_workspace_layout(dp)
        xg = ws[lay["xn"]:lay["xn"] + T * H * 2].view(torch.bfloat16).float().cpu().numpy()
        xn, _ = validated_prenorm_x(xg.reshape(T, H)[toks], h64, None, 1e-6)
        r = O.dense_mlp_forward(xn, host(wg), host(wu), host(wd), pre_norm=False)
        want = O.residual_step(h64, r["out"], residual_k) if residual_k else r["out"]
    else:
        r = O.dense_mlp_forward(h64, host(wg), host(wu), host(wd), pre_norm=False,
                                residual_k=residual_k)
        want = r["h"] if residual_k else r["out"]
    err = rel_err(host(out)[toks], want)
    assert err <= OUT_REL_TOL, f"rel err {err}"
    return err


@pytest.mark.parametrize("T,H,I", [(1, 256, 128), (7, 256, 384), (24, 512, 128),
                                   (64, 256, 256), (300, 512, 128), (1000, 256, 384),
                                   (333, 384, 256), (600, 512, 512), (1000, 768, 256)])
def test_dense_shapes(B, T, H, I):
    _check(B, T, H, I, seed=T + I, fp32_out=True)


@pytest.mark.parametrize("T", [5, 700])
def test_dense_prenorm_residual(B, T):
    _check(B, T, 512, 256, seed=3 + T, pre_norm=True, residual_k=5)


def test_dense_full_size_prefill(B):
    """Beam hidden size 5120, intermediate 12288 (a stand-in: the pages do not
    give it), T=8192; sampled tokens checked one by one."""
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(8192, 24, replace=False))
    err = _check(B, 8192, 5120, 12288, seed=5, pre_norm=True, residual_k=3, sample=sample)
    print(f"dense T=8192: rel err {err:.2e}")


def test_dense_full_size_decode(B):
    err = _check(B, 64, 5120, 12288, seed=6, fp32_out=True)
    print(f"dense T=64: rel err {err:.2e}")
