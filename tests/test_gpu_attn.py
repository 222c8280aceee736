"""GPU parity of the attention sublayer (fused Q/K/V/gate projection on the
2-SM tcgen05 GEMM, QK-RMSNorm, RoPE or the global query scale, tcgen05 flash
attention with causal and sliding-window masks, sigmoid gate, output
projection, post-norm and residual) against the oracle. All calls go
through the C ABI."""
import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O
from _helpers import host, rel_err

pytestmark = pytest.mark.gpu

# Tolerance derived from the arithmetic (the oracle is FP64 throughout): P
# enters the P V tensor-core product as BF16 (relative 2^-9 per weight) and
# the gated output is rounded to BF16 (2^-9), so each element of the output
# projection's input differs by about 2^-8 relative and flips BF16 roundings
# of the large outputs of early rows (row 0 attends to one key); the output
# projection sums 6144 such terms with random signs: about 0.4% per output
# element, 2% at the tails. Bound: max |err| / RMS <= 5e-2 and RMS(err) /
# RMS <= 1e-2.
ATT_MAX_TOL = 5e-2
ATT_RMS_TOL = 1e-2


def _rms_rel(got, want):
    want = np.asarray(want, dtype=np.float64)
    d = np.asarray(got, dtype=np.float64) - want
    return float(np.sqrt(np.mean(d * d)) / np.sqrt(np.mean(want * want)))


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    return B


def _check(B, T, H, nq, nkv, window, seed, pre_norm=False, residual_k=0, rows=None, gain=None):
    d = S.attn_inputs(T, H, nq, nkv, seed, "cuda")
    if gain is not None:   # constant q and k gains (sets the layer's logit bound)
        d["q_gain"] = torch.full((128,), gain, dtype=torch.float32, device="cuda")
        d["k_gain"] = torch.full((128,), gain, dtype=torch.float32, device="cuda")
    flags = (B.FLAG_PRE_NORM if pre_norm else 0) | (0 if residual_k else B.FLAG_FP32_OUT)
    p = B.make_attn_params(T, H, nq, nkv, 128, window, 10000.0, 1e-6, residual_k, flags)
    out = B.attention_forward(p, d["x"], d["w_qkvg"], d["w_o"], d["q_gain"], d["k_gain"])
    assert B.status() == 0, B.last_error()
    ref = O.attention_forward(host(d["x"]), host(d["w_qkvg"]), host(d["w_o"]), host(d["q_gain"]),
                              host(d["k_gain"]), n_q=nq, n_kv=nkv, window=window,
                              pre_norm=pre_norm, residual_k=residual_k, query_rows=rows)
    want = ref["h"] if residual_k else ref["out"]
    got = host(out) if rows is None else host(out)[rows]
    err, rms = rel_err(got, want), _rms_rel(got, want)
    assert err <= ATT_MAX_TOL and rms <= ATT_RMS_TOL, f"max err {err}, rms err {rms}"
    return err


@pytest.mark.parametrize("T", [1, 100, 128, 129, 300])
@pytest.mark.parametrize("window", [512, 0])
def test_attention_small(B, T, window):
    _check(B, T, 256, 48, 8, window, seed=T + window)


@pytest.mark.parametrize("T,window", [(300, 64), (700, 512), (700, 0), (1000, 200)])
def test_attention_windows_across_tiles(B, T, window):
    """Windows that start inside earlier key tiles and causal masks over
    several query and key tiles."""
    _check(B, T, 256, 48, 8, window, seed=T + 7)


def test_attention_other_head_grouping(B):
    _check(B, 200, 512, 6, 2, 96, seed=3)
    _check(B, 200, 256, 16, 16, 0, seed=4)


def test_attention_prenorm_residual(B):
    _check(B, 260, 256, 48, 8, 512, seed=5, pre_norm=True, residual_k=4)
    _check(B, 260, 256, 48, 8, 0, seed=6, pre_norm=True, residual_k=30)


@pytest.mark.parametrize("T,window", [(500, 512), (2000, 0)])
def test_attention_run_to_run(B, T, window):
    """Bitwise repeatable: the flash kernel's TMEM hand-offs (P written over
    its S buffer, the next S issued behind P V) leave no ordering race."""
    d = S.attn_inputs(T, 256, 48, 8, 9, "cuda")
    p = B.make_attn_params(T, 256, 48, 8, 128, window, 10000.0, 1e-6, 0, B.FLAG_FP32_OUT)
    a = B.attention_forward(p, d["x"], d["w_qkvg"], d["w_o"], d["q_gain"], d["k_gain"])
    for _ in range(3):
        b = B.attention_forward(p, d["x"], d["w_qkvg"], d["w_o"], d["q_gain"], d["k_gain"])
        assert B.status() == 0 and torch.equal(a, b)


@pytest.mark.parametrize("window", [512, 0])
def test_attention_full_width(B, window):
    """Hidden 5120, 48/8 heads, T = 2048 with pre-norm and residual: sampled
    query rows (all keys) against the oracle."""
    rows = np.array([0, 1, 127, 128, 511, 512, 513, 1000, 1500, 2047])
    _check(B, 2048, 5120, 48, 8, window, seed=11 + window, pre_norm=True, residual_k=8, rows=rows)


@pytest.mark.parametrize("name,window,k,seed", [("swa", 512, 10, 12), ("global", 0, 12, 13)])
def test_attention_bench_configuration(B, name, window, k, seed):
    """The benchmark's attention workloads exactly (T = 8192, hidden 5120,
    48/8 heads, pre-norm, residual k, the bench's seed and input recipe):
    sampled query rows -- the first rows, both sides of the window edge and
    of key tiles, the last row -- against the oracle with every key."""
    rows = np.array([0, 1, 127, 128, 511, 512, 513, 2047, 4096, 6143, 8000, 8191])
    _check(B, 8192, 5120, 48, 8, window, seed=seed, pre_norm=True, residual_k=k, rows=rows)


@pytest.mark.parametrize("gain", [1.68, 3.0])
@pytest.mark.parametrize("window", [512, 0])
def test_attention_large_gains(B, gain, window):
    """Constant q/k gains well above 1 make the logits large and the softmax
    peaked (|s| up to sqrt(128) * gain^2), so the online reference moves and
    the O rows are rescaled on many tiles."""
    _check(B, 700, 256, 4, 2, window, seed=17, gain=gain)
