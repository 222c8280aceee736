"""Pins for the oracle's FP8 (E4M3) expert-weight path, each against
something other than the oracle itself: torch's float8_e4m3fn type (an
independent implementation of the same format), hand-derived grid values and
ties, a hand-computed one-expert case whose operands are exactly
representable, and properties of the format. No GPU needed.
"""
import math

import numpy as np
import torch

import oracle as O


def test_decode_all_codes_matches_torch():
    c = np.arange(256, dtype=np.uint8)
    got = O.e4m3_decode(c)
    ref = torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.isnan(got).sum() == 2                      # 0x7F and 0xFF only
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert O.e4m3_decode(np.uint8(0x7E)) == 448.0        # largest finite
    assert O.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9    # smallest subnormal
    assert O.e4m3_decode(np.uint8(0x08)) == 2.0 ** -6    # smallest normal
    assert O.e4m3_decode(np.uint8(0x38)) == 1.0          # exponent field 7 = bias


def test_encode_round_trips_every_finite_code():
    c = np.arange(256, dtype=np.uint8)
    v = O.e4m3_decode(c)
    ok = ~np.isnan(v)
    assert np.array_equal(O.e4m3_encode(v[ok]), c[ok])   # includes -0.0 -> 0x80


def test_round_matches_torch_in_range():
    g = torch.Generator().manual_seed(3)
    v = torch.randn(200000, generator=g) * torch.exp(torch.empty(200000).uniform_(-14, 6, generator=g))
    v = v.clamp(-448, 448)
    ref = v.to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_round(v.numpy()), ref)


def test_round_ties_go_to_even_at_every_midpoint():
    grid = O.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))   # 0 .. 448, ascending
    mids = (grid[:-1] + grid[1:]) / 2                             # exact in float32
    got = O.e4m3_round(mids.astype(np.float32))
    ref = torch.from_numpy(mids.astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(got, ref)
    codes = O.e4m3_encode(got)
    assert np.all((codes & 1) == 0)                               # even mantissa


def test_round_hand_values():
    cases = {
        2.0 ** -10: 0.0,              # half the smallest subnormal: tie to 0
        3 * 2.0 ** -10: 2.0 ** -8,    # between 1 and 2 units of 2^-9: tie to 2
        1.0625: 1.0,                  # between 1 and 1.125: tie to mantissa 0
        1.1875: 1.25,                 # between 1.125 and 1.25: tie to mantissa 2
        240.0: 240.0,                 # 1.875 * 2^7, exact
        447.0: 448.0,
        460.0: 448.0,
        500.0: 448.0,                 # saturates (torch's conversion gives NaN here)
        1e6: 448.0,
        -1e6: -448.0,
        -0.3: -0.3125,                # 1.25 * 2^-2
    }
    for v, want in cases.items():
        assert O.e4m3_round(np.float32(v)) == want, v


def test_quantize_rows_against_torch_steps():
    # the same definition carried out with torch's FP32 arithmetic and its
    # float8 conversion (clamped first: torch maps overflow to NaN)
    g = torch.Generator().manual_seed(5)
    a = (torch.randn(64, 320, generator=g) * torch.exp(torch.randn(64, 1, generator=g) * 3))
    a = a.to(torch.bfloat16).float()
    a[7] = 0.0
    codes, scale = O.quantize_rows_e4m3(a.numpy())
    amax = a.abs().amax(dim=1)
    nz = amax > 0
    inv = torch.where(nz, torch.tensor(448.0) / torch.where(nz, amax, torch.ones_like(amax)), torch.ones_like(amax))
    sc = torch.where(nz, amax / torch.tensor(448.0), torch.ones_like(amax))
    q = (a * inv[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn)
    assert np.array_equal(codes, q.view(torch.uint8).numpy())
    assert np.array_equal(scale, sc.numpy())
    assert np.all(codes[7] == 0) and scale[7] == 1.0


def test_quantize_rows_properties():
    g = np.random.default_rng(11)
    a = (g.standard_normal((32, 512)) * 0.02).astype(np.float32)
    codes, scale = O.quantize_rows_e4m3(a)
    vals = O.e4m3_decode(codes)
    # the row's largest magnitude lands on +-448
    j = np.argmax(np.abs(a), axis=1)
    assert np.all(np.abs(vals[np.arange(32), j]) == 448.0)
    # dequantised within half a grid step: relative 2^-4 for normal values,
    # absolute 2^-10 * scale in the subnormal range
    deq = O.dequantize_rows_e4m3(codes, scale)
    err = np.abs(deq - a)
    bound = np.maximum(np.abs(a) * 2.0 ** -4, scale[:, None].astype(np.float64) * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.all(np.sign(deq) * np.sign(a) >= 0)


def test_fp8_expert_hand_case():
    # H = 2, I = 1; every operand is exact in E4M3 with power-of-two scales
    x = np.array([[0.5, 1.75]])                 # amax 1.75: inv 256, codes 128, 448
    wg = np.array([[0.875, -0.4375]])           # amax 0.875: inv 512, codes 448, -224
    wu = np.array([[1.75, 0.875]])              # inv 256: codes 448, 224
    wd = np.array([[0.875], [1.75]])            # one element per row: code 448
    qg, qu, qd = (O.quantize_rows_e4m3(w) for w in (wg, wu, wd))
    assert np.array_equal(O.dequantize_rows_e4m3(*qg), wg)
    assert np.array_equal(O.dequantize_rows_e4m3(*qd), wd)
    y = O.swiglu_expert_fp8(x, qg, qu, qd)
    g = 0.5 * 0.875 - 1.75 * 0.4375             # -0.328125
    u = 0.5 * 1.75 + 1.75 * 0.875               # 2.40625
    a = g / (1 + math.exp(-g)) * u
    a_bf16 = float(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).float())
    # A has one element: it quantises to -448 with scale fp32(|a|/448)
    want = a_bf16 * np.array([0.875, 1.75])
    assert np.allclose(y[0], want, rtol=2 ** -22, atol=0)
    assert not np.allclose(y[0], a * np.array([0.875, 1.75]), rtol=1e-4, atol=0)   # BF16 step matters


def test_fp8_activation_is_quantised_per_row():
    """x is quantised per row before the gate/up products. Row 1: amax 448,
    scale 1, and 1.03125 (= 1 + 2^-5, between E4M3 grid points 1 and 1.125)
    rounds to 1. Row 2 is row 1 halved: scale 1/2, the same codes, values
    224 and 0.5. Gate and up weights read element 1 with code 0x38 (= 1.0)
    and scale 1, so g = u = the quantised element: 1 and 0.5."""
    x = np.array([[448.0, 1.03125], [224.0, 0.515625]])
    one = (np.array([[0x00, 0x38]], dtype=np.uint8), np.array([1.0], dtype=np.float32))
    a = O.swiglu_act_fp8(x, one, one)
    silu = lambda z: z / (1.0 + math.exp(-z))
    assert np.allclose(a[:, 0], [silu(1.0) * 1.0, silu(0.5) * 0.5], rtol=1e-15, atol=0)


def test_fp8_activation_row_quantised_before_down_projection():
    """x = [4, 1]: scale 1/112, codes 448 and 112 (both on the grid), so the
    expert sees x exactly. Identity gate/up rows (code 0x38 = 1, scale 1)
    give g = u = [4, 1]; A = bf16(silu(g) * u) = [3.921875, 0.73046875].
    A's row is quantised with inv = fp32(448 / 3.921875): element 1 becomes
    83.44..., whose nearest E4M3 values are 80 and 88, so it is coded 80
    and comes back as 80 * 3.921875 / 448. A down row that reads element 1
    returns exactly that."""
    x = np.array([[4.0, 1.0]])
    eye = (np.array([[0x38, 0x00], [0x00, 0x38]], dtype=np.uint8), np.ones(2, dtype=np.float32))
    down = (np.array([[0x00, 0x38]], dtype=np.uint8), np.ones(1, dtype=np.float32))
    y = O.swiglu_expert_fp8(x, eye, eye, down)
    assert np.allclose(y[0, 0], 80.0 * 3.921875 / 448.0, rtol=1e-6, atol=0)


def test_fp8_forward_residual_keeps_the_layer_input():
    """All-zero FP8 experts (codes 0, scale 1) give out = 0 and
    h_k = sqrt((k-1)/k) * h_{k-1} exactly, with h_{k-1} the layer input
    rather than its pre-normed copy."""
    rng = np.random.default_rng(15)
    T, H, E, I, k = 4, 32, 8, 4, 9
    h = rng.normal(size=(T, H)) * 5.0
    zq = tuple(O.quantize_rows_e4m3(np.zeros(shape)) for shape in ((I, H), (I, H), (H, I)))
    r = O.moe_forward_fp8(h, rng.normal(size=(E, H)), None, lambda e: zq, n_group=2,
                          topk_group=1, top_k=2, pre_norm=True, residual_k=k)
    assert np.array_equal(r["out"], np.zeros((T, H)))
    assert np.allclose(r["h"], math.sqrt((k - 1) / k) * h, rtol=1e-15, atol=0)


def test_fp8_forward_gains():
    """Pre- and post-norm gains of powers of two in the FP8 sublayer: the
    BF16 pre-norm output scales exactly per channel and the post-norm branch
    h_k - sqrt((k-1)/k) h_{k-1} scales by the post-norm gain."""
    rng = np.random.default_rng(20)
    T, H, E, I, k = 4, 32, 8, 8, 5
    h = rng.normal(size=(T, H)) * 2.0
    wr = rng.normal(size=(E, H))
    Q = [tuple(O.quantize_rows_e4m3(rng.normal(size=s) * 0.2) for s in ((I, H), (I, H), (H, I)))
         for _ in range(E)]
    g = np.tile([0.5, 1.0, 2.0, 4.0], H // 4)
    run = lambda pg, qg: O.moe_forward_fp8(h, wr, None, lambda e: Q[e], n_group=2, topk_group=1,
                                           top_k=2, pre_norm=True, pre_gain=pg, residual_k=k,
                                           post_gain=qg)
    base, pre, post = run(None, None), run(g, None), run(None, g)
    assert np.array_equal(pre["x"], base["x"] * g[None, :])
    keep = math.sqrt((k - 1) / k) * h
    assert np.allclose(post["h"] - keep, (base["h"] - keep) * g[None, :], rtol=1e-13, atol=1e-13)


def test_fp8_forward_close_to_bf16_forward():
    # FP8 weights and activations stay within E4M3's relative precision of
    # the unquantised sublayer (a wrong scale or operand would be far off)
    g = np.random.default_rng(2)
    T, H, I, E = 12, 256, 128, 32
    x = O.bf16_round(g.standard_normal((T, H))).astype(np.float64)
    wr = g.standard_normal((E, H)) * 0.05
    W = [(O.bf16_round(g.standard_normal((I, H)) * 0.02).astype(np.float64),
          O.bf16_round(g.standard_normal((I, H)) * 0.02).astype(np.float64),
          O.bf16_round(g.standard_normal((H, I)) * 0.02).astype(np.float64)) for _ in range(E)]
    Q = [tuple(O.quantize_rows_e4m3(w) for w in ws) for ws in W]
    kw = dict(n_group=4, topk_group=2, top_k=4, scale=2.5)
    ref = O.moe_forward(x, wr, None, lambda e: W[e], **kw)
    got = O.moe_forward_fp8(x, wr, None, lambda e: Q[e], **kw)
    assert np.array_equal(ref["sel"]["idx"], got["sel"]["idx"])      # router unquantised
    rel = np.sqrt(np.mean((got["out"] - ref["out"]) ** 2)) / np.sqrt(np.mean(ref["out"] ** 2))
    assert 0.005 < rel < 0.08, rel


def test_fp8_checkpoint_counts():
    # [P5] 四套权重的账: F8_E4M3 + BF16 + F32 counts of the FP8 checkpoint sum
    # to the model's parameter total, and every routed-expert weight
    # (49 layers x 256 experts x 3 x 5120 x 2560) fits in the F8 share
    f8, bf16, f32 = 499_646_464_000, 1_556_910_528, 64_237_824
    assert f8 + bf16 + f32 == 501_267_612_352
    experts = 49 * 256 * 3 * 5120 * 2560
    assert experts == 493_250_150_400 and experts < f8
