"""Pins for the oracle's NVFP4 (E2M1 + E4M3 block scales) expert-weight
path, each against something other than the oracle: the format's value
table written out, brute-force nearest-value search with the tie rule,
hand-built exactly representable blocks, error bounds of the format and the
checkpoint's published sizes. No GPU needed."""
import numpy as np

import oracle as O

# E2M1 magnitudes for the codes 0..7, written out from the format definition
# (exponent bias 1, one mantissa bit, subnormal 0.5 step)
TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_decode_table():
    got = O.e2m1_decode(np.arange(16))
    assert list(got[:8]) == TABLE
    assert list(-got[8:]) == TABLE and np.signbit(got[8])


def _nearest_even(v):
    """Brute force: the grid value nearest to v; on a tie the one whose code
    has mantissa bit 0; beyond 6 the saturated value."""
    grid = np.array(TABLE)
    out = []
    for x in np.asarray(v, dtype=np.float64):
        a = min(abs(x), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        k = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        out.append(np.copysign(grid[k], x))
    return np.array(out)


def test_round_matches_brute_force_and_ties():
    grid = np.array(TABLE)
    mids = (grid[:-1] + grid[1:]) / 2
    rng = np.random.default_rng(4)
    v = np.concatenate([mids, -mids, rng.uniform(-8, 8, 5000), [0.0, 6.0, 6.5, 100.0, -1e9]])
    v = v.astype(np.float32).astype(np.float64)
    assert np.array_equal(O.e2m1_round(v), _nearest_even(v))
    # ties written out: 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4
    assert list(O.e2m1_round(mids)) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_encode_decode_pack_round_trip():
    c = np.arange(16, dtype=np.uint8)
    assert np.array_equal(O.e2m1_encode(O.e2m1_decode(c)), c)
    assert O.pack_e2m1(np.array([1, 2], dtype=np.uint8))[0] == 0x21   # even element low
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 16, size=(5, 64)).astype(np.uint8)
    assert np.array_equal(O.unpack_e2m1(O.pack_e2m1(codes)), codes)


def test_quantize_exact_block():
    # one row, one block: the values are E2M1 grid points times 2^-3, so the
    # row maximum gives block scale 448 and every element lands on its code
    vals = np.array([6, 3, -1.5, 0.5, 0, -6, 4, 2, 1, -0.5, 1.5, -3, -4, 0, 2, -1.0])
    a = (vals * 2.0 ** -3).astype(np.float32)[None, :]
    packed, sb, g = O.quantize_nvfp4(a, 1)
    assert sb[0, 0] == 0x7E                                # E4M3 code of 448
    assert np.isclose(g[0], 0.75 / 2688.0, rtol=1e-7)
    assert np.array_equal(O.e2m1_decode(O.unpack_e2m1(packed))[0], vals)
    deq = O.dequantize_nvfp4(packed, sb, g, 1)
    assert np.allclose(deq, a, rtol=1e-6, atol=0)


def test_quantize_group_scale_and_bounds():
    rng = np.random.default_rng(7)
    a = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    a[5] = 0.0
    packed, sb, g = O.quantize_nvfp4(a, 32)                # two groups of 32 rows
    assert g.shape == (2,)
    for k in range(2):
        grp = a[32 * k:32 * (k + 1)]
        assert np.float32(g[k]) == np.float32(np.abs(grp).max() / np.float32(2688.0))
    # the largest element of each group is coded +-6 with block scale 448
    vals = O.e2m1_decode(O.unpack_e2m1(packed))
    for k in range(2):
        r, j = np.unravel_index(np.argmax(np.abs(a[32 * k:32 * (k + 1)])), (32, 256))
        assert abs(vals[32 * k + r, j]) == 6.0 and sb[32 * k + r, j // 16] == 0x7E
    assert np.all(vals[5] == 0)
    # dequantised within one unit of the block's scale (half the top grid
    # step is 1; saturation after the E4M3 rounding of the block scale adds
    # at most 0.4)
    deq = O.dequantize_nvfp4(packed, sb, g, 32)
    unit = (O.e4m3_decode(sb) * np.repeat(g, 32)[:, None]).repeat(16, axis=1)
    assert np.all(np.abs(deq - a) <= unit * (1 + 1e-6))


def test_nvfp4_forward_close_to_bf16_forward():
    g = np.random.default_rng(3)
    T, H, I, E = 10, 256, 128, 16
    x = O.bf16_round(g.standard_normal((T, H))).astype(np.float64)
    W = [(O.bf16_round(g.standard_normal((I, H)) * 0.02).astype(np.float64),
          O.bf16_round(g.standard_normal((I, H)) * 0.02).astype(np.float64),
          O.bf16_round(g.standard_normal((H, I)) * 0.02).astype(np.float64)) for _ in range(E)]
    Q = [(O.quantize_nvfp4(w[0], I), O.quantize_nvfp4(w[1], I), O.quantize_nvfp4(w[2], H))
         for w in W]
    idx = np.stack([g.choice(E, 4, replace=False) for _ in range(T)])
    wts = np.full((T, 4), 2.5 / 4)
    ref = O.moe_combine(x, idx, wts, lambda e: W[e])
    got = O.moe_combine_nvfp4(x, idx, wts, lambda e: Q[e])
    rel = np.sqrt(np.mean((got - ref) ** 2)) / np.sqrt(np.mean(ref ** 2))
    assert 0.02 < rel < 0.3, rel


def test_nvfp4_checkpoint_size():
    # [P5] 四套权重的账: U8 + BF16 + F32 bytes plus one E4M3 byte per 16
    # routed-expert weights give the 293.63 GB on disk
    u8, bf16, f32 = 246_625_075_200, 7_953_224_128, 64_237_824
    experts = 49 * 256 * 3 * 5120 * 2560
    assert 2 * u8 == experts
    total = u8 + 2 * bf16 + 4 * f32 + experts // 16
    assert abs(total - 293.63e9) < 0.02e9


def test_expert_quantises_x_and_the_activation_row():
    """H = I = 16, one token. x = [1.5, 1.1875, 0, ...]: per-row group scale
    1.5/2688, block scale 448, so x is coded at scale 1/4: 1.5 -> 6 and
    1.1875 -> 4.75, whose nearest E2M1 value is 4, i.e. back to 1. Gate and
    up weights are the identity on the first two channels (coded exactly):
    g = u = [1.5, 1], A = bf16(silu(g) * u) = [1.8359375, 0.73046875]
    (silu(1.5) * 1.5 = 1.83954..., silu(1) = 0.73106...). A's row is coded
    at scale 1.8359375/6: 0.73046875 -> 2.387..., nearest E2M1 value 2, i.e.
    back to 2 * 1.8359375 / 6. A down matrix that swaps the two channels
    returns [2 * 1.8359375 / 6, 1.8359375] in its first two rows."""
    H = I = 16
    x = np.zeros((1, H))
    x[0, :2] = [1.5, 1.1875]
    eye2 = np.zeros((I, H))
    eye2[0, 0] = eye2[1, 1] = 1.0
    swap = np.zeros((H, I))
    swap[0, 1] = swap[1, 0] = 1.0
    gq = O.quantize_nvfp4(eye2, I)
    dq = O.quantize_nvfp4(swap, H)
    y = O.swiglu_expert_nvfp4(x, gq, gq, dq)
    assert np.allclose(y[0, :2], [2.0 * 1.8359375 / 6.0, 1.8359375], rtol=1e-6, atol=0)
    assert np.array_equal(y[0, 2:], np.zeros(H - 2))


def test_expert_hand_case_closed_form():
    """One token through one NVFP4 expert (H = I = 16, one block per row),
    with operands chosen so that every quantisation is exact: each row's
    block holds E2M1 grid values times a power of two, and each weight row's
    block maximum is the matrix maximum over a power of two (block scale 448,
    224, 112, 56). Only gate/up row 0 and down column 0 are non-zero, so the
    activation row has one non-zero element, which its own quantisation keeps.
    Closed form: y_h = bf16(silu(x . Wg[0]) * (x . Wu[0])) * Wd[h, 0]. Swapping
    gate and up, dropping the BF16 step or transposing W_d changes the value."""
    import torch
    H = I = 16
    x = np.zeros((1, H))
    x[0, :9] = np.array([6, -4, 3, 0, 2, -1.5, 1, 0.5, -2]) * 0.25
    wg = np.zeros((I, H))
    wg[0, :6] = np.array([6, 2, -3, 1, 0.5, -1]) / 16
    wu = np.zeros((I, H))
    wu[0, :6] = np.array([1, -1, 0.5, 4, 6, 1.5]) / 8
    wd = np.zeros((H, I))
    wd[:6, 0] = np.array([6, -3, 1.5, -6, 0.75, 3]) / 4
    gq = O.quantize_nvfp4(wg, I)
    uq = O.quantize_nvfp4(wu, I)
    dq = O.quantize_nvfp4(wd, H)
    assert list(O.e4m3_decode(dq[1][:6, 0])) == [448, 224, 112, 448, 56, 224]
    y = O.swiglu_expert_nvfp4(x, gq, uq, dq)
    g0 = float(x[0] @ wg[0])
    u0 = float(x[0] @ wu[0])
    a0 = g0 / (1.0 + np.exp(-g0)) * u0
    a0 = float(torch.tensor(a0, dtype=torch.float64).to(torch.bfloat16).to(torch.float64))
    want = a0 * wd[:, 0]
    assert np.allclose(y[0], want, rtol=1e-6, atol=1e-12)
    # the BF16 step is visible at this size
    assert abs(a0 - g0 / (1.0 + np.exp(-g0)) * u0) > 1e-6 * abs(a0)
