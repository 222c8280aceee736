"""The parity checkers of the GPU tests accept what is correct and reject
what is not.

The GPU tests compare routing with compare_routing (exact sets except at
near ties, where another FP32-correct selection is allowed) and validate
quantised SwiGLU rows with check_act_codes_fp8 / check_act_codes_nvfp4
(every code and scale must lie between the decisions taken at the two ends
of an error interval). A checker that accepted anything would make those
tests vacuous, so here each one is fed the oracle's own result, which it must
accept, and results with one planted mistake each, which it must reject. No
GPU needed.
"""
import numpy as np
import pytest

import _helpers as Hp
import oracle as O


class _Wl:                      # the routing fields compare_routing reads
    n_group, topk_group, top_k, routed_scale = 8, 4, 8, 2.5


def _select(s64):
    s32 = s64.astype(np.float32)
    sel = O.group_limited_topk(s32, 8, 4, 8)
    sel["weights"] = O.combine_weights(s64, sel["idx"], 2.5)
    sel["s64"], sel["s32"] = s64, s32
    return sel


def _scores(seed, T=12):
    return np.random.default_rng(seed).uniform(0.02, 0.98, size=(T, 256))


def _kept_order(s32, groups):
    cand = np.concatenate([np.arange(g * 32, (g + 1) * 32) for g in sorted(groups)])
    return cand[np.lexsort((cand, -s32[cand].astype(np.float64)))]


def test_routing_checker_accepts_the_oracle_and_rejects_changes():
    sel = _select(_scores(0))
    assert not O.near_ties(sel).any()
    idx, w = sel["idx"].copy(), sel["weights"].astype(np.float32)
    Hp.compare_routing(sel, idx, w, _Wl)
    t = 3
    outside = next(e for e in range(256) if e not in idx[t])
    bad = idx.copy()
    bad[t, 7] = outside                                   # a wrong expert
    with pytest.raises(AssertionError):
        Hp.compare_routing(sel, bad, w, _Wl)
    bad_w = w.copy()
    bad_w[t, 2] += 1e-4                                   # a weight off by 1e-4
    with pytest.raises(AssertionError):
        Hp.compare_routing(sel, idx, bad_w, _Wl)
    rev = idx.copy()
    rev[t] = rev[t][::-1]                                 # ascending order
    with pytest.raises(AssertionError):
        Hp.compare_routing(sel, rev, w[:, ::-1].copy(), _Wl)


def test_routing_checker_allows_only_the_near_tie_swap():
    """Token 0's best unselected candidate is put 2e-6 below its 8th: the
    selection with the two swapped is also FP32-correct and must pass;
    swapping in the next candidate instead must not."""
    s64 = _scores(1)
    base = _select(s64)
    order = _kept_order(base["s32"][0], base["kept"][0])
    s64[0, order[8]] = s64[0, order[7]] - 2e-6
    sel = _select(s64)
    assert O.near_ties(sel)[0]
    alt = sel["idx"].copy()
    alt[0, 7] = order[8]
    w = sel["weights"].astype(np.float32).copy()
    w[0] = 2.5 * s64[0, alt[0]] / s64[0, alt[0]].sum()
    Hp.compare_routing(sel, alt, w, _Wl)
    wrong = sel["idx"].copy()
    wrong[0, 7] = order[9]
    w2 = w.copy()
    w2[0] = 2.5 * s64[0, wrong[0]] / s64[0, wrong[0]].sum()
    with pytest.raises(AssertionError):
        Hp.compare_routing(sel, wrong, w2, _Wl)


def test_routing_checker_allows_the_group_boundary_swap():
    """Token 0's fifth group is given a top-2 sum 1e-6 below the fourth's:
    keeping it instead is also FP32-correct. The alternative selection is
    worked out here by plain sorting, not by the checker's own helper."""
    s64 = _scores(2)
    base = _select(s64)
    gs = base["gscore"][0].astype(np.float64)
    gorder = np.lexsort((np.arange(8), -gs))
    g4, g5 = int(gorder[3]), int(gorder[4])
    s64[0, g5 * 32:(g5 + 1) * 32] = 0.01
    s64[0, g5 * 32:g5 * 32 + 2] = (gs[g4] - 1e-6) / 2
    sel = _select(s64)
    assert sel["group_margin"][0] < 1e-5
    groups = [int(g) for g in gorder[:3]] + [g5]
    alt_set = _kept_order(sel["s32"][0], groups)[:8]
    alt = sel["idx"].copy()
    alt[0] = alt_set
    w = sel["weights"].astype(np.float32).copy()
    w[0] = 2.5 * s64[0, alt_set] / s64[0, alt_set].sum()
    Hp.compare_routing(sel, alt, w, _Wl)


def _act_rows(seed):
    rng = np.random.default_rng(seed)
    a = rng.normal(size=(6, 64)) * np.array([1e-3, 0.1, 1.0, 7.0, 300.0, 1.0])[:, None]
    a[5] = 0.0                                            # an all-zero row
    return a


def _mid_element(v):
    """Column of the largest |v| below half the row's maximum."""
    m = np.abs(v)
    return int(np.argmax(np.where(m < 0.5 * m.max(), m, -1.0)))


def test_fp8_activation_checker():
    a64 = _act_rows(3)
    codes, scale = O.quantize_rows_e4m3(O.bf16_round(a64))
    Hp.check_act_codes_fp8(a64, codes, scale)
    r = 3
    j = _mid_element(a64[r])
    bad = codes.copy()
    bad[r, j] = (bad[r, j] & 0x80) | ((bad[r, j] & 0x7F) + 1)   # one grid step up
    with pytest.raises(AssertionError):
        Hp.check_act_codes_fp8(a64, bad, scale)
    bad_s = scale.copy()
    bad_s[2] *= np.float32(1.01)
    with pytest.raises(AssertionError):
        Hp.check_act_codes_fp8(a64, codes, bad_s)
    zero_s = scale.copy()
    zero_s[5] = 2.0                                       # a zero row must have scale 1
    with pytest.raises(AssertionError):
        Hp.check_act_codes_fp8(a64, codes, zero_s)


def test_nvfp4_activation_checker():
    a64 = _act_rows(4)
    packed, sf, g = O.quantize_nvfp4(O.bf16_round(a64), 1)
    Hp.check_act_codes_nvfp4(a64, packed, sf, g)
    r = 4
    # the largest element of block 0 is coded 6 (index 7): recode it as 4
    j = int(np.argmax(np.abs(a64[r, :16])))
    codes = O.unpack_e2m1(packed)
    assert codes[r, j] & 0x7 == 7
    codes[r, j] = (codes[r, j] & 0x8) | 6
    with pytest.raises(AssertionError):
        Hp.check_act_codes_nvfp4(a64, O.pack_e2m1(codes), sf, g)
    bad_sf = sf.copy()
    bad_sf[r, 1] += 1                                     # block scale one E4M3 step up
    with pytest.raises(AssertionError):
        Hp.check_act_codes_nvfp4(a64, packed, bad_sf, g)
    bad_g = g.copy()
    bad_g[2] *= np.float32(1.01)
    with pytest.raises(AssertionError):
        Hp.check_act_codes_nvfp4(a64, packed, sf, bad_g)


def test_prenorm_ambiguity_flags_an_exact_midpoint():
    """Row [a, b] with a = (1 + 2^-8) r and b chosen so that the row's RMS
    (with eps) is r: the normalised a is 1 + 2^-8, exactly halfway between
    the BF16 values 1 and 1 + 2^-7, so either rounding is correct."""
    r, eps = 100.0, 1e-6
    a = (1.0 + 2.0 ** -8) * r
    b = np.sqrt(2 * r * r - a * a - 2 * eps)
    flags = Hp.prenorm_ambiguous(np.array([[a, b]]), None, eps)
    assert flags[0, 0]
    rng = np.random.default_rng(5)
    h = rng.normal(size=(64, 256))
    frac = Hp.prenorm_ambiguous(h, None, eps).mean()
    assert frac < 1e-3                                    # rare on random rows


# ------------------------------------------------ pre-norm x and unit cover
def test_bf16_neighbour_matches_torch_nextafter():
    """The other rounding candidate is torch's BF16 nextafter toward v."""
    import torch
    rng = np.random.default_rng(3)
    v = rng.standard_normal(4000) * np.exp2(rng.integers(-20, 20, 4000))
    lo = O.bf16_round(v).astype(np.float64)
    keep = lo != v
    got = Hp.bf16_neighbour_toward(lo[keep], v[keep])
    # torch's nextafter toward a target well beyond lo on the side of v (v
    # itself would round to lo or to the neighbour in BF16)
    away = np.sign(v[keep] - lo[keep]) * np.sign(lo[keep]) > 0
    tgt = np.where(away, lo[keep] * 2.0, lo[keep] / 2.0)
    want = torch.nextafter(torch.tensor(lo[keep]).to(torch.bfloat16),
                           torch.tensor(tgt).to(torch.bfloat16)).double().numpy()
    assert np.array_equal(got, want)


def _prenorm_case(seed=11, T=40, H=256):
    rng = np.random.default_rng(seed)
    h = O.bf16_round(rng.standard_normal((T, H))).astype(np.float64)
    x = O.bf16_round(O.rms_norm(h, None, 1e-6)).astype(np.float64)
    return h, x


def test_validated_prenorm_accepts_oracle_and_other_rounding_at_midpoints():
    h, x = _prenorm_case()
    got, n_other = Hp.validated_prenorm_x(x, h, None, 1e-6)
    assert np.array_equal(got, x) and n_other == 0
    # flip an element the checker calls ambiguous (make one by widening `rel`)
    amb = Hp.prenorm_ambiguous(h, None, 1e-6, rel=1e-3)
    r, c = np.argwhere(amb)[0]
    v = O.rms_norm(h, None, 1e-6)
    y = x.copy()
    y[r, c] = Hp.bf16_neighbour_toward(x[r, c], v[r, c])
    _, n_other = Hp.validated_prenorm_x(y, h, None, 1e-6, rel=1e-3)
    assert n_other == 1


def test_validated_prenorm_rejects_wrong_rounding():
    h, x = _prenorm_case()
    v = O.rms_norm(h, None, 1e-6)
    amb = Hp.prenorm_ambiguous(h, None, 1e-6)
    r, c = np.argwhere(~amb)[5]
    for bad in (Hp.bf16_neighbour_toward(x[r, c], v[r, c]),          # the other rounding
                Hp.bf16_neighbour_toward(x[r, c], -3 * v[r, c])):      # the far neighbour
        y = x.copy()
        y[r, c] = bad
        with pytest.raises(AssertionError):
            Hp.validated_prenorm_x(y, h, None, 1e-6)


def _groups_brute(n, size):
    """Balanced groups written out: ceil(n/size) groups, sizes differing by
    at most one, the larger ones first."""
    g = -(-n // size)
    sizes = [n // g + (1 if i < n % g else 0) for i in range(g)]
    out, s = [], 0
    for z in sizes:
        out.append(range(s, s + z))
        s += z
    return out


@pytest.mark.parametrize("tiling,size", [("groups", 256), ("tiles", 128), ("tiles", 32)])
def test_unit_cover_hits_every_group(tiling, size):
    rng = np.random.default_rng(5)
    T, E, K = 3000, 16, 8
    gi = np.stack([rng.choice(E, K, replace=False) for _ in range(T)])
    gi[:1200, 0] = 3                         # one hot expert: several groups
    gi[:1200] = np.stack([np.concatenate([[3], rng.choice(np.delete(np.arange(E), 3), K - 1,
                                                          replace=False)]) for _ in range(1200)])
    picks = set(Hp.unit_cover_tokens(gi, E, tiling, size).tolist())
    for e in range(E):
        toks = np.nonzero((gi == e).any(axis=1))[0]
        groups = (_groups_brute(len(toks), size) if tiling == "groups" else
                  [range(j, min(j + size, len(toks))) for j in range(0, len(toks), size)])
        for grp in groups:
            assert any(int(toks[p]) in picks for p in grp), (e, grp)
            assert int(toks[grp[-1]]) in picks          # the group's last row
    assert len(picks) <= sum(-(-int((gi == e).any(1).sum()) // size) for e in range(E))
