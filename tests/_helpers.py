"""Shared helpers for the parity tests: run the oracle on the same seeded
inputs the CUDA path gets, and compare results the way the layer allows.

Routing: the selected expert SET must be identical except on near-tie tokens
(group or top-k boundary closer than 1e-5 in FP32 score), which are counted.
The output order (descending score) is unique only between scores more than
1e-5 apart, so the order is checked to be non-increasing in the oracle's
score up to that margin. For those the
oracle lists the alternative selections another correct FP32 evaluation may
make (swap the k-th and (k+1)-th candidate, or the 4th and 5th group); the
CUDA result must be one of them, and its output is compared with the oracle's
output for that alternative. Nothing the CUDA path computes is fed to the
oracle.
"""
import numpy as np
import torch

import oracle as O

ROUTE_W_TOL = 1e-5       # absolute, on the combine weights
OUT_REL_TOL = 2e-2       # max |err| / RMS(oracle output)
TIE_MARGIN = 1e-5


def expert_getter(d):
    """Oracle access to the expert weights (copies one expert to the host)."""
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = tuple(d[k][e].float().cpu().numpy() for k in ("w_gate", "w_up", "w_down"))
            if len(cache) > 48:
                cache.pop(next(iter(cache)))
        return cache[e]
    return get


def host(t):
    return None if t is None else t.float().cpu().numpy()


def alternatives(sel, t, n_group, topk_group, top_k, scale, margin=TIE_MARGIN):
    """Valid selections for token t: the oracle's own plus the near-tie swaps.
    Returns list of (idx array, weights array)."""
    s32 = sel["s32"][t]
    s64 = sel["s64"][t]
    E = s32.shape[0]
    gsize = E // n_group
    out = [(sel["idx"][t], sel["weights"][t])]

    def topk_in(groups):
        cand = np.concatenate([np.arange(g * gsize, (g + 1) * gsize) for g in sorted(groups)])
        order = cand[np.lexsort((cand, -s32[cand].astype(np.float64)))]
        return order

    gs = sel["gscore"][t]
    gorder = np.lexsort((np.arange(n_group), -gs.astype(np.float64)))
    group_sets = [list(gorder[:topk_group])]
    if topk_group < n_group and sel["group_margin"][t] < margin:
        alt = list(gorder[:topk_group - 1]) + [gorder[topk_group]]
        group_sets.append(alt)
    for gset in group_sets:
        order = topk_in(gset)
        cands = [order[:top_k]]
        if len(order) > top_k and float(s32[order[top_k - 1]]) - float(s32[order[top_k]]) < margin:
            swapped = np.concatenate([order[:top_k - 1], order[top_k:top_k + 1]])
            cands.append(swapped)
        for c in cands:
            w = scale * s64[c] / s64[c].sum()
            out.append((c.astype(np.int32), w))
    return out


def compare_routing(sel, gpu_idx, gpu_w, wl, allow_alternatives=True):
    """Returns (near_tie_mask, chosen) where chosen[t] = (idx, weights) of the
    oracle selection the GPU matched. Asserts exactness elsewhere."""
    gpu_idx = np.asarray(gpu_idx)
    gpu_w = np.asarray(gpu_w, dtype=np.float64)
    T = gpu_idx.shape[0]
    ties = O.near_ties(sel, TIE_MARGIN)
    chosen = []
    for t in range(T):
        if not ties[t]:
            assert sorted(gpu_idx[t].tolist()) == sorted(sel["idx"][t].tolist()), \
                f"token {t}: gpu {gpu_idx[t]} oracle {sel['idx'][t]}"
            wmap = dict(zip(sel["idx"][t].tolist(), sel["weights"][t].tolist()))
            want_w = np.array([wmap[e] for e in gpu_idx[t].tolist()])
            assert np.max(np.abs(gpu_w[t] - want_w)) <= ROUTE_W_TOL, \
                f"token {t}: weights {gpu_w[t]} vs {want_w}"
            sc = sel["s32"][t][gpu_idx[t]].astype(np.float64)
            assert np.all(np.diff(sc) <= TIE_MARGIN), f"token {t}: order {gpu_idx[t]}"
            chosen.append((sel["idx"][t], sel["weights"][t]))
            continue
        assert allow_alternatives
        alts = alternatives(sel, t, wl.n_group, wl.topk_group, wl.top_k, wl.routed_scale)
        hit = None
        for ai, aw in alts:
            if set(ai.tolist()) == set(gpu_idx[t].tolist()):
                hit = (ai, aw)
                break
        assert hit is not None, f"near-tie token {t}: gpu {gpu_idx[t]} is none of {alts}"
        # weights: match by expert
        wmap = dict(zip(hit[0].tolist(), hit[1].tolist()))
        for j, e in enumerate(gpu_idx[t].tolist()):
            assert abs(gpu_w[t, j] - wmap[e]) <= ROUTE_W_TOL
        # order: non-increasing in the oracle's score, up to the margin
        sc = sel["s32"][t][gpu_idx[t]].astype(np.float64)
        assert np.all(np.diff(sc) <= TIE_MARGIN)
        chosen.append((gpu_idx[t].copy(), np.array([wmap[e] for e in gpu_idx[t].tolist()])))
    return ties, chosen


def oracle_outputs(x64, chosen_rows, tokens, get_expert):
    """Oracle combine for the given tokens using the (oracle-made) selections."""
    idx = np.stack([chosen_rows[i][0] for i in range(len(tokens))])
    w = np.stack([chosen_rows[i][1] for i in range(len(tokens))])
    return O.moe_combine(x64[tokens], idx, w, get_expert)


def expert_getter_fp8(gq, uq, dq):
    """Oracle access to E4M3 expert weights: ((codes, scales) x 3) per expert,
    copied from the device tensors the quantiser wrote."""
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = tuple((q[0][e].cpu().numpy(), q[1][e].cpu().numpy()) for q in (gq, uq, dq))
            if len(cache) > 48:
                cache.pop(next(iter(cache)))
        return cache[e]
    return get


def _bf16_grid_between(lo, hi):
    """BF16 values in [lo, hi] for 0 <= lo <= hi (both BF16 values)."""
    b0 = int(np.float32(lo).view(np.uint32)) >> 16
    b1 = int(np.float32(hi).view(np.uint32)) >> 16
    assert b1 - b0 <= 4096, "interval too wide"
    bits = (np.arange(b0, b1 + 1, dtype=np.uint32) << np.uint32(16))
    return bits.view(np.float32).astype(np.float64)


def check_act_codes_fp8(a64, gpu_codes, gpu_scale, rel=1e-5, row_abs=1e-5):
    """Validate the GPU's E4M3 codes and row scales of SwiGLU rows a64 [n, I]
    (FP64, before rounding) against the oracle's quantiser.

    The GPU's FP32 value of each element lies within m = rel*|a| +
    row_abs*max|a_row| of a64 (its FP32 accumulation and SwiGLU err far less).
    BF16 rounding, the FP32 product with the row's 448/amax and the E4M3
    rounding are all monotone, so a correct code lies between the codes of
    the interval's two ends; the row maximum lies between the largest lower
    and upper ends, and the GPU's scale must be amax/448 (FP32) for a BF16
    value amax there. Returns (checked mask [n] (all rows), codes, scale):
    the validated GPU codes and scales, each of them an oracle-admitted
    result."""
    a64 = np.asarray(a64, dtype=np.float64)
    gpu_codes = np.asarray(gpu_codes)
    gpu_scale = np.asarray(gpu_scale, dtype=np.float32)
    n = a64.shape[0]
    m = rel * np.abs(a64) + row_abs * np.max(np.abs(a64), axis=1, keepdims=True)
    lo_v = O.bf16_round(a64 - m).astype(np.float64)
    hi_v = O.bf16_round(a64 + m).astype(np.float64)
    absmin = np.where(lo_v > 0, lo_v, np.where(hi_v < 0, -hi_v, 0.0))
    absmax = np.maximum(np.abs(lo_v), np.abs(hi_v))
    amax_lo, amax_hi = absmin.max(axis=1), absmax.max(axis=1)
    inv = np.empty(n, dtype=np.float32)
    f448 = np.float32(O.E4M3_MAX)
    for r in range(n):
        if amax_hi[r] == 0:
            assert gpu_scale[r] == 1.0, f"row {r}: zero row with scale {gpu_scale[r]}"
            inv[r] = 1.0
            continue
        cands = _bf16_grid_between(amax_lo[r], amax_hi[r])
        cands = cands[cands > 0].astype(np.float32)
        hit = cands[(cands / f448).astype(np.float32) == gpu_scale[r]]
        assert len(hit) >= 1, (f"row {r}: scale {gpu_scale[r]} is amax/448 for no amax in "
                               f"[{amax_lo[r]}, {amax_hi[r]}]")
        inv[r] = np.float32(f448 / hit[0])
    inv2 = inv[:, None]
    c_lo = O.e4m3_round((lo_v.astype(np.float32) * inv2).astype(np.float32))
    c_hi = O.e4m3_round((hi_v.astype(np.float32) * inv2).astype(np.float32))
    gv = O.e4m3_decode(gpu_codes)
    ok = (gv >= c_lo) & (gv <= c_hi)
    if not ok.all():
        r, j = map(int, np.argwhere(~ok)[0])
        raise AssertionError(
            f"{(~ok).sum()} act codes outside the oracle's interval; first at row {r} "
            f"col {j}: a64={a64[r, j]!r} code value {gv[r, j]!r} not in "
            f"[{c_lo[r, j]!r}, {c_hi[r, j]!r}] (scale {gpu_scale[r]!r})")
    return np.ones(n, dtype=bool), gpu_codes, gpu_scale


def oracle_outputs_fp8_checked(x64, gpu_idx, weight_of, get_expert_q, act_rows, E,
                               tokens=None):
    """Oracle FP8 combine for `tokens` (default: all), with each pair row's
    SwiGLU codes and scale validated against the GPU's
    (check_act_codes_fp8). Rows are in the expert order the permutation of
    gpu_idx gives (stable by token, slot); act_rows(rows) returns the GPU's
    (codes [n, I], scales [n]) of those rows; weight_of(t, e) is the oracle's
    combine weight. Returns (out [len(tokens), H], all-checked mask)."""
    gpu_idx = np.asarray(gpu_idx)
    T, K = gpu_idx.shape
    perm = O.permutation(gpu_idx, E)
    row_of_pair = np.empty(T * K, dtype=np.int64)
    row_of_pair[perm["row_pair"]] = np.arange(T * K)
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    pos = {int(t): i for i, t in enumerate(toks)}
    pairs = (toks[:, None] * K + np.arange(K)[None, :]).ravel()
    experts = gpu_idx.ravel()[pairs]
    out = np.zeros((len(toks), x64.shape[1]))
    for e in np.unique(experts):
        pe = pairs[experts == e]
        rows, tk = row_of_pair[pe], pe // K
        gq, uq, dq = get_expert_q(int(e))
        a64 = O.swiglu_act_fp8(x64[tk], gq, uq)
        codes_g, scale_g = act_rows(rows)
        _, codes, scale = check_act_codes_fp8(a64, codes_g, scale_g)
        y = O.dequantize_rows_e4m3(codes, scale) @ O.dequantize_rows_e4m3(*dq).T
        for i, t in enumerate(tk):
            out[pos[int(t)]] += weight_of(int(t), int(e)) * y[i]
    return out, np.ones(len(toks), dtype=bool)


def act_rows_reader(ws, lay, I):
    """act_rows callable for oracle_outputs_fp8_checked: copies the GPU's
    E4M3 SwiGLU rows and their scales out of the workspace."""
    def read(rows):
        rows = np.asarray(rows, dtype=np.int64)
        codes = np.stack([ws[lay["act_q"] + r * I:lay["act_q"] + (r + 1) * I].cpu().numpy()
                          for r in rows])
        sc = ws[lay["act_scale"]:lay["act_scale"] + (int(rows.max()) + 1) * 4]
        sc = sc.view(torch.float32).cpu().numpy()[rows]
        return codes, sc
    return read


def weights_from_chosen(chosen, tokens=None):
    """weight_of(t, e) from compare_routing's chosen selections (listed in
    the order of `tokens`, default 0..T-1)."""
    toks = range(len(chosen)) if tokens is None else tokens
    maps = {int(t): dict(zip(c[0].tolist(), c[1].tolist())) for t, c in zip(toks, chosen)}
    return lambda t, e: maps[t][e]


def oracle_outputs_fp8(x64, chosen_rows, tokens, get_expert_q):
    """Oracle FP8 combine for the given tokens using the selections."""
    idx = np.stack([chosen_rows[i][0] for i in range(len(tokens))])
    w = np.stack([chosen_rows[i][1] for i in range(len(tokens))])
    return O.moe_combine_fp8(x64[tokens], idx, w, get_expert_q)


def rel_err(got, want):
    want = np.asarray(want, dtype=np.float64)
    got = np.asarray(got, dtype=np.float64)
    rms = np.sqrt(np.mean(want * want))
    return float(np.max(np.abs(got - want)) / rms)


def bf16_ulp(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 1e-38)))
    return np.exp2(e - 7)


def prenorm_ambiguous(h64, gain, eps, rel=4e-7):
    """Elements whose FP64 pre-norm value lies within `rel` (relative) of a
    BF16 rounding midpoint: an FP32 evaluation may round them either way, so
    both BF16 neighbours are correct. Returns a boolean mask."""
    v = O.rms_norm(h64, gain, eps)
    lo = O.bf16_round(v).astype(np.float64)
    # midpoint to the neighbour on the side of v
    ulp = bf16_ulp(lo)
    mid = lo + np.sign(v - lo) * ulp / 2
    return (v != lo) & (np.abs(v - mid) <= rel * np.abs(v))


def bf16_neighbour_toward(lo, v):
    """The BF16 value next to lo (a BF16 value) on the side of v."""
    lo = np.asarray(lo, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    b = (lo.astype(np.float32).view(np.uint32) >> 16).astype(np.int64)
    step = np.where(np.abs(v) > np.abs(lo), 1, -1)       # BF16 is sign-magnitude
    nb = np.where(lo != 0, b + step, b)
    return ((nb.astype(np.uint32) << 16).view(np.float32)).astype(np.float64)


def validated_prenorm_x(x_gpu, h64, gain, eps, rel=4e-7):
    """The GPU's BF16 pre-norm output, checked element by element: each
    element must equal the oracle's BF16 rounding of the FP64 value, or --
    where that value lies within `rel` of a rounding midpoint, so that FP32
    arithmetic may round either way (prenorm_ambiguous) -- the BF16 neighbour
    on the other side of the midpoint. Returns (the validated x as FP64, the
    number of elements that took the other rounding); the oracle routes and
    runs the experts on this x, so no token needs to be left out."""
    v = O.rms_norm(np.asarray(h64, dtype=np.float64), gain, eps)
    lo = O.bf16_round(v).astype(np.float64)
    amb = prenorm_ambiguous(h64, gain, eps, rel)
    other = bf16_neighbour_toward(lo, v)
    xg = np.asarray(x_gpu, dtype=np.float64)
    ok = (xg == lo) | (amb & (xg == other))
    if not ok.all():
        r, c = np.argwhere(~ok)[0]
        raise AssertionError(f"{(~ok).sum()} pre-norm elements are neither rounding; first "
                             f"[{r}, {c}]: gpu {xg[r, c]!r}, oracle {lo[r, c]!r}, exact {v[r, c]!r}")
    return xg, int((ok & (xg != lo)).sum())


def unit_cover_tokens(gpu_idx, E, tiling, size):
    """Tokens whose outputs together pass through every expert-GEMM work unit
    of a call: for every expert, the last token (in the expert's row order,
    ascending token) of each of its row groups. tiling 'groups': the 2-SM
    wide kernel's ceil(n / size) balanced groups (sizes differing by at most
    one); 'tiles': consecutive tiles of `size` rows (token-major and
    weight-major kernels). The last token of a group also lies in its last,
    possibly partial, 16-row MMA block."""
    gpu_idx = np.asarray(gpu_idx)
    picks = set()
    for e in range(E):
        toks = np.nonzero((gpu_idx == e).any(axis=1))[0]
        n = len(toks)
        if n == 0:
            continue
        if tiling == "groups":
            g = (n + size - 1) // size
            q, extra = divmod(n, g)
            ends = [i * q + min(i, extra) + q + (1 if i < extra else 0) - 1 for i in range(g)]
        else:
            ends = [min((j + 1) * size, n) - 1 for j in range((n + size - 1) // size)]
        picks.update(int(toks[p]) for p in ends)
    return np.array(sorted(picks), dtype=np.int64)


# ---------------------------------------------------------------- NVFP4
def sf_index(r, b, K, tile=128):
    """Byte of row r, 16-element block b in the library's SF-group layout
    (512-byte groups per row tile of `tile` rows and K = 64 step)."""
    return ((r // tile) * (K // 64) + b // 4) * 512 + (r % 32) * 16 + ((r % tile) // 32) * 4 + b % 4


def sf_groups_to_plain(sf, rows, K, tile=128):
    """Block scales from the SF-group layout to a plain [rows, K/16] array;
    `sf` starts at a tile boundary."""
    sf = np.asarray(sf)
    r = np.arange(rows)[:, None]
    b = np.arange(K // 16)[None, :]
    return sf[sf_index(r, b, K, tile)]


def expert_getter_nvfp4(gq, uq, dq):
    """Oracle access to NVFP4 expert weights quantised by the library:
    per expert ((codes, plain block scales, group scale) x 3)."""
    cache = {}

    def one(q, e):
        codes, sf, g = q
        n, kh = codes.shape[1], codes.shape[2]
        K = 2 * kh
        start = e * n * K // 16
        sfe = sf[start:start + n * K // 16].cpu().numpy()
        return (codes[e].cpu().numpy(), sf_groups_to_plain(sfe, n, K), g[e:e + 1].cpu().numpy())

    def get(e):
        if e not in cache:
            cache[e] = tuple(one(q, e) for q in (gq, uq, dq))
            if len(cache) > 48:
                cache.pop(next(iter(cache)))
        return cache[e]
    return get


def check_act_codes_nvfp4(a64, gpu_codes, gpu_sf, gpu_g, rel=1e-5, row_abs=1e-5):
    """Validate the GPU's NVFP4 quantisation of SwiGLU rows a64 [n, I] (FP64,
    before rounding): per-row scale, block scales and codes. As for E4M3,
    each element's GPU FP32 value lies within m = rel*|a| + row_abs*max|a_row|
    of a64; BF16 rounding, the block and row maxima, the E4M3 block scale and
    the E2M1 code are monotone in it, so every GPU decision must lie between
    the decisions taken at the interval's two ends (given the GPU's own
    scales for the later steps). Returns (codes, plain block scales, row
    scales) validated."""
    a64 = np.asarray(a64, dtype=np.float64)
    n, I = a64.shape
    m = rel * np.abs(a64) + row_abs * np.max(np.abs(a64), axis=1, keepdims=True)
    lo_v = O.bf16_round(a64 - m).astype(np.float64)
    hi_v = O.bf16_round(a64 + m).astype(np.float64)
    absmin = np.where(lo_v > 0, lo_v, np.where(hi_v < 0, -hi_v, 0.0))
    absmax = np.maximum(np.abs(lo_v), np.abs(hi_v))
    g = np.asarray(gpu_g, dtype=np.float32)
    f2688 = np.float32(2688.0)
    for r in range(n):
        lo_a, hi_a = absmin[r].max(), absmax[r].max()
        if hi_a == 0:
            assert g[r] == 1.0
            continue
        cands = _bf16_grid_between(lo_a, hi_a)
        cands = cands[cands > 0].astype(np.float32)
        assert ((cands / f2688).astype(np.float32) == g[r]).any(), \
            f"row {r}: scale {g[r]} is amax/2688 for no amax in [{lo_a}, {hi_a}]"
    six_g = (np.float32(6.0) * g).astype(np.float32)[:, None]
    bmin = absmin.reshape(n, I // 16, 16).max(axis=2)
    bmax = absmax.reshape(n, I // 16, 16).max(axis=2)
    s_lo = O.e4m3_round((bmin.astype(np.float32) / six_g).astype(np.float32))
    s_hi = O.e4m3_round((bmax.astype(np.float32) / six_g).astype(np.float32))
    sbv = O.e4m3_decode(np.asarray(gpu_sf))
    ok_s = (sbv >= s_lo) & (sbv <= s_hi)
    assert ok_s.all(), f"{(~ok_s).sum()} block scales outside the oracle's interval"
    denom = (sbv.astype(np.float32) * g[:, None]).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(sbv > 0, np.float32(1.0) / np.where(sbv > 0, denom, np.float32(1.0)),
                       np.float32(0.0)).astype(np.float32)
    inv_e = np.repeat(inv, 16, axis=1)
    c_lo = O.e2m1_round((lo_v.astype(np.float32) * inv_e).astype(np.float32))
    c_hi = O.e2m1_round((hi_v.astype(np.float32) * inv_e).astype(np.float32))
    gv = O.e2m1_decode(O.unpack_e2m1(np.asarray(gpu_codes)))
    ok = (gv >= c_lo) & (gv <= c_hi)
    if not ok.all():
        r, j = map(int, np.argwhere(~ok)[0])
        raise AssertionError(f"{(~ok).sum()} act codes outside the oracle's interval; first at "
                             f"row {r} col {j}: a64={a64[r, j]!r} code value {gv[r, j]} not in "
                             f"[{c_lo[r, j]}, {c_hi[r, j]}]")
    return np.asarray(gpu_codes), np.asarray(gpu_sf), g


def nvfp4_pad(T, top_k, E):
    """Token-tile padding of the NVFP4 expert-ordered layout (32 rows on the
    decode tiles, 128 when there are many tokens per expert)."""
    return 32 if T * top_k <= 24 * E else 128


def oracle_outputs_nvfp4_checked(x64, gpu_idx, weight_of, get_expert_q, act_rows, E, pad,
                                 tokens=None):
    """Oracle NVFP4 combine for `tokens`, with each pair row's SwiGLU
    quantisation validated (check_act_codes_nvfp4). Rows are in the
    library's padded expert order: expert e's rows start at the sum of the
    earlier experts' counts each rounded up to `pad`, in pair order.
    act_rows(rows) -> (codes [n, I/2], plain block scales [n, I/16],
    row scales [n])."""
    gpu_idx = np.asarray(gpu_idx)
    T, K = gpu_idx.shape
    perm = O.permutation(gpu_idx, E)
    counts = perm["counts"]
    padded = (counts + pad - 1) // pad * pad
    poff = np.concatenate([[0], np.cumsum(padded)])
    row_of_pair = np.empty(T * K, dtype=np.int64)
    for e in np.nonzero(counts)[0]:
        pr = perm["row_pair"][perm["offsets"][e]:perm["offsets"][e + 1]]
        row_of_pair[pr] = poff[e] + np.arange(len(pr))
    toks = np.arange(T) if tokens is None else np.asarray(tokens)
    pos = {int(t): i for i, t in enumerate(toks)}
    pairs = (toks[:, None] * K + np.arange(K)[None, :]).ravel()
    experts = gpu_idx.ravel()[pairs]
    out = np.zeros((len(toks), x64.shape[1]))
    for e in np.unique(experts):
        pe = pairs[experts == e]
        rows, tk = row_of_pair[pe], pe // K
        gq, uq, dq = get_expert_q(int(e))
        a64 = O.swiglu_act_nvfp4(x64[tk], gq, uq)
        codes_g, sf_g, g_g = act_rows(rows)
        codes, sf, g = check_act_codes_nvfp4(a64, codes_g, sf_g, g_g)
        H = dq[0].shape[0]
        y = O.dequantize_nvfp4(codes, sf, g, 1) @ O.dequantize_nvfp4(*dq, H).T
        for i, t in enumerate(tk):
            out[pos[int(t)]] += weight_of(int(t), int(e)) * y[i]
    return out


def act_rows_reader_nvfp4(ws, lay, I, tile):
    """act_rows callable for oracle_outputs_nvfp4_checked: the GPU's NVFP4
    SwiGLU codes, block scales (token tiles of `tile` rows) and row scales
    from the workspace."""
    def read(rows):
        rows = np.asarray(rows, dtype=np.int64)
        tiles = int(rows.max()) // tile + 1
        sf_all = ws[lay["act_sf"]:lay["act_sf"] + tiles * (I // 64) * 512].cpu().numpy()
        g_all = ws[lay["act_scale"]:lay["act_scale"] + tiles * tile * 4].view(torch.float32).cpu().numpy()
        codes = np.stack([ws[lay["act_q"] + r * (I // 2):lay["act_q"] + (r + 1) * (I // 2)].cpu().numpy()
                          for r in rows])
        idx = sf_index(rows[:, None], np.arange(I // 16)[None, :], I, tile)
        return codes, sf_all[idx], g_all[rows]
    return read
