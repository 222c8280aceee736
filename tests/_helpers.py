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
