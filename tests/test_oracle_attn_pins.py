"""Pins for the oracle's attention sublayer, each against something other
than the oracle: closed forms of RoPE and the global query scale, a
brute-force per-query loop, special cases (window 1, equal scores), a
one-hot check of the query-to-key/value head mapping, and torch's
scaled_dot_product_attention. No GPU needed."""
import math

import numpy as np
import torch

import oracle as O


def test_rope_closed_forms():
    # d = 2: the pair (x, y) turns by pos * theta^0 = pos radians
    v = np.array([[[1.0, 0.0]]] * 3).reshape(1, 3, 2)
    out = O.rope_rotate(v, np.array([0, 1, 2]))
    assert np.allclose(out[0], [[1, 0], [math.cos(1), math.sin(1)], [math.cos(2), math.sin(2)]])
    rng = np.random.default_rng(0)
    q, k = rng.standard_normal((2, 1, 5, 128))
    # norms of the (i, i + 64) pairs are kept
    rq = O.rope_rotate(q, np.arange(5))
    assert np.allclose(q[..., :64] ** 2 + q[..., 64:] ** 2, rq[..., :64] ** 2 + rq[..., 64:] ** 2)
    # position 0 is the identity; dot products depend only on the position difference
    assert np.allclose(rq[0, 0], q[0, 0])
    a = (O.rope_rotate(q, np.array([3, 3, 3, 3, 3]))[0, 0] @ O.rope_rotate(k, np.array([1] * 5))[0, 0])
    b = (O.rope_rotate(q, np.array([10] * 5))[0, 0] @ O.rope_rotate(k, np.array([8] * 5))[0, 0])
    assert np.isclose(a, b)
    # channel pair i turns with frequency 10000^(-2i/128): pair 32 at position 1
    e = np.zeros((1, 1, 128)); e[0, 0, 32] = 1.0
    r = O.rope_rotate(e, np.array([1]))[0, 0]
    ang = 10000.0 ** (-64 / 128)
    assert np.isclose(r[32], math.cos(ang)) and np.isclose(r[96], math.sin(ang))


def test_global_query_scale_closed_form():
    assert O.global_query_scale(np.array([-1.0]))[0] == 1.0
    assert np.isclose(O.global_query_scale(np.array([2047.0]))[0], 2.0 ** 0.1)
    assert np.isclose(O.global_query_scale(np.array([6143.0]))[0], 4.0 ** 0.1)


def _brute(q, k, v, window):
    nq, T, d = q.shape
    g = nq // k.shape[0]
    out = np.zeros_like(q)
    for h in range(nq):
        for i in range(T):
            keys = [j for j in range(T) if j <= i and (window == 0 or i - j < window)]
            s = np.array([q[h, i] @ k[h // g, j] / math.sqrt(d) for j in keys])
            w = np.exp(s - s.max())
            w /= w.sum()
            out[h, i] = sum(wj * v[h // g, j] for wj, j in zip(w, keys))
    return out


def test_core_brute_force_and_special_cases():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, 9, 8))
    k = rng.standard_normal((2, 9, 8))
    v = rng.standard_normal((2, 9, 8))
    for window in (0, 1, 3, 100):
        assert np.allclose(O.attention_core(q, k, v, window), _brute(q, k, v, window))
    # window 1: every query sees only itself
    o = O.attention_core(q, k, v, 1)
    assert np.allclose(o[0], v[0]) and np.allclose(o[3], v[1])
    # equal scores: the mean of the visible values (causal prefix / last w)
    z = np.zeros_like(q)
    o = O.attention_core(z, k, v, 0)
    assert np.allclose(o[0, 4], v[0, :5].mean(axis=0))
    o = O.attention_core(z, k, v, 3)
    assert np.allclose(o[2, 6], v[1, 4:7].mean(axis=0))


def test_query_head_to_kv_head_mapping():
    T, d = 5, 4
    q = np.random.default_rng(2).standard_normal((48, T, d))
    k = np.zeros((8, T, d))
    v = np.zeros((8, T, d))
    v[3] = 1.0                                   # only key/value head 3 carries ones
    o = O.attention_core(q, k, v, 0)
    ones = np.array([np.allclose(o[h], 1.0) for h in range(48)])
    assert ones.sum() == 6 and np.all(ones[18:24])   # query heads 18..23 = 3 * 6 .. 3 * 6 + 5


def test_core_matches_torch_sdpa():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, 12, 40, 32, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, 40, 32, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, 40, 32, generator=g, dtype=torch.float64)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, enable_gqa=True)
    got = O.attention_core(q[0].numpy(), k[0].numpy(), v[0].numpy(), 0)
    assert np.allclose(got, ref[0].numpy(), atol=1e-12)
    i = torch.arange(40)[:, None]
    j = torch.arange(40)[None, :]
    mask = (j <= i) & (i - j < 7)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, enable_gqa=True)
    assert np.allclose(O.attention_core(q[0].numpy(), k[0].numpy(), v[0].numpy(), 7), ref[0].numpy(),
                       atol=1e-12)


def test_forward_gate_and_layout():
    """Zero gate weights give a gate of 1/2 everywhere; the fused weight's
    row blocks are read as [W_q; W_k; W_v; W_g]."""
    rng = np.random.default_rng(4)
    T, H, nq, nkv, d = 12, 64, 6, 2, 16
    w = rng.standard_normal(((nq + 2 * nkv + nq) * d, H)) * 0.1
    w[(nq + 2 * nkv) * d:] = 0.0
    wo = np.eye(H, nq * d)
    r = O.attention_forward(rng.standard_normal((T, H)), w, wo, np.ones(d), np.ones(d), n_q=nq,
                            n_kv=nkv, head_dim=d, window=4)
    assert np.allclose(r["gate"], 0.5)
    o = O.attention_core(r["q"], r["k"], r["v"], 4).transpose(1, 0, 2).reshape(T, nq * d)
    assert np.allclose(r["attn"], O.bf16_round(0.5 * o), rtol=0, atol=0)
    # K rows come right after the query rows: a zero K block gives equal scores
    w2 = w.copy()
    w2[nq * d:(nq + nkv) * d] = 0.0
    r2 = O.attention_forward(np.ones((T, H)), w2, wo, np.ones(d), np.ones(d), n_q=nq, n_kv=nkv,
                             head_dim=d, window=0)
    assert np.allclose(r2["k"], 0.0)


def test_forward_query_row_subset_equals_full():
    rng = np.random.default_rng(5)
    T, H, nq, nkv, d = 30, 64, 4, 2, 16
    w = rng.standard_normal(((nq + 2 * nkv + nq) * d, H)) * 0.1
    wo = rng.standard_normal((H, nq * d)) * 0.1
    h = rng.standard_normal((T, H))
    for window in (0, 7):
        full = O.attention_forward(h, w, wo, np.ones(d), np.ones(d), n_q=nq, n_kv=nkv,
                                   head_dim=d, window=window, residual_k=5)
        rows = np.array([0, 3, 17, 29])
        sub = O.attention_forward(h, w, wo, np.ones(d), np.ones(d), n_q=nq, n_kv=nkv,
                                  head_dim=d, window=window, residual_k=5, query_rows=rows)
        assert np.allclose(sub["out"], full["out"][rows], rtol=1e-12, atol=1e-12)
        assert np.allclose(sub["h"], full["h"][rows], rtol=1e-12, atol=1e-12)


def test_forward_single_token_closed_form():
    """T = 1: the softmax has one key, so every head's output is its KV
    head's value row, whatever q and k are. Closed form:
    out = bf16(v[kv(h)] * sigmoid(x W_g^T)) W_o^T with x = bf16(RMSNorm(h_in)),
    v = bf16(x W_v^T) -- it fixes the third block of the fused weight as W_v,
    the fourth as the gate, the gate's per-channel product with the head
    outputs, the query-head to KV-head grouping and W_o's orientation."""
    import torch
    rng = np.random.default_rng(6)
    H, nq, nkv, d = 32, 4, 2, 8
    h_in = rng.standard_normal((1, H))
    wq, wk, wv, wg = (rng.standard_normal((n * d, H)) * 0.3 for n in (nq, nkv, nkv, nq))
    wo = rng.standard_normal((H, nq * d)) * 0.3
    w = np.concatenate([wq, wk, wv, wg])
    for window in (0, 16):
        r = O.attention_forward(h_in, w, wo, np.ones(d) * 1.5, np.ones(d) * 0.5, n_q=nq,
                                n_kv=nkv, head_dim=d, window=window)
        bf = lambda a: torch.tensor(a, dtype=torch.float64).to(torch.bfloat16).to(torch.float64).numpy()
        x = bf(h_in / np.sqrt(np.mean(h_in ** 2) + 1e-6))
        v = bf(x @ wv.T).reshape(nkv, d)
        heads = np.concatenate([v[hd // (nq // nkv)] for hd in range(nq)])
        gate = 1.0 / (1.0 + np.exp(-(x @ wg.T)[0]))
        want = bf(heads * gate) @ wo.T
        assert np.allclose(r["out"][0], want, rtol=1e-12, atol=1e-12)


def test_forward_global_query_scale_follows_the_norms():
    """Global layer: q = (1 + (pos+1)/2048)^0.1 * RMSNorm(x W_q^T) * q_gain
    and k = RMSNorm(x W_k^T) * k_gain, per head. With q_gain = 2 and
    k_gain = 1/2 the RMS over a head's channels is 2 * scale(pos) for
    queries and 1/2 for keys, up to BF16 rounding (relative 2^-9): at
    position 2047 the scale is 2^0.1, so a scale applied before the norm,
    or the key gain used for queries, is far off."""
    rng = np.random.default_rng(16)
    T, H, nq, nkv, d = 2048, 32, 2, 1, 16
    w = rng.standard_normal(((nq + 2 * nkv + nq) * d, H)) * 0.3
    wo = rng.standard_normal((H, nq * d)) * 0.3
    rows = np.array([0, 1023, 2047])
    r = O.attention_forward(rng.standard_normal((T, H)), w, wo, np.full(d, 2.0), np.full(d, 0.5),
                            n_q=nq, n_kv=nkv, head_dim=d, window=0, query_rows=rows)
    rms_q = np.sqrt(np.mean(r["q"] ** 2, axis=-1))               # [nq, rows]
    want = 2.0 * (1.0 + (rows + 1.0) / 2048.0) ** 0.1
    assert np.allclose(rms_q, want[None, :], rtol=2.0 ** -8, atol=0)
    assert np.allclose(np.sqrt(np.mean(r["k"] ** 2, axis=-1)), 0.5, rtol=2.0 ** -8, atol=0)


def test_forward_rope_acts_after_the_norm_gains():
    """Sliding layer, every token the same input row: before RoPE the
    normalised, gained q and k are the same at every position, and RoPE only
    turns each (i, i + d/2) pair, so each pair's length is the same at every
    position (up to BF16 rounding). The gains differ between the two halves
    (1 and 2), so a norm or gain applied after the rotation would change the
    pair lengths with the position."""
    rng = np.random.default_rng(17)
    T, H, nq, nkv, d = 12, 32, 2, 1, 16
    w = rng.standard_normal(((nq + 2 * nkv + nq) * d, H)) * 0.3
    wo = rng.standard_normal((H, nq * d)) * 0.3
    h_in = np.tile(rng.standard_normal((1, H)), (T, 1))
    g_q = np.concatenate([np.ones(d // 2), np.full(d // 2, 2.0)])
    r = O.attention_forward(h_in, w, wo, g_q, g_q[::-1].copy(), n_q=nq, n_kv=nkv, head_dim=d,
                            window=8)
    for a in (r["q"], r["k"]):
        pair = np.sqrt(a[..., : d // 2] ** 2 + a[..., d // 2:] ** 2)   # [heads, T, d/2]
        assert np.allclose(pair, pair[:, :1, :], rtol=2.0 ** -7, atol=0)


def test_forward_gains_and_residual_branch():
    """The pre-norm gain scales each channel of the BF16 input x exactly
    (powers of two); the post-norm gain scales the branch
    h_k - sqrt((k-1)/k) h_{k-1}; and with W_o = 0 the output is 0, so
    h_k = sqrt((k-1)/k) h_{k-1} with h_{k-1} the layer input itself (RMS 4
    here, so not its normalised copy)."""
    rng = np.random.default_rng(19)
    T, H, nq, nkv, d, k = 10, 32, 2, 1, 16, 7
    w = rng.standard_normal(((nq + 2 * nkv + nq) * d, H)) * 0.3
    wo = rng.standard_normal((H, nq * d)) * 0.3
    h = rng.standard_normal((T, H)) * 4.0
    g = np.tile([0.5, 1.0, 2.0, 4.0], H // 4)
    run = lambda wo_, pg, qg: O.attention_forward(h, w, wo_, np.ones(d), np.ones(d), n_q=nq,
                                                  n_kv=nkv, head_dim=d, window=4, pre_gain=pg,
                                                  residual_k=k, post_gain=qg)
    base, pre, post = run(wo, None, None), run(wo, g, None), run(wo, None, g)
    assert np.array_equal(pre["x"], base["x"] * g[None, :])
    keep = math.sqrt((k - 1) / k) * h
    assert np.allclose(post["h"] - keep, (base["h"] - keep) * g[None, :], rtol=1e-13, atol=1e-13)
    zero = run(np.zeros_like(wo), None, None)
    assert np.array_equal(zero["out"], np.zeros((T, H)))
    assert np.allclose(zero["h"], keep, rtol=1e-15, atol=0)
