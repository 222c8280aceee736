"""Expert parallelism on CPU ranks (gloo): the orchestration in
sparse_moe_transformer_limited_b300.expert_parallel -- dispatch order, the
row-count and row exchanges, the owners' local expert ids, the return path
and the source-side combine -- with 2 and 4 ranks, each holding E/P experts
and its own tokens. The compute steps are the oracle's (FP64, test-only),
so every rank's result must equal the single-process oracle sublayer on its
tokens with all experts, to FP64 rounding. The library's CUDA steps of the
same protocol are checked on a GPU in test_gpu_ep.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O

H, I, E, TOPK = 64, 32, 256, 8


class OracleOps:
    """The expert_parallel compute steps written with the oracle, on CPU
    FP64 tensors."""

    def route(self, p, h, w_router, bias, pre_gain):
        h64 = h.numpy()
        x = (O.bf16_round(O.rms_norm(h64, None, p.rms_eps)).astype(np.float64)
             if p.flags & 1 else h64)
        sel = O.route(x, w_router.numpy(), None if bias is None else bias.numpy(), p.n_group,
                      p.topk_group, p.top_k, p.routed_scale)
        return (torch.tensor(sel["idx"], dtype=torch.int32), torch.tensor(sel["weights"]),
                torch.tensor(x))

    def dispatch(self, p, P, x, idx):
        # pairs by expert, stable by pair index; rank d owns experts [d E/P, (d+1) E/P)
        flat = idx.numpy().ravel()
        order = np.argsort(flat, kind="stable")
        pair_row = np.empty_like(order)
        pair_row[order] = np.arange(len(order))
        per = p.E // P
        counts = np.array([np.sum((flat >= d * per) & (flat < (d + 1) * per)) for d in range(P)])
        return (x[torch.tensor(order // p.top_k)], torch.tensor(flat[order], dtype=torch.int32),
                torch.tensor(pair_row, dtype=torch.int32), torch.tensor(counts, dtype=torch.int64))

    def empty_rows(self, n, H_, like, dtype=None):
        return torch.empty((n, H_), dtype=torch.float64)

    def experts(self, p, rows, local_idx, experts):
        y = torch.zeros((rows.shape[0], p.H), dtype=torch.float64)
        li = local_idx.numpy()
        for e in np.unique(li):
            sel = np.nonzero(li == e)[0]
            y[sel] = torch.tensor(O.swiglu_expert(rows.numpy()[sel], experts.w_gate[e].numpy(),
                                                  experts.w_up[e].numpy(),
                                                  experts.w_down[e].numpy()))
        return y

    def combine(self, p, back, pair_row, w, h, post_gain):
        T, k = w.shape
        rows = back.numpy()[pair_row.numpy().reshape(T, k)]          # [T, k, H]
        o = np.einsum("tk,tkh->th", w.numpy(), rows)
        if p.residual_k >= 2:
            o = O.residual_step(h.numpy(), o, p.residual_k, None, p.rms_eps, True)
        return torch.tensor(o)


def _weights():
    g = np.random.default_rng(7)
    wr = g.normal(0, 0.05, (E, H))
    wg = O.bf16_round(g.normal(0, 0.02, (E, I, H))).astype(np.float64)
    wu = O.bf16_round(g.normal(0, 0.02, (E, I, H))).astype(np.float64)
    wd = O.bf16_round(g.normal(0, 0.02, (E, H, I))).astype(np.float64)
    return wr, wg, wu, wd


def _rank(rank, world, port, results, Ts=None):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from sparse_moe_transformer_limited_b300 import _native as N
        from sparse_moe_transformer_limited_b300.expert_parallel import (LocalExperts,
                                                                          moe_forward_ep)
        wr, wg, wu, wd = _weights()
        per = E // world
        mine = slice(rank * per, (rank + 1) * per)
        local = LocalExperts(torch.tensor(wg[mine]), torch.tensor(wu[mine]), torch.tensor(wd[mine]))
        T = 40 + 17 * rank if Ts is None else Ts[rank]   # ranks hold different token counts
        h = O.bf16_round(np.random.default_rng(100 + rank).standard_normal((T, H))).astype(np.float64)
        worst = 0.0
        for flags, k in ((0, 0), (1, 9)):            # plain output; pre-norm + residual k = 9
            p = N.make_params(T, H, E, I, 8, 4, TOPK, 2.5, 1e-6, k, flags)
            got = moe_forward_ep(p, torch.tensor(h), torch.tensor(wr), local, ops=OracleOps())
            ref = O.moe_forward(h, wr, None, lambda e: (wg[e], wu[e], wd[e]), n_group=8,
                                topk_group=4, top_k=TOPK, scale=2.5, eps=1e-6,
                                pre_norm=bool(flags), residual_k=k)
            want = ref["h"] if k else ref["out"]
            assert got.shape == (T, H)
            if T:
                worst = max(worst, float(np.max(np.abs(got.numpy() - want)) / np.sqrt(np.mean(want ** 2))))
        results[rank] = worst
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_matches_single_process_oracle(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world, join=True,
                           start_method="spawn")
        worst = dict(results)
    assert sorted(worst) == list(range(world))
    assert max(worst.values()) < 1e-9, worst


def test_expert_parallel_with_a_rank_without_tokens():
    """A rank with no tokens still takes part in every exchange (zero-row
    splits both ways) and its owners' experts serve the other ranks."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank, args=(2, _free_port(), results, (0, 73)), nprocs=2, join=True,
                           start_method="spawn")
        worst = dict(results)
    assert sorted(worst) == [0, 1]
    assert max(worst.values()) < 1e-9, worst


def test_expert_parallel_rejects_a_wrong_local_expert_count():
    """A rank must hold exactly E / P experts: the call raises before any
    exchange."""
    from sparse_moe_transformer_limited_b300 import _native as N
    from sparse_moe_transformer_limited_b300.expert_parallel import LocalExperts, moe_forward_ep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    dist.init_process_group("gloo", rank=0, world_size=1)
    try:
        wr, wg, wu, wd = _weights()
        local = LocalExperts(torch.tensor(wg[:3]), torch.tensor(wu[:3]), torch.tensor(wd[:3]))
        p = N.make_params(4, H, E, I, 8, 4, TOPK, 2.5, 1e-6, 0, 0)
        with pytest.raises(ValueError, match="holds 3 experts"):
            moe_forward_ep(p, torch.zeros((4, H), dtype=torch.float64), torch.tensor(wr), local,
                           ops=OracleOps())
    finally:
        dist.destroy_process_group()
