"""Expert parallelism on one GPU: the library's steps of the protocol
(beam_ep_dispatch, beam_moe_forward_routed, beam_ep_combine) with P ranks
emulated in one process -- each rank's tokens routed and dispatched, the
all-to-all done by slicing the send buffers, each owner running its E/P
experts on the rows it received, the outputs returned and combined -- must
give what beam_moe_forward gives with all experts on one device. The
orchestration module itself runs over a one-rank NCCL group. All calls go
through the C ABI."""
import os
import socket

import numpy as np
import pytest
import torch

import beam_synth as S
import oracle as O
from _helpers import OUT_REL_TOL, bf16_ulp, compare_routing, expert_getter, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    return B


def _rank_inputs(P, H, I, E, seeds, Ts):
    wl, d = S.make_custom(T=Ts[0], H=H, E=E, I=I, n_group=8, topk_group=4, top_k=8, seed=seeds[0],
                          device="cuda")

    def x_of(T, s):
        if T == 0:          # a rank without tokens
            return torch.empty((0, H), dtype=torch.bfloat16, device="cuda")
        return S.make_custom(T=T, H=H, E=E, I=I, n_group=8, topk_group=4, top_k=8, seed=s,
                             device="cuda")[1]["x"]
    xs = [d["x"]] + [x_of(T, s) for T, s in zip(Ts[1:], seeds[1:])]
    return wl, d, xs


def _ep_emulated(B, P, wl, d, xs, flags, k):
    """The protocol with P ranks in one process; returns each rank's output
    and routing."""
    per = wl.E // P
    sends = []
    for x in xs:
        p = B.make_params(x.shape[0], wl.H, wl.E, wl.I, 8, 4, 8, 2.5, 1e-6, k, flags)
        ws = B.alloc_workspace(p)
        idx, w, _ = B.route(p, x, d["w_router"], workspace=ws)
        xs_send = x
        if flags & B.FLAG_PRE_NORM:
            off = B.workspace_layout(p)["xn"]
            xs_send = ws[off:off + p.T * p.H * 2].view(torch.bfloat16).view(p.T, p.H)
        sx, se, prow, sc = B.ep_dispatch(p, P, xs_send, idx)
        assert B.status() == 0, B.last_error()
        cum = np.concatenate([[0], np.cumsum(sc.cpu().numpy())])
        sends.append(dict(p=p, idx=idx, w=w, sx=sx, se=se, prow=prow, cum=cum, x=x))
    # all-to-all: owner d receives, in source order, every source's block d
    ys = []
    for dst in range(P):
        rx = torch.cat([s["sx"][s["cum"][dst]:s["cum"][dst + 1]] for s in sends])
        re = torch.cat([s["se"][s["cum"][dst]:s["cum"][dst + 1]] for s in sends])
        R = rx.shape[0]
        q = B.make_params(R, wl.H, per, wl.I, 1, 1, 1, 1.0, 1e-6, 0, B.FLAG_FP32_OUT)
        ones = torch.ones((R, 1), dtype=torch.float32, device="cuda")
        local = (re - dst * per).view(R, 1).contiguous()
        sl = slice(dst * per, (dst + 1) * per)
        y = B.forward_routed(q, rx.contiguous(), local, ones, d["w_gate"][sl], d["w_up"][sl],
                             d["w_down"][sl])
        assert B.status() == 0, B.last_error()
        ys.append(y)
    outs = []
    for si, s in enumerate(sends):
        # owner dst returns rows in the order received: source si's part of y_dst
        parts = []
        for dst in range(P):
            before = sum(int(t["cum"][dst + 1] - t["cum"][dst]) for t in sends[:si])
            n = int(s["cum"][dst + 1] - s["cum"][dst])
            parts.append(ys[dst][before:before + n])
        back = torch.cat(parts).contiguous()
        out = B.ep_combine(back, s["prow"], s["w"], h_prev=s["x"], residual_k=k,
                           out_f32=not k)
        assert B.status() == 0, B.last_error()
        outs.append((out, s["idx"], s["w"]))
    return outs


@pytest.mark.parametrize("P,Ts", [(2, (300, 77)), (4, (300, 77, 512, 5)), (4, (300, 0, 512, 5))])
@pytest.mark.parametrize("resid", [False, True])
def test_ep_emulated_matches_single_device(B, P, Ts, resid):
    """(the last case has a rank without tokens: it sends and receives zero
    rows, and its experts still serve the others)"""
    wl, d, xs = _rank_inputs(P, 256, 256, 256, [11, 12, 13, 14][:P], list(Ts))
    flags, k = (B.FLAG_PRE_NORM, 9) if resid else (B.FLAG_FP32_OUT, 0)
    outs = _ep_emulated(B, P, wl, d, xs, flags, k)
    for x, (out, idx, w) in zip(xs, outs):
        if x.shape[0] == 0:
            assert out.shape == (0, wl.H) and idx.shape[0] == 0
            continue
        p = B.make_params(x.shape[0], wl.H, wl.E, wl.I, 8, 4, 8, 2.5, 1e-6, k, flags)
        i2 = torch.empty_like(idx)
        w2 = torch.empty_like(w)
        ref = B.forward(p, x, d["w_router"], d["w_gate"], d["w_up"], d["w_down"], topk_idx=i2,
                        topk_w=w2)
        assert B.status() == 0, B.last_error()
        assert torch.equal(idx, i2) and torch.equal(w, w2)
        a, b = host(out), host(ref)
        # The owners' GEMMs (decode- or prefill-shaped, by their row counts)
        # accumulate in another order than the one-device GEMMs, so a SwiGLU
        # element may take the other BF16 rounding: that moves an output
        # element by about 2^-9 of one expert's term. Bound: 1e-3 of the
        # largest output, plus one BF16 rounding step of the residual output.
        if resid:
            assert np.all(np.abs(a - b) <= bf16_ulp(np.maximum(np.abs(a), np.abs(b))) + 1e-3)
        else:
            assert np.max(np.abs(a - b)) <= 1e-3 * np.max(np.abs(b))
    # and one rank against the oracle
    x64 = host(xs[0]).astype(np.float64)
    if not resid:
        sel = O.route(x64, host(d["w_router"]), None, 8, 4, 8, 2.5)
        _, chosen = compare_routing(sel, outs[0][1].cpu().numpy(), outs[0][2].cpu().numpy(), wl)
        want = O.moe_combine(x64, np.stack([c[0] for c in chosen]),
                             np.stack([c[1] for c in chosen]), expert_getter(d))
        assert rel_err(host(outs[0][0]), want) <= OUT_REL_TOL


def test_ep_dispatch_order_is_the_expert_permutation(B):
    """Send order = pairs by expert, stable by pair; per-rank counts and the
    expert of each sent row follow from it."""
    wl, d = S.make_custom(T=333, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8, seed=3,
                          device="cuda")
    p = B.make_params(wl.T, wl.H, wl.E, wl.I)
    idx, w, _ = B.route(p, d["x"], d["w_router"])
    sx, se, prow, sc = B.ep_dispatch(p, 8, d["x"], idx)
    assert B.status() == 0, B.last_error()
    perm = O.permutation(idx.cpu().numpy(), wl.E)
    flat = idx.cpu().numpy().ravel()
    assert np.array_equal(prow.cpu().numpy()[perm["row_pair"]], np.arange(wl.T * 8))
    assert np.array_equal(se.cpu().numpy(), flat[perm["row_pair"]])
    assert np.array_equal(sc.cpu().numpy(), np.bincount(flat // 32, minlength=8))
    assert torch.equal(sx, d["x"][torch.as_tensor(perm["row_pair"] // 8, device="cuda")])


def test_routed_forward_rejects_bad_index_without_fault(B):
    """An expert index outside [0, E) is dropped with the device error flag
    raised; the call completes and the context keeps working."""
    wl, d = S.make_custom(T=40, H=256, E=32, I=256, n_group=1, topk_group=1, top_k=2, seed=9,
                          device="cuda")
    p = B.make_params(40, 256, 32, 256, 1, 1, 2, 1.0, 1e-6, 0, B.FLAG_FP32_OUT)
    idx = torch.randint(0, 32, (40, 2), dtype=torch.int32, device="cuda")
    idx[5, 1] = 32
    idx[7, 0] = -1
    w = torch.ones((40, 2), dtype=torch.float32, device="cuda")
    B.forward_routed(p, d["x"], idx, w, d["w_gate"], d["w_up"], d["w_down"])
    assert B.status() == 6                       # BEAM_ERR_DEVICE_FLAG
    assert "outside [0, E)" in B.last_error()
    B.forward_routed(p, d["x"], idx.clamp(0, 31), w, d["w_gate"], d["w_up"], d["w_down"])
    assert B.status() == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_orchestration_over_one_rank_nccl_group(B):
    """expert_parallel.moe_forward_ep with the library's ops over a one-rank
    NCCL group equals beam_moe_forward (the exchanges are identities)."""
    import torch.distributed as dist
    from sparse_moe_transformer_limited_b300.expert_parallel import LocalExperts, moe_forward_ep
    wl, d = S.make_custom(T=200, H=256, E=256, I=256, n_group=8, topk_group=4, top_k=8, seed=21,
                          device="cuda")
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        p = B.make_params(wl.T, wl.H, wl.E, wl.I, 8, 4, 8, 2.5, 1e-6, 9, B.FLAG_PRE_NORM)
        got = moe_forward_ep(p, d["x"], d["w_router"],
                             LocalExperts(d["w_gate"], d["w_up"], d["w_down"]))
        ref = B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"])
        assert B.status() == 0, B.last_error()
        a, b = host(got), host(ref)
        assert np.all(np.abs(a - b) <= bf16_ulp(np.maximum(np.abs(a), np.abs(b))) + 1e-6)
    finally:
        dist.destroy_process_group()
