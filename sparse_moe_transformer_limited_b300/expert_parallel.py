"""Expert parallelism for the Beam MoE sublayer: the layer split by expert
across the ranks of a torch.distributed group.

"Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文", section 多 GPU 和多节点:
each expert lives on one device and the device count divides the 256
experts. Rank d owns experts [d E/P, (d+1) E/P) and their weights; the
router weight is replicated. One call, on every rank, for that rank's own
tokens:

  1. route its tokens (pre-norm, FP32 router, group-limited top-k);
  2. order the token-expert pairs by expert, hence by owning rank;
  3. exchange per-rank row counts, then the rows and their expert ids
     (all-to-all);
  4. run the local experts on the received rows (FP32 outputs);
  5. send the outputs back the same way (all-to-all, reversed splits);
  6. combine them with the router weights, then post-norm and the scaled
     residual (section 残差流).

Steps 1, 2, 4 and 6 are the library's kernels (DeviceOps); the exchanges
are torch.distributed all-to-alls on the group (NCCL on GPUs). The compute
steps are passed in as an object with the DeviceOps methods, so the same
orchestration can run over gloo on the CPU with other implementations.
The row counts are read on the host to size the exchanges (one
device-to-host copy of P integers per call).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch
import torch.distributed as dist

from . import _native as N


@dataclass
class LocalExperts:
    """This rank's experts: w_gate, w_up [E/P, I, H], w_down [E/P, H, I]."""
    w_gate: torch.Tensor
    w_up: torch.Tensor
    w_down: torch.Tensor


class DeviceOps:
    """The library calls of each compute step, on CUDA tensors."""

    def route(self, p, h, w_router, bias, pre_gain):
        """(topk_idx [T,k] int32, topk_w [T,k] fp32, x [T,H] bf16 rows to send)."""
        ws = N.alloc_workspace(p, h.device)
        idx, w, _ = N.route(p, h, w_router, bias=bias, pre_gain=pre_gain, workspace=ws)
        if p.flags & N.FLAG_PRE_NORM:
            off = N.workspace_layout(p)["xn"]
            x = ws[off:off + p.T * p.H * 2].view(torch.bfloat16).view(p.T, p.H)
        else:
            x = h
        return idx, w, x

    def dispatch(self, p, n_ranks, x, idx):
        """(send_x, send_expert, pair_row, send_counts) in send order."""
        return N.ep_dispatch(p, n_ranks, x, idx)

    def empty_rows(self, n, H, like, dtype=None):
        return torch.empty((n, H), dtype=dtype or like.dtype, device=like.device)

    def experts(self, p, rows, local_idx, experts: LocalExperts):
        """FP32 output of each received row's (local) expert."""
        R = rows.shape[0]
        if R == 0:
            return torch.empty((0, p.H), dtype=torch.float32, device=rows.device)
        E_local = experts.w_gate.shape[0]
        q = N.make_params(R, p.H, E_local, p.I, 1, 1, 1, 1.0, p.rms_eps, 0, N.FLAG_FP32_OUT)
        ones = torch.ones((R, 1), dtype=torch.float32, device=rows.device)
        return N.forward_routed(q, rows, local_idx.view(R, 1), ones, experts.w_gate,
                                experts.w_up, experts.w_down)

    def combine(self, p, back, pair_row, w, h, post_gain):
        out_f32 = bool(p.flags & N.FLAG_FP32_OUT)
        return N.ep_combine(back, pair_row, w, h_prev=h, post_gain=post_gain, eps=p.rms_eps,
                            residual_k=p.residual_k, out_f32=out_f32)


def moe_forward_ep(p: N.Params, h: torch.Tensor, w_router: torch.Tensor, experts: LocalExperts,
                   group=None, bias: Optional[torch.Tensor] = None,
                   pre_gain: Optional[torch.Tensor] = None,
                   post_gain: Optional[torch.Tensor] = None, ops=None) -> torch.Tensor:
    """The MoE sublayer for this rank's tokens h [T,H] (p.T = T) with the
    experts split across `group` (every rank calls it, with its own tokens;
    T may differ between ranks). `experts` holds this rank's E/P experts.
    Returns out [T,H] as beam_moe_forward would with all experts local."""
    ops = ops or DeviceOps()
    P = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if p.E % P:
        raise ValueError(f"{P} ranks do not divide {p.E} experts")
    E_local = p.E // P
    if experts.w_gate.shape[0] != E_local:
        raise ValueError(f"rank {rank} holds {experts.w_gate.shape[0]} experts, expected {E_local}")
    # 1-2. route this rank's tokens, order the pairs for sending
    idx, w, x = ops.route(p, h, w_router, bias, pre_gain)
    send_x, send_expert, pair_row, send_counts = ops.dispatch(p, P, x, idx)
    # 3. counts, then rows and expert ids
    recv_counts = torch.empty_like(send_counts)
    dist.all_to_all_single(recv_counts, send_counts, group=group)
    sc = [int(v) for v in send_counts.tolist()]
    rc = [int(v) for v in recv_counts.tolist()]
    recv_x = ops.empty_rows(sum(rc), p.H, send_x)
    dist.all_to_all_single(recv_x, send_x, rc, sc, group=group)
    recv_expert = torch.empty(sum(rc), dtype=send_expert.dtype, device=send_expert.device)
    dist.all_to_all_single(recv_expert, send_expert, rc, sc, group=group)
    # 4. the local experts on the received rows
    y = ops.experts(p, recv_x, recv_expert - rank * E_local, experts)
    # 5. outputs back to their source ranks, in send order
    back = ops.empty_rows(sum(sc), p.H, y)
    dist.all_to_all_single(back, y, sc, rc, group=group)
    # 6. weighted combine, post-norm and residual
    return ops.combine(p, back, pair_row, w, h, post_gain)
