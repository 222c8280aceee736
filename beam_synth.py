"""Seeded synthetic inputs for the Beam MoE sublayer.

This module only draws random tensors of the right shapes, dtypes and value
distributions. It holds none of the layer's arithmetic, so both the CUDA
path (through the binding) and the CPU oracle can take their inputs from it.

Shapes follow the layer as the release pages state it:
  * hidden size 5120, 256 experts per MoE layer, 8 routed per token,
    expert SwiGLU intermediate 2560 -- "Reflection 发布 Beam 501B 开源模型，
    支持 1M tokens 上下文", sections 注意力 and 专家混合模型;
  * 8 groups, 4 kept groups, scaling factor 2.5 -- "Reflection 放出 501B 的
    Beam 权重：四套精度、滑动窗口和一场榜单落差", section
    "config.json 里还有六处能直接抄的细节".

Workloads (value distributions and seeds):
  tiny          T=64,    H=256,  I=128,  seed 0; expert weights FP32 N(0,0.02)
                rounded to BF16, router FP32 N(0,0.05), x N(0,1) in BF16.
  decode        T=64,    H=5120, I=2560, seed 1; expert weights BF16 N(0,0.02),
                router FP32 N(0,0.02), x BF16 N(0,1).
  prefill       T=8192,  same shapes, seed 2.
  skew          T=4096,  same shapes, seed 3; additive router-logit bias
                b_e = 3 * rank_e^-1.1 over a seeded permutation of experts.
  long_prefill  T=16384, same shapes, seed 4; h_prev BF16 N(0,1), pre-norm,
                post-norm and the scaled residual at step k=50.

Large tensors are drawn on the target device with a seeded torch.Generator of
that device (the CPU and CUDA generators give different streams, so a test
that needs the same values on both sides copies them from one to the other).
Small workloads (the tiny one and the shape sweeps) are always drawn on the
CPU and then moved.
"""
from __future__ import annotations

import dataclasses
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int = 5120
    E: int = 256
    I: int = 2560
    n_group: int = 8
    topk_group: int = 4
    top_k: int = 8
    routed_scale: float = 2.5
    rms_eps: float = 1e-6
    seed: int = 0
    w_std: float = 0.02          # expert weight std
    wr_std: float = 0.02         # router weight std
    skew_bias: bool = False      # Zipf-like router-logit bias
    pre_norm: bool = False       # input is h_prev, normalised inside the layer
    residual_k: int = 0          # 0: no residual; else the step index k >= 2

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", T=64, H=256, I=128, seed=0, wr_std=0.05),
    "decode": Workload("decode", T=64, seed=1),
    "prefill": Workload("prefill", T=8192, seed=2),
    "skew": Workload("skew", T=4096, seed=3, skew_bias=True),
    "long_prefill": Workload("long_prefill", T=16384, seed=4, pre_norm=True,
                             residual_k=50),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, std, gen, device, chunk_rows=None):
    """N(0, std) drawn in FP32 then rounded once to BF16, in row chunks."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    step = chunk_rows or shape[0]
    for r0 in range(0, shape[0], step):
        r1 = min(shape[0], r0 + step)
        v = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                        dtype=torch.float32)
        flat[r0:r1].copy_(v.mul_(std))
    return out


def skew_bias(E: int, seed: int, device="cpu") -> torch.Tensor:
    """b_e = 3 * rank_e^-1.1, rank_e = 1 + position of e in a seeded permutation."""
    g = _gen("cpu", seed)
    perm = torch.randperm(E, generator=g)
    rank = torch.empty(E, dtype=torch.float64)
    rank[perm] = torch.arange(1, E + 1, dtype=torch.float64)
    return (3.0 * rank.pow(-1.1)).to(torch.float32).to(device)


def make_inputs(wl: Workload, device="cpu", router_mode: str = "random"):
    """Draw every input of one MoE-sublayer call.

    Returns a dict of torch tensors:
      x         [T,H] bf16   layer input (h_prev when wl.pre_norm)
      w_router  [E,H] f32
      bias      [E]   f32 or None
      w_gate    [E,I,H] bf16
      w_up      [E,I,H] bf16
      w_down    [E,H,I] bf16
    router_mode shapes the routing for edge cases:
      "random"      plain N(0, wr_std)
      "dup_rows"    router rows 1, 33 and 200 copy rows 0, 0 and 199 (exact
                    score ties inside one group and across groups)
      "hot_expert"  a logit bias of +20 on expert 5: every token selects it
      "hot_group"   a logit bias of +20 on experts 0..7: every token selects
                    exactly those eight and the other experts stay empty
    Small workloads (< 64M elements in all) are drawn on the CPU whatever the
    target device, so their values are the same on every machine.
    """
    dev = torch.device(device)
    E, H, I, T = wl.E, wl.H, wl.I, wl.T
    small = (3 * E * I * H + T * H + E * H) < (1 << 26)
    gen_dev = "cpu" if small or dev.type == "cpu" else dev
    g = _gen(gen_dev, wl.seed)

    w_router = torch.randn((E, H), generator=g, device=gen_dev,
                           dtype=torch.float32).mul_(wl.wr_std)
    rows = max(1, min(E, (1 << 26) // max(1, I * H)))
    # Expert weights: FP32 N(0, std) rounded once to BF16.
    w_gate = _randn_bf16((E, I, H), wl.w_std, g, gen_dev, rows)
    w_up = _randn_bf16((E, I, H), wl.w_std, g, gen_dev, rows)
    w_down = _randn_bf16((E, H, I), wl.w_std, g, gen_dev, rows)
    x = _randn_bf16((T, H), 1.0, g, gen_dev, max(1, min(T, (1 << 26) // H)))

    bias = skew_bias(E, wl.seed, gen_dev) if wl.skew_bias else None
    if router_mode == "dup_rows":
        # (indices folded into range for small E)
        w_router[1 % E] = w_router[0]
        w_router[33 % E] = w_router[0]
        w_router[200 % E] = w_router[199 % E]
    elif router_mode in ("hot_expert", "hot_group"):
        if bias is None:
            bias = torch.zeros(E, dtype=torch.float32, device=gen_dev)
        hot = [5] if router_mode == "hot_expert" else list(range(8))
        bias[hot] += 20.0
    elif router_mode != "random":
        raise ValueError(router_mode)
    out = dict(x=x, w_router=w_router, bias=bias, w_gate=w_gate, w_up=w_up,
               w_down=w_down)
    return {k: (v.to(dev) if v is not None else None) for k, v in out.items()}


def make_custom(T, H, E, I, n_group, topk_group, top_k, seed=0, device="cpu",
                wr_std=0.05, **kw) -> tuple:
    """A small workload of arbitrary shape, drawn on the CPU (for shape sweeps)."""
    router_mode = kw.pop("router_mode", "random")
    wl = Workload("custom", T=T, H=H, E=E, I=I, n_group=n_group,
                  topk_group=topk_group, top_k=top_k, seed=seed, wr_std=wr_std,
                  **kw)
    return wl, make_inputs(wl, device, router_mode)


def residual_inputs(T: int, H: int, seed: int, device="cpu"):
    """h_prev BF16 N(0,1) and a sublayer output BF16 N(0,1)."""
    g = _gen("cpu", seed)
    h = torch.randn((T, H), generator=g).to(torch.bfloat16)
    o = torch.randn((T, H), generator=g).to(torch.bfloat16)
    return h.to(device), o.to(device)


def dense_inputs(T: int, H: int, I: int, seed: int, device="cpu"):
    """Dense SwiGLU MLP inputs: x BF16 N(0,1); w_gate, w_up [I,H] and w_down
    [H,I] FP32 N(0, 0.02) rounded to BF16. Small sizes are drawn on the CPU."""
    dev = torch.device(device)
    small = (3 * I * H + T * H) < (1 << 26)
    gen_dev = "cpu" if small or dev.type == "cpu" else dev
    g = _gen(gen_dev, seed)
    w_gate = _randn_bf16((I, H), 0.02, g, gen_dev)
    w_up = _randn_bf16((I, H), 0.02, g, gen_dev)
    w_down = _randn_bf16((H, I), 0.02, g, gen_dev)
    x = _randn_bf16((T, H), 1.0, g, gen_dev, max(1, min(T, (1 << 26) // H)))
    return tuple(t.to(dev) for t in (x, w_gate, w_up, w_down))


def attn_inputs(T: int, H: int, n_q: int, n_kv: int, seed: int, device="cpu", head_dim=128):
    """Attention sublayer inputs: h BF16 N(0,1) [T,H]; the fused weight
    [W_q; W_k; W_v; W_g] [(2 n_q + 2 n_kv) * head_dim, H] and W_o
    [H, n_q * head_dim], FP32 N(0, 0.02) rounded to BF16; q/k RMSNorm gains
    1 + 0.1 N(0,1) (FP32). Small sizes are drawn on the CPU."""
    dev = torch.device(device)
    rows = (2 * n_q + 2 * n_kv) * head_dim
    small = (rows * H + H * n_q * head_dim + T * H) < (1 << 26)
    gen_dev = "cpu" if small or dev.type == "cpu" else dev
    g = _gen(gen_dev, seed)
    w_qkvg = _randn_bf16((rows, H), 0.02, g, gen_dev)
    w_o = _randn_bf16((H, n_q * head_dim), 0.02, g, gen_dev)
    x = _randn_bf16((T, H), 1.0, g, gen_dev, max(1, min(T, (1 << 26) // H)))
    q_gain = 1.0 + 0.1 * torch.randn(head_dim, generator=g, device=gen_dev)
    k_gain = 1.0 + 0.1 * torch.randn(head_dim, generator=g, device=gen_dev)
    return dict(x=x.to(dev), w_qkvg=w_qkvg.to(dev), w_o=w_o.to(dev), q_gain=q_gain.to(dev),
                k_gain=k_gain.to(dev))
