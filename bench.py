"""Benchmark of the Beam MoE sublayer on B300 GPUs.

One step = one pass of the whole sublayer over one batch: pre-RMSNorm, FP32
router with group-limited top-8, permutation, SwiGLU experts, weighted
combine, post-RMSNorm and the scaled residual update at k=50. Inputs are
synthetic (seeded; see beam_synth.py), weights random-init of the layer's
shapes (20.1 GB of BF16 expert weights, larger than the 126 MB L2, so no L2
flush is needed between steps).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode|prefill|skew|long_prefill]
                  [--impl ours|reference]

Prints one JSON line on rank 0. With N > 1 (torchrun) every rank runs an
independent replica on its own batch (weak scaling, no data-path
collective); `value` is the tokens/s of all ranks over the slowest rank's
time. `--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import beam_synth as S  # noqa: E402

METRIC = "MoE-layer tokens/s at T=64 and T=8192; % of HBM or BF16 tensor roofline"
RESIDUAL_K = 50


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=6400.0, bf16=1800.0, bf16_sustained=1400.0, source="fallback")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "25", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- ranks
def combine_ranks(ms_total: float, e2e_s: float, world: int, device) -> tuple:
    """Slowest rank's device time and end-to-end time (each rank ran its own
    batch; the job finishes when the slowest rank does)."""
    if world <= 1:
        return ms_total, e2e_s
    t = torch.tensor([ms_total, e2e_s], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t[0].item()), float(t[1].item())


def weak_scaling_value(world: int, tokens_per_rank: int, steps: int, seconds: float) -> float:
    """Tokens/s of the whole job: all ranks' tokens over the slowest time."""
    return world * tokens_per_rank * steps / seconds


def timed_steps(B, step, steps, stream, barrier, gpu_index, prof_steps=10):
    """Time `steps` calls of step() with CUDA events on `stream` while the
    clocks are sampled (the library's per-launch events off), then run up to
    prof_steps more with the per-launch events on for the per-kernel split.
    Returns (ms over the timed steps, per-kernel record, clocks, profiled steps)."""
    clocks = ClockSampler(gpu_index)
    barrier()
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    n_prof = max(1, min(steps, prof_steps))
    B.profile_read()
    B.profile_enable(True)
    for _ in range(n_prof):
        step()
    barrier()
    B.profile_enable(False)
    prof = B.profile_read()
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    return ms, prof, clk, n_prof


# ------------------------------------------------------------ workload
def _workload(name):
    wl = S.WORKLOADS[name]
    return wl


def _config(wl, world):
    """The workload description both arms print."""
    return {"workload": _describe(wl), "T": wl.T, "H": wl.H, "E": wl.E, "I": wl.I,
            "top_k": wl.top_k, "seed": wl.seed,
            "parallelism": "replicas" if world > 1 else "single GPU",
            "l2": "no flush: 20.1 GB of expert weights per step exceed the 126 MB L2"}


def _describe(wl):
    return (f"Beam MoE sublayer, {wl.name}: T={wl.T} tokens, hidden {wl.H}, {wl.E} experts "
            f"(8 groups x 32, keep 4), top-{wl.top_k}, SwiGLU intermediate {wl.I}; "
            f"pre-RMSNorm -> FP32 sigmoid router -> permute -> experts -> x2.5 weighted "
            f"combine -> post-RMSNorm -> residual k={RESIDUAL_K}")


# bytes per weight element and per weight row, by expert weight type:
# BF16; E4M3 codes + one FP32 scale per row; NVFP4 packed codes + one E4M3
# block scale per 16 elements (the per-matrix FP32 scale is negligible)
WEIGHT_BYTES = {"bf16": (2.0, 0), "fp8": (1.0, 4), "nvfp4": (0.5 + 1.0 / 16, 0)}
# nominal dense tensor rate relative to BF16 (2.25 / 4.5 / 13.5 PFLOP/s)
TENSOR_RATIO = {"bf16": 1, "fp8": 2, "nvfp4": 6}


def _algorithmic(wl, counts, kind="bf16"):
    """Algorithmic bytes / FLOPs (what the method must move and compute): each
    touched expert's weights once (WEIGHT_BYTES) plus the layer's BF16 input
    or output; the intermediates (permuted x, SwiGLU activations, the FP32
    combine rows) are not counted."""
    touched = int((counts > 0).sum())
    R = wl.T * wl.top_k
    eb, sc = WEIGHT_BYTES[kind]
    gu_bytes = int(touched * 2 * wl.I * (wl.H * eb + sc)) + wl.T * wl.H * 2
    dn_bytes = int(touched * wl.H * (wl.I * eb + sc)) + wl.T * wl.H * 2
    gu_flops = 2.0 * R * 2 * wl.I * wl.H
    dn_flops = 2.0 * R * wl.I * wl.H
    layer_bytes = (int(touched * (3 * wl.I * wl.H * eb + (2 * wl.I + wl.H) * sc))
                   + 2 * wl.T * wl.H * 2 + wl.E * wl.H * 4)
    return dict(touched=touched, gu_bytes=gu_bytes, dn_bytes=dn_bytes, gu_flops=gu_flops,
                dn_flops=dn_flops, layer_bytes=layer_bytes,
                layer_flops=gu_flops + dn_flops + 2.0 * wl.T * wl.H * wl.E)


def gemm_roofline(kname, nbytes, flops, launch_ms, peaks, dtype, traffic):
    """Roofline of one GEMM launch against the bound that binds it: the larger
    of the two least times, algorithmic bytes / measured copy rate and
    algorithmic FLOPs / measured sustained tensor rate (the expert GEMMs run
    inside loops of back-to-back steps, seconds under the board's power cap).
    Decode-sized launches are bound by their weight bytes; prefill BF16 by
    FLOPs; with few tokens per expert (skewed routing) or packed 4-bit
    weights the bytes can bind at prefill sizes too. The other bound's
    fraction is given beside it."""
    s = launch_ms / 1e3
    hbm = {"bound": "hbm", "achieved": round(nbytes / s / 1e9, 1), "peak": peaks["hbm"],
           "unit": "GB/s", "frac": round(nbytes / s / 1e9 / peaks["hbm"], 4),
           "peak_source": peaks["source"] + " hbm_gbs", "algorithmic_bytes_per_launch": nbytes}
    tc = {"bound": "tensor", "achieved": round(flops / s / 1e12, 1),
          "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
          "frac": round(flops / s / 1e12 / peaks["bf16_sustained"], 4),
          "peak_source": (peaks["source"] + " bf16_tflops_sustained (timed inside a long step)"
                          + peaks.get("tensor_note", "")),
          "frac_of_burst": round(flops / s / 1e12 / peaks["bf16"], 4),
          "algorithmic_flops_per_launch": flops}
    t_bytes = nbytes / (peaks["hbm"] * 1e9)
    t_flops = flops / (peaks["bf16_sustained"] * 1e12)
    roof, other = (hbm, tc) if t_bytes >= t_flops else (tc, hbm)
    roof = dict({"kernel": kname}, **roof)
    roof.update(dtype=dtype, traffic=traffic, launch_ms=round(launch_ms, 4),
                other_bound={"bound": other["bound"], "frac": other["frac"]})
    return roof


def _traffic_for(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    for r in rec.get("entries", []):
        if r.get("kernel") != kernel or r.get("workload") != workload:
            continue
        src = os.path.join(ROOT, "sparse_moe_transformer_limited_b300", "csrc", r["src_file"])
        try:
            with open(src, "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()[:16]
        except OSError:
            return None
        return r.get("dram_bytes_per_launch") if r.get("src_sha") == sha else None
    return None


# ------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank, kind="bf16"):
    """The sublayer with BF16 expert weights, or E4M3 / NVFP4 expert weights
    quantised once on the device before any timing."""
    fp8, f4 = kind == "fp8", kind == "nvfp4"
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = _workload(args.config)
    wl_rank = wl.replace(seed=wl.seed + 1000 * rank) if rank else wl
    d = S.make_inputs(wl_rank, dev)
    flags = (B.FLAG_PRE_NORM | (B.FLAG_FP8_EXPERTS if fp8 else 0)
             | (B.FLAG_NVFP4_EXPERTS if f4 else 0))
    p = B.make_params(wl.T, wl.H, wl.E, wl.I, wl.n_group, wl.topk_group, wl.top_k,
                      wl.routed_scale, wl.rms_eps, RESIDUAL_K, flags)
    ws = B.alloc_workspace(p, dev)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    if fp8 or f4:
        quant = B.quantize_e4m3_rows if fp8 else B.quantize_nvfp4
        q = tuple(quant(d[k]) for k in ("w_gate", "w_up", "w_down"))
        for k in ("w_gate", "w_up", "w_down"):
            d[k] = None
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()

    def fwd(x_in, o=None):
        o = out if o is None else o
        if fp8:
            B.forward_fp8(p, x_in, d["w_router"], *q, bias=d["bias"], out=o, workspace=ws)
        elif f4:
            B.forward_nvfp4(p, x_in, d["w_router"], *q, bias=d["bias"], out=o, workspace=ws)
        else:
            B.forward(p, x_in, d["w_router"], d["w_gate"], d["w_up"], d["w_down"],
                      bias=d["bias"], out=o, workspace=ws)

    def step():
        fwd(d["x"])

    for _ in range(max(args.warmup, 3)):
        step()
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    lay = B.workspace_layout(p)
    counts = ws[lay["counts"]:lay["counts"] + wl.E * 4].view(torch.int32).cpu().numpy()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    # ---- device-timed region (inputs resident in HBM), per-launch events off;
    # then the per-kernel split in a second pass of the same steps
    ms_total, prof, clk, prof_steps = timed_steps(B, step, args.steps, stream, barrier, local_rank)

    # ---- end-to-end through the public API with host buffers: every step
    # uploads its input from pinned host memory and downloads its output.
    # The copies run on their own streams with two device buffers each, so
    # step i+1's upload and step i-1's download overlap step i's forward
    # (what a serving loop does); events order each buffer's reuse.
    h_host = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    h_host.copy_(d["x"].cpu())
    o_host = [torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(d["x"]) for _ in range(2)]
    o_dev = [torch.empty_like(out) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp = torch.cuda.current_stream(dev)
    x_ready, x_free, o_ready, o_free = ([torch.cuda.Event() for _ in range(2)] for _ in range(4))
    for e in x_free + o_free:
        e.record(comp)

    def e2e_step(i):
        b = i & 1
        up.wait_event(x_free[b])
        with torch.cuda.stream(up):
            x_dev[b].copy_(h_host, non_blocking=True)
        x_ready[b].record(up)
        comp.wait_event(x_ready[b])
        comp.wait_event(o_free[b])
        fwd(x_dev[b], o_dev[b])
        x_free[b].record(comp)
        o_ready[b].record(comp)
        down.wait_event(o_ready[b])
        with torch.cuda.stream(down):
            o_host[b].copy_(o_dev[b], non_blocking=True)
        o_free[b].record(down)

    for i in range(3):
        e2e_step(i)
    barrier()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    barrier()
    e2e_s = time.perf_counter() - t0
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    ms_total, e2e_s = combine_ranks(ms_total, e2e_s, world, dev)
    ms_step = ms_total / args.steps
    value = weak_scaling_value(world, wl.T, args.steps, ms_total / 1e3)
    e2e_value = weak_scaling_value(world, wl.T, args.steps, e2e_s)

    alg = _algorithmic(wl, counts, kind)
    peaks = _peaks()
    if kind != "bf16":
        # E4M3 / NVFP4 contraction: the measured BF16 peaks times the nominal
        # dense ratio to BF16 (4.5 / 2.25 and 13.5 / 2.25 PFLOP/s)
        rt = TENSOR_RATIO[kind]
        peaks = dict(peaks, bf16=rt * peaks["bf16"], bf16_sustained=rt * peaks["bf16_sustained"],
                     tensor_note=f" x {rt} (nominal {kind}/BF16 dense ratio)")
    gu_ms = prof["expert_gemm_gateup_swiglu"][0] / prof["expert_gemm_gateup_swiglu"][1]
    kname = "expert_gemm_gateup_swiglu"
    roof = gemm_roofline(kname, alg["gu_bytes"], alg["gu_flops"], gu_ms, peaks,
                         {"bf16": "bf16", "fp8": "e4m3", "nvfp4": "nvfp4"}[kind],
                         _traffic_for(kname, wl.name if kind == "bf16" else f"{wl.name}_{kind}"))
    layer = {"hbm_frac": round(alg["layer_bytes"] / (ms_step / 1e3) / 1e9 / peaks["hbm"], 4),
             "tensor_frac": round(alg["layer_flops"] / (ms_step / 1e3) / 1e12
                                  / peaks["bf16_sustained"], 4),
             "tensor_frac_of_burst": round(alg["layer_flops"] / (ms_step / 1e3) / 1e12
                                           / peaks["bf16"], 4),
             "touched_experts": alg["touched"], "max_tokens_per_expert": int(counts.max())}
    kernels = {k: round(v[0] / v[1], 4) for k, v in sorted(prof.items(), key=lambda kv: -kv[1][0])}
    # the library's launches in the timed region: per step (from the profiled
    # pass, which runs the same steps) times the timed steps
    launches = sum(v[1] for v in prof.values()) // prof_steps * args.steps
    return dict(value=value, ms_step=ms_step, e2e=e2e_value, clocks=clk, roofline=roof,
                layer=layer, kernels_ms=kernels, wl=wl, launches=launches,
                h2d=wl.T * wl.H * 2, d2h=wl.T * wl.H * 2)


# ------------------------------------------------------- dense MLP arm
# The dense SwiGLU MLP of the first layers. Its intermediate size is not on
# the pages; 12288 (2.4 x hidden) stands in for it. Layer 0's MLP is residual
# step k = 3 (the embedding is step 1, layer 0's attention step 2).
DENSE = {"dense_prefill": dict(T=8192, H=5120, I=12288, seed=5),
         "dense_decode": dict(T=64, H=5120, I=12288, seed=6)}
DENSE_K = 3


def run_dense(args, rank, world, local_rank, name):
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = DENSE[name]
    T, H, I = cfg["T"], cfg["H"], cfg["I"]
    x, wg, wu, wd = S.dense_inputs(T, H, I, cfg["seed"] + 1000 * rank, dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    n = B.lib().beam_dense_workspace_size(ctypes.byref(B.DenseParams(T, H, I, 1e-6, DENSE_K,
                                                                     B.FLAG_PRE_NORM)))
    ws = torch.empty(n, dtype=torch.uint8, device=dev)

    def step():
        B.dense_forward(T, H, I, x, wg, wu, wd, residual_k=DENSE_K, flags=B.FLAG_PRE_NORM,
                        out=out, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    ms, prof, clk, _ = timed_steps(B, step, args.steps, torch.cuda.current_stream(dev),
                                   lambda: torch.cuda.synchronize(dev), local_rank)
    ms /= args.steps
    peaks = _peaks()
    gu_ms = prof["expert_gemm_gateup_swiglu"][0] / prof["expert_gemm_gateup_swiglu"][1]
    flops = 2.0 * T * 3 * H * I
    wbytes = 3 * H * I * 2 + 2 * T * H * 2
    if T <= 24:
        bound, ach, peak, unit = "hbm", 2 * I * H * 2 / (gu_ms / 1e3) / 1e9, peaks["hbm"], "GB/s"
    else:
        bound, ach, peak, unit = ("tensor", 2.0 * T * 2 * I * H / (gu_ms / 1e3) / 1e12,
                                  peaks["bf16_sustained"], "TFLOP/s")
    return {"workload": f"dense SwiGLU MLP sublayer T={T}, hidden {H}, intermediate {I} "
                        f"(stand-in size), pre-norm + residual k={DENSE_K}",
            "value": round(T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "layer_tflops": round(flops / (ms / 1e3) / 1e12, 1),
            "layer_hbm_gbs": round(wbytes / (ms / 1e3) / 1e9, 1),
            "roofline": {"kernel": "expert_gemm_gateup_swiglu", "bound": bound,
                         "achieved": round(ach, 1), "peak": peak, "unit": unit,
                         "frac": round(ach / peak, 4), "launch_ms": round(gu_ms, 4),
                         **({"frac_of_burst": round(ach / peaks["bf16"], 4),
                             "peak_source": peaks["source"] + " bf16_tflops_sustained"}
                            if bound == "tensor" else {})},
            "kernels_ms": {k: round(v[0] / v[1], 4) for k, v in prof.items()}, "clocks": clk}


# ------------------------------------------------------- attention arm
# The attention sublayer over one sequence of 8192 tokens (hidden 5120, 48
# query / 8 key-value heads of 128, pre-norm, post-norm and residual): a
# sliding-window layer (window 512, RoPE; layer 4, residual step k = 10) and a
# global layer (layer 5, k = 12).
ATTN = {"attn_swa": dict(T=8192, window=512, k=10, seed=12),
        "attn_global": dict(T=8192, window=0, k=12, seed=13)}


def run_attn(args, rank, world, local_rank, name):
    import sparse_moe_transformer_limited_b300 as B
    B.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = ATTN[name]
    T, H, nq, nkv, D = cfg["T"], 5120, 48, 8, 128
    d = S.attn_inputs(T, H, nq, nkv, cfg["seed"] + 1000 * rank, dev)
    p = B.make_attn_params(T, H, nq, nkv, D, cfg["window"], 10000.0, 1e-6, cfg["k"],
                           B.FLAG_PRE_NORM)
    ws = torch.empty(B.attention_workspace_size(p), dtype=torch.uint8, device=dev)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def step():
        B.attention_forward(p, d["x"], d["w_qkvg"], d["w_o"], d["q_gain"], d["k_gain"], out=out,
                            workspace=ws)

    for _ in range(max(args.warmup, 3)):
        step()
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    steps = max(1, args.steps // 2)
    ms, prof, clk, _ = timed_steps(B, step, steps, torch.cuda.current_stream(dev),
                                   lambda: torch.cuda.synchronize(dev), local_rank)
    ms /= steps
    w = cfg["window"]
    pairs = sum(min(i + 1, w) for i in range(T)) if w else T * (T + 1) // 2
    attn_flops = 4.0 * nq * D * pairs                        # Q K^T and P V over visible pairs
    proj_flops = 2.0 * T * H * (2 * nq + 2 * nkv) * D + 2.0 * T * nq * D * H
    peaks = _peaks()
    k_ms = {k: v[0] / v[1] for k, v in prof.items()}
    top = "flash_attn" if k_ms.get("flash_attn", 0) > k_ms.get("attn_qkvg_proj", 0) else "attn_qkvg_proj"
    top_flops = attn_flops if top == "flash_attn" else 2.0 * T * H * (2 * nq + 2 * nkv) * D
    ach = top_flops / (k_ms[top] / 1e3) / 1e12
    return {"workload": f"attention sublayer, one sequence of T={T}, hidden {H}, {nq}/{nkv} heads x "
                        f"{D}, {'sliding window ' + str(w) + ' + RoPE' if w else 'global + query scale'}, "
                        f"pre-norm, post-norm, residual k={cfg['k']}",
            "value": round(T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
            "layer_tflops": round((attn_flops + proj_flops) / (ms / 1e3) / 1e12, 1),
            "roofline": {"kernel": top, "bound": "tensor", "achieved": round(ach, 1),
                         "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                         "frac": round(ach / peaks["bf16_sustained"], 4),
                         "frac_of_burst": round(ach / peaks["bf16"], 4),
                         "algorithmic_flops_per_launch": top_flops, "launch_ms": round(k_ms[top], 4),
                         "peak_source": peaks["source"] + " bf16_tflops_sustained"},
            "kernels_ms": {k: round(v, 4) for k, v in sorted(k_ms.items(), key=lambda kv: -kv[1])},
            "clocks": clk}


# ---------------------------------------------------------- oracle arm
def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def oracle_sample(wl, n_tokens, device):
    """Stage the oracle (as it stands) on the first n_tokens of the batch and
    return a callable that runs it once: pre-norm, routing, experts, combine,
    post-norm and residual. Expert weights are copied to host memory here,
    before any clock starts."""
    import oracle as O
    d = S.make_inputs(wl, device)
    x = d["x"][:n_tokens].float().cpu().numpy()
    wr = d["w_router"].float().cpu().numpy()
    bias = None if d["bias"] is None else d["bias"].float().cpu().numpy()
    xn = O.bf16_round(O.rms_norm(x.astype(np.float64), None, wl.rms_eps)).astype(np.float64)
    sel = O.route(xn, wr, bias, wl.n_group, wl.topk_group, wl.top_k, wl.routed_scale)
    weights = {int(e): tuple(d[k][int(e)].float().cpu().numpy()
                             for k in ("w_gate", "w_up", "w_down"))
               for e in np.unique(sel["idx"])}
    del d

    def run():
        O.moe_forward(x, wr, bias, lambda e: weights[e], n_group=wl.n_group,
                      topk_group=wl.topk_group, top_k=wl.top_k, scale=wl.routed_scale,
                      eps=wl.rms_eps, pre_norm=True, residual_k=RESIDUAL_K)
    return run, len(weights)


def time_oracle(run, n_tok, min_s=10.0, max_runs=20):
    """Repeat the staged oracle sample until it has taken at least min_s
    seconds of CPU work (at least once, at most max_runs times). Returns
    (tokens/s, runs, seconds)."""
    runs, t0 = 0, time.perf_counter()
    while True:
        run()
        runs += 1
        dt = time.perf_counter() - t0
        if dt >= min_s or runs >= max_runs:
            return n_tok * runs / dt, runs, dt


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, each step a bounded sample (2
    tokens) of the same workload, on the host cores of rank 0 only."""
    if rank != 0:
        return None
    wl = _workload(args.config)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    n_tok = 2
    run, ne = oracle_sample(wl, n_tok, dev)
    for _ in range(min(args.warmup, 1)):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    total = time.perf_counter() - t0
    value = n_tok * args.steps / total
    sample = (f"{n_tok} tokens of the {wl.name} batch per step (full sublayer path: pre-norm, "
              f"routing, {wl.top_k} experts each ({ne} distinct), combine, post-norm, "
              f"residual); weights staged on host before timing")
    return dict(value=value, ms_step=1e3 * total / args.steps, cores=_blas_threads(),
                sample=sample)


# ------------------------------------------------------------ ncu cases
def run_ncu_case(kind, experts="bf16"):
    """A small case for profiler captures: the full layer path with the real
    H=5120 / I=2560 shapes but 32 experts (one group, plain top-8), so the
    expert weights take 2.5 GB -- more than the L2, little device memory.
    kind 'decode': T=64 (16 tokens/expert, token tile 32);
    kind 'prefill': T=2048 (512 tokens/expert, token tile 128).
    Runs four forward calls (pre-norm + residual k=50) and exits; with
    experts fp8 / nvfp4 the expert weights are quantised first."""
    import sparse_moe_transformer_limited_b300 as B
    T = 64 if kind == "decode" else 2048
    wl = S.Workload("ncu_" + kind, T=T, E=32, n_group=1, topk_group=1, seed=7)
    d = S.make_inputs(wl, "cuda")
    fp8, f4 = experts == "fp8", experts == "nvfp4"
    flags = (B.FLAG_PRE_NORM | (B.FLAG_FP8_EXPERTS if fp8 else 0)
             | (B.FLAG_NVFP4_EXPERTS if f4 else 0))
    p = B.make_params(wl.T, wl.H, wl.E, wl.I, wl.n_group, wl.topk_group, wl.top_k,
                      wl.routed_scale, wl.rms_eps, RESIDUAL_K, flags)
    ws = B.alloc_workspace(p)
    out = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device="cuda")
    quant = B.quantize_e4m3_rows if fp8 else B.quantize_nvfp4
    q = tuple(quant(d[k]) for k in ("w_gate", "w_up", "w_down")) if (fp8 or f4) else None
    for _ in range(4):
        if fp8:
            B.forward_fp8(p, d["x"], d["w_router"], *q, out=out, workspace=ws)
        elif f4:
            B.forward_nvfp4(p, d["x"], d["w_router"], *q, out=out, workspace=ws)
        else:
            B.forward(p, d["x"], d["w_router"], d["w_gate"], d["w_up"], d["w_down"], out=out,
                      workspace=ws)
    if B.status() != 0:
        raise RuntimeError(B.last_error())
    print(f"ncu case {kind}: ok")


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="decode",
                    choices=sorted(S.WORKLOADS) + sorted(DENSE) + sorted(ATTN))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--experts", default="bf16", choices=["bf16", "fp8", "nvfp4"],
                    help="expert weight type of the timed sublayer (fp8: E4M3 + row scales; "
                         "nvfp4: E2M1 + E4M3 block scales + FP32 matrix scales)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the secondary T=8192 measurement")
    ap.add_argument("--ncu-case", choices=["decode", "prefill"],
                    help="run the small profiler case and exit")
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args.ncu_case, args.experts)
        return

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if world > 1 and args.impl == "ours":
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    if args.config in DENSE or args.config in ATTN:
        fn = run_dense if args.config in DENSE else run_attn
        r = fn(args, rank, world, local_rank, args.config)
        if rank == 0:
            print(json.dumps(dict(metric=METRIC, n_gpus=world, steps=args.steps, **r)), flush=True)
        return
    wl = _workload(args.config)
    if args.impl == "reference":
        r = run_reference(args, rank, world)
        if r is None:
            return
        line = {"impl": "reference", "metric": METRIC, "value": round(r["value"], 4),
                "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(r["ms_step"], 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": _config(wl, world),
                "cpu_baseline": {"value": round(r["value"], 4), "unit": "tokens/s",
                                 "cores": r["cores"], "kind": "oracle", "sample": r["sample"]},
                "e2e": {"value": round(r["value"], 4), "unit": "tokens/s",
                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    kind = args.experts
    r = run_ours(args, rank, world, local_rank, kind)
    extra = {}
    if rank == 0 and world == 1 and args.config == "decode" and not args.no_prefill:
        a2 = argparse.Namespace(**vars(args))
        a2.config = "prefill"

        def summary(rr):
            """A secondary workload's line: value, step time, e2e, roofline of
            its dominant kernel, layer fractions and clocks (the per-kernel
            split of the secondaries is left out to keep the line short)."""
            ro = rr["roofline"]
            keep = ("bound", "achieved", "peak", "unit", "frac", "frac_of_burst", "traffic",
                    "launch_ms", "dtype", "other_bound")
            return {"value": round(rr["value"], 1), "unit": "tokens/s",
                    "ms_per_step": round(rr["ms_step"], 4), "e2e": round(rr["e2e"], 1),
                    "roofline": {k: ro[k] for k in keep if k in ro},
                    "layer": {k: rr["layer"][k] for k in ("hbm_frac", "tensor_frac",
                                                          "tensor_frac_of_burst")},
                    "clocks": None if rr["clocks"] is None else
                    {k: rr["clocks"][k] for k in ("sm_mhz", "reasons")}}
        # the BF16 T = 8192 line is measured right after the headline and
        # printed last, where a reader keeping the end of the line sees it
        torch.cuda.empty_cache()
        rp = run_ours(a2, rank, world, local_rank)
        prefill = summary(rp)
        prefill["kernels_ms"] = dict(list(rp["kernels_ms"].items())[:4])
        torch.cuda.empty_cache()
        extra["dense_mlp_T8192"] = run_dense(a2, rank, world, local_rank, "dense_prefill")
        # the skewed-routing and long-prefill-with-residual workloads
        for cfg, key in (("skew", "skew_T4096"), ("long_prefill", "long_prefill_T16384")):
            a4 = argparse.Namespace(**vars(args))
            a4.config = cfg
            torch.cuda.empty_cache()
            extra[key] = summary(run_ours(a4, rank, world, local_rank))
        for an in ("attn_swa", "attn_global"):
            torch.cuda.empty_cache()
            extra[f"attention_{an[5:]}_T8192"] = run_attn(a2, rank, world, local_rank, an)
        if kind == "bf16":
            # the same sublayers with E4M3 and NVFP4 expert weights (secondary lines)
            a3 = argparse.Namespace(**vars(args))
            for k2 in ("fp8", "nvfp4"):
                torch.cuda.empty_cache()
                extra[f"{k2}_experts_T64"] = summary(run_ours(a3, rank, world, local_rank, k2))
                torch.cuda.empty_cache()
                extra[f"{k2}_experts_T8192"] = summary(run_ours(a2, rank, world, local_rank, k2))
            torch.cuda.empty_cache()
        extra["prefill_T8192"] = prefill
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        torch.cuda.empty_cache()
        n_tok = 4
        run, ne = oracle_sample(wl, n_tok, "cuda")
        v, runs, dt = time_oracle(run, n_tok)
        cpu = {"value": round(v, 4), "unit": "tokens/s", "cores": _blas_threads(),
               "kind": "oracle",
               "sample": f"{n_tok} tokens of the {wl.name} batch (full sublayer path, {ne} "
                         f"experts), run {runs} times: {dt:.1f} s of CPU work; weights staged "
                         f"on host before timing"}
    if rank != 0:
        return
    line = {"metric": METRIC, "value": round(r["value"], 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(r["ms_step"], 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"bf16": "bf16", "fp8": "e4m3", "nvfp4": "nvfp4"}[kind],
            "data": "synthetic",
            "config": _config(wl, world),
            "roofline": r["roofline"], "layer": r["layer"], "kernels_ms": r["kernels_ms"],
            "clocks": r["clocks"],
            "e2e": {"value": round(r["e2e"], 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": r["launches"],
            "cpu_baseline": cpu}
    line.update(extra)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
