"""The C-ABI library loads without a GPU, exports every symbol the public
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

import sparse_moe_transformer_limited_b300 as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_moe.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(beam_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    names = _declared()
    assert "beam_moe_forward" in names and len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.EXPORTED)


def test_params_struct_matches_header():
    src = open(HEADER).read()
    body = re.search(r"typedef struct \{(.*?)\} beam_moe_params;", src, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b([A-Za-z_][A-Za-z_0-9]*)\s*[,;]", body)
    assert fields == [f for f, _ in B.Params._fields_]


def test_dense_params_struct_matches_header():
    src = open(HEADER).read()
    body = re.search(r"typedef struct \{([^{}]*)\} beam_dense_params;", src).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b([A-Za-z_][A-Za-z_0-9]*)\s*[,;]", body)
    assert fields == [f for f, _ in B.DenseParams._fields_]


@pytest.mark.parametrize("T,H,I,k,flags,code", [
    (8, 5120, 2500, 0, 0, 2), (8, 5000, 2560, 0, 0, 2), (8, 5120, 2560, 1, 0, 1),
    (8, 5120, 2560, 50, 2, 1), (-1, 5120, 2560, 0, 0, 1), (8, 5120, 2560, 0, 4, 1),
])
def test_dense_invalid_params_rejected(T, H, I, k, flags, code):
    p = B.DenseParams(T, H, I, 1e-6, k, flags)
    assert B.lib().beam_dense_workspace_size(ctypes.byref(p)) == 0
    r = B.lib().beam_dense_mlp_forward(ctypes.byref(p), *([None] * 8), 0, None)
    assert r == code, B.last_error()


def _p(**kw):
    base = dict(T=64, H=5120, E=256, I=2560)
    base.update(kw)
    return B.make_params(**base)


def test_workspace_size_and_layout():
    p = _p()
    n = B.workspace_size(p)
    lay = B.workspace_layout(p)
    assert list(lay) == list(B._native.LAYOUT_NAMES)
    offs = list(lay.values())
    assert offs == sorted(offs) and offs[-1] <= n
    assert all(o % 1024 == 0 for o in offs)
    # the permuted copy of x and the SwiGLU buffer are sized for T*top_k rows
    assert lay["act"] - lay["xperm"] >= 64 * 8 * 5120 * 2
    big = B.workspace_size(_p(T=16384, flags=B.FLAG_PRE_NORM, residual_k=50))
    assert big > 16384 * 8 * (5120 + 2560) * 2


@pytest.mark.parametrize("kw,code", [
    (dict(residual_k=1), 1), (dict(residual_k=-3), 1), (dict(E=48, n_group=8), 2),
    (dict(H=5000), 2), (dict(I=2500), 2), (dict(top_k=0), 1), (dict(top_k=33), 1),
    (dict(topk_group=9), 1), (dict(n_group=3), 1), (dict(E=256, n_group=16), 2),
    (dict(routed_scale=-1.0), 1), (dict(flags=64), 1),
    (dict(flags=B.FLAG_FP32_OUT, residual_k=50), 1), (dict(T=-1), 1),
])
def test_invalid_params_rejected(kw, code):
    p = _p(**kw)
    assert B.lib().beam_moe_workspace_size(ctypes.byref(p)) == 0
    r = B.lib().beam_moe_forward(ctypes.byref(p), *([None] * 12), 0, None)
    assert r == code, B.last_error()
    assert B.last_error()


def test_null_pointers_rejected():
    p = _p()
    r = B.lib().beam_moe_forward(ctypes.byref(p), *([None] * 12), 0, None)
    assert r == 1
    r = B.lib().beam_moe_route(ctypes.byref(p), *([None] * 8), 0, None)
    assert r == 1


def test_route_static_host_checks():
    """The allocation-free router checks its arguments and its scratch size
    on the host and returns before any CUDA call: bad sizes, NULL pointers,
    misaligned x, and a batch whose scratch exceeds the fixed array
    (T = 16384 with pre-norm needs far more than 8 MiB). Addresses here are
    never dereferenced: every call fails before it would launch."""
    lib = B.lib()
    fake = ctypes.c_void_p(1 << 20)                 # 16-byte aligned, never read
    args = lambda x: (x, fake, None, None, fake, fake, None, None)
    assert lib.beam_moe_route_static(ctypes.byref(_p(top_k=0)), *args(fake)) == 1
    assert lib.beam_moe_route_static(ctypes.byref(_p(H=5000)), *args(fake)) == 2
    assert lib.beam_moe_route_static(ctypes.byref(_p()), *args(None)) == 1
    assert lib.beam_moe_route_static(ctypes.byref(_p()), *args(ctypes.c_void_p((1 << 20) + 8))) == 1
    assert "16-byte aligned" in B.last_error()
    p = _p(flags=B.FLAG_RETURN_SCORES)
    assert lib.beam_moe_route_static(ctypes.byref(p), *args(fake)) == 1     # no scores buffer
    big = _p(T=16384, flags=B.FLAG_PRE_NORM)
    assert lib.beam_moe_route_static(ctypes.byref(big), *args(fake)) == 2
    assert "static scratch holds 8388608 bytes" in B.last_error()
    assert lib.beam_moe_route_static(ctypes.byref(_p(T=0)), *args(None)) == 0


def test_residual_step_args_rejected():
    lib = B.lib()
    assert lib.beam_residual_step(None, None, 4, 5120, 1, None, 1e-6, 1, 0, None, None) == 1
    assert lib.beam_residual_step(None, None, 4, 5121, 2, None, 1e-6, 1, 0, None, None) == 1
    assert lib.beam_residual_step(None, None, 4, 5120, 2, None, 1e-6, 1, 0, None, None) == 1


def test_empty_batch_is_a_no_op():
    p = _p(T=0)
    assert B.lib().beam_moe_forward(ctypes.byref(p), *([None] * 12), 0, None) == 0


@pytest.mark.parametrize("flags", [0, B.FLAG_PRE_NORM, B.FLAG_FP8_EXPERTS, B.FLAG_NVFP4_EXPERTS,
                                   B.FLAG_RETURN_SCORES])
def test_empty_batch_workspace_queries(flags):
    """Sizing a workspace for T = 0 (a rank without tokens, say) returns a
    size and a layout; routing an empty batch is a no-op."""
    p = _p(T=0, flags=flags)
    assert B.workspace_size(p) > 0
    assert len(B.workspace_layout(p)) > 0
    assert B.lib().beam_moe_route(ctypes.byref(p), *([None] * 8), ctypes.c_size_t(0), None) == 0


def test_fp8_workspace_holds_e4m3_buffers():
    plain = B.workspace_layout(_p())
    f8 = B.workspace_layout(_p(flags=B.FLAG_FP8_EXPERTS))
    assert plain["act_q"] == plain["act_scale"]          # absent without the flag
    assert f8["act_scale"] - f8["act_q"] >= 64 * 8 * 2560  # one code per activation
    assert f8["act_q"] - f8["x_scale"] >= 64 * 8 * 4       # one scale per pair row
    assert B.workspace_size(_p(flags=B.FLAG_FP8_EXPERTS)) > B.workspace_size(_p())


def test_fp8_entry_points_reject_bad_args():
    lib = B.lib()
    p = _p()                                   # FLAG_FP8_EXPERTS missing
    assert lib.beam_moe_forward_fp8(ctypes.byref(p), *([None] * 15), 0, None) == 1
    assert "FP8_EXPERTS" in B.last_error()
    p = _p(flags=B.FLAG_FP8_EXPERTS)           # pointers missing
    assert lib.beam_moe_forward_fp8(ctypes.byref(p), *([None] * 15), 0, None) == 1
    p = _p(T=0, flags=B.FLAG_FP8_EXPERTS)
    assert lib.beam_moe_forward_fp8(ctypes.byref(p), *([None] * 15), 0, None) == 0
    d = B.DenseParams(8, 5120, 2560, 1e-6, 0, 0)
    assert lib.beam_dense_mlp_forward_fp8(ctypes.byref(d), *([None] * 11), 0, None) == 1
    # the quantiser wants K a positive multiple of 16 and rows >= 0
    assert lib.beam_quantize_e4m3_rows(None, 4, 10, None, None, None) == 1
    assert lib.beam_quantize_e4m3_rows(None, -1, 16, None, None, None) == 1
    assert lib.beam_quantize_e4m3_rows(None, 0, 16, None, None, None) == 0
    assert lib.beam_quantize_e4m3_rows(None, 4, 16, None, None, None) == 1


def test_nvfp4_entry_points_reject_bad_args():
    lib = B.lib()
    p = _p()                                   # FLAG_NVFP4_EXPERTS missing
    assert lib.beam_moe_forward_nvfp4(ctypes.byref(p), *([None] * 18), 0, None) == 1
    p = _p(flags=B.FLAG_NVFP4_EXPERTS | B.FLAG_FP8_EXPERTS)
    assert B.lib().beam_moe_workspace_size(ctypes.byref(p)) == 0
    p = _p(I=2560 + 128, flags=B.FLAG_NVFP4_EXPERTS)   # I % 256 != 0
    assert lib.beam_moe_forward_nvfp4(ctypes.byref(p), *([None] * 18), 0, None) == 2
    p = _p(T=0, flags=B.FLAG_NVFP4_EXPERTS)
    assert lib.beam_moe_forward_nvfp4(ctypes.byref(p), *([None] * 18), 0, None) == 0
    # the quantiser wants rows a multiple of 128 and of rows_per_group, K of 64
    assert lib.beam_quantize_nvfp4(None, 100, 64, 1, None, None, None, None) == 1
    assert lib.beam_quantize_nvfp4(None, 128, 48, 1, None, None, None, None) == 1
    assert lib.beam_quantize_nvfp4(None, 256, 64, 100, None, None, None, None) == 1
    assert lib.beam_quantize_nvfp4(None, 0, 64, 1, None, None, None, None) == 0


def test_nvfp4_workspace_pads_expert_rows():
    f4 = B.workspace_layout(_p(flags=B.FLAG_NVFP4_EXPERTS))
    plain = B.workspace_layout(_p())
    # T=64, top-8: up to 256 experts each padded to 32 rows -> far more rows
    assert f4["act"] - f4["xperm"] > plain["act"] - plain["xperm"]
    assert f4["act_sf"] > f4["x_sf"] > f4["act_scale"]


def test_attn_params_struct_matches_header():
    src = open(HEADER).read()
    body = re.search(r"typedef struct \{([^{}]*)\} beam_attn_params;", src).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = re.findall(r"\b([A-Za-z_][A-Za-z_0-9]*)\s*[,;]", body)
    assert fields == [f for f, _ in B.AttnParams._fields_]


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), 2), (dict(H=5000), 2), (dict(n_q=48, n_kv=5), 2), (dict(n_q=7, n_kv=2), 2),
    (dict(window=-1), 1), (dict(residual_k=1), 1), (dict(flags=64), 1),
    (dict(flags=2, residual_k=50), 1), (dict(T=-1), 1),
])
def test_attn_invalid_params_rejected(kw, code):
    base = dict(T=64)
    base.update(kw)
    p = B.make_attn_params(**base)
    assert B.lib().beam_attention_workspace_size(ctypes.byref(p)) == 0
    assert B.lib().beam_attention_forward(ctypes.byref(p), *([None] * 9), 0, None) == code


def test_attn_workspace_and_empty_sequence():
    assert B.attention_workspace_size(B.make_attn_params(T=8192)) > 8192 * 14336 * 4
    p = B.make_attn_params(T=0)
    assert B.lib().beam_attention_forward(ctypes.byref(p), *([None] * 9), 0, None) == 0


def test_header_is_plain_c_and_links(tmp_path):
    """include/beam_moe.h compiles as pedantic C99, and a C program links
    against the library and runs a host-only entry point (argument checks;
    no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    import sparse_moe_transformer_limited_b300 as pkg
    from sparse_moe_transformer_limited_b300 import _native
    lib = _native.LIB_PATH
    if not os.path.exists(lib):
        pytest.skip("library not built")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = tmp_path / "abi.c"
    src.write_text(
        '#include "beam_moe.h"\n'
        '#include <stdio.h>\n'
        'int main(void) {\n'
        '  beam_moe_params p = {0};\n'
        '  /* T = 64 but H = 0: rejected on the host */\n'
        '  p.T = 64; p.E = 256; p.I = 2560;\n'
        '  beam_status_t s = beam_moe_route(&p, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0);\n'
        '  printf("%d %s\\n", (int)s, beam_last_error_string());\n'
        '  return s == BEAM_ERR_INVALID_ARG ? 0 : 1;\n'
        '}\n')
    exe = tmp_path / "abi"
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
           "-I", os.path.join(root, "include"), str(src), "-o", str(exe),
           lib, "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("1 ")


def _list_bytes(lay):
    """Sizes of the gate/up and down work lists (entries are 1 KB aligned)."""
    return lay["units_dn"] - lay["units_gu"], lay["pair_row"] - lay["units_dn"]


def _kb(nbytes):
    return (nbytes + 1023) // 1024 * 1024


@pytest.mark.parametrize("flags,T,want_gu,want_dn", [
    # decode, 512 pairs <= 24 per expert: weight-major token tiles of 32;
    # one list of (512/32 + E) tiles, expanded by the I/128 gate/up and H/128
    # down weight tiles
    (0, 64, 16 * (16 + 256) * 20, 16 * (16 + 256) * 40),
    # prefill BF16: wide 2-SM units, at most 65536/256 + E token groups, one
    # unit per group and weight slice (I/256 gate/up, H/512 down slices)
    (0, 8192, 16 * 512 * 10, 16 * 512 * 10),
    ("fp8", 8192, 16 * 512 * 10, 16 * 512 * 10),
    # the weight-major flag: 128-token tiles for both GEMMs
    ("wm", 8192, 16 * (512 + 256) * 20, 16 * (512 + 256) * 40),
    # prefill NVFP4: both GEMMs on the token-major cluster kernel
    ("nvfp4", 8192, 16 * 2 * (512 * 20 + 256 * 11), 16 * 2 * (512 * 20 + 256 * 11)),
    # NVFP4 with the weight-major flag: 128-token tiles
    ("nvfp4+wm", 8192, 16 * (512 + 256) * 20, 16 * (512 + 256) * 40),
])
def test_gemm_regime_follows_tokens_and_flag(flags, T, want_gu, want_dn):
    """The expert-GEMM regime is chosen on the host from tokens per expert,
    the expert weight type and BEAM_FLAG_PREFILL_WEIGHT_MAJOR; each regime's
    work-list format fixes the size of its workspace entries (read here
    without a GPU)."""
    f = 0
    if flags and "nvfp4" in flags:
        f |= B.FLAG_NVFP4_EXPERTS
    if flags and "fp8" in flags:
        f |= B.FLAG_FP8_EXPERTS
    if flags and "wm" in flags:
        f |= B.FLAG_PREFILL_WEIGHT_MAJOR
    gu, dn = _list_bytes(B.workspace_layout(_p(T=T, flags=f)))
    assert (gu, dn) == (_kb(want_gu), _kb(want_dn))


def test_combined_output_buffer_is_per_token():
    """The down projection adds into one FP32 row per token (no per-pair
    expert outputs), followed by one arrival counter per token."""
    for T in (64, 8192):
        lay = B.workspace_layout(_p(T=T))
        assert lay["n_units"] - lay["oacc"] == _kb(T * 5120 * 4)
        n = B.workspace_size(_p(T=T))
        assert n - lay["arrive"] >= T * 4


def test_expert_parallel_entry_points_check_args_on_host():
    """The expert-parallel entry points reject bad arguments before any CUDA
    call (no GPU here): a rank count that does not divide E, NULL or
    misaligned pointers, quantised-expert flags on the routed forward, a
    residual step of 1 or an FP32 output with the residual in the combine.
    Empty batches are no-ops."""
    lib = B.lib()
    fake = ctypes.c_void_p(1 << 20)                 # 16-byte aligned, never read
    p = ctypes.byref(_p())
    assert lib.beam_ep_dispatch(p, 3, *([fake] * 7), 1 << 30, None) == 1
    assert "must divide" in B.last_error()
    assert lib.beam_ep_dispatch(p, 8, None, *([fake] * 6), 1 << 30, None) == 1
    assert lib.beam_ep_dispatch(p, 8, ctypes.c_void_p((1 << 20) + 4), *([fake] * 6), 1 << 30,
                                None) == 1
    assert lib.beam_ep_dispatch(ctypes.byref(_p(T=0)), 8, *([None] * 7), 0, None) == 0
    routed = lambda q, x: lib.beam_moe_forward_routed(q, x, *([fake] * 9), 1 << 30, None)
    assert routed(ctypes.byref(_p(flags=B.FLAG_FP8_EXPERTS)), fake) == 2
    assert routed(p, None) == 1
    assert routed(ctypes.byref(_p(T=0)), None) == 0
    comb = lambda T, k, H, rk, f32: lib.beam_ep_combine(T, k, H, fake, fake, fake, fake, None,
                                                        1e-6, rk, f32, fake, None)
    assert comb(4, 8, 5120, 1, 0) == 1
    assert comb(4, 8, 5120, 50, 1) == 1
    assert comb(4, 33, 5120, 0, 0) == 1
    assert comb(4, 8, 5000, 0, 0) == 2
    assert comb(0, 8, 5120, 50, 0) == 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every entry point raises; nothing falls back
    to another implementation."""
    from sparse_moe_transformer_limited_b300 import _native
    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "libbeam_moe.so"))
    with pytest.raises(ImportError, match="is missing"):
        _native.lib()
    with pytest.raises(ImportError):
        _native.workspace_size(_p())
    import torch
    x = torch.zeros((4, 256), dtype=torch.bfloat16)
    with pytest.raises(ImportError):
        _native.route(_p(T=4, H=256), x, torch.zeros((256, 256)))


def test_empty_batch_every_entry_point():
    """T = 0 (or zero rows) returns BEAM_OK from every compute entry point
    with NULL buffers: nothing is enqueued."""
    lib = B.lib()
    n0 = ctypes.c_size_t(0)
    L0 = ctypes.c_longlong(0)
    f8 = _p(T=0, flags=B.FLAG_FP8_EXPERTS)
    f4 = _p(T=0, flags=B.FLAG_NVFP4_EXPERTS)
    dense = B.DenseParams(0, 5120, 12288, 1e-6, 3, 0)
    dense8 = B.DenseParams(0, 5120, 12288, 1e-6, 3, B.FLAG_FP8_EXPERTS)
    dense4 = B.DenseParams(0, 5120, 12288, 1e-6, 3, B.FLAG_NVFP4_EXPERTS)
    attn = B.make_attn_params(T=0)
    calls = {
        "route": lib.beam_moe_route(ctypes.byref(_p(T=0)), *([None] * 8), n0, None),
        "forward": lib.beam_moe_forward(ctypes.byref(_p(T=0)), *([None] * 12), n0, None),
        "forward_fp8": lib.beam_moe_forward_fp8(ctypes.byref(f8), *([None] * 15), n0, None),
        "forward_nvfp4": lib.beam_moe_forward_nvfp4(ctypes.byref(f4), *([None] * 18), n0, None),
        "dense": lib.beam_dense_mlp_forward(ctypes.byref(dense), *([None] * 8), n0, None),
        "dense_fp8": lib.beam_dense_mlp_forward_fp8(ctypes.byref(dense8), *([None] * 11), n0, None),
        "dense_nvfp4": lib.beam_dense_mlp_forward_nvfp4(ctypes.byref(dense4), *([None] * 14), n0,
                                                        None),
        "attention": lib.beam_attention_forward(ctypes.byref(attn), *([None] * 9), n0, None),
        "quantize_e4m3": lib.beam_quantize_e4m3_rows(None, L0, 5120, None, None, None),
        "quantize_nvfp4": lib.beam_quantize_nvfp4(None, L0, 5120, 128, None, None, None, None),
        "residual": lib.beam_residual_step(None, None, 0, 5120, 2, None, ctypes.c_float(1e-6), 1,
                                           0, None, None),
        "ep_combine": lib.beam_ep_combine(0, 8, 5120, None, None, None, None, None,
                                          ctypes.c_float(1e-6), 9, 0, None, None),
    }
    assert all(v == 0 for v in calls.values()), calls
