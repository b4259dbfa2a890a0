"""The C-ABI library builds, loads and exports every symbol its header
declares; the Python binding passes arguments with the header's types; host
argument checks reject bad calls before anything reaches a GPU.  CPU only."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")

import nvfp4_precision_moe_gb300 as nv  # noqa: E402
from nvfp4_precision_moe_gb300.build import build_library  # noqa: E402

OK, INVALID, UNSUP, ALIGN, ARCH = 0, 1, 2, 3, 7


def _decls():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(int|const char \*)\s*(nvfp4_\w+)\s*\(([^)]*)\)\s*;", txt):
        args = [a.strip() for a in m.group(3).split(",") if a.strip() and a.strip() != "void"]
        sig = ""
        for a in args:
            if "*" in a:
                sig += "p"
            elif a.startswith("int64_t"):
                sig += "q"
            elif a.startswith("int32_t") or a.startswith("int "):
                sig += "i"
            else:
                raise AssertionError("unknown argument type: " + a)
        out[m.group(2)] = (m.group(1), sig)
    return out


@pytest.fixture(scope="module")
def lib():
    build_library()
    return nv.load()


def test_header_declares_the_boundary():
    d = _decls()
    for name in ["nvfp4_quantize", "nvfp4_amax", "nvfp4_fake_quant", "nvfp4_prepare_weights",
                 "nvfp4_w4a4_rac_grouped_gemm", "nvfp4_bf16_grouped_gemm", "nvfp4_route_topk",
                 "nvfp4_moe_combine", "nvfp4_rac_select_channels", "nvfp4_status_str"]:
        assert name in d


def test_library_exports_every_declared_symbol(lib):
    for name in _decls():
        assert hasattr(lib, name), name


def test_binding_signatures_match_header(lib):
    d = _decls()
    for name, (ret, sig) in d.items():
        if ret != "int":
            continue
        assert nv._SIGS.get(name) == sig, (name, nv._SIGS.get(name), sig)


def test_status_strings(lib):
    for code, name in nv.STATUS.items():
        assert lib.nvfp4_status_str(code).decode() == name


# a fake, 16-byte aligned "device" address: the host checks never dereference it
P = 0x10000
PM = 0x10008  # misaligned


def test_host_checks_without_gpu(lib):
    q = lib.nvfp4_quantize
    # x, M, K, ldx, amax, gs, S, k, dst, fanout, rows_out, codes, scales, resid, row_limit, status, stream
    assert q(None, 4, 64, 64, P, None, None, 0, None, 1, 4, P, P, None, None, None, None) == INVALID
    assert q(P, 4, 48, 48, P, None, None, 0, None, 1, 4, P, P, None, None, None, None) == UNSUP  # K % 32
    assert q(PM, 4, 64, 64, P, None, None, 0, None, 1, 4, P, P, None, None, None, None) == ALIGN
    assert q(P, 4, 64, 64, P, None, P, 8, None, 1, 4, P, P, None, None, None, None) == INVALID  # k>0, no resid
    assert q(P, 4, 64, 64, P, None, None, 0, None, 2, 4, P, P, None, None, None, None) == INVALID  # fanout w/o map
    # a row's destinations live in 32 per-warp slots: more than 32 is refused before any launch
    assert q(P, 4, 64, 64, P, None, None, 0, P, 33, 4 * 33, P, P, None, None, None, None) == UNSUP
    fq = lib.nvfp4_fake_quant_noalloc
    # w, ntensors, rows, cols, w_hat, gs_out, dev_status, stream
    assert fq(P, 2, 16, 48, P, None, None, None) == UNSUP  # cols % 32
    assert fq(P, 4097, 16, 64, P, None, None, None) == UNSUP  # beyond its 4096-slot array
    assert b"4096" in lib.nvfp4_last_error()
    assert fq(PM, 2, 16, 64, P, None, None, None) == ALIGN
    g = lib.nvfp4_w4a4_rac_grouped_gemm
    args = [P, P, None, P, P, P, P, None, 0, P, 1, 128, 256, 256, 0, 0, P, 256, None, None, None]
    bad_k = list(args)
    bad_k[13] = 192  # K % 256
    assert g(*bad_k) == UNSUP
    bad_n = list(args)
    bad_n[12] = 128  # N % 256
    assert g(*bad_n) == UNSUP
    swiglu_f32 = list(args)
    swiglu_f32[14] = 1  # SwiGLU needs BF16 output
    assert g(*swiglu_f32) == INVALID
    mis = list(args)
    mis[16] = PM
    assert g(*mis) == ALIGN
    # a valid call reaches the device check: there is no CPU path
    import torch
    if not torch.cuda.is_available():
        assert g(*args) == ARCH
        assert lib.nvfp4_init() == ARCH
    r = lib.nvfp4_route_topk
    assert r(P, 16, 8, 9, P, P, P, P, P, None) == UNSUP  # topk > E
    c = lib.nvfp4_moe_combine
    assert c(P, 3, 64, P, P, 4, 2, 64, P, None) == INVALID  # bad dtype


def test_host_checks_of_the_trainer_and_online_entry_points(lib):
    d = lib.nvfp4_bf16_grouped_gemm_dgrad
    # dy, w_hat, offsets, E, rows_cap, N, K, out_dtype, epilogue, gu, y, ldy, dev_status, stream
    args = [P, P, P, 2, 256, 256, 128, 1, 0, None, P, 256, None, None]
    bad = list(args)
    bad[6] = 96  # K % 64
    assert d(*bad) == UNSUP
    bad = list(args)
    bad[5] = 128  # N % 256
    assert d(*bad) == UNSUP
    bad = list(args)
    bad[8] = 2  # the SwiGLU backward needs the saved pre-activations
    assert d(*bad) == INVALID
    bad = list(args)
    bad[8], bad[9], bad[7], bad[11] = 2, P, 0, 512  # ... and BF16 output
    assert d(*bad) == INVALID
    bad = list(args)
    bad[8], bad[9], bad[11] = 2, P, 256  # ... and a row of 2N
    assert d(*bad) == INVALID
    bad = list(args)
    bad[8] = 1  # the forward SwiGLU is not an input-gradient epilogue
    assert d(*bad) == INVALID
    bad = list(args)
    bad[1] = PM
    assert d(*bad) == ALIGN
    w = lib.nvfp4_bf16_grouped_gemm_wgrad_rows
    # a, b, offsets, E, R, M, N, out_dtype, dw, dev_status, stream
    assert w(P, P, P, 2, 256, 96, 256, 0, P, None, None) == UNSUP  # M % 128
    assert w(P, P, P, 2, 256, 128, 128, 0, P, None, None) == UNSUP  # N % 256
    assert w(P, P, P, 2, 200, 128, 256, 0, P, None, None) == UNSUP  # R % 128
    assert w(PM, P, P, 2, 256, 128, 256, 0, P, None, None) == ALIGN
    gw = lib.nvfp4_gather_selected_weights
    # w_codes, w_scales, E, N, K, S, k, w_sel, dev_status, stream
    assert gw(P, P, 2, 256, 96, P, 8, P, None, None) == UNSUP  # K % 64
    assert gw(P, P, 2, 200, 256, P, 8, P, None, None) == UNSUP  # N % 128
    assert gw(P, P, 2, 256, 256, P, 12, P, None, None) == UNSUP  # k % 8
    assert gw(P, P, 2, 256, 256, P, 300, P, None, None) == INVALID  # k > K
    cb = lib.nvfp4_moe_combine_backward
    # dout, y, dst_row, weights, T, topk, H, counts, offsets, E, rows_cap, dy, dweights, stream
    assert cb(P, P, P, P, 4, 33, 64, P, P, 2, 256, P, None, None) == UNSUP  # topk > 32


def test_empty_batch_buffers_may_be_null(lib):
    """A batch of no tokens passes the argument checks with NULL token-sized
    buffers (on a machine without an sm_103 device the call then stops at the
    architecture check; nothing is dereferenced)."""
    ok = (OK, ARCH)
    # x, M, K, ldx, ntensors, tensor_stride, amax_out, stream
    assert lib.nvfp4_amax(None, 0, 64, 64, 1, 0, P, None) in ok
    # x, M, K, ldx, amax, gs, S, k, dst, fanout, rows_out, codes, scales, resid, row_limit, status, stream
    assert lib.nvfp4_quantize(None, 0, 64, 64, P, None, P, 8, None, 8, 128, P, P, P, None, None, None) in ok
    # logits, T, E, topk, ids, weights, counts, offsets, dst_row, stream
    assert lib.nvfp4_route_topk(None, 0, 16, 4, None, None, P, P, None, None) in ok
    # y, y_dtype, ldy, dst_row, weights, T, topk, H, out, stream
    assert lib.nvfp4_moe_combine(P, 1, 64, None, None, 0, 4, 64, None, None) in ok
    # with tokens the same buffers are required
    assert lib.nvfp4_route_topk(None, 3, 16, 4, None, None, P, P, None, None) == INVALID
    assert lib.nvfp4_moe_combine(P, 1, 64, None, None, 3, 4, 64, None, None) == INVALID


def test_bf16_gemm_pre_activation_buffer(lib):
    b = lib.nvfp4_bf16_grouped_gemm
    # x, w_hat, offsets, E, rows_cap, N, K, out_dtype, epilogue, y, ldy, gu, status, stream
    assert b(P, P, P, 1, 128, 256, 64, 1, nv.NVFP4_EPI_SWIGLU_SAVE, P, 128, None, None, None) == INVALID  # no gu
    assert b(P, P, P, 1, 128, 256, 64, 1, nv.NVFP4_EPI_SWIGLU, P, 128, P, None, None) == INVALID  # gu unused
    assert b(P, P, P, 1, 128, 256, 64, 0, nv.NVFP4_EPI_SWIGLU_SAVE, P, 128, P, None, None) == INVALID  # F32 out
    assert b(P, P, P, 1, 128, 256, 64, 1, nv.NVFP4_EPI_SWIGLU_SAVE, P, 128, PM, None, None) == ALIGN


def test_gemm_pipeline_selector(lib):
    prev = ctypes.c_int32(-1)
    assert lib.nvfp4_gemm_pipeline(7, None) == INVALID
    assert lib.nvfp4_gemm_pipeline(nv.NVFP4_PIPELINE_PAIR, ctypes.byref(prev)) == OK
    assert prev.value == nv.NVFP4_PIPELINE_AUTO
    assert nv.nvfp4_gemm_pipeline(nv.NVFP4_PIPELINE_AUTO) == nv.NVFP4_PIPELINE_PAIR


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import importlib
    monkeypatch.setattr(nv, "_lib", None)
    monkeypatch.setattr(nv, "LIB", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError):
        nv.load()


def test_every_entry_point_cites_its_passage():
    """Each declaration's own comment names the passage that defines it (QUADS
    section / equation) or says that the paper has no counterpart."""
    import re

    h = open(HEADER).read()
    for m in re.finditer(r"\n(?:int|const char \*)\s+(nvfp4_\w+)\(", h):
        start, end = h.rfind("/*", 0, m.start()), h.rfind("*/", 0, m.start())
        comment = h[start:end]
        assert start >= 0 and end > start and (
            "QUADS" in comment or "no counterpart" in comment or "not described" in comment), m.group(1)
