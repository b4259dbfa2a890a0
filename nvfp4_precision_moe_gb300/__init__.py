"""Python binding of libnvfp4moe, the NVFP4 W4A4 + RAC MoE hot path for GB300.

Argument marshalling only: each function here has the name of a C entry point
of ``include/nvfp4moe.h``, takes torch tensors, passes their device pointers,
sizes and the current CUDA stream to that entry point, and raises
``NVFP4Error`` when it returns a non-zero status.  Every step of the path runs
in the library's CUDA kernels; there is no CPU path, and importing the
functions without the built library fails loudly.

"QUADS" is the paper "QUADS: Stabilizing NVFP4 Reinforcement Learning for MoE
via QUantization-error Alignment across Dual Sides"; the header cites, per
entry point, the section or equation it implements.
"""
import ctypes
import os

import torch

from .build import LIB, build_library

NVFP4_OUT_F32, NVFP4_OUT_BF16 = 0, 1
NVFP4_EPI_NONE, NVFP4_EPI_SWIGLU, NVFP4_EPI_SWIGLU_BWD, NVFP4_EPI_SWIGLU_SAVE = 0, 1, 2, 3
NVFP4_PIPELINE_AUTO, NVFP4_PIPELINE_SINGLE, NVFP4_PIPELINE_PAIR = 0, 1, 2
STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED",
          3: "NVFP4_ERR_ALIGNMENT", 4: "NVFP4_ERR_CUDA", 5: "NVFP4_ERR_TIMEOUT",
          6: "NVFP4_ERR_NONFINITE", 7: "NVFP4_ERR_ARCH"}

# entry point -> argument types (p = pointer, q = int64, i = int32)
_SIGS = {
    "nvfp4_init": "",
    "nvfp4_amax": "pqqqiqpp",
    "nvfp4_quantize": "pqqqpppipiqpppppp",
    "nvfp4_fake_quant": "piqqppppp",
    "nvfp4_fake_quant_noalloc": "piqqpppp",
    "nvfp4_fake_quant_transposed": "piqqpppppp",
    "nvfp4_prepare_weights": "piqqpiippppppp",
    "nvfp4_rac_select_channels": "pqqpippp",
    "nvfp4_rac_requant_residual": "pqipipppp",
    "nvfp4_rac_select_channels_online": "pqqpipippp",
    "nvfp4_gather_selected_weights": "ppiqqpippp",
    "nvfp4_transpose_weight_pack": "ppiqqppp",
    "nvfp4_gather_selected_weights_t": "ppiqqpipp",
    "nvfp4_transpose_bf16": "piqqpp",
    "nvfp4_swiglu": "pqqpp",
    "nvfp4_swiglu_backward": "ppqqpp",
    "nvfp4_moe_combine_backward": "ppppiiqppiqppp",
    "nvfp4_bf16_grouped_gemm_wgrad": "pppiqqqippp",
    "nvfp4_bf16_grouped_gemm_wgrad_rows": "pppiqqqippp",
    "nvfp4_bf16_grouped_gemm_dgrad": "pppiqqqiippqpp",
    "nvfp4_w4a4_rac_grouped_gemm": "ppppppppipiqqqiipqppp",
    "nvfp4_bf16_grouped_gemm": "pppiqqqiipqppp",
    "nvfp4_gemm_pipeline": "ip",
    "nvfp4_route_topk": "piiipppppp",
    "nvfp4_moe_clear_padding": "ppiqqipppp",
    "nvfp4_moe_scatter_rows": "piqipppiqpp",
    "nvfp4_moe_combine": "piqppiiqpp",
    "nvfp4_selftest_wait_timeout": "ipp",
    "nvfp4_mismatch_norm": "ppqpp",
}
_CT = {"p": ctypes.c_void_p, "q": ctypes.c_int64, "i": ctypes.c_int32}


class NVFP4Error(RuntimeError):
    def __init__(self, fn, status, detail=""):
        self.status = status
        super().__init__("%s -> %s%s" % (fn, STATUS.get(status, status), (": " + detail) if detail else ""))


_lib = None


def library_path():
    return LIB


def load(build: bool = False):
    """Load libnvfp4moe.so (compiling it first if `build`); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        build_library()
    if not os.path.exists(LIB):
        raise RuntimeError("libnvfp4moe.so is not built (%s); run __graft_entry__.build() "
                           "or python -m nvfp4_precision_moe_gb300.build" % LIB)
    L = ctypes.CDLL(LIB)
    for name, sig in _SIGS.items():
        fn = getattr(L, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [_CT[c] for c in sig]
    L.nvfp4_status_str.restype = ctypes.c_char_p
    L.nvfp4_status_str.argtypes = [ctypes.c_int]
    L.nvfp4_last_error.restype = ctypes.c_char_p
    L.nvfp4_last_error.argtypes = []
    _lib = L
    return L


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    assert t.is_cuda, "device tensor expected"
    return t.data_ptr()


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _call(name, *args):
    L = load()
    st = getattr(L, name)(*args)
    if st != 0:
        raise NVFP4Error(name, st, L.nvfp4_last_error().decode())


def nvfp4_init():
    _call("nvfp4_init")


def nvfp4_amax(x, amax_out, ntensors=1, stream=None):
    """A1: amax_out[t] = max|x[t]| for x [ntensors*M, K] (or [ntensors, M, K]) BF16."""
    K = x.shape[-1]
    M = x.numel() // (K * ntensors)
    _call("nvfp4_amax", _p(x), M, K, K, ntensors, M * K, _p(amax_out), _s(stream))


def nvfp4_quantize(x, amax, codes, scales, resid=None, S=None, gs_out=None, dst_row=None,
                   fanout=1, rows_out=None, row_limit=None, dev_status=None, stream=None):
    """A1-A5, A9: NVFP4 codes, block scales and the RAC residual of x [M, K]
    (rows below the device int32 *row_limit only, if given)."""
    M, K = x.shape
    k = 0 if S is None else S.numel()
    if rows_out is None:
        rows_out = codes.shape[0]
    _call("nvfp4_quantize", _p(x), M, K, x.stride(0), _p(amax), _p(gs_out), _p(S), k,
          _p(dst_row), fanout, rows_out, _p(codes), _p(scales), _p(resid), _p(row_limit),
          _p(dev_status), _s(stream))


def nvfp4_fake_quant(w, w_hat, amax_ws, gs_out=None, dev_status=None, stream=None):
    """A16: QDQ_W of each w[t] (w: [ntensors, rows, cols] BF16); amax_ws holds
    at least 2 * ntensors + 1 32-bit words of scratch."""
    nt, rows, cols = w.shape
    if amax_ws.numel() * amax_ws.element_size() < 4 * (2 * nt + 1):
        raise ValueError("nvfp4_fake_quant: amax_ws needs 2 * ntensors + 1 words")
    _call("nvfp4_fake_quant", _p(w), nt, rows, cols, _p(w_hat), _p(gs_out), _p(amax_ws),
          _p(dev_status), _s(stream))


def nvfp4_fake_quant_transposed(w, w_hat, w_hat_t, amax_ws, gs_out=None, dev_status=None, stream=None):
    """QDQ_W of each w[t] and its transpose w_hat_t[t] = w_hat[t]^T, from one read of w."""
    nt, rows, cols = w.shape
    _call("nvfp4_fake_quant_transposed", _p(w), nt, rows, cols, _p(w_hat), _p(w_hat_t), _p(gs_out), _p(amax_ws),
          _p(dev_status), _s(stream))


def nvfp4_fake_quant_noalloc(w, w_hat, gs_out=None, dev_status=None, stream=None):
    """A16 without caller scratch: the library's own fixed array (<= 4096 tensors)."""
    nt, rows, cols = w.shape
    _call("nvfp4_fake_quant_noalloc", _p(w), nt, rows, cols, _p(w_hat), _p(gs_out), _p(dev_status),
          _s(stream))


def nvfp4_rac_requant_residual(resid, amax_ws, offsets=None, E=0, gs_out=None, dev_status=None, stream=None):
    """Literal Eq. 21 residual: resid [rows_cap, k] BF16 replaced in place by
    its own NVFP4 quantize-dequantize (rows [0, offsets[E]) when offsets is given)."""
    rows_cap, k = resid.shape
    _call("nvfp4_rac_requant_residual", _p(resid), rows_cap, k, _p(offsets), E, _p(amax_ws), _p(gs_out),
          _p(dev_status), _s(stream))


def nvfp4_rac_select_channels_online(x, amax, k, S_out, score_ws, offsets=None, E=0, stream=None):
    """Eq. 23-24 on the batch at hand (rows [0, offsets[E]) of x when offsets is
    given); score_ws: device float64[257 * K]."""
    rows_cap, K = x.shape
    _call("nvfp4_rac_select_channels_online", _p(x), rows_cap, K, _p(offsets), E, _p(amax), k, _p(S_out),
          _p(score_ws), _s(stream))


def nvfp4_gather_selected_weights(w_codes, w_scales, E, N, K, S, w_sel, dev_status=None, stream=None):
    """w_sel [E, N, k] of a weight pack for the channel set S."""
    _call("nvfp4_gather_selected_weights", _p(w_codes), _p(w_scales), E, N, K, _p(S), S.numel(), _p(w_sel),
          _p(dev_status), _s(stream))


def nvfp4_transpose_weight_pack(w_codes, w_scales, E, N, K, codes_t, scales_t, stream=None):
    """Channel-major copy of a weight pack: codes_t [E, K, N/2], scales_t [E, K/16, N] (uint8)."""
    _call("nvfp4_transpose_weight_pack", _p(w_codes), _p(w_scales), E, N, K, _p(codes_t), _p(scales_t), _s(stream))


def nvfp4_gather_selected_weights_t(codes_t, scales_t, E, N, K, S, w_sel, stream=None):
    """w_sel [E, N, k] for the channel set S from the channel-major copy of a weight pack."""
    _call("nvfp4_gather_selected_weights_t", _p(codes_t), _p(scales_t), E, N, K, _p(S), S.numel(), _p(w_sel),
          _s(stream))


def nvfp4_prepare_weights(w, w_codes, w_scales, gs_w, amax_ws, S=None, w_sel=None, interleave=0,
                          dev_status=None, stream=None):
    """A7: rollout weight pack of w [E, N, K] BF16."""
    E, N, K = w.shape
    k = 0 if S is None else S.numel()
    _call("nvfp4_prepare_weights", _p(w), E, N, K, _p(S), k, interleave, _p(w_codes),
          _p(w_scales), _p(gs_w), _p(w_sel), _p(amax_ws), _p(dev_status), _s(stream))


def nvfp4_rac_select_channels(x, amax, k, S_out, score_ws, stream=None):
    """A6: channel calibration (Eq. 23-24) on a calibration batch x [M, K]."""
    M, K = x.shape
    _call("nvfp4_rac_select_channels", _p(x), M, K, _p(amax), k, _p(S_out), _p(score_ws),
          _s(stream))


def nvfp4_w4a4_rac_grouped_gemm(a_codes, a_scales, a_resid, gs_a, w_codes, w_scales, gs_w, w_sel,
                                k, offsets, E, N, K, y, epilogue=NVFP4_EPI_NONE,
                                out_dtype=NVFP4_OUT_F32, amax_out=None, dev_status=None,
                                stream=None):
    """A10-A13: y = gs_a*gs_w*(A.W^T) + gs_w*(r.W_sel^T) per expert segment."""
    rows_cap = a_codes.shape[0]
    _call("nvfp4_w4a4_rac_grouped_gemm", _p(a_codes), _p(a_scales), _p(a_resid), _p(gs_a),
          _p(w_codes), _p(w_scales), _p(gs_w), _p(w_sel), k, _p(offsets), E, rows_cap, N, K,
          epilogue, out_dtype, _p(y), y.stride(0), _p(amax_out), _p(dev_status), _s(stream))


def nvfp4_bf16_grouped_gemm(x, w_hat, offsets, E, N, K, y, out_dtype=NVFP4_OUT_F32,
                            epilogue=NVFP4_EPI_NONE, gu=None, dev_status=None, stream=None):
    """A17: y = x . w_hat[e]^T per expert segment (BF16 in, FP32 accumulate);
    NVFP4_EPI_SWIGLU_SAVE also stores the BF16 pre-activations to gu."""
    rows_cap = x.shape[0]
    _call("nvfp4_bf16_grouped_gemm", _p(x), _p(w_hat), _p(offsets), E, rows_cap, N, K, out_dtype,
          epilogue, _p(y), y.stride(0), _p(gu), _p(dev_status), _s(stream))


def nvfp4_bf16_grouped_gemm_dgrad(dy, w_hat, offsets, E, N, K, y, out_dtype=NVFP4_OUT_F32,
                                  epilogue=NVFP4_EPI_NONE, gu=None, dev_status=None, stream=None):
    """Eq. 13 dX: y = dy . w_hat[e] per expert segment, dy [rows_cap, K], w_hat [E, K, N] as stored;
    with epilogue=NVFP4_EPI_SWIGLU_BWD and the saved pre-activations gu [rows_cap, 2N], y = [dg | du]."""
    rows_cap = dy.shape[0]
    _call("nvfp4_bf16_grouped_gemm_dgrad", _p(dy), _p(w_hat), _p(offsets), E, rows_cap, N, K, out_dtype, epilogue,
          _p(gu), _p(y), y.stride(0), _p(dev_status), _s(stream))


def nvfp4_transpose_bf16(x, y, stream=None):
    """y[b] = x[b]^T for BF16 x [batch, rows, cols] (or [rows, cols])."""
    b, r, c = (1, *x.shape) if x.dim() == 2 else x.shape
    _call("nvfp4_transpose_bf16", _p(x), b, r, c, _p(y), _s(stream))


def nvfp4_swiglu(gu, h, stream=None):
    """h = bf16(silu(g) * u), gu = [g | u] BF16 [rows, 2I]."""
    rows, n2 = gu.shape
    _call("nvfp4_swiglu", _p(gu), rows, n2 // 2, _p(h), _s(stream))


def nvfp4_swiglu_backward(gu, dh, dgu, stream=None):
    """dgu = [dg | du] from gu = [g | u] and dh."""
    rows, n2 = gu.shape
    _call("nvfp4_swiglu_backward", _p(gu), _p(dh), rows, n2 // 2, _p(dgu), _s(stream))


def nvfp4_moe_combine_backward(dout, y, dst_row, weights, counts, offsets, E, dy, dweights=None, stream=None):
    """Routed gradient dy (BF16 [rows_cap, H]) and the combine weights' gradient."""
    T, topk = dst_row.shape
    _call("nvfp4_moe_combine_backward", _p(dout), _p(y), _p(dst_row), _p(weights), T, topk, dout.shape[1],
          _p(counts), _p(offsets), E, dy.shape[0], _p(dy), _p(dweights), _s(stream))


def nvfp4_bf16_grouped_gemm_wgrad(a_t, b_t, offsets, E, dw, out_dtype=NVFP4_OUT_F32, dev_status=None, stream=None):
    """dw[e] = a_t[:, seg e] . b_t[:, seg e]^T; a_t [M, R], b_t [N, R] BF16, dw [E, M, N]."""
    M, R = a_t.shape
    N = b_t.shape[0]
    _call("nvfp4_bf16_grouped_gemm_wgrad", _p(a_t), _p(b_t), _p(offsets), E, R, M, N, out_dtype, _p(dw),
          _p(dev_status), _s(stream))


def nvfp4_bf16_grouped_gemm_wgrad_rows(a, b, offsets, E, dw, out_dtype=NVFP4_OUT_F32, dev_status=None, stream=None):
    """dw[e] = a[seg e, :]^T . b[seg e, :]; a [R, M], b [R, N] BF16 routed rows, dw [E, M, N]."""
    R, M = a.shape
    N = b.shape[1]
    _call("nvfp4_bf16_grouped_gemm_wgrad_rows", _p(a), _p(b), _p(offsets), E, R, M, N, out_dtype, _p(dw),
          _p(dev_status), _s(stream))


def nvfp4_gemm_pipeline(which):
    """Selects the grouped-GEMM pipeline (NVFP4_PIPELINE_AUTO / _SINGLE / _PAIR)
    for later calls, process-wide; returns the previous setting."""
    prev = ctypes.c_int32(0)
    _call("nvfp4_gemm_pipeline", which, ctypes.byref(prev))
    return prev.value


def nvfp4_route_topk(logits, topk, ids, weights, counts, offsets, dst_row, stream=None):
    """A8: top-k softmax routing and the padded routed-row layout."""
    T, E = logits.shape
    _call("nvfp4_route_topk", _p(logits), T, E, topk, _p(ids), _p(weights), _p(counts),
          _p(offsets), _p(dst_row), _s(stream))


def nvfp4_moe_clear_padding(counts, offsets, E, K, k, codes, scales, resid=None, stream=None):
    """Zero the padding rows of a routed NVFP4 activation."""
    _call("nvfp4_moe_clear_padding", _p(counts), _p(offsets), E, codes.shape[0], K, k, _p(codes),
          _p(scales), _p(resid), _s(stream))


def nvfp4_moe_scatter_rows(x, topk, dst_row, counts, offsets, E, y, stream=None):
    """BF16 dispatch of token rows to routed rows (QAT path)."""
    T, K = x.shape
    _call("nvfp4_moe_scatter_rows", _p(x), T, K, topk, _p(dst_row), _p(counts), _p(offsets), E,
          y.shape[0], _p(y), _s(stream))


def nvfp4_moe_combine(y, dst_row, weights, topk, out, stream=None):
    """A15: out[t] = sum_s weights[t,s] * y[dst_row[t,s]] (FP32)."""
    y_dtype = NVFP4_OUT_BF16 if y.dtype == torch.bfloat16 else NVFP4_OUT_F32
    T, H = out.shape
    _call("nvfp4_moe_combine", _p(y), y_dtype, y.stride(0), _p(dst_row), _p(weights), T, topk, H,
          _p(out), _s(stream))


def nvfp4_selftest_wait_timeout(limit_us, dev_status, stream=None):
    """Bounded-wait self test: dev_status becomes NVFP4_ERR_TIMEOUT."""
    _call("nvfp4_selftest_wait_timeout", limit_us, _p(dev_status), _s(stream))


def nvfp4_mismatch_norm(y_infer, y_train, acc, stream=None):
    """QUADS §3.1 Eq. 11: (||y_infer - y_train||_2, ||y_train||_2) of two FP32
    layer outputs; `acc` is a device float64[2] work buffer."""
    assert y_infer.shape == y_train.shape
    _call("nvfp4_mismatch_norm", _p(y_infer), _p(y_train), y_train.numel(), _p(acc), _s(stream))
    a = acc.cpu().tolist()
    return a[0] ** 0.5, a[1] ** 0.5


from .layer import RolloutMoE, QatMoE, scale_bytes, rows_capacity  # noqa: E402
