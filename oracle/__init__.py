"""CPU oracle for the NVFP4 W4A4 + RAC hot path -- TEST INFRASTRUCTURE ONLY.

A plain, slow restatement of what the path computes, used to check the CUDA
library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` import it; the library itself never does.  It shares no code
with the CUDA path: the numeric core is ``nvfp4_oracle.c`` (plain C, loaded
with ctypes) and the bookkeeping below is numpy.

"QUADS" is the paper "QUADS: Stabilizing NVFP4 Reinforcement Learning for MoE
via QUantization-error Alignment across Dual Sides".  BF16 tensors cross this
interface as numpy ``uint16`` bit patterns.

Parity status: every function is pinned by ``tests/test_oracle_*.py`` except
the scale layout, which is pinned only by the GPU GEMM parity tests (a wrong
layout gives errors far above their tolerance; on the CPU it is checked to be
a bijection with zero padding).
"""
import ctypes
import numpy as np

from .build import build_oracle

_lib = None

_f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(np.uint8, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build_oracle())
        sig = {
            "orc_e2m1_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_e4m3_value": (ctypes.c_double, [ctypes.c_int]),
            "orc_e2m1_encode": (ctypes.c_int, [ctypes.c_float]),
            "orc_e4m3_encode": (ctypes.c_int, [ctypes.c_float]),
            "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_float]),
            "orc_e2m1_encode_array": (None, [_f32p, _i64, _u8p]),
            "orc_e4m3_encode_array": (None, [_f32p, _i64, _u8p]),
            "orc_bf16_round_array": (None, [_f32p, _i64, _u16p]),
            "orc_amax": (ctypes.c_float, [_u16p, _i64, _i64, _i64]),
            "orc_tensor_scale": (ctypes.c_float, [ctypes.c_float]),
            "orc_quantize": (None, [_u16p, _i64, _i64, _i64, ctypes.c_float, _u8p, _u8p,
                                    ctypes.c_void_p, _i32, ctypes.c_void_p]),
            "orc_dequantize_exact": (None, [_u8p, _u8p, _i64, _i64, ctypes.c_float, _f64p]),
            "orc_dequantize_f32": (None, [_u8p, _u8p, _i64, _i64, ctypes.c_float, _f32p]),
            "orc_scale_layout": (None, [_u8p, _i64, _i64, _u8p]),
            "orc_fake_quant": (None, [_u16p, _i64, _i64, _u16p, ctypes.POINTER(ctypes.c_float)]),
            "orc_rac_gemm": (None, [_f64p, ctypes.c_void_p, ctypes.c_void_p, _i32, ctypes.c_double,
                                    _f64p, _i64, _i64, _i64, _f64p]),
            "orc_bf16_gemm": (None, [_u16p, _u16p, _i64, _i64, _i64, _f64p]),
            "orc_channel_scores": (None, [_u16p, _i64, _i64, ctypes.c_float, _f64p]),
            "orc_select_channels": (None, [_f64p, _i64, _i32, _i32p]),
            "orc_route_topk": (None, [_f32p, _i32, _i32, _i32, _i32p, _f64p]),
            "orc_swiglu": (None, [_f64p, _i64, _i64, _f64p]),
            "orc_combine": (None, [_f64p, _i64, _i32p, _f64p, _i32, _i32, _i64, _f64p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- formats --

def e2m1_value(code):
    """E2M1 code -> value (QUADS §2.2 "FP4.")."""
    return lib().orc_e2m1_value(int(code))


def e4m3_value(code):
    """E4M3 code -> value (QUADS §2.2 "FP8."); NaN for 0x7F / 0xFF."""
    return lib().orc_e4m3_value(int(code))


def e2m1_encode(v):
    """float32 array -> E2M1 codes (RNE, saturating, sign kept)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e2m1_encode_array(v.reshape(-1), v.size, out.reshape(-1))
    return out


def e4m3_encode(v):
    """non-negative float32 array -> E4M3 codes (RNE, saturating at 448)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_e4m3_encode_array(v.reshape(-1), v.size, out.reshape(-1))
    return out


def bf16_round(v):
    """float32 array -> bfloat16 bit patterns (RNE)."""
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_round_array(v.reshape(-1), v.size, out.reshape(-1))
    return out


def bf16_to_f32(b):
    """bfloat16 bit patterns -> float32 (exact)."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# -------------------------------------------------------------- quantizer --

def amax(x):
    """max |x| of a BF16 matrix."""
    x = _c(x, np.uint16)
    M, K = x.shape
    return float(lib().orc_amax(x, M, K, K))


def tensor_scale(a):
    """Per-tensor FP32 scale: the smallest power of two >= fl(amax / 2688)
    (1 for an all-zero tensor)."""
    return float(np.float32(lib().orc_tensor_scale(float(a))))


def quantize(x, gs=None, S=None):
    """NVFP4 quantize of a BF16 matrix [M,K] (QUADS §2.2, Eq. 9 / Eq. 20).

    Returns (codes [M,K/2] u8, scales [M,K/16] u8 canonical, resid [M,k] u16
    bf16 bits of the residual in units of gs, gs float).  gs defaults to the
    tensor scale of x's amax.
    """
    x = _c(x, np.uint16)
    M, K = x.shape
    assert K % 16 == 0
    if gs is None:
        gs = tensor_scale(amax(x))
    S = np.zeros(0, np.int32) if S is None else _c(S, np.int32)
    k = S.size
    codes = np.zeros((M, K // 2), np.uint8)
    scales = np.zeros((M, K // 16), np.uint8)
    resid = np.zeros((M, k), np.uint16)
    lib().orc_quantize(x, M, K, K, float(gs), codes, scales, _ptr(S) if k else None, k,
                       _ptr(resid) if k else None)
    return codes, scales, resid, float(gs)


def dequantize_exact(codes, scales, gs):
    """codes/scales -> exact real values code*sb*gs as float64 [M,K]."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    M = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((M, K), np.float64)
    lib().orc_dequantize_exact(codes, scales, M, K, float(gs), out)
    return out


def dequantize_f32(codes, scales, gs):
    """codes/scales -> binary32 dequantized values fl(fl(code*sb)*gs)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    M = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((M, K), np.float32)
    lib().orc_dequantize_f32(codes, scales, M, K, float(gs), out)
    return out


def scale_bytes(M, K):
    """Size of the scale layout: ceil(M/128) * ceil(K/256) * 2048 bytes."""
    return ((M + 127) // 128) * ((K // 16 + 15) // 16) * 2048


def scale_layout(scales, K):
    """Canonical [M,K/16] scales -> the scale layout shared by the quantizer
    and the GEMM (1-D u8)."""
    scales = _c(scales, np.uint8)
    M = scales.shape[0]
    out = np.empty(scale_bytes(M, K), np.uint8)
    lib().orc_scale_layout(scales, M, K, out)
    return out


def scale_offsets(K):
    """Byte offsets [128, K/16] of every (row, block) of one 128-row tile in
    the scale layout, found by laying out two index patterns (row ids,
    block-in-slice ids) with the layout function itself."""
    nb = K // 16
    Lr = scale_layout(np.repeat(np.arange(1, 129, dtype=np.uint8)[:, None], nb, axis=1), K)
    Lb = scale_layout(np.tile((np.arange(nb) % 16 + 1).astype(np.uint8), (128, 1)), K)
    per_slice = Lr.size // ((nb + 15) // 16)
    where = np.full((128, nb), -1, np.int64)
    o = np.nonzero(Lr)[0]
    where[Lr[o].astype(np.int64) - 1, (o // per_slice) * 16 + Lb[o].astype(np.int64) - 1] = o
    assert (where >= 0).all()
    return where


def scale_rows(layout, rows, K):
    """The canonical block scales [len(rows), K/16] of `rows`, read back from
    a scale buffer in the scale layout."""
    rows = np.asarray(rows, np.int64)
    return np.asarray(layout)[(rows // 128)[:, None] * scale_bytes(128, K) + scale_offsets(K)[rows % 128]]


def requant_residual(resid, gs_a):
    """The literal second-pass form of QUADS §3.3 Eq. 21: the residual on the
    selected channels is itself NVFP4-quantized, Q_A(r) with r = resid*gs_a
    (resid as quantize() returns it, in units of gs_a).  Reading: Q_A acts on
    the gathered [M, k] residual -- 16-element blocks along the gathered
    channel axis -- with a tensor scale of its own (from amax |r| over all M
    rows).  Returns Q_A(r)/gs_a as BF16 bits [M, k] (exact: FP4-grid values
    need at most 6 significant bits) and the residual's tensor scale."""
    resid = _c(resid, np.uint16)
    r = bf16_round((bf16_to_f32(resid).astype(np.float64) * gs_a).astype(np.float32))
    codes, scales, _, gs_r = quantize(r)
    q = dequantize_exact(codes, scales, gs_r) / gs_a
    out = bf16_round(q.astype(np.float32))
    assert np.array_equal(bf16_to_f32(out).astype(np.float64), q), "Q_A(r)/gs_a not exact in BF16"
    return out, gs_r


def fake_quant(w):
    """QDQ_W of QUADS §3.2 Eq. 12: returns (w_hat bf16 bits [M,K], gs)."""
    w = _c(w, np.uint16)
    M, K = w.shape
    out = np.empty((M, K), np.uint16)
    gs = ctypes.c_float()
    lib().orc_fake_quant(w, M, K, out, ctypes.byref(gs))
    return out, float(gs.value)


# ----------------------------------------------------------------- GEMMs --

def rac_gemm(xq, wq, resid=None, S=None, gs_a=1.0):
    """W4A4 + RAC product (QUADS §3.3 Eq. 21), binary64.

    xq [M,K], wq [N,K]: exact dequantized operands (float64);
    resid [M,k] bf16 bits on channels S, in units of gs_a (as quantize()
    returns it).  Returns float64 [M,N].
    """
    xq = _c(xq, np.float64)
    wq = _c(wq, np.float64)
    M, K = xq.shape
    N = wq.shape[0]
    k = 0 if S is None else len(S)
    Sa = _c(S, np.int32) if k else None
    ra = _c(resid, np.uint16) if k else None
    y = np.empty((M, N), np.float64)
    lib().orc_rac_gemm(xq, _ptr(ra), _ptr(Sa), k, float(gs_a), wq, M, N, K, y)
    return y


def bf16_gemm(x, w):
    """Asymmetric-QAT forward (QUADS §3.2 Eq. 12): x [M,K] @ w [N,K]^T in binary64."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    y = np.empty((M, N), np.float64)
    lib().orc_bf16_gemm(x, w, M, N, K, y)
    return y


# -------------------------------------------------------- channel choice --

def channel_scores_sq(x, gs=None):
    """Squared Eq. 23 score per channel over the batch, float64 [K]."""
    x = _c(x, np.uint16)
    M, K = x.shape
    if gs is None:
        gs = tensor_scale(amax(x))
    out = np.empty(K, np.float64)
    lib().orc_channel_scores(x, M, K, float(gs), out)
    return out


def select_channels(ssq, k):
    """Eq. 24 with a channel count: top-k by score, ties to lower index, sorted."""
    ssq = _c(ssq, np.float64)
    S = np.zeros(k, np.int32)
    lib().orc_select_channels(ssq, ssq.size, k, S)
    return S


# --------------------------------------------------------------- MoE glue --

def route_topk(logits, topk):
    """Top-k softmax router: (ids int32 [T,topk], weights float64 [T,topk])."""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float64)
    lib().orc_route_topk(logits, T, E, topk, ids, w)
    return ids, w


def route_layout(ids, E, pad=128):
    """Routed-row layout of the grouped GEMM (a layout choice of this library).

    Rows are ordered by (expert, token, slot); each expert's segment starts at
    a multiple of ``pad``.  Returns (counts [E], offsets [E+1] padded row
    starts, dst_row [T,topk]).
    """
    ids = np.asarray(ids)
    T, topk = ids.shape
    counts = np.bincount(ids.reshape(-1), minlength=E).astype(np.int64)
    padded = (counts + pad - 1) // pad * pad
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(padded)
    dst = np.empty((T, topk), np.int64)
    fill = offsets[:-1].copy()
    for t in range(T):
        for s in range(topk):
            e = ids[t, s]
            dst[t, s] = fill[e]
            fill[e] += 1
    return counts, offsets, dst


def swiglu(y, I):
    """h = silu(gate) * up, gate = y[:, :I], up = y[:, I:2I], binary64."""
    y = _c(y, np.float64)
    M = y.shape[0]
    h = np.empty((M, I), np.float64)
    lib().orc_swiglu(y, M, I, h)
    return h


def combine(y, rows, weights):
    """out[t] = sum_s weights[t,s] * y[rows[t,s]] (binary64)."""
    y = _c(y, np.float64)
    rows = _c(rows, np.int32)
    weights = _c(weights, np.float64)
    T, topk = rows.shape
    H = y.shape[1]
    out = np.empty((T, H), np.float64)
    lib().orc_combine(y, H, rows, weights, T, topk, H, out)
    return out


# ------------------------------------------------ trainer backward (Eq. 13) --
# The asymmetric-QAT learner's backward with the straight-through estimator
# (QUADS §3.2 Eq. 13): the weight fake-quantizer passes gradients unchanged,
# so these are the plain derivatives of the layer's forward, in binary64.

def swiglu_grad(gu, dh):
    """Backward of h = silu(g) * u for gu = [g | u] ([M, 2I]): returns
    [dg | du] with dg = dh * u * s * (1 + g * (1 - s)), du = dh * g * s,
    s = 1 / (1 + exp(-g))."""
    gu = _c(gu, np.float64)
    dh = _c(dh, np.float64)
    I = dh.shape[1]
    g, u = gu[:, :I], gu[:, I:2 * I]
    s = 1.0 / (1.0 + np.exp(-g))
    return np.concatenate([dh * u * s * (1.0 + g * (1.0 - s)), dh * g * s], axis=1)


def combine_grad(dout, y, rows, weights, R):
    """Backward of combine(): for out[t] = sum_s w[t,s] y[rows[t,s]], returns
    dy [R, H] (dy[rows[t,s]] = w[t,s] dout[t], other rows 0) and
    dw[t,s] = <y[rows[t,s]], dout[t]>."""
    dout = _c(dout, np.float64)
    y = _c(y, np.float64)
    rows = np.asarray(rows)
    w = _c(weights, np.float64)
    T, topk = rows.shape
    dy = np.zeros((R, dout.shape[1]))
    dw = np.zeros((T, topk))
    for t in range(T):
        for s in range(topk):
            dy[rows[t, s]] = w[t, s] * dout[t]
            dw[t, s] = y[rows[t, s]] @ dout[t]
    return dy, dw


def segment_wgrad(a, b, offsets):
    """Per-expert weight gradient: dW[e] = a[seg e]^T . b[seg e] over the row
    segments seg e = [offsets[e], offsets[e+1]) of a [R, M] and b [R, N]."""
    a = _c(a, np.float64)
    b = _c(b, np.float64)
    E = len(offsets) - 1
    out = np.zeros((E, a.shape[1], b.shape[1]))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        out[e] = a[r0:r1].T @ b[r0:r1]
    return out
