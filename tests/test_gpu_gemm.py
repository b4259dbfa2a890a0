"""GPU parity of the tcgen05 grouped GEMMs against the CPU oracle.

* Exact case (all block scales 1.0, gs = 1): sums of products of E2M1 values
  are exact in FP32, so the FP4 tensor-core GEMM must match integer
  arithmetic bit for bit; this pins operand layout, nibble order and the MMA.
* W4A4 + RAC (QUADS §3.3 Eq. 21) on the dense workloads: max relative error
  1e-3 against the oracle's binary64 product, the error measured per element
  against max(|ref|, rms of the reference row).
* BF16 output equals the BF16 rounding of the FP32 output of the same kernel.
* Grouping: ragged expert segments (1, 127, 128, 129 rows, an empty expert).
* SwiGLU epilogue and the fused amax of its output.
* BF16 GEMM of the asymmetric-QAT forward (QUADS §3.2 Eq. 12).
Every test runs on both tcgen05 pipelines (one CTA per 128x256 tile; a CTA
pair per 256x256 tile), which must give the same results.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu as G

pytestmark = pytest.mark.gpu
TOL = 1e-3

nv = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global nv
    import nvfp4_precision_moe_gb300 as m
    m.load(build=True)
    nv = m


@pytest.fixture(autouse=True, params=["single", "pair"])
def pipeline(request, _lib):
    which = {"single": nv.NVFP4_PIPELINE_SINGLE, "pair": nv.NVFP4_PIPELINE_PAIR}[request.param]
    prev = nv.nvfp4_gemm_pipeline(which)
    yield request.param
    nv.nvfp4_gemm_pipeline(prev)


def _lut2():
    return np.array([int(round(2 * oracle.e2m1_value(c))) for c in range(16)], np.int64)


def _unpack(codes):
    return np.stack([codes & 15, codes >> 4], -1).reshape(codes.shape[0], -1)


def test_exact_integer_fp4_gemm():
    rng = np.random.default_rng(1)
    E, N, K = 2, 256, 512
    counts = [128, 256]
    offsets = np.array([0, 128, 384], np.int32)
    rows = 384
    ca = rng.integers(0, 256, (rows, K // 2), dtype=np.uint8)
    cw = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    a_codes = torch.from_numpy(ca).to(G.DEV)
    w_codes = torch.from_numpy(cw).to(G.DEV)
    a_scales = torch.full((oracle.scale_bytes(rows, K),), 0x38, dtype=torch.uint8, device=G.DEV)
    w_scales = torch.full((E * N * K // 16,), 0x38, dtype=torch.uint8, device=G.DEV)
    one = torch.ones(1, dtype=torch.float32, device=G.DEV)
    gs_w = torch.ones(E, dtype=torch.float32, device=G.DEV)
    y = G.zeros((rows, N), torch.float32)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_w4a4_rac_grouped_gemm(a_codes, a_scales, None, one, w_codes, w_scales, gs_w, None, 0,
                                   torch.from_numpy(offsets).to(G.DEV), E, N, K, y, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    lut = _lut2()
    ia = lut[_unpack(ca)]
    got = y.cpu().numpy().astype(np.float64)
    for e in range(E):
        r0, r1 = offsets[e], offsets[e + 1]
        iw = lut[_unpack(cw[e])]
        want = (ia[r0:r1] @ iw.T).astype(np.float64) / 4.0
        bad = np.argwhere(got[r0:r1] != want)
        assert bad.size == 0, "expert %d: %d mismatches, first %s gpu %r want %r" % (
            e, len(bad), bad[0], got[r0 + bad[0][0], bad[0][1]], want[bad[0][0], bad[0][1]])


class Dense:
    """One dense layer through the library: amax, quantize, prepare, GEMM."""

    def __init__(self, x_u16, w_u16, S, out_dtype=0):
        M, K = x_u16.shape
        N = w_u16.shape[0]
        self.M, self.N, self.K = M, N, K
        Mp = (M + 127) // 128 * 128
        k = 0 if S is None else len(S)
        self.k = k
        x = G.bf16_from_u16(x_u16)
        w = G.bf16_from_u16(w_u16)[None]
        Sd = torch.tensor(np.asarray(S), dtype=torch.int32, device=G.DEV) if k else None
        amax = G.zeros(1, torch.float32)
        nv.nvfp4_amax(x, amax)
        self.codes = G.zeros((Mp, K // 2), torch.uint8)
        self.scales = G.zeros(oracle.scale_bytes(Mp, K), torch.uint8)
        self.resid = G.zeros((Mp, k), torch.bfloat16) if k else None
        self.gs = G.zeros(1, torch.float32)
        nv.nvfp4_quantize(x, amax, self.codes, self.scales, resid=self.resid, S=Sd, gs_out=self.gs)
        self.wc = G.zeros((1, N, K // 2), torch.uint8)
        self.ws = G.zeros(N * K // 16, torch.uint8)
        self.gw = G.zeros(1, torch.float32)
        self.sel = G.zeros((1, N, k), torch.bfloat16) if k else None
        nv.nvfp4_prepare_weights(w, self.wc, self.ws, self.gw, G.zeros(1, torch.float32), S=Sd,
                                 w_sel=self.sel)
        self.offsets = torch.tensor([0, Mp], dtype=torch.int32, device=G.DEV)
        self.Mp = Mp

    def run(self, out_dtype=0):
        dt = torch.float32 if out_dtype == 0 else torch.bfloat16
        y = G.zeros((self.Mp, self.N), dt)
        st = G.zeros(1, torch.int32)
        nv.nvfp4_w4a4_rac_grouped_gemm(self.codes, self.scales, self.resid, self.gs, self.wc, self.ws,
                                       self.gw, self.sel, self.k, self.offsets, 1, self.N, self.K, y,
                                       out_dtype=out_dtype, dev_status=st)
        torch.cuda.synchronize()
        G.status_ok(st)
        return y


def _oracle_dense(x_u16, w_u16, S):
    ca, sa, r, ga = oracle.quantize(x_u16, S=S)
    cw, sw, _, gw = oracle.quantize(w_u16)
    xq = oracle.dequantize_exact(ca, sa, ga)
    wq = oracle.dequantize_exact(cw, sw, gw)
    return oracle.rac_gemm(xq, wq, r, S, ga), xq, wq


def _cfg_S(cfg, k):
    xc = synth.u16(synth.activations(cfg, batch=1))
    return oracle.select_channels(oracle.channel_scores_sq(xc), k)


@pytest.mark.parametrize("cfg", [1, 2])
def test_rac_gemm_dense_parity(cfg):
    c = synth.CONFIGS[cfg]
    x = synth.u16(synth.activations(cfg))
    w = synth.u16(synth.dense_weight(cfg))
    S = _cfg_S(cfg, c["k"])
    d = Dense(x, w, S)
    y = d.run(0)[: d.M].cpu().numpy()
    ref, xq, wq = _oracle_dense(x, w, S)
    err = G.rel_err(y, ref)
    assert err <= TOL, err
    # RAC makes a difference well above the tolerance on these inputs
    plain = oracle.rac_gemm(xq, wq)
    assert G.rel_err(plain, ref) > 10 * TOL
    # BF16 output is the BF16 rounding of the FP32 output of the same kernel
    yb = d.run(1)[: d.M]
    yf = torch.from_numpy(y).to(G.DEV).to(torch.bfloat16)
    assert torch.equal(yb.view(torch.int16), yf.view(torch.int16))


def test_rac_k0_and_all_channels():
    x = synth.u16(synth.activations(1))
    w = synth.u16(synth.dense_weight(1))
    # k = 0: plain W4A4
    d0 = Dense(x, w, None)
    ref0, xq, wq = _oracle_dense(x, w, None)
    assert G.rel_err(d0.run(0)[:64].cpu().numpy(), ref0) <= TOL
    # S = every channel (K = 256): W4A16 within the BF16 rounding of the residual
    x2 = np.ascontiguousarray(x[:, :256])
    w2 = np.ascontiguousarray(w[:, :256])
    S = np.arange(256, dtype=np.int32)
    dk = Dense(x2, w2, S)
    refk, _, wq2 = _oracle_dense(x2, w2, S)
    yk = dk.run(0)[:64].cpu().numpy()
    assert G.rel_err(yk, refk) <= TOL
    w4a16 = oracle.bf16_to_f32(x2).astype(np.float64) @ wq2.T
    assert G.rel_err(yk, w4a16) <= 2 * TOL


def test_rac_half_and_all_channels_of_a_wide_layer():
    """k beyond 256 (more RAC slices): half of the channels -- the pages' k = 50% setting
    (QUADS §4.4.1) -- and all of them, where the RAC GEMM reproduces W4A16 within the BF16
    rounding of the residual (the oracle's own pin, here on the GPU)."""
    x = synth.u16(synth.activations(1))  # 64 x 512
    w = synth.u16(synth.dense_weight(1))  # 512 x 512
    sc = oracle.channel_scores_sq(x)
    for k in (256, 512):
        S = oracle.select_channels(sc, k)
        d = Dense(x, w, S)
        ref, _, wq = _oracle_dense(x, w, S)
        y = d.run(0)[:64].cpu().numpy()
        assert G.rel_err(y, ref) <= TOL, k
        if k == 512:
            w4a16 = oracle.bf16_to_f32(x).astype(np.float64) @ wq.T
            assert G.rel_err(y, w4a16) <= 2 * TOL


def test_grouped_ragged_segments():
    rng = np.random.default_rng(3)
    E, N, K, k = 5, 256, 512, 32
    counts = np.array([1, 127, 0, 128, 129])
    offsets = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    rows = int(offsets[-1]) + 128  # one spare tile that no segment covers
    xs = synth.activations(1)  # 64 x 512
    x_all = torch.cat([xs] * 7)[: counts.sum()]
    xu = synth.u16(x_all)
    S = np.sort(rng.choice(K, k, replace=False)).astype(np.int32)
    # place each expert's rows at its segment; the rest stays zero (padding)
    dst = np.concatenate([offsets[e] + np.arange(counts[e]) for e in range(E)])
    x = G.bf16_from_u16(xu)
    amax = G.zeros(1, torch.float32)
    nv.nvfp4_amax(x, amax)
    codes = G.zeros((rows, K // 2), torch.uint8)
    scales = G.zeros(oracle.scale_bytes(rows, K), torch.uint8)
    resid = G.zeros((rows, k), torch.bfloat16)
    gs = G.zeros(1, torch.float32)
    Sd = torch.tensor(S, device=G.DEV)
    nv.nvfp4_quantize(x, amax, codes, scales, resid=resid, S=Sd, gs_out=gs,
                      dst_row=torch.tensor(dst, dtype=torch.int32, device=G.DEV), fanout=1, rows_out=rows)
    ws = torch.stack([synth.dense_weight(1)[:N] * (1 + 0.5 * e) for e in range(E)])
    wc = G.zeros((E, N, K // 2), torch.uint8)
    wsc = G.zeros(E * N * K // 16, torch.uint8)
    gw = G.zeros(E, torch.float32)
    sel = G.zeros((E, N, k), torch.bfloat16)
    nv.nvfp4_prepare_weights(ws.to(G.DEV), wc, wsc, gw, G.zeros(E, torch.float32), S=Sd, w_sel=sel)
    y = torch.full((rows, N), float("nan"), dtype=torch.float32, device=G.DEV)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_w4a4_rac_grouped_gemm(codes, scales, resid, gs, wc, wsc, gw, sel, k,
                                   torch.tensor(offsets, device=G.DEV), E, N, K, y, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    got = y.cpu().numpy()
    ca, sa, r, ga = oracle.quantize(xu, S=S)
    xq = oracle.dequantize_exact(ca, sa, ga)
    pos = 0
    for e in range(E):
        cw, sw, _, g = oracle.quantize(synth.u16(ws[e]))
        wq = oracle.dequantize_exact(cw, sw, g)
        n = counts[e]
        if n:
            ref = oracle.rac_gemm(xq[pos:pos + n], wq, r[pos:pos + n], S, ga)
            assert G.rel_err(got[offsets[e]:offsets[e] + n], ref) <= TOL, e
        # padding rows of a segment are exactly zero
        assert (got[offsets[e] + n:offsets[e + 1]] == 0).all()
        pos += n
    # rows beyond the last segment are never written
    assert np.isnan(got[offsets[-1]:]).all()


def test_swiglu_epilogue_and_fused_amax():
    rng = np.random.default_rng(4)
    E, I, H, k = 2, 128, 512, 16
    N = 2 * I
    counts = np.array([100, 160])
    offsets = np.array([0, 128, 384], np.int32)
    rows = 384
    xs = torch.cat([synth.activations(1)] * 5)[: counts.sum()]
    xu = synth.u16(xs)
    S = np.sort(rng.choice(H, k, replace=False)).astype(np.int32)
    dst = np.concatenate([offsets[e] + np.arange(counts[e]) for e in range(E)])
    x = G.bf16_from_u16(xu)
    amax = G.zeros(1, torch.float32)
    nv.nvfp4_amax(x, amax)
    codes = G.zeros((rows, H // 2), torch.uint8)
    scales = G.zeros(oracle.scale_bytes(rows, H), torch.uint8)
    resid = G.zeros((rows, k), torch.bfloat16)
    gs = G.zeros(1, torch.float32)
    Sd = torch.tensor(S, device=G.DEV)
    nv.nvfp4_quantize(x, amax, codes, scales, resid=resid, S=Sd, gs_out=gs,
                      dst_row=torch.tensor(dst, dtype=torch.int32, device=G.DEV), rows_out=rows)
    w13 = torch.stack([synth.dense_weight(1)[:N] * (1 + e) for e in range(E)])
    wc = G.zeros((E, N, H // 2), torch.uint8)
    wsc = G.zeros(E * N * H // 16, torch.uint8)
    gw = G.zeros(E, torch.float32)
    sel = G.zeros((E, N, k), torch.bfloat16)
    nv.nvfp4_prepare_weights(w13.to(G.DEV), wc, wsc, gw, G.zeros(E, torch.float32), S=Sd, w_sel=sel,
                             interleave=1)
    h = G.zeros((rows, I), torch.bfloat16)
    hmax = G.zeros(1, torch.float32)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_w4a4_rac_grouped_gemm(codes, scales, resid, gs, wc, wsc, gw, sel, k,
                                   torch.tensor(offsets, device=G.DEV), E, N, H, h, epilogue=1,
                                   out_dtype=1, amax_out=hmax, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    got = h.float().cpu().numpy()
    ca, sa, r, ga = oracle.quantize(xu, S=S)
    xq = oracle.dequantize_exact(ca, sa, ga)
    pos = 0
    for e in range(E):
        cw, sw, _, g = oracle.quantize(synth.u16(w13[e]))
        wq = oracle.dequantize_exact(cw, sw, g)
        n = counts[e]
        y = oracle.rac_gemm(xq[pos:pos + n], wq, r[pos:pos + n], S, ga)
        ref = oracle.swiglu(y, I)
        # BF16 output: the unit roundoff 2^-8 of BF16 plus the GEMM tolerance
        assert G.rel_err(got[offsets[e]:offsets[e] + n], ref) <= 2.0 ** -8 + TOL
        assert (got[offsets[e] + n:offsets[e + 1]] == 0).all()
        pos += n
    assert hmax.item() == np.abs(got).max()


@pytest.mark.parametrize("pipe", [1, 2])
def test_bf16_swiglu_epilogue_that_keeps_the_pre_activations(pipe):
    """NVFP4_EPI_SWIGLU_SAVE: its h equals the NVFP4_EPI_SWIGLU output and its
    pre-activations the BF16 NVFP4_EPI_NONE output, bit for bit, on both GEMM
    pipelines, over ragged and empty experts and two 256-column tiles."""
    E, N, K = 3, 512, 192
    counts = np.array([50, 0, 300])
    offsets = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    rows = int(offsets[-1])
    rng = np.random.default_rng(16)
    xr = np.zeros((rows, K), np.float32)
    for e in range(E):
        xr[offsets[e]:offsets[e] + counts[e]] = rng.standard_normal((counts[e], K))
    x = G.bf16_from_u16(oracle.bf16_round(xr))
    w = G.bf16_from_u16(oracle.bf16_round((rng.standard_normal((E, N, K)) * 0.05).astype(np.float32)))
    offs = torch.tensor(offsets, device=G.DEV)
    st = G.zeros(1, torch.int32)
    h_ref = G.zeros((rows, N // 2), torch.bfloat16)
    gu_ref = G.zeros((rows, N), torch.bfloat16)
    h = torch.full((rows, N // 2), 7.0, dtype=torch.bfloat16, device=G.DEV)
    gu = torch.full((rows, N), 7.0, dtype=torch.bfloat16, device=G.DEV)
    prev = nv.nvfp4_gemm_pipeline(pipe)
    try:
        nv.nvfp4_bf16_grouped_gemm(x, w, offs, E, N, K, h_ref, out_dtype=1, epilogue=nv.NVFP4_EPI_SWIGLU, dev_status=st)
        nv.nvfp4_bf16_grouped_gemm(x, w, offs, E, N, K, gu_ref, out_dtype=1, dev_status=st)
        nv.nvfp4_bf16_grouped_gemm(x, w, offs, E, N, K, h, out_dtype=1, epilogue=nv.NVFP4_EPI_SWIGLU_SAVE, gu=gu,
                                   dev_status=st)
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_gemm_pipeline(prev)
    G.status_ok(st)
    assert torch.equal(h, h_ref) and torch.equal(gu, gu_ref)


@pytest.mark.parametrize("swiglu", [False, True])
def test_bf16_grouped_gemm_parity(swiglu):
    E, N, K = 3, 256, 192
    counts = np.array([50, 0, 200])
    offsets = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    rows = int(offsets[-1])
    rng = np.random.default_rng(6)
    xr = np.zeros((rows, K), np.float32)
    for e in range(E):
        xr[offsets[e]:offsets[e] + counts[e]] = rng.standard_normal((counts[e], K))
    xu = oracle.bf16_round(xr)
    wu = oracle.bf16_round((rng.standard_normal((E, N, K)) * 0.05).astype(np.float32))
    x = G.bf16_from_u16(xu)
    w = G.bf16_from_u16(wu)
    st = G.zeros(1, torch.int32)
    offs = torch.tensor(offsets, device=G.DEV)
    if swiglu:
        y = G.zeros((rows, N // 2), torch.bfloat16)
        nv.nvfp4_bf16_grouped_gemm(x, w, offs, E, N, K, y, out_dtype=1, epilogue=1, dev_status=st)
    else:
        y = G.zeros((rows, N), torch.float32)
        nv.nvfp4_bf16_grouped_gemm(x, w, offs, E, N, K, y, out_dtype=0, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    got = y.float().cpu().numpy()
    for e in range(E):
        n = counts[e]
        if not n:
            continue
        ref = oracle.bf16_gemm(xu[offsets[e]:offsets[e] + n], wu[e])
        if swiglu:
            ref = oracle.swiglu(ref, N // 2)
            assert G.rel_err(got[offsets[e]:offsets[e] + n], ref) <= 2.0 ** -8 + TOL
        else:
            assert G.rel_err(got[offsets[e]:offsets[e] + n], ref) <= TOL
