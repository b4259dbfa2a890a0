"""GPU parity of the quantization kernels against the CPU oracle.

Codes, block scales (in the header's scale layout), residuals, per-tensor scales, fake-quantized weights
and selected channels must be bit-exact (QUADS §2.2 "FP4.", Eq. 12, Eq. 20-21,
Eq. 23-24).  Every input is a seeded synthetic tensor; the oracle computes
its expected values from the same inputs on its own.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu as G
from tests.test_oracle_quant import _rand_x

pytestmark = pytest.mark.gpu

nv = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global nv
    import nvfp4_precision_moe_gb300 as m
    m.load(build=True)
    nv = m


def _gpu_quantize(x_u16, S=None, rows_out=None, dst=None, fanout=1, amax_override=None):
    M, K = x_u16.shape
    rows_out = M if rows_out is None else rows_out
    x = G.bf16_from_u16(x_u16)
    k = 0 if S is None else len(S)
    amax = G.zeros(1, torch.float32)
    if amax_override is None:
        nv.nvfp4_amax(x, amax)
    else:
        amax.fill_(amax_override)
    codes = G.zeros((rows_out, K // 2), torch.uint8)
    scales = G.zeros(oracle.scale_bytes(rows_out, K), torch.uint8)
    resid = G.zeros((rows_out, max(k, 1)), torch.bfloat16)[:, :k].contiguous() if k else None
    gs = G.zeros(1, torch.float32)
    st = G.zeros(1, torch.int32)
    Sd = torch.tensor(np.asarray(S), dtype=torch.int32, device=G.DEV) if k else None
    dd = torch.tensor(np.asarray(dst), dtype=torch.int32, device=G.DEV) if dst is not None else None
    nv.nvfp4_quantize(x, amax, codes, scales, resid=resid, S=Sd, gs_out=gs, dst_row=dd, fanout=fanout,
                      rows_out=rows_out, dev_status=st)
    torch.cuda.synchronize()
    return dict(amax=amax.item(), gs=gs.item(), codes=codes.cpu().numpy(), scales=scales.cpu().numpy(),
                resid=G.u16(resid) if k else np.zeros((rows_out, 0), np.uint16), status=st.item())


def _check_against_oracle(x_u16, S=None):
    got = _gpu_quantize(x_u16, S)
    M, K = x_u16.shape
    a = oracle.amax(x_u16)
    assert got["amax"] == a
    codes, scales, resid, gs = oracle.quantize(x_u16, S=S)
    assert got["gs"] == np.float32(gs)
    assert got["status"] == 0
    bad = np.flatnonzero(got["codes"].reshape(-1) != codes.reshape(-1))
    assert bad.size == 0, "codes differ at %d bytes, first %s: gpu %02x oracle %02x" % (
        bad.size, bad[:4], got["codes"].reshape(-1)[bad[0]], codes.reshape(-1)[bad[0]])
    sw = oracle.scale_layout(scales, K)
    assert np.array_equal(got["scales"], sw)
    if S is not None and len(S):
        assert np.array_equal(got["resid"], resid)


def _cfg_S(cfg, k):
    """RAC channels chosen by the oracle on the workload's calibration batch."""
    xc = synth.u16(synth.activations(cfg, batch=1))
    return oracle.select_channels(oracle.channel_scores_sq(xc), k)


def test_amax_exact():
    x = synth.u16(synth.activations(2))
    got = _gpu_quantize(x)
    assert got["amax"] == oracle.amax(x)
    # batched: three tensors, each its own amax
    w = torch.stack([synth.dense_weight(1), synth.dense_weight(1) * 3, synth.dense_weight(1) * 0])
    amax = G.zeros(3, torch.float32)
    nv.nvfp4_amax(w.to(G.DEV), amax, ntensors=3)
    ref = [oracle.amax(synth.u16(w[i])) for i in range(3)]
    assert amax.cpu().tolist() == ref


@pytest.mark.parametrize("cfg", [1, 2])
def test_quantize_activation_parity(cfg):
    x = synth.u16(synth.activations(cfg))
    _check_against_oracle(x, _cfg_S(cfg, synth.CONFIGS[cfg]["k"]))


def test_quantize_weight_alone_parity():
    _check_against_oracle(synth.u16(synth.dense_weight(2)))
    _check_against_oracle(synth.u16(synth.dense_weight(1)))


@pytest.mark.parametrize("M,K", [(1, 32), (17, 96), (129, 160), (300, 512), (128, 64)])
def test_quantize_ragged_shapes(M, K):
    rng = np.random.default_rng(M * 1000 + K)
    x = torch.from_numpy(rng.standard_t(3, (M, K)).astype(np.float32)).to(torch.bfloat16)
    S = np.sort(rng.choice(K, 8 if K >= 8 else K, replace=False)).astype(np.int32)
    _check_against_oracle(synth.u16(x), S)


def test_quantize_maximum_width_and_unstaged_residual():
    """K = 16384 (the largest row the quantizer takes) with k = 1040 selected
    channels: more than the per-warp stage holds, so the residual goes straight
    to the destination rows from the row's block scales."""
    rng = np.random.default_rng(77)
    M, K, k = 40, 16384, 1040
    x = torch.from_numpy(rng.standard_t(3, (M, K)).astype(np.float32)).to(torch.bfloat16)
    S = np.sort(rng.choice(K, k, replace=False)).astype(np.int32)
    _check_against_oracle(synth.u16(x), S)


def test_element_encoder_all_bf16_values():
    # gs = 1 (amax 2688) and every block's first element 6 -> block scale 1.0,
    # so each element is rounded to E2M1 as is: this covers every BF16 value in
    # [-6, 6] and all E2M1 ties.
    vals = np.arange(0, 65536, dtype=np.uint32)
    f = (vals << 16).view(np.float32)
    f = f[np.isfinite(f) & (np.abs(f) <= 6.0)]
    per = 15
    nblk = (f.size + per - 1) // per
    blk = np.zeros((nblk, 16), np.float32)
    blk[:, 0] = 6.0
    flat = np.zeros(nblk * per, np.float32)
    flat[: f.size] = f
    blk[:, 1:] = flat.reshape(nblk, per)
    K = 512
    rows = (nblk * 16 + K - 1) // K
    x = np.zeros(rows * K, np.float32)
    x[: nblk * 16] = blk.reshape(-1)
    x = x.reshape(rows, K)
    x = np.vstack([x, np.full((1, K), 2688.0, np.float32)])
    xb = oracle.bf16_round(x)
    _check_against_oracle(xb)


def test_block_scale_ties_and_subnormals():
    # gs = 1; block amax = 6 * m for m every E4M3 value and every midpoint
    # between neighbours (including the subnormal range): the scale is the
    # E4M3 rounding of m, ties to even.
    vals = np.array([oracle.e4m3_value(c) for c in range(127)])
    mids = (vals[:-1] + vals[1:]) / 2
    ms = np.concatenate([vals, mids, [vals[-1] * 1.01, 1e-4, 3e-3]])
    K = 64
    rows = (ms.size * 16 + K - 1) // K
    x = np.zeros((rows * K // 16, 16), np.float32)
    rng = np.random.default_rng(5)
    x[: ms.size, 0] = 6.0 * ms
    x[: ms.size, 1:] = rng.uniform(-1, 1, (ms.size, 15)) * 6.0 * ms[:, None]
    x = x.reshape(rows, K)
    x = np.vstack([x, np.full((1, K), 2688.0, np.float32)])
    _check_against_oracle(oracle.bf16_round(x))


def test_zero_tensor_and_signed_zeros():
    x = np.zeros((4, 64), np.uint16)
    x[1, :] = 0x8000  # -0
    S = np.array([0, 5, 9, 20, 33, 40, 50, 63], np.int32)
    got = _gpu_quantize(x, S=S)
    assert got["gs"] == 1.0 and got["amax"] == 0.0
    codes, _, _, _ = oracle.quantize(x, S=S)
    assert np.array_equal(got["codes"], codes)
    assert not got["scales"].any() and not got["resid"].any()
    assert (got["codes"][1] == 0x88).all()


def test_scatter_to_routed_rows():
    rng = np.random.default_rng(9)
    x = synth.u16(synth.activations(1))[:40]
    S = np.array([3, 100, 101, 200, 300, 301, 400, 511], np.int32)
    fan = 3
    rows_out = 256
    dst = rng.permutation(rows_out)[: 40 * fan].reshape(40, fan)
    got = _gpu_quantize(x, S, rows_out=rows_out, dst=dst, fanout=fan)
    codes, scales, resid, gs = oracle.quantize(x, S=S)
    # scatter the oracle's rows the same way in the test (plain indexing)
    oc = np.zeros((rows_out, 256), np.uint8)
    osc = np.zeros((rows_out, 32), np.uint8)
    ores = np.zeros((rows_out, 8), np.uint16)
    for t in range(40):
        for f in range(fan):
            oc[dst[t, f]] = codes[t]
            osc[dst[t, f]] = scales[t]
            ores[dst[t, f]] = resid[t]
    assert np.array_equal(got["codes"], oc)
    assert np.array_equal(got["scales"], oracle.scale_layout(osc, 512))
    assert np.array_equal(got["resid"], ores)


def test_nonfinite_amax_is_reported():
    x = synth.u16(synth.activations(1))
    got = _gpu_quantize(x, amax_override=float("nan"))
    assert got["status"] == 6  # NVFP4_ERR_NONFINITE


def test_fake_quant_parity():
    ws = [synth.dense_weight(1), synth.dense_weight(1) * 7, torch.cat([synth.activations(1)] * 8)]
    w = torch.stack([t.contiguous() for t in ws])
    wd = w.to(G.DEV)
    w_hat = torch.empty_like(wd)
    gs = G.zeros(3, torch.float32)
    amax = G.zeros(7, torch.float32)  # 2 * 3 + 1 words of scratch
    st = G.zeros(1, torch.int32)
    nv.nvfp4_fake_quant(wd, w_hat, amax, gs_out=gs, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    got = G.u16(w_hat)
    for i in range(3):
        ref, g = oracle.fake_quant(synth.u16(w[i]))
        assert gs[i].item() == np.float32(g)
        assert np.array_equal(got[i], ref), i


def test_fake_quant_equals_rollout_dequant():
    # Eq. 16: the learner's W_hat equals the rollout's dequantized weight,
    # both computed on the GPU: fake_quant(W) == bf16((code*sb)*gs) of
    # prepare_weights(W), with S = all channels giving code*sb directly.
    w = synth.dense_weight(1)[:256]
    wd = w.to(G.DEV)[None]
    w_hat = torch.empty_like(wd)
    nv.nvfp4_fake_quant(wd, w_hat, G.zeros(3, torch.float32))
    K = 512
    S = torch.arange(K, dtype=torch.int32, device=G.DEV)
    codes = G.zeros((1, 256, K // 2), torch.uint8)
    scales = G.zeros(256 * K // 16, torch.uint8)
    gs = G.zeros(1, torch.float32)
    sel = G.zeros((1, 256, K), torch.bfloat16)
    nv.nvfp4_prepare_weights(wd, codes, scales, gs, G.zeros(1, torch.float32), S=S, w_sel=sel)
    deq = (sel.float() * gs).to(torch.bfloat16)  # (code*sb)*gs in FP32, then BF16
    assert torch.equal(deq.view(torch.int16), w_hat.view(torch.int16))


@pytest.mark.parametrize("interleave", [0, 1])
def test_prepare_weights_parity(interleave):
    E, N, K = 3, 256, 512
    ws = torch.stack([synth.dense_weight(1)[:N] * (e + 1) for e in range(E)])
    S = np.array([0, 17, 64, 65, 300, 511, 128, 2], np.int32)
    S.sort()
    wd = ws.to(G.DEV)
    codes = G.zeros((E, N, K // 2), torch.uint8)
    scales = G.zeros(E * N * K // 16, torch.uint8)
    gs = G.zeros(E, torch.float32)
    sel = G.zeros((E, N, len(S)), torch.bfloat16)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_prepare_weights(wd, codes, scales, gs, G.zeros(E, torch.float32),
                             S=torch.tensor(S, device=G.DEV), w_sel=sel, interleave=interleave,
                             dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    if interleave:
        t = np.arange(N) // 256
        i = np.arange(N) % 256
        perm = np.where(i < 128, t * 128 + i, N // 2 + t * 128 + (i - 128))
    else:
        perm = np.arange(N)
    gsel = G.u16(sel)
    for e in range(E):
        we = synth.u16(ws[e])[perm]
        c, s, _, g = oracle.quantize(we)
        assert gs[e].item() == np.float32(g)
        assert np.array_equal(codes[e].cpu().numpy(), c)
        sc = scales.cpu().numpy()[e * N * K // 16:(e + 1) * N * K // 16]
        assert np.array_equal(sc, oracle.scale_layout(s, K))
        unscaled = oracle.dequantize_exact(c, s, 1.0)[:, S]
        assert np.array_equal(gsel[e], oracle.bf16_round(unscaled.astype(np.float32)))


@pytest.mark.parametrize("cfg", [1, 2])
def test_channel_selection_parity(cfg):
    xc = synth.activations(cfg, batch=1)
    xu = synth.u16(xc)
    M, K = xu.shape
    k = synth.CONFIGS[cfg]["k"]
    x = xc.to(G.DEV)
    amax = G.zeros(1, torch.float32)
    nv.nvfp4_amax(x, amax)
    S = G.zeros(k, torch.int32)
    ws = torch.zeros(K, dtype=torch.float64, device=G.DEV)
    nv.nvfp4_rac_select_channels(x, amax, k, S, ws)
    torch.cuda.synchronize()
    ssq = oracle.channel_scores_sq(xu)
    assert np.array_equal(ws.cpu().numpy(), ssq)  # same binary64 sums, same order
    assert np.array_equal(S.cpu().numpy(), oracle.select_channels(ssq, k))
    # the seeded outlier channels are among the selected ones
    assert set(synth.outlier_channels(cfg).tolist()) <= set(S.cpu().tolist())


@pytest.mark.parametrize("limit", [0, 1, 131, 300, 400, -5])
def test_row_limit(limit):
    """With a device-side row bound only the source rows below it are
    quantized (bit-exact against the oracle, which quantizes those rows with
    the whole tensor's amax); codes, scales and residuals of later rows are
    never written (their sentinel bytes survive).  The bound is clamped to
    [0, M]."""
    M, K = 300, 512
    x = _rand_x(M, K, seed=90)
    S = np.array([3, 17, 200, 201, 300, 301, 302, 511], np.int32)
    xd = G.bf16_from_u16(x)
    amax = G.zeros(1, torch.float32)
    nv.nvfp4_amax(xd, amax)
    codes = torch.full((M, K // 2), 0xAB, dtype=torch.uint8, device=G.DEV)
    scales = torch.full((oracle.scale_bytes(M, K),), 0xAB, dtype=torch.uint8, device=G.DEV)
    resid = torch.full((M, len(S)), 7.0, dtype=torch.bfloat16, device=G.DEV)
    lim = torch.tensor([limit], dtype=torch.int32, device=G.DEV)
    Sd = torch.tensor(S, dtype=torch.int32, device=G.DEV)
    nv.nvfp4_quantize(xd, amax, codes, scales, resid=resid, S=Sd, row_limit=lim)
    torch.cuda.synchronize()
    n = min(max(limit, 0), M)
    c_ref, s_ref, r_ref, _ = oracle.quantize(x, S=S)
    got_c, got_s, got_r = codes.cpu().numpy(), scales.cpu().numpy(), G.u16(resid)
    assert np.array_equal(got_c[:n], c_ref[:n]) and (got_c[n:] == 0xAB).all()
    assert np.array_equal(got_r[:n], r_ref[:n])
    assert (resid[n:].float().cpu().numpy() == 7.0).all()
    rows = np.arange(M)
    sc = oracle.scale_rows(got_s, rows, K)
    assert np.array_equal(sc[:n], s_ref[:n]) and (sc[n:] == 0xAB).all()


@pytest.mark.parametrize("k", [3, 16, 40, 100])
def test_channel_selection_ties_and_early_stop(k):
    """Top-k on scores with exact ties: channels 32..63 copy channel 32 (two
    whole blocks of equal columns, so equal binary64 scores) and a wider
    outlier set; k values put the boundary inside the tied group (ties to the
    lower channels) and inside distinct scores, where the radix search stops
    once the k-th key's bucket is kept whole."""
    g = torch.Generator().manual_seed(71 + k)
    M, K = 96, 512
    x = torch.randn((M, K), generator=g)
    x[:, 32:64] = x[:, 32:33] * 3.0
    x[:, 200:208] *= 5.0
    xu = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xd = x.to(torch.bfloat16).to(G.DEV)
    amax = G.zeros(1, torch.float32)
    nv.nvfp4_amax(xd, amax)
    S = G.zeros(k, torch.int32)
    ws = torch.zeros(K, dtype=torch.float64, device=G.DEV)
    nv.nvfp4_rac_select_channels(xd, amax, k, S, ws)
    torch.cuda.synchronize()
    ssq = oracle.channel_scores_sq(xu)
    assert np.array_equal(ws.cpu().numpy(), ssq)
    assert len(set(ssq[32:64].tolist())) == 1  # the tied group
    assert np.array_equal(S.cpu().numpy(), oracle.select_channels(ssq, k))


def test_bounded_wait_times_out_cleanly():
    st = G.zeros(1, torch.int32)
    nv.nvfp4_selftest_wait_timeout(2000, st)  # 2 ms
    torch.cuda.synchronize()
    assert st.item() == 5  # NVFP4_ERR_TIMEOUT
    # the context is still usable afterwards
    x = synth.u16(synth.activations(1))
    assert _gpu_quantize(x)["status"] == 0
