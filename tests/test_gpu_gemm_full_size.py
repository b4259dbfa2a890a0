"""The grouped GEMMs with FP32 output at the MoE workloads' full launch shapes,
against the oracle at a maximum relative error of 1e-3, on both GEMM
pipelines.  The error of an element is |y - ref| / max(|ref|, rms of the
sampled reference row), so that cancellation near zero is measured against
the row's scale.

* W4A4 + RAC (QUADS §3.3 Eq. 21) at the prefill workload (16384 tokens top-8
  over 128 experts with Zipf routing, hidden 4096, intermediate 1536, k = 128)
  and the decode workload (2048 tokens top-8 over 64 experts, hidden 2048,
  intermediate 768, k = 64).  After one layer forward, both projections run
  again with FP32 output -- gate_up without the SwiGLU epilogue, so its
  columns come out in the weight pack's gate/up tile order -- on the layer's
  own routed NVFP4 activations (x, and the quantized h of the forward).  Every
  expert's segment is sampled at its first and last rows and at its rows 127,
  128 and 129; columns at the first, second, 128th, 129th and last column of
  every 256-column tile, plus random ones.  The reference quantizes the same
  BF16 inputs (x, or the GPU's h) and the expert's weight rows behind the
  sampled columns with the oracle (the weight's tensor scale from its whole
  amax), then takes the binary64 W4A4 + RAC product.  Padding rows are zero.
* BF16 grouped GEMM of the asymmetric-QAT forward (QUADS §3.2 Eq. 12) at the
  QAT workload (4096 tokens top-8 over 128 experts, W13 3072 x 4096, down
  4096 x 1536): the routed x and the GPU's h against oracle.bf16_gemm with
  the fake-quantized weights, on the same row and column samples.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu as G

pytestmark = pytest.mark.gpu
TOL = 1e-3
PIPES = {"single": 1, "pair": 2}


def _rows(offs, counts, e):
    r0, r1 = int(offs[e]), int(offs[e]) + int(counts[e])
    return np.array(sorted({r for r in (r0, r0 + 127, r0 + 128, r0 + 129, r1 - 1) if r0 <= r < r1}), np.int64)


def _cols(N, rng, extra=32):
    c = set()
    for t in range(0, N, 256):
        c |= {t, t + 1, t + 127, t + 128, t + 255}
    c |= set(rng.integers(0, N, extra).tolist())
    return np.array(sorted(x for x in c if x < N), np.int64)


def _gate_up_source_rows(j, I):
    """Source row of W13 ([gate; up], 2I rows) behind output column j of the
    interleaved pack: 256-column tiles of 128 gate then 128 up rows."""
    t, i = j // 256, j % 256
    return np.where(i < 128, t * 128 + i, I + t * 128 + (i - 128))


def _run_pipes(fn):
    import nvfp4_precision_moe_gb300 as nv

    out = {}
    try:
        for name, which in PIPES.items():
            nv.nvfp4_gemm_pipeline(which)
            out[name] = fn()
            torch.cuda.synchronize()
    finally:
        nv.nvfp4_gemm_pipeline(0)
    return out


@pytest.fixture(scope="module", params=[5, 3], ids=["moe_prefill", "moe_decode"])
def moe(request):
    import nvfp4_precision_moe_gb300 as nv
    import bench

    cfg = request.param
    nv.load(build=True)
    dev = torch.device(G.DEV)
    c, layer, x, logits, _ = bench.build_workload(dev, cfg)
    layer.forward(x, logits)
    torch.cuda.synchronize()
    G.status_ok(layer.dev_status)
    st = G.zeros(1, torch.int32)

    def gemms():
        xa, ha, W13, Wd = layer.xa, layer.ha, layer.w13, layer.wd
        y13 = torch.full((layer.rows_cap, W13.N), float("nan"), dtype=torch.float32, device=dev)
        yd = torch.full((layer.rows_cap, Wd.N), float("nan"), dtype=torch.float32, device=dev)
        r = layer.route
        nv.nvfp4_w4a4_rac_grouped_gemm(xa.codes, xa.scales, xa.resid, xa.gs, W13.codes, W13.scales, W13.gs,
                                       W13.sel, W13.k, r.offsets, layer.E, W13.N, W13.K, y13, dev_status=st)
        nv.nvfp4_w4a4_rac_grouped_gemm(ha.codes, ha.scales, ha.resid, ha.gs, Wd.codes, Wd.scales, Wd.gs,
                                       Wd.sel, Wd.k, r.offsets, layer.E, Wd.N, Wd.K, yd, dev_status=st)
        return y13, yd

    ys = _run_pipes(gemms)
    G.status_ok(st)
    return cfg, c, layer, x, ys


def test_w4a4_rac_gemm_fp32_every_expert(moe):
    cfg, c, layer, x, ys = moe
    T, H, E, I, topk = c["T"], c["H"], c["E"], c["I"], c["topk"]
    r = layer.route
    counts, offs, dst = r.counts.cpu().numpy(), r.offsets.cpu().numpy(), r.dst_row.cpu().numpy()
    S13, Sd = layer.S13.cpu().numpy(), layer.Sd.cpu().numpy()
    xu = G.u16(x)
    h_all = G.u16(layer.h)
    gs_x = oracle.tensor_scale(oracle.amax(xu))
    gs_h = oracle.tensor_scale(oracle.amax(h_all))
    assert float(layer.xa.gs.item()) == gs_x and float(layer.ha.gs.item()) == gs_h
    tok_of_row = np.full(layer.rows_cap, -1, np.int64)
    tok_of_row[dst.reshape(-1)] = np.repeat(np.arange(T), topk)
    rng = np.random.default_rng(100 + cfg)
    y13 = {k: v[0] for k, v in ys.items()}
    yd = {k: v[1] for k, v in ys.items()}
    worst = {k: 0.0 for k in ys}
    checked = 0
    for e in range(E):
        rows = _rows(offs, counts, e)
        if rows.size == 0:
            continue
        tk = tok_of_row[rows]
        assert (tk >= 0).all()
        ridx = torch.from_numpy(rows).to(G.DEV)
        # gate_up: sampled columns of the interleaved pack
        w13 = synth.u16(synth.expert_weight(cfg, e, "w13"))
        g13 = oracle.tensor_scale(oracle.amax(w13))
        J = _cols(2 * I, rng)
        cw, sw, _, _ = oracle.quantize(w13[_gate_up_source_rows(J, I)], gs=g13)
        ca, sa, ra, _ = oracle.quantize(xu[tk], gs=gs_x, S=S13)
        ref = oracle.rac_gemm(oracle.dequantize_exact(ca, sa, gs_x), oracle.dequantize_exact(cw, sw, g13),
                              ra, S13, gs_x)
        jidx = torch.from_numpy(J).to(G.DEV)
        for name in ys:
            got = y13[name][ridx][:, jidx].cpu().numpy()
            err = G.rel_err(got, ref)
            worst[name] = max(worst[name], err)
            assert err <= TOL, (name, "gate_up", e, err)
        # down: sampled columns, the GPU's h re-quantized by the oracle
        wd = synth.u16(synth.expert_weight(cfg, e, "down"))
        gd = oracle.tensor_scale(oracle.amax(wd))
        J = _cols(H, rng)
        cw, sw, _, _ = oracle.quantize(wd[J], gs=gd)
        ch, sh, rh, _ = oracle.quantize(h_all[rows], gs=gs_h, S=Sd)
        ref = oracle.rac_gemm(oracle.dequantize_exact(ch, sh, gs_h), oracle.dequantize_exact(cw, sw, gd),
                              rh, Sd, gs_h)
        jidx = torch.from_numpy(J).to(G.DEV)
        for name in ys:
            got = yd[name][ridx][:, jidx].cpu().numpy()
            err = G.rel_err(got, ref)
            worst[name] = max(worst[name], err)
            assert err <= TOL, (name, "down", e, err)
        checked += 1
    assert checked == int((counts > 0).sum())
    print("max rel err", worst)
    # padding rows of the segments (zero codes, scales and residual) give zeros
    live = np.zeros(layer.rows_cap, bool)
    live[dst.reshape(-1)] = True
    pad = np.nonzero(~live[: int(offs[-1])])[0]
    if pad.size:
        pidx = torch.from_numpy(rng.choice(pad, min(512, pad.size), replace=False)).to(G.DEV)
        for name in ys:
            assert not y13[name][pidx].any().item() and not yd[name][pidx].any().item(), name


@pytest.fixture(scope="module")
def qat():
    import nvfp4_precision_moe_gb300 as nv
    import bench

    nv.load(build=True)
    dev = torch.device(G.DEV)
    c, w13, wd, x, logits = bench.build_qat_workload(dev)
    L = nv.QatMoE(w13, wd, c["topk"], c["T"])
    L.forward(x, logits)
    torch.cuda.synchronize()
    G.status_ok(L.dev_status)
    st = G.zeros(1, torch.int32)
    E, H, I = c["E"], c["H"], c["I"]

    def gemms():
        y13 = torch.full((L.rows_cap, 2 * I), float("nan"), dtype=torch.float32, device=dev)
        yd = torch.full((L.rows_cap, H), float("nan"), dtype=torch.float32, device=dev)
        nv.nvfp4_bf16_grouped_gemm(L.xr, L.w13_hat, L.route.offsets, E, 2 * I, H, y13, dev_status=st)
        nv.nvfp4_bf16_grouped_gemm(L.h, L.wd_hat, L.route.offsets, E, H, I, yd, dev_status=st)
        return y13, yd

    ys = _run_pipes(gemms)
    G.status_ok(st)
    return c, L, ys


def test_bf16_grouped_gemm_fp32_every_expert(qat):
    c, L, ys = qat
    E, H, I = c["E"], c["H"], c["I"]
    counts, offs = L.route.counts.cpu().numpy(), L.route.offsets.cpu().numpy()
    rng = np.random.default_rng(44)
    worst = {k: 0.0 for k in ys}
    for e in range(E):
        rows = _rows(offs, counts, e)
        if rows.size == 0:
            continue
        ridx = torch.from_numpy(rows).to(G.DEV)
        for proj, a, w, N, which in (("gate_up", L.xr, L.w13_hat, 2 * I, 0), ("down", L.h, L.wd_hat, H, 1)):
            J = _cols(N, rng)
            ref = oracle.bf16_gemm(G.u16(a[ridx]), G.u16(w[e][torch.from_numpy(J).to(G.DEV)]))
            jidx = torch.from_numpy(J).to(G.DEV)
            for name in ys:
                got = ys[name][which][ridx][:, jidx].cpu().numpy()
                err = G.rel_err(got, ref)
                worst[name] = max(worst[name], err)
                assert err <= TOL, (name, proj, e, err)
    print("max rel err", worst)
