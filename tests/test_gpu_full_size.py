"""Parity at full size, in the launch configuration bench.py times: the
prefill workload (16384 tokens, hidden 4096, 128 experts top-8 with Zipf
routing, intermediate 1536, k = 128 on both projections) and the decode
workload (2048 tokens, hidden 2048, 64 experts top-8, intermediate 768,
k = 64) through RolloutMoE.forward, checked stage by stage on sampled rows.  Each stage's GPU
output is compared with the oracle applied to the previous stage's GPU output:

* quantize x: gs exact; codes, block scales (read back through the tiled
  layout of the header) and residual bit-exact for sampled tokens at all 8 of
  their routed rows; padding rows of the routed codes are zero.
* gate_up W4A4 + RAC GEMM + SwiGLU (QUADS §3.3 Eq. 21): sampled rows of the
  first, last, largest and smallest experts -- each segment's first and last
  rows included -- within 2^-8 + 1e-3 of the oracle; the fused amax of h
  equals max|h| over all rows; padding rows of h are zero.
* quantize h: gs exact; codes, scales and residual bit-exact on the sampled rows.
* down GEMM: the same rows, within 2^-8 + 1e-3 (BF16 output).
* combine: sampled tokens, within 1e-5 of the weighted sum of the GPU's rows.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _gpu as G

pytestmark = pytest.mark.gpu
TOL_BF16 = 2.0 ** -8 + 1e-3


def _scale_rows(sw, rows, K):
    """Canonical [len(rows), K/16] block scales of `rows` read back from the
    scale layout of the header (through the oracle's layout)."""
    return oracle.scale_rows(sw, rows, K)


@pytest.fixture(scope="module", params=[5, 3], ids=["moe_prefill", "moe_decode"])
def layer_run(request):
    import nvfp4_precision_moe_gb300 as nv
    import bench

    nv.load(build=True)
    dev = torch.device(G.DEV)
    c, layer, x, logits, _ = bench.build_workload(dev, request.param)
    out = layer.forward(x, logits)
    torch.cuda.synchronize()
    G.status_ok(layer.dev_status)
    return request.param, c, layer, x, out


def test_full_size_stage_parity(layer_run):
    cfg, c, layer, x, out = layer_run
    T, H, E, I, topk, k = c["T"], c["H"], c["E"], c["I"], c["topk"], c["k"]
    r = layer.route
    ids = r.ids.cpu().numpy()
    w = r.weights.cpu().numpy()
    counts = r.counts.cpu().numpy()
    offs = r.offsets.cpu().numpy()
    dst = r.dst_row.cpu().numpy()
    S13 = layer.S13.cpu().numpy()
    Sd = layer.Sd.cpu().numpy()
    xu = G.u16(x)
    rng = np.random.default_rng(2024)

    # ---- quantize x (dispatched to the routed rows)
    gs_x = oracle.tensor_scale(oracle.amax(xu))
    assert float(layer.xa.gs.item()) == gs_x
    toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 62, replace=False)]))
    qc, qs, qr, _ = oracle.quantize(xu[toks], gs=gs_x, S=S13)
    xa_scales = layer.xa.scales.cpu().numpy()
    rows = dst[toks].reshape(-1)
    gc = layer.xa.codes[torch.from_numpy(rows).to(G.DEV)].cpu().numpy()
    gr = G.u16(layer.xa.resid[torch.from_numpy(rows).to(G.DEV)])
    gsc = _scale_rows(xa_scales, rows, H)
    rep = np.repeat(np.arange(len(toks)), topk)
    assert np.array_equal(gc, qc[rep])
    assert np.array_equal(gsc, qs[rep])
    assert np.array_equal(gr, qr[rep])
    live = np.zeros(layer.rows_cap, bool)
    live[dst.reshape(-1)] = True
    pad = np.nonzero(~live[: int(offs[-1])])[0]
    pad_s = rng.choice(pad, min(256, pad.size), replace=False)
    assert not layer.xa.codes[torch.from_numpy(pad_s).to(G.DEV)].any().item()

    # ---- sampled rows of four experts: first and last rows of each segment
    nz = np.nonzero(counts)[0]
    experts = sorted({0, E - 1, int(np.argmax(counts)), int(nz[np.argmin(counts[nz])])})
    tok_of_row = np.full(layer.rows_cap, -1, np.int64)
    tok_of_row[dst.reshape(-1)] = np.repeat(np.arange(T), topk)
    samples = []
    for e in experts:
        r0, r1 = int(offs[e]), int(offs[e]) + int(counts[e])
        if r1 == r0:
            continue
        pick = {r0, r1 - 1, min(r0 + 127, r1 - 1), min(r0 + 128, r1 - 1)}
        pick |= set(rng.integers(r0, r1, 4).tolist())
        samples.append((e, np.array(sorted(pick))))

    # ---- gate_up GEMM + SwiGLU, and the fused amax of h
    h_all = G.u16(layer.h)
    assert float(layer.ha.amax.item()) == oracle.amax(h_all)
    hpad = pad_s[pad_s < layer.rows_cap]
    assert not h_all[hpad].any()
    for e, rr in samples:
        tk = tok_of_row[rr]
        assert (tk >= 0).all()
        ca, sa, ra, _ = oracle.quantize(xu[tk], gs=gs_x, S=S13)
        cw, sw, _, gw = oracle.quantize(synth.u16(synth.expert_weight(cfg, e, "w13")))
        y = oracle.rac_gemm(oracle.dequantize_exact(ca, sa, gs_x), oracle.dequantize_exact(cw, sw, gw), ra, S13, gs_x)
        ref = oracle.swiglu(y, I)
        assert G.rel_err(oracle.bf16_to_f32(h_all[rr]), ref) <= TOL_BF16, e

    # ---- quantize h
    gs_h = oracle.tensor_scale(oracle.amax(h_all))
    assert float(layer.ha.gs.item()) == gs_h
    ha_scales = layer.ha.scales.cpu().numpy()
    all_rows = np.concatenate([rr for _, rr in samples])
    hc, hs, hr, _ = oracle.quantize(h_all[all_rows], gs=gs_h, S=Sd)
    idx = torch.from_numpy(all_rows).to(G.DEV)
    assert np.array_equal(layer.ha.codes[idx].cpu().numpy(), hc)
    assert np.array_equal(_scale_rows(ha_scales, all_rows, I), hs)
    assert np.array_equal(G.u16(layer.ha.resid[idx]), hr)

    # ---- down GEMM
    y_all = layer.y
    for e, rr in samples:
        ch, sh, rh, _ = oracle.quantize(h_all[rr], gs=gs_h, S=Sd)
        cw, sw, _, gw = oracle.quantize(synth.u16(synth.expert_weight(cfg, e, "down")))
        ref = oracle.rac_gemm(oracle.dequantize_exact(ch, sh, gs_h), oracle.dequantize_exact(cw, sw, gw), rh, Sd, gs_h)
        got = y_all[torch.from_numpy(rr).to(G.DEV)].float().cpu().numpy()
        assert G.rel_err(got, ref) <= TOL_BF16, e

    # ---- combine
    ct = toks[:16]
    yrows = y_all[torch.from_numpy(dst[ct].reshape(-1)).to(G.DEV)].float().cpu().numpy().astype(np.float64)
    ref = oracle.combine(yrows, np.arange(len(ct) * topk, dtype=np.int32).reshape(len(ct), topk),
                         w[ct].astype(np.float64))
    assert G.rel_err(out[torch.from_numpy(ct).to(G.DEV)].cpu().numpy(), ref) <= 1e-5
