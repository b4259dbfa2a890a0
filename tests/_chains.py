"""Oracle chains of one MoE layer forward, for the mismatch tests (QUADS §3.1
Eq. 11, §3.2 Eq. 12, §3.3 Eq. 21, §4.3.1 Fig. 7): the trainer (weights BF16 or
fake-quantized; activations BF16, or fake-quantized too for the symmetric W4A4
QAT ablation) and the rollout (W4A4, optionally with the RAC residual).
Rounding points follow the library's layers: BF16 routed inputs, binary64
GEMM sums, BF16 h and y, binary64 combine."""
import numpy as np

import oracle
import synth


def route(logits, E, topk):
    ids, rw = oracle.route_topk(logits, topk)
    counts, offs, dst = oracle.route_layout(ids, E)
    return ids, rw, counts, offs, dst


def _combine(y_rows, dst, rw):
    yb = oracle.bf16_to_f32(oracle.bf16_round(y_rows.astype(np.float32))).astype(np.float64)
    return oracle.combine(yb, dst.astype(np.int32), rw)


def trainer(x_u16, logits, w13, wd, topk, fake, sym=False):
    """W16A16 (fake=False), W4A16 (fake=True) or, with sym=True, symmetric W4A4
    QAT (x and h fake-quantized as well, one tensor scale each) trainer forward
    -> out [T, H] binary64."""
    E, N13, H = w13.shape
    I = N13 // 2
    ids, rw, counts, offs, dst = route(logits, E, topk)
    R = int(offs[-1])
    if sym:
        x_u16, _ = oracle.fake_quant(x_u16)
    xf = oracle.bf16_to_f32(x_u16).astype(np.float64)
    h = np.zeros((R, I))
    yd = np.zeros((R, H))
    wq13, wqd = [], []
    for e in range(E):
        a, b = synth.u16(w13[e]), synth.u16(wd[e])
        if fake:
            a, _ = oracle.fake_quant(a)
            b, _ = oracle.fake_quant(b)
        wq13.append(oracle.bf16_to_f32(a).astype(np.float64))
        wqd.append(oracle.bf16_to_f32(b).astype(np.float64))
    for e in range(E):
        toks = np.nonzero((ids == e).any(1))[0]
        if toks.size:
            rows = dst[toks, np.argmax(ids[toks] == e, 1)]
            h[rows] = oracle.swiglu(xf[toks] @ wq13[e].T, I)
    hu = oracle.bf16_round(h.astype(np.float32))
    if sym:
        hu, _ = oracle.fake_quant(hu)
    hb = oracle.bf16_to_f32(hu).astype(np.float64)
    for e in range(E):
        r0, r1 = offs[e], offs[e] + counts[e]
        if r1 > r0:
            yd[r0:r1] = hb[r0:r1] @ wqd[e].T
    return _combine(yd, dst, rw)


def rollout(x_u16, logits, w13, wd, topk, S13=None, Sd=None, fp4_resid=False):
    """W4A4 rollout forward, with the RAC residual on S13 / Sd when given (BF16,
    or with fp4_resid the literal Eq. 21 second NVFP4 pass) -> out [T, H]."""
    E, N13, H = w13.shape
    I = N13 // 2
    ids, rw, counts, offs, dst = route(logits, E, topk)
    R = int(offs[-1])
    ca, sa, ra, ga = oracle.quantize(x_u16, S=S13)
    if fp4_resid and S13 is not None:
        ra, _ = oracle.requant_residual(ra, ga)
    xq = oracle.dequantize_exact(ca, sa, ga)
    h = np.zeros((R, I))
    for e in range(E):
        toks = np.nonzero((ids == e).any(1))[0]
        if toks.size:
            cw, sw, _, gw = oracle.quantize(synth.u16(w13[e]))
            y = oracle.rac_gemm(xq[toks], oracle.dequantize_exact(cw, sw, gw), ra[toks] if S13 is not None else None,
                                S13, ga)
            rows = dst[toks, np.argmax(ids[toks] == e, 1)]
            h[rows] = oracle.swiglu(y, I)
    hu = oracle.bf16_round(h.astype(np.float32))
    ch, sh, rh, gh = oracle.quantize(hu, S=Sd)
    if fp4_resid and Sd is not None:
        rh, _ = oracle.requant_residual(rh, gh)
    hq = oracle.dequantize_exact(ch, sh, gh)
    yd = np.zeros((R, H))
    for e in range(E):
        r0, r1 = offs[e], offs[e] + counts[e]
        if r1 > r0:
            cw, sw, _, gw = oracle.quantize(synth.u16(wd[e]))
            yd[r0:r1] = oracle.rac_gemm(hq[r0:r1], oracle.dequantize_exact(cw, sw, gw),
                                        rh[r0:r1] if Sd is not None else None, Sd, gh)
    return _combine(yd, dst, rw)


def inputs(cfg, T):
    c = synth.CONFIGS[cfg]
    x = synth.activations(cfg)[:T].contiguous()
    logits = synth.router_logits(cfg)[:T].contiguous()
    import torch

    w13 = torch.stack([synth.expert_weight(cfg, e, "w13") for e in range(c["E"])])
    wd = torch.stack([synth.expert_weight(cfg, e, "down") for e in range(c["E"])])
    return c, x, logits, w13, wd


def valid_topk(S, scores, k, rel=1e-6):
    """S is a top-k of `scores` (ties within `rel` either way), sorted, distinct."""
    S = np.asarray(S)
    if len(S) != k or np.any(np.diff(S) <= 0):
        return False
    t = np.sort(scores)[::-1][k - 1]
    sel = np.zeros(len(scores), bool)
    sel[S] = True
    return bool(np.all(scores[sel] >= t * (1 - rel)) and np.all(scores[~sel] <= t * (1 + rel)))


def rollout_online(x_u16, logits, w13, wd, topk, k13, kd, S13=None, Sd=None):
    """W4A4 + RAC rollout forward with Eq. 23-24 applied to this batch: S13 from
    the scores of x, Sd from the scores of the routed rows of h (padding rows
    included: they are zero).  S13 / Sd, when given (e.g. the library's own
    choice), replace the oracle's choice downstream; the oracle's scores are
    returned either way -> (out, S13, Sd, scores13, scoresd)."""
    E, N13, H = w13.shape
    I = N13 // 2
    sc13 = oracle.channel_scores_sq(x_u16)
    S13 = oracle.select_channels(sc13, k13) if S13 is None else np.asarray(S13, np.int32)
    ids, rw, counts, offs, dst = route(logits, E, topk)
    R = int(offs[-1])
    ca, sa, ra, ga = oracle.quantize(x_u16, S=S13)
    xq = oracle.dequantize_exact(ca, sa, ga)
    h = np.zeros((R, I))
    for e in range(E):
        toks = np.nonzero((ids == e).any(1))[0]
        if toks.size:
            cw, sw, _, gw = oracle.quantize(synth.u16(w13[e]))
            y = oracle.rac_gemm(xq[toks], oracle.dequantize_exact(cw, sw, gw), ra[toks], S13, ga)
            rows = dst[toks, np.argmax(ids[toks] == e, 1)]
            h[rows] = oracle.swiglu(y, I)
    hu = oracle.bf16_round(h.astype(np.float32))
    scd = oracle.channel_scores_sq(hu)
    Sd = oracle.select_channels(scd, kd) if Sd is None else np.asarray(Sd, np.int32)
    ch, sh, rh, gh = oracle.quantize(hu, S=Sd)
    hq = oracle.dequantize_exact(ch, sh, gh)
    yd = np.zeros((R, H))
    for e in range(E):
        r0, r1 = offs[e], offs[e] + counts[e]
        if r1 > r0:
            cw, sw, _, gw = oracle.quantize(synth.u16(wd[e]))
            yd[r0:r1] = oracle.rac_gemm(hq[r0:r1], oracle.dequantize_exact(cw, sw, gw), rh[r0:r1], Sd, gh)
    return _combine(yd, dst, rw), S13, Sd, sc13, scd
