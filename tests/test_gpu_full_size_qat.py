"""Parity at the QAT workload's full size, in the launch configuration bench.py
times (128 experts, W13 3072 x 4096 and down 4096 x 1536 fake-quantized every
step, 4096 tokens top-8; QUADS §3.2 Eq. 12-13):

* fake-quant: three experts' W13_hat and W_down_hat bit-exact;
* the forward (fused SwiGLU epilogue): sampled routed rows of h and y of those
  experts within 2^-8 + 1e-3 of the oracle on the GPU's own previous stage, and
  sampled tokens of the output within 1e-5 of the weighted sum of the GPU's rows;
* the training step (QatMoE(train=True).backward): the three experts' whole
  weight gradients dW_down and dW_13 within 1e-5 (FP32 accumulation), sampled
  rows of dh and d(x routed) within 2^-8 + 1e-3, sampled tokens of dx within
  1e-5 -- each against the oracle applied to the GPU's previous stage.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import _gpu as G

pytestmark = pytest.mark.gpu
TOL_BF16 = 2.0 ** -8 + 1e-3


def f64(t):
    return t.detach().float().cpu().double().numpy()


@pytest.fixture(scope="module")
def qat():
    import nvfp4_precision_moe_gb300 as nv
    import bench

    nv.load(build=True)
    dev = torch.device(G.DEV)
    c, w13, wd, x, logits = bench.build_qat_workload(dev)
    T, topk = c["T"], c["topk"]
    plain = nv.QatMoE(w13, wd, topk, T)
    out = plain.forward(x, logits).clone()
    train = nv.QatMoE(w13, wd, topk, T, train=True)
    train.forward(x, logits)
    g = torch.Generator(device=dev)
    g.manual_seed(45)
    dout = torch.randn((T, c["H"]), device=dev, generator=g)
    dx, dw13, dwd, _ = train.backward(dout)
    torch.cuda.synchronize()
    G.status_ok(plain.dev_status)
    G.status_ok(train.dev_status)
    counts = plain.route.counts.cpu().numpy()
    experts = sorted({0, c["E"] - 1, int(np.argmax(counts))})
    return dict(c=c, w13=w13, wd=wd, x=x, plain=plain, out=out, train=train, dout=dout, dx=dx.clone(),
                dw13=dw13, dwd=dwd, experts=experts)


def _rows(layer, e, rng, n=6):
    offs, counts = layer.route.offsets.cpu().numpy(), layer.route.counts.cpu().numpy()
    r0, r1 = int(offs[e]), int(offs[e]) + int(counts[e])
    return np.array(sorted({r0, r1 - 1} | set(rng.integers(r0, r1, n).tolist())))


def test_fake_quant_bit_exact(qat):
    for e in qat["experts"]:
        for w, w_hat in ((qat["w13"], qat["plain"].w13_hat), (qat["wd"], qat["plain"].wd_hat)):
            ref, _ = oracle.fake_quant(G.u16(w[e]))
            assert np.array_equal(G.u16(w_hat[e]), ref), e


def test_training_fake_quant_matches_the_forward(qat):
    P, L = qat["plain"], qat["train"]
    assert torch.equal(L.w13_hat, P.w13_hat) and torch.equal(L.wd_hat, P.wd_hat)


def test_forward_sampled_rows(qat):
    L, I = qat["plain"], qat["c"]["I"]
    rng = np.random.default_rng(40)
    xr, h, y = L.xr, L.h, L.y
    for e in qat["experts"]:
        rr = torch.from_numpy(_rows(L, e, rng)).to(G.DEV)
        ref_h = oracle.swiglu(oracle.bf16_gemm(G.u16(xr[rr]), G.u16(L.w13_hat[e])), I)
        assert G.rel_err(f64(h[rr]), ref_h) <= TOL_BF16, e
        assert G.rel_err(f64(y[rr]), oracle.bf16_gemm(G.u16(h[rr]), G.u16(L.wd_hat[e]))) <= TOL_BF16, e
    T, topk = qat["c"]["T"], qat["c"]["topk"]
    toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    dst = L.route.dst_row.cpu().numpy()[toks]
    w = L.route.weights.cpu().numpy()[toks].astype(np.float64)
    yrows = f64(y[torch.from_numpy(dst.reshape(-1)).to(G.DEV)])
    ref = oracle.combine(yrows, np.arange(len(toks) * topk, dtype=np.int32).reshape(len(toks), topk), w)
    assert G.rel_err(f64(qat["out"][torch.from_numpy(toks).to(G.DEV)]), ref) <= 1e-5


def test_training_step_gradients(qat):
    L = qat["train"]
    offs = L.route.offsets.cpu().numpy()
    rng = np.random.default_rng(41)
    for e in qat["experts"]:
        r0, r1 = int(offs[e]), int(offs[e + 1])  # the whole segment, padding rows included (zero)
        seg = torch.arange(r0, r1, device=G.DEV)
        dy, h, dgu, xr = f64(L.dy[seg]), f64(L.h[seg]), f64(L.dgu[seg]), f64(L.xr[seg])
        one = np.array([0, r1 - r0])
        assert G.rel_err(f64(qat["dwd"][e]), oracle.segment_wgrad(dy, h, one)[0]) <= 1e-5, e
        assert G.rel_err(f64(qat["dw13"][e]), oracle.segment_wgrad(dgu, xr, one)[0]) <= 1e-5, e
        rr = torch.from_numpy(_rows(L, e, rng)).to(G.DEV)
        # d(gate|up) = the SwiGLU gradient of dh = dY . Wd_hat (rounded to BF16 in the GEMM's epilogue;
        # the oracle's product may round to the neighbouring BF16 value), dx = d(gate|up) . W13_hat
        dh_ref = oracle.bf16_gemm(G.u16(L.dy[rr]), G.u16(L.wd_hat[e].t().contiguous()))
        dh_ref = oracle.bf16_to_f32(oracle.bf16_round(dh_ref.astype(np.float32))).astype(np.float64)
        ref_dgu = oracle.swiglu_grad(f64(L.gu[rr]), dh_ref)
        assert G.rel_err(f64(L.dgu[rr]), ref_dgu) <= 2.0 ** -7 + 1e-3, e
        assert G.rel_err(f64(L.dxr[rr]), oracle.bf16_gemm(G.u16(L.dgu[rr]), G.u16(L.w13_hat[e].t().contiguous()))) <= TOL_BF16, e
    T, topk = qat["c"]["T"], qat["c"]["topk"]
    toks = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    dst = L.route.dst_row.cpu().numpy()[toks]
    rows = f64(L.dxr[torch.from_numpy(dst.reshape(-1)).to(G.DEV)])
    ref = oracle.combine(rows, np.arange(len(toks) * topk, dtype=np.int32).reshape(len(toks), topk),
                         np.ones((len(toks), topk)))
    assert G.rel_err(f64(qat["dx"][torch.from_numpy(toks).to(G.DEV)]), ref) <= 1e-5
