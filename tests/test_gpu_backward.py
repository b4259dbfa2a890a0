"""GPU parity of the trainer backward (QUADS §3.2 Eq. 13, straight-through
estimator) against the oracle's binary64 derivatives: the transposes
bit-exact, the SwiGLU forward/backward within one BF16 rounding, the combine
backward's routed gradient bit-exact, the grouped weight gradient (an empty
expert included) within FP32 accumulation error from transposed operands and
from the routed rows as stored, the grouped input gradient from the weights as
stored on both GEMM pipelines, and QatMoE(train=True).backward stage by stage
-- each stage against the oracle applied to the GPU's previous stage."""
import numpy as np
import pytest
import torch

import oracle
from tests import _gpu as G

pytestmark = pytest.mark.gpu
TOL = 1e-3
TOL_BF16 = 2.0 ** -8 + 1e-3


@pytest.fixture(scope="module")
def nv():
    import nvfp4_precision_moe_gb300 as m

    m.load(build=True)
    return m


def f64(t):
    return t.detach().float().cpu().double().numpy()


def bf16_of(a):
    return oracle.bf16_to_f32(oracle.bf16_round(np.asarray(a, np.float32))).astype(np.float64)


@pytest.mark.parametrize("shape", [(3, 37, 70), (2, 130, 200), (1, 64, 4096)])
def test_transpose_is_exact(nv, shape):
    g = torch.Generator().manual_seed(3)
    x = torch.randn(shape, generator=g).to(torch.bfloat16).to(G.DEV)
    y = torch.empty((shape[0], shape[2], shape[1]), dtype=torch.bfloat16, device=G.DEV)
    nv.nvfp4_transpose_bf16(x, y)
    torch.cuda.synchronize()
    assert torch.equal(y, x.transpose(1, 2))


def test_fake_quant_transposed(nv):
    g = torch.Generator().manual_seed(17)
    w = (torch.randn((3, 192, 320), generator=g) * 0.02).to(torch.bfloat16).to(G.DEV)
    w[1, 5, 7] = 3.0  # an outlier block
    ref = torch.empty_like(w)
    got = torch.empty_like(w)
    got_t = torch.empty((3, 320, 192), dtype=torch.bfloat16, device=G.DEV)
    gs_ref, gs_got = G.zeros(3, torch.float32), G.zeros(3, torch.float32)
    nv.nvfp4_fake_quant(w, ref, G.zeros(7, torch.float32), gs_out=gs_ref)
    nv.nvfp4_fake_quant_transposed(w, got, got_t, G.zeros(3, torch.float32), gs_out=gs_got)
    torch.cuda.synchronize()
    assert torch.equal(got, ref) and torch.equal(gs_got, gs_ref)
    assert torch.equal(got_t, ref.transpose(1, 2))


def test_swiglu_forward_and_backward(nv):
    g = torch.Generator().manual_seed(5)
    rows, I = 300, 192
    gu = (torch.randn((rows, 2 * I), generator=g) * 3).to(torch.bfloat16)
    dh = torch.randn((rows, I), generator=g).to(torch.bfloat16)
    gud, dhd = gu.to(G.DEV), dh.to(G.DEV)
    h = torch.empty((rows, I), dtype=torch.bfloat16, device=G.DEV)
    dgu = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=G.DEV)
    nv.nvfp4_swiglu(gud, h)
    nv.nvfp4_swiglu_backward(gud, dhd, dgu)
    torch.cuda.synchronize()
    for got, ref in ((f64(h), oracle.swiglu(f64(gu), I)), (f64(dgu), oracle.swiglu_grad(f64(gu), f64(dh)))):
        # one BF16 rounding of a binary32 evaluation: within 2^-8 relative (plus a tiny absolute floor)
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


def _routing(nv, T, E, topk, seed, empty=None):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn((T, E), generator=g)
    if empty is not None:
        logits[:, empty] -= 100.0
    ids, rw = oracle.route_topk(logits.numpy(), topk)
    counts, offs, dst = oracle.route_layout(ids, E)
    return logits, rw, counts, offs, dst


def test_combine_backward(nv):
    T, E, topk, H = 50, 4, 2, 256
    logits, rw, counts, offs, dst = _routing(nv, T, E, topk, 7)
    R = int(offs[-1]) + 128  # rows past offsets[E] too
    g = torch.Generator().manual_seed(8)
    y = torch.randn((R, H), generator=g).to(torch.bfloat16)
    dout = torch.randn((T, H), generator=g)
    dy = torch.full((R, H), 7.0, dtype=torch.bfloat16, device=G.DEV)  # stale values everywhere
    dw = torch.empty((T, topk), dtype=torch.float32, device=G.DEV)
    d = lambda a, dt=None: torch.as_tensor(a).to(G.DEV) if dt is None else torch.as_tensor(a, dtype=dt).to(G.DEV)
    nv.nvfp4_moe_combine_backward(d(dout), d(y), d(dst, torch.int32), d(rw, torch.float32), d(counts, torch.int32),
                                  d(offs, torch.int32), E, dy, dweights=dw)
    torch.cuda.synchronize()
    ref_dy, ref_dw = oracle.combine_grad(f64(dout), f64(y), dst, rw, R)
    live = np.zeros(R, bool)
    live[dst.reshape(-1)] = True
    got = f64(dy)
    rows = np.arange(int(offs[-1]))
    # routed rows: bf16(fp32(w * dout)), exactly; padding rows inside the segments: zero
    want = bf16_of(np.float32(rw)[:, :, None] * np.float32(f64(dout))[:, None, :]).reshape(-1, H)
    assert np.array_equal(got[dst.reshape(-1)], want)
    assert not got[rows[~live[rows]]].any()
    assert np.allclose(f64(dw), ref_dw, rtol=1e-5, atol=1e-5)
    assert np.allclose(got[dst.reshape(-1)], ref_dy[dst.reshape(-1)], rtol=2.0 ** -8, atol=0)


@pytest.mark.parametrize("out_dtype", [0, 1])
def test_grouped_weight_gradient(nv, out_dtype):
    T, E, topk, M, N = 200, 5, 2, 384, 512
    _, _, counts, offs, dst = _routing(nv, T, E, topk, 11, empty=3)
    assert counts[3] == 0
    R = int(offs[-1]) + 128
    g = torch.Generator().manual_seed(12)
    a = torch.randn((R, M), generator=g).to(torch.bfloat16)
    b = torch.randn((R, N), generator=g).to(torch.bfloat16)
    a[int(offs[-1]):] = 1e4  # rows past offsets[E] must not be read
    at, bt = a.t().contiguous().to(G.DEV), b.t().contiguous().to(G.DEV)
    dw = torch.full((E, M, N), 5.0, dtype=torch.float32 if out_dtype == 0 else torch.bfloat16, device=G.DEV)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_bf16_grouped_gemm_wgrad(at, bt, torch.as_tensor(offs, dtype=torch.int32).to(G.DEV), E, dw,
                                     out_dtype=out_dtype, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    ref = oracle.segment_wgrad(f64(a)[:int(offs[-1])], f64(b)[:int(offs[-1])], offs)
    got = f64(dw)
    assert not got[3].any()
    tol = 1e-5 if out_dtype == 0 else TOL_BF16
    assert G.rel_err(got, ref) <= tol


@pytest.mark.parametrize("M,N", [(384, 512), (128, 256), (256, 768)])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_grouped_weight_gradient_from_rows(nv, out_dtype, M, N):
    """The same weight gradient with both operands read as the routed rows
    themselves (MN-major tiles: no transposes); one output tile per expert
    and an odd number of 256-column tiles included."""
    T, E, topk = 200, 5, 2
    _, _, counts, offs, dst = _routing(nv, T, E, topk, 21, empty=1)
    assert counts[1] == 0
    R = int(offs[-1]) + 128
    g = torch.Generator().manual_seed(22)
    a = torch.randn((R, M), generator=g).to(torch.bfloat16)
    b = torch.randn((R, N), generator=g).to(torch.bfloat16)
    a[int(offs[-1]):] = 1e4  # rows past offsets[E] must not be read
    dw = torch.full((E, M, N), 5.0, dtype=torch.float32 if out_dtype == 0 else torch.bfloat16, device=G.DEV)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_bf16_grouped_gemm_wgrad_rows(a.to(G.DEV), b.to(G.DEV), torch.as_tensor(offs, dtype=torch.int32).to(G.DEV),
                                          E, dw, out_dtype=out_dtype, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    ref = oracle.segment_wgrad(f64(a)[:int(offs[-1])], f64(b)[:int(offs[-1])], offs)
    got = f64(dw)
    assert not got[1].any()
    tol = 1e-5 if out_dtype == 0 else TOL_BF16
    assert G.rel_err(got, ref) <= tol


@pytest.mark.parametrize("pipe", ["single", "pair"])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_grouped_input_gradient(nv, pipe, out_dtype):
    """dX = W_hat^T dY with W_hat read as stored ([E, K, N], MN-major tiles):
    ragged experts, an empty one, three 256-column tiles and K over several
    64-element slices; rows past each expert's tokens are zero and give zeros."""
    E, K, N = 4, 320, 768
    counts = np.array([70, 0, 300, 129])
    offsets = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    rows = int(offsets[-1])
    rng = np.random.default_rng(23)
    dy = np.zeros((rows, K), np.float32)
    for e in range(E):
        dy[offsets[e]:offsets[e] + counts[e]] = rng.standard_normal((counts[e], K))
    dyu = oracle.bf16_round(dy)
    wu = oracle.bf16_round((rng.standard_normal((E, K, N)) * 0.05).astype(np.float32))
    y = G.zeros((rows, N), torch.float32 if out_dtype == 0 else torch.bfloat16)
    y.fill_(7.0)
    st = G.zeros(1, torch.int32)
    prev = nv.nvfp4_gemm_pipeline({"single": 1, "pair": 2}[pipe])
    try:
        nv.nvfp4_bf16_grouped_gemm_dgrad(G.bf16_from_u16(dyu), G.bf16_from_u16(wu), torch.tensor(offsets, device=G.DEV),
                                         E, N, K, y, out_dtype=out_dtype, dev_status=st)
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_gemm_pipeline(prev)
    G.status_ok(st)
    got = y.float().cpu().numpy()
    tol = TOL if out_dtype == 0 else TOL_BF16
    for e in range(E):
        r0, n = int(offsets[e]), int(counts[e])
        if n:
            ref = oracle.bf16_gemm(dyu[r0:r0 + n], np.ascontiguousarray(wu[e].T))
            assert G.rel_err(got[r0:r0 + n], ref) <= tol, e
        assert not got[r0 + n:int(offsets[e + 1])].any(), e


@pytest.mark.parametrize("pipe", ["single", "pair"])
def test_input_gradient_with_fused_swiglu_backward(nv, pipe):
    """The input-gradient GEMM with the SwiGLU backward in its epilogue equals,
    bit for bit, the unfused chain on the GPU (the product stored in BF16, then
    nvfp4_swiglu_backward), and that chain matches the oracle's SwiGLU
    gradient of the stored product."""
    E, K, I = 3, 192, 512
    counts = np.array([100, 0, 260])
    offsets = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    rows = int(offsets[-1])
    rng = np.random.default_rng(24)
    dy = np.zeros((rows, K), np.float32)
    gu = np.zeros((rows, 2 * I), np.float32)
    for e in range(E):
        dy[offsets[e]:offsets[e] + counts[e]] = rng.standard_normal((counts[e], K))
        gu[offsets[e]:offsets[e] + counts[e]] = rng.standard_normal((counts[e], 2 * I)) * 2
    dyd, gud = G.bf16_from_u16(oracle.bf16_round(dy)), G.bf16_from_u16(oracle.bf16_round(gu))
    wd = G.bf16_from_u16(oracle.bf16_round((rng.standard_normal((E, K, I)) * 0.05).astype(np.float32)))
    offs = torch.tensor(offsets, device=G.DEV)
    dh = G.zeros((rows, I), torch.bfloat16)
    dgu_ref = G.zeros((rows, 2 * I), torch.bfloat16)
    dgu = torch.full((rows, 2 * I), 3.0, dtype=torch.bfloat16, device=G.DEV)
    st = G.zeros(1, torch.int32)
    prev = nv.nvfp4_gemm_pipeline({"single": 1, "pair": 2}[pipe])
    try:
        nv.nvfp4_bf16_grouped_gemm_dgrad(dyd, wd, offs, E, I, K, dh, out_dtype=1, dev_status=st)
        nv.nvfp4_swiglu_backward(gud, dh, dgu_ref)
        nv.nvfp4_bf16_grouped_gemm_dgrad(dyd, wd, offs, E, I, K, dgu, out_dtype=1, epilogue=nv.NVFP4_EPI_SWIGLU_BWD,
                                         gu=gud, dev_status=st)
        torch.cuda.synchronize()
    finally:
        nv.nvfp4_gemm_pipeline(prev)
    G.status_ok(st)
    live = np.concatenate([np.arange(offsets[e], offsets[e] + counts[e]) for e in range(E)])
    li = torch.from_numpy(live).to(G.DEV)
    assert torch.equal(dgu[li], dgu_ref[li])
    ref = oracle.swiglu_grad(f64(gud[li]), f64(dh[li]))
    got = f64(dgu[li])
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


def test_qat_layer_empty_batch(nv):
    """The training layer on a batch of no tokens: an empty output and input
    gradient, and zero weight gradients for every expert."""
    from tests.test_oracle_mismatch import small_moe

    x, logits, w13, wd = small_moe()
    dev = lambda a: torch.as_tensor(a).to(G.DEV)
    E, N13, H = w13.shape
    layer = nv.QatMoE(dev(w13), dev(wd), 2, x.shape[0], fake=True, train=True)
    out = layer.forward(dev(x)[:0], dev(logits)[:0])
    dx, dw13, dwd, dweights = layer.backward(torch.zeros((0, H), dtype=torch.float32, device=G.DEV))
    torch.cuda.synchronize()
    G.status_ok(layer.dev_status)
    assert out.shape == (0, H) and dx.shape == (0, H) and dweights.shape == (0, 2)
    assert not dw13.any().item() and not dwd.any().item()


def test_qat_layer_backward_stage_by_stage(nv):
    from tests.test_oracle_mismatch import small_moe

    x, logits, w13, wd = small_moe()
    logits[:, 3] -= 100.0  # one expert without tokens: its weight gradients are zero
    T, topk = x.shape[0], 2
    E, N13, H = w13.shape
    I = N13 // 2
    dev = lambda a: torch.as_tensor(a).to(G.DEV)
    layer = nv.QatMoE(dev(w13), dev(wd), topk, T, fake=True, train=True)
    out = layer.forward(dev(x), dev(logits))
    g = torch.Generator().manual_seed(13)
    dout = torch.randn((T, H), generator=g)
    dx, dw13, dwd, dweights = layer.backward(dout.to(G.DEV))
    torch.cuda.synchronize()
    G.status_ok(layer.dev_status)
    r = layer.route
    offs = r.offsets.cpu().numpy()
    dst = r.dst_row.cpu().numpy()[:T]
    rw = r.weights.cpu().numpy()[:T].astype(np.float64)
    Rl = int(offs[-1])
    xr, gu, h, y = f64(layer.xr)[:Rl], f64(layer.gu)[:Rl], f64(layer.h)[:Rl], f64(layer.y)[:Rl]

    def per_expert(a, w_of):  # the BF16 rows of expert e times w_of(e) [N, K]^T: oracle.bf16_gemm
        n = w_of(0).shape[0]
        o = np.zeros((Rl, n))
        for e in range(E):
            r0, r1 = int(offs[e]), int(offs[e + 1])
            if r1 > r0:
                o[r0:r1] = oracle.bf16_gemm(G.u16(a[r0:r1]), G.u16(w_of(e)))
        return o

    # forward with saved pre-activations: the BF16 pre-activations and h, which the gate_up GEMM's
    # epilogue computes from its FP32 products (as the inference-mode forward does)
    gu64 = per_expert(layer.xr, lambda e: layer.w13_hat[e])
    assert G.rel_err(gu, gu64) <= TOL_BF16
    assert G.rel_err(h, oracle.swiglu(gu64, I)) <= TOL_BF16
    assert G.rel_err(f64(out), oracle.combine(y, dst.astype(np.int32), rw)) <= 1e-5
    # backward
    dy = f64(layer.dy)[:Rl]
    ref_dy, ref_dw = oracle.combine_grad(f64(dout), y, dst, rw, Rl)
    assert G.rel_err(dy, ref_dy) <= 2.0 ** -8
    assert np.allclose(f64(dweights), ref_dw, rtol=1e-5, atol=1e-5)
    assert G.rel_err(f64(dwd), oracle.segment_wgrad(dy, h, offs)) <= 1e-5
    # d(gate|up): the SwiGLU gradient of dh = dY . Wd_hat, which the GEMM's epilogue rounds to BF16
    # (the oracle's product may round to the neighbouring BF16 value: one more 2^-8)
    dgu = f64(layer.dgu)[:Rl]
    ref_dgu = oracle.swiglu_grad(gu, bf16_of(per_expert(layer.dy, lambda e: layer.wd_hat[e].t().contiguous())))
    assert G.rel_err(dgu, ref_dgu) <= 2.0 ** -7 + 1e-3
    dxr = f64(layer.dxr)[:Rl]
    assert G.rel_err(dxr, per_expert(layer.dgu, lambda e: layer.w13_hat[e].t().contiguous())) <= TOL_BF16
    assert G.rel_err(f64(dw13), oracle.segment_wgrad(dgu, xr, offs)) <= 1e-5
    assert not f64(dw13)[3].any() and not f64(dwd)[3].any()
    assert G.rel_err(f64(dx), oracle.combine(dxr, dst.astype(np.int32), np.ones(dst.shape))) <= 1e-5
