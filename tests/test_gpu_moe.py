"""GPU parity of the MoE glue and of whole layers against the CPU oracle.

Routing ids, counts, segment offsets and routed rows are integers and must be
bit-exact; router weights and the combine are FP32 against binary64.  Whole
layers are checked stage by stage on the workloads' shapes, and end to end on
a reduced token count with a tolerance that allows an occasional 1-code
difference in the re-quantized intermediate (the GPU's BF16 h and the
oracle's may differ by one BF16 ulp, which can move an element across an E2M1
rounding boundary).
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


def _route_gpu(logits, topk):
    T, E = logits.shape
    ld = logits.to(G.DEV)
    ids = G.zeros((T, topk), torch.int32)
    w = G.zeros((T, topk), torch.float32)
    counts = G.zeros(E, torch.int32)
    offs = G.zeros(E + 1, torch.int32)
    dst = G.zeros((T, topk), torch.int32)
    nv.nvfp4_route_topk(ld, topk, ids, w, counts, offs, dst)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy(), counts.cpu().numpy(), offs.cpu().numpy(), dst.cpu().numpy()


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_routing_parity_full_size(cfg):
    c = synth.CONFIGS[cfg]
    logits = synth.router_logits(cfg)
    ids, w, counts, offs, dst = _route_gpu(logits, c["topk"])
    rid, rw = oracle.route_topk(logits.numpy(), c["topk"])
    assert np.array_equal(ids, rid)
    assert np.allclose(w, rw, rtol=1e-5, atol=0)
    rc, ro, rd = oracle.route_layout(rid, c["E"])
    assert np.array_equal(counts, rc)
    assert np.array_equal(offs, ro)
    assert np.array_equal(dst, rd)


def test_routing_ties_and_small_shapes():
    logits = torch.zeros((5, 40))  # all ties: experts 0..topk-1, in order
    logits[3, 39] = 1.0
    ids, w, counts, offs, dst = _route_gpu(logits, 6)
    rid, rw = oracle.route_topk(logits.numpy(), 6)
    assert np.array_equal(ids, rid)
    assert ids[0].tolist() == [0, 1, 2, 3, 4, 5] and ids[3, 0] == 39
    assert np.allclose(w, rw, rtol=1e-6)
    rc, ro, rd = oracle.route_layout(rid, 40)
    assert np.array_equal(offs, ro) and np.array_equal(dst, rd)


@pytest.mark.parametrize("T,E,topk,skew", [(300, 200, 8, 0.0), (257, 600, 5, 0.0), (12000, 64, 6, 8.0),
                                             (16384, 128, 8, 8.0), (20000, 128, 8, 8.0)])
def test_routing_wide_and_skewed(T, E, topk, skew):
    """Expert counts that take the 8- and 32-key-per-lane selections, a slot
    count that is not a multiple of 4, and routing so skewed that every id of
    a thread's run of tokens matches (every token prefers the same topk
    experts), with runs of 128 ids (kept as a match mask) and of 160 (counted,
    then read again)."""
    g = torch.Generator().manual_seed(T + E)
    logits = torch.randn((T, E), generator=g)
    logits[:, :topk] += skew
    ids, w, counts, offs, dst = _route_gpu(logits, topk)
    rid, rw = oracle.route_topk(logits.numpy(), topk)
    assert np.array_equal(ids, rid)
    assert np.allclose(w, rw, rtol=1e-5, atol=0)
    rc, ro, rd = oracle.route_layout(rid, E)
    assert np.array_equal(counts, rc) and np.array_equal(offs, ro) and np.array_equal(dst, rd)


@pytest.mark.parametrize("ydt", [torch.float32, torch.bfloat16])
def test_combine_parity(ydt):
    T, topk, E, H = 300, 8, 64, 512
    logits = torch.randn((T, E), generator=torch.Generator().manual_seed(3))
    ids, w, counts, offs, dst = _route_gpu(logits, topk)
    rows = int(offs[-1])
    y = torch.randn((rows, H), generator=torch.Generator().manual_seed(4)).to(ydt)
    out = G.zeros((T, H), torch.float32)
    nv.nvfp4_moe_combine(y.to(G.DEV), torch.from_numpy(dst).to(G.DEV), torch.from_numpy(w).to(G.DEV), topk, out)
    torch.cuda.synchronize()
    ref = oracle.combine(y.float().numpy().astype(np.float64), dst.astype(np.int32), w.astype(np.float64))
    assert G.rel_err(out.cpu().numpy(), ref) <= 1e-5


def _layer_inputs(cfg, T):
    c = synth.CONFIGS[cfg]
    x = synth.activations(cfg)[:T].contiguous()
    logits = synth.router_logits(cfg)[:T].contiguous()
    w13 = torch.stack([synth.expert_weight(cfg, e, "w13") for e in range(c["E"])])
    wd = torch.stack([synth.expert_weight(cfg, e, "down") for e in range(c["E"])])
    return c, x, logits, w13, wd


def _seeded_channels(K, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.sort(torch.randperm(K, generator=g)[:k]).values.to(torch.int32).numpy()


def test_rollout_layer_empty_batch():
    """A batch of no tokens leaves nothing to route: the forward returns an
    empty output without error, and the next batch is unaffected (its output
    equals a fresh layer's)."""
    cfg, T = 3, 64
    c, x, logits, w13, wd = _layer_inputs(cfg, T)
    S13, Sd = _seeded_channels(c["H"], c["k"], 5), _seeded_channels(c["I"], c["k"], 6)
    mk = lambda: nv.RolloutMoE(w13.to(G.DEV), wd.to(G.DEV), torch.from_numpy(S13).to(G.DEV),
                               torch.from_numpy(Sd).to(G.DEV), c["topk"], T)
    layer = mk()
    xd, ld = x.to(G.DEV), logits.to(G.DEV)
    out = layer.forward(xd[:0], ld[:0])
    torch.cuda.synchronize()
    G.status_ok(layer.dev_status)
    assert out.shape == (0, c["H"])
    got = layer.forward(xd, ld).clone()
    ref = mk().forward(xd, ld)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


@pytest.mark.parametrize("T", [1, 64])
def test_rollout_layer_end_to_end_reduced(T):
    cfg = 3
    c, x, logits, w13, wd = _layer_inputs(cfg, T)
    E, H, I, topk, k = c["E"], c["H"], c["I"], c["topk"], c["k"]
    S13 = oracle.select_channels(oracle.channel_scores_sq(synth.u16(synth.activations(cfg, batch=1)[:256])), k)
    Sd = _seeded_channels(I, k, 77)
    layer = nv.RolloutMoE(w13.to(G.DEV), wd.to(G.DEV), torch.from_numpy(S13).to(G.DEV),
                          torch.from_numpy(Sd).to(G.DEV), topk, T)
    out = layer.forward(x.to(G.DEV), logits.to(G.DEV)).cpu().numpy()
    G.status_ok(layer.dev_status)
    # ---- oracle chain
    ids, rw = oracle.route_topk(logits.numpy(), topk)
    counts, offs, dst = oracle.route_layout(ids, E)
    xu = synth.u16(x)
    ca, sa, ra, ga = oracle.quantize(xu, S=S13)
    xq = oracle.dequantize_exact(ca, sa, ga)
    R = int(offs[-1])
    h_ref = np.zeros((R, I))
    for e in range(E):
        toks = np.nonzero((ids == e).any(1))[0]
        if toks.size == 0:
            continue
        cw, sw, _, g = oracle.quantize(synth.u16(w13[e]))
        y = oracle.rac_gemm(xq[toks], oracle.dequantize_exact(cw, sw, g), ra[toks], S13, ga)
        rows = dst[toks, np.argmax(ids[toks] == e, 1)]
        h_ref[rows] = oracle.swiglu(y, I)
    # stage check: the GPU's h on every routed row
    h_gpu = layer.h[:R].float().cpu().numpy()
    live = np.zeros(R, bool)
    live[dst.reshape(-1)] = True
    assert G.rel_err(h_gpu[live], h_ref[live]) <= 2.0 ** -8 + TOL
    assert (h_gpu[~live] == 0).all()
    # continue the oracle chain from its own BF16 h
    hu = oracle.bf16_round(h_ref.astype(np.float32))
    ch, sh, rh, gh = oracle.quantize(hu, S=Sd)
    hq = oracle.dequantize_exact(ch, sh, gh)
    y_ref = np.zeros((R, H))
    for e in range(E):
        r0, r1 = offs[e], offs[e] + counts[e]
        if r1 == r0:
            continue
        cw, sw, _, g = oracle.quantize(synth.u16(wd[e]))
        y_ref[r0:r1] = oracle.rac_gemm(hq[r0:r1], oracle.dequantize_exact(cw, sw, g), rh[r0:r1], Sd, gh)
    y_ref_b = oracle.bf16_to_f32(oracle.bf16_round(y_ref.astype(np.float32))).astype(np.float64)
    out_ref = oracle.combine(y_ref_b, dst.astype(np.int32), rw)
    err = G.rel_err(out, out_ref)
    assert err <= 2e-2, err
