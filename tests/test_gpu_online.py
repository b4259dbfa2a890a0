"""Online channel selection (QUADS §3.3 Eq. 23-24 on every forward pass):
nvfp4_rac_select_channels_online against the oracle's scores (its sums are
taken in a different, faster order, so scores agree to ~1e-6 and S must be a
valid top-k: ties that close may go either way), the row bound of routed
activations, the weight-column gather against nvfp4_prepare_weights and the
oracle, and the rollout layer in online mode against the oracle chain."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _chains
from tests import _gpu as G
from tests.test_oracle_quant import _rand_x

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_precision_moe_gb300 as m

    m.load(build=True)
    return m


def _select(nv, x_u16, k, offsets=None, E=0):
    x = G.bf16_from_u16(x_u16)
    M, K = x_u16.shape
    amax = G.zeros(1, torch.float32)
    rows = M if offsets is None else int(offsets[-1])
    nv.nvfp4_amax(x[:rows], amax)
    S = G.zeros(k, torch.int32)
    ws = G.zeros(257 * K, torch.float64)
    off = None if offsets is None else torch.tensor(offsets, dtype=torch.int32, device=G.DEV)
    nv.nvfp4_rac_select_channels_online(x, amax, k, S, ws, offsets=off, E=E)
    torch.cuda.synchronize()
    return S.cpu().numpy(), ws[:K].cpu().numpy()


@pytest.mark.parametrize("M,K,k", [(300, 512, 64), (2048, 4096, 128), (77, 1536, 16)])
def test_online_scores_and_selection(nv, M, K, k):
    x = _rand_x(M, K, seed=K + k)
    S, ssq = _select(nv, x, k)
    ref = oracle.channel_scores_sq(x)
    assert np.allclose(ssq, ref, rtol=1e-6, atol=0)
    assert _chains.valid_topk(S, ref, k)


def test_online_selection_reads_routed_rows_only(nv):
    M, K, k, live = 512, 512, 32, 301
    x = _rand_x(M, K, seed=9)
    x[live:] = oracle.bf16_round(np.full((M - live, K), 3.0e4, np.float32))  # stale rows
    S, ssq = _select(nv, x, k, offsets=[0, 128, live], E=2)
    ref = oracle.channel_scores_sq(x[:live])
    assert np.allclose(ssq, ref, rtol=1e-6, atol=0)
    assert _chains.valid_topk(S, ref, k)


@pytest.mark.parametrize("interleave,E,N,K,k", [(0, 3, 512, 768, 48), (1, 3, 512, 768, 48), (0, 2, 384, 960, 160),
                                                (1, 2, 256, 4096, 136)])
def test_gather_equals_the_weight_pack(nv, interleave, E, N, K, k):
    g = torch.Generator().manual_seed(21)
    w = (torch.randn((E, N, K), generator=g) * 0.02).to(torch.bfloat16)
    wd = w.to(G.DEV)
    rng = np.random.default_rng(4)
    Sa = np.sort(rng.choice(K, k, replace=False)).astype(np.int32)
    Sb = np.sort(rng.choice(K, k, replace=False)).astype(np.int32)

    def pack(S):
        codes = G.zeros((E, N, K // 2), torch.uint8)
        scales = G.zeros(E * nv.scale_bytes(N, K), torch.uint8)
        sel = G.zeros((E, N, k), torch.bfloat16)
        nv.nvfp4_prepare_weights(wd, codes, scales, G.zeros(E, torch.float32), G.zeros(E, torch.float32),
                                 S=torch.tensor(S, device=G.DEV), w_sel=sel, interleave=interleave)
        return codes, scales, sel

    codes, scales, _ = pack(Sa)
    _, _, want = pack(Sb)
    got = G.zeros((E, N, k), torch.bfloat16)
    st = G.zeros(1, torch.int32)
    nv.nvfp4_gather_selected_weights(codes, scales, E, N, K, torch.tensor(Sb, device=G.DEV), got, dev_status=st)
    torch.cuda.synchronize()
    G.status_ok(st)
    assert torch.equal(got, want)
    if not interleave:  # rows in source order: the oracle's unscaled dequantized weights on Sb
        for e in range(E):
            c, s, _, _ = oracle.quantize(synth.u16(w[e]))
            ref = oracle.bf16_round(oracle.dequantize_exact(c, s, 1.0)[:, Sb].astype(np.float32))
            assert np.array_equal(G.u16(got[e]), ref)


@pytest.mark.parametrize("interleave,E,N,K,k", [(0, 3, 512, 768, 48), (1, 2, 256, 4096, 136), (0, 2, 384, 960, 160)])
def test_gather_from_the_channel_major_pack(nv, interleave, E, N, K, k):
    """nvfp4_transpose_weight_pack + nvfp4_gather_selected_weights_t give the
    same w_sel as the gather from the pack itself, bit for bit; the
    channel-major copy holds every code and block scale of the pack."""
    g = torch.Generator().manual_seed(31)
    w = (torch.randn((E, N, K), generator=g) * 0.02).to(torch.bfloat16).to(G.DEV)
    codes = G.zeros((E, N, K // 2), torch.uint8)
    scales = G.zeros(E * nv.scale_bytes(N, K), torch.uint8)
    nv.nvfp4_prepare_weights(w, codes, scales, G.zeros(E, torch.float32), G.zeros(E, torch.float32),
                             interleave=interleave)
    rng = np.random.default_rng(32)
    S = torch.tensor(np.sort(rng.choice(K, k, replace=False)).astype(np.int32), device=G.DEV)
    codes_t = G.zeros((E, K, N // 2), torch.uint8)
    scales_t = G.zeros((E, K // 16, N), torch.uint8)
    nv.nvfp4_transpose_weight_pack(codes, scales, E, N, K, codes_t, scales_t)
    want = G.zeros((E, N, k), torch.bfloat16)
    got = torch.full((E, N, k), 7.0, dtype=torch.bfloat16, device=G.DEV)
    nv.nvfp4_gather_selected_weights(codes, scales, E, N, K, S, want)
    nv.nvfp4_gather_selected_weights_t(codes_t, scales_t, E, N, K, S, got)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    # the copy itself: every code and block scale, by the layouts' definitions
    c = codes.cpu().numpy()
    lo, hi = c & 15, c >> 4
    full = np.empty((E, N, K), np.uint8)
    full[:, :, 0::2], full[:, :, 1::2] = lo, hi
    ct = codes_t.cpu().numpy()
    tfull = np.empty((E, K, N), np.uint8)
    tfull[:, :, 0::2], tfull[:, :, 1::2] = ct & 15, ct >> 4
    assert np.array_equal(tfull, full.transpose(0, 2, 1))
    sc = scales.cpu().numpy().reshape(E, -1)
    st = scales_t.cpu().numpy()
    for e in range(E):
        assert np.array_equal(st[e].T, oracle.scale_rows(sc[e], np.arange(N), K))


def test_rollout_layer_online(nv):
    from tests.test_oracle_mismatch import small_moe

    x, logits, w13, wd = small_moe()
    T, topk, k13, kd = x.shape[0], 2, 32, 16
    xu, l = synth.u16(x), logits.numpy()
    dev = lambda a: torch.as_tensor(a).to(G.DEV)
    S0 = lambda k: torch.arange(k, dtype=torch.int32, device=G.DEV)  # a first set only fixes k
    layer = nv.RolloutMoE(dev(w13), dev(wd), S0(k13), S0(kd), topk, T, online=True)
    assert layer.LAUNCHES == 17
    y = layer.forward(dev(x), dev(logits)).cpu().double().numpy()
    G.status_ok(layer.dev_status)
    S13, Sd = layer.S13.cpu().numpy(), layer.Sd.cpu().numpy()
    ref, _, _, sc13, scd = _chains.rollout_online(xu, l, w13, wd, topk, k13, kd, S13=S13, Sd=Sd)
    assert _chains.valid_topk(S13, sc13, k13) and _chains.valid_topk(Sd, scd, kd)
    y_qat = _chains.trainer(xu, l, w13, wd, topk, fake=True)
    d_ref = np.linalg.norm(ref - y_qat)
    assert np.linalg.norm(y - ref) <= 0.05 * d_ref
    assert d_ref < np.linalg.norm(_chains.rollout(xu, l, w13, wd, topk) - y_qat)
    # a second batch re-selects: the sets follow the data
    x2 = x.clone()
    x2[:, :k13] = 0
    layer.forward(dev(x2), dev(logits))
    torch.cuda.synchronize()
    assert _chains.valid_topk(layer.S13.cpu().numpy(), oracle.channel_scores_sq(synth.u16(x2)), k13)
