"""GPU parity of the literal second-pass residual of QUADS §3.3 Eq. 21
(nvfp4_rac_requant_residual) against the oracle's requant_residual: bit-exact
in place, rows past offsets[E] untouched and kept out of the amax, zero and
non-finite residuals, and the rollout layer with resid_fp4 against the
oracle's rollout chain."""
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


def _resid_of(nv, x_u16, S):
    """The GPU quantizer's residual of x on S (bit-exact with the oracle's)."""
    M, K = x_u16.shape
    x = G.bf16_from_u16(x_u16)
    amax, gs = G.zeros(1, torch.float32), G.zeros(1, torch.float32)
    nv.nvfp4_amax(x, amax)
    resid = G.zeros((M, len(S)), torch.bfloat16)
    nv.nvfp4_quantize(x, amax, G.zeros((M, K // 2), torch.uint8),
                      G.zeros(oracle.scale_bytes(M, K), torch.uint8), resid=resid,
                      S=torch.tensor(S, dtype=torch.int32, device=G.DEV), gs_out=gs)
    return resid, float(gs.item())


@pytest.mark.parametrize("M,K,k", [(300, 512, 64), (37, 256, 16), (1024, 1024, 128)])
def test_requant_is_bit_exact(nv, M, K, k):
    x = _rand_x(M, K, seed=M + k)
    S = oracle.select_channels(oracle.channel_scores_sq(x), k)
    resid, gs_a = _resid_of(nv, x, S)
    _, _, r_ref, g_ref = oracle.quantize(x, S=S)
    assert gs_a == g_ref and np.array_equal(G.u16(resid), r_ref)
    want, gs_r = oracle.requant_residual(r_ref, gs_a)
    ws, gs_out, st = G.zeros(1, torch.float32), G.zeros(1, torch.float32), G.zeros(1, torch.int32)
    nv.nvfp4_rac_requant_residual(resid, ws, gs_out=gs_out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(G.u16(resid), want)
    assert float(gs_out.item()) * gs_a == gs_r
    assert float(ws.item()) == oracle.amax(r_ref)


def test_rows_past_offsets_are_untouched_and_unread(nv):
    rows_cap, k, live = 512, 32, 300
    rng = np.random.default_rng(11)
    r = oracle.bf16_round(rng.standard_normal((rows_cap, k)).astype(np.float32))
    r[live:] = oracle.bf16_round(np.full((rows_cap - live, k), 1000.0, np.float32))  # stale rows
    resid = G.bf16_from_u16(r)
    offsets = torch.tensor([0, 128, live], dtype=torch.int32, device=G.DEV)
    ws = G.zeros(1, torch.float32)
    nv.nvfp4_rac_requant_residual(resid, ws, offsets=offsets, E=2)
    torch.cuda.synchronize()
    got = G.u16(resid)
    want, _ = oracle.requant_residual(r[:live], 1.0)
    assert np.array_equal(got[:live], want)
    assert np.array_equal(got[live:], r[live:])
    assert float(ws.item()) == oracle.amax(r[:live])


def test_zero_and_nonfinite_residuals(nv):
    z = G.zeros((256, 16), torch.bfloat16)
    ws, st = G.zeros(1, torch.float32), G.zeros(1, torch.int32)
    nv.nvfp4_rac_requant_residual(z, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0 and not z.any().item()
    bad = torch.ones((128, 16), dtype=torch.bfloat16, device=G.DEV)
    bad[5, 3] = float("inf")
    before = bad.clone()
    nv.nvfp4_rac_requant_residual(bad, ws, dev_status=st)
    torch.cuda.synchronize()
    assert nv.STATUS[st.item()] == "NVFP4_ERR_NONFINITE"
    assert torch.equal(bad, before)


def test_rollout_layer_with_the_second_pass(nv):
    from tests.test_oracle_mismatch import small_moe

    x, logits, w13, wd = small_moe()
    T, topk = x.shape[0], 2
    xu, l = synth.u16(x), logits.numpy()
    S13 = oracle.select_channels(oracle.channel_scores_sq(xu), 32)
    Sd = np.arange(0, 256, 16, dtype=np.int32)
    dev = lambda a: torch.as_tensor(a).to(G.DEV)
    layer = nv.RolloutMoE(dev(w13), dev(wd), dev(S13), dev(Sd), topk, T, resid_fp4=True)
    assert layer.LAUNCHES == 13
    y = layer.forward(dev(x), dev(logits)).cpu().double().numpy()
    G.status_ok(layer.dev_status)
    ref = _chains.rollout(xu, l, w13, wd, topk, S13, Sd, fp4_resid=True)
    y_qat = _chains.trainer(xu, l, w13, wd, topk, fake=True)
    # the layer against the oracle chain, measured against the chain's own mismatch
    d_ref = np.linalg.norm(ref - y_qat)
    assert np.linalg.norm(y - ref) <= 0.05 * d_ref
    assert abs(np.linalg.norm(y - y_qat) - d_ref) <= 0.05 * d_ref
