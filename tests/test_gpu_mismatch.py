"""The layer-mismatch diagnostic (QUADS §3.1 Eq. 11, Fig. 4b) through the
library: the trainer layer (QatMoE, W16A16 or W4A16) and the rollout layer
(RolloutMoE, W4A4 with or without RAC) on the same small MoE layer, and
nvfp4_mismatch_norm on their outputs.  Each dY matches the oracle chains'
dY within 5% (the layers' own GEMM errors are ~1e-3 of ||Y||), and the order
no QAT > W4A16 QAT > W4A16 QAT + RAC holds on the GPU as in the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests import _chains
from tests import _gpu as G
from tests.test_oracle_mismatch import small_moe

pytestmark = pytest.mark.gpu


def test_mismatch_norm_matches_the_oracle_chains():
    import nvfp4_precision_moe_gb300 as nv

    nv.load(build=True)
    x, logits, w13, wd = small_moe()
    T, H = x.shape
    topk = 2
    xu = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    S13 = oracle.select_channels(oracle.channel_scores_sq(xu), 32)
    Sd = np.arange(0, 256, 16, dtype=np.int32)
    xd, ld = x.to(G.DEV), logits.to(G.DEV)
    w13d, wdd = w13.to(G.DEV), wd.to(G.DEV)
    s13d, sdd = torch.from_numpy(S13).to(G.DEV), torch.from_numpy(Sd).to(G.DEV)
    outs = {}
    for name, layer in [("w16a16", nv.QatMoE(w13d, wdd, topk, T, fake=False)),
                        ("w4a16", nv.QatMoE(w13d, wdd, topk, T, fake=True)),
                        ("w4a4", nv.RolloutMoE(w13d, wdd, None, None, topk, T)),
                        ("w4a4_rac", nv.RolloutMoE(w13d, wdd, s13d, sdd, topk, T))]:
        outs[name] = layer.forward(xd, ld).clone()
        G.status_ok(layer.dev_status)
    acc = torch.zeros(2, dtype=torch.float64, device=G.DEV)
    pairs = {"no_qat": ("w4a4", "w16a16"), "qat": ("w4a4", "w4a16"), "qat_rac": ("w4a4_rac", "w4a16")}
    gpu = {k: nv.nvfp4_mismatch_norm(outs[a], outs[b], acc) for k, (a, b) in pairs.items()}
    # the norm itself against numpy on the same two buffers
    a, b = outs["w4a4"].cpu().double().numpy(), outs["w16a16"].cpu().double().numpy()
    assert gpu["no_qat"][0] == pytest.approx(np.linalg.norm(a - b), rel=1e-12)
    assert gpu["no_qat"][1] == pytest.approx(np.linalg.norm(b), rel=1e-12)
    # the oracle chains
    l = logits.numpy()
    ref = {"w16a16": _chains.trainer(xu, l, w13, wd, topk, fake=False),
           "w4a16": _chains.trainer(xu, l, w13, wd, topk, fake=True),
           "w4a4": _chains.rollout(xu, l, w13, wd, topk),
           "w4a4_rac": _chains.rollout(xu, l, w13, wd, topk, S13, Sd)}
    for k, (p, q) in pairs.items():
        d_ref = np.linalg.norm(ref[p] - ref[q])
        assert abs(gpu[k][0] - d_ref) <= 0.05 * d_ref, (k, gpu[k][0], d_ref)
    assert gpu["no_qat"][0] > gpu["qat"][0] > gpu["qat_rac"][0] > 0


def test_symmetric_qat_on_the_gpu():
    """Symmetric W4A4 QAT (QUADS §4.3.1 Fig. 7) through QatMoE(sym=True): it
    matches the oracle's symmetric chain, and with eta = 0 it nearly equals
    the library's own W4A4 rollout (the two differ only where the BF16 and
    FP4 GEMMs' FP32 sums round h differently) -- far closer than the W4A16
    trainer.  With the ~2^-10 synthetic drift of Eq. 8 on the rollout's input
    the symmetric mismatch is many times the drift's effect on the BF16 layer."""
    import synth
    import nvfp4_precision_moe_gb300 as nv

    nv.load(build=True)
    x, logits, w13, wd = small_moe()
    T = x.shape[0]
    topk = 2
    xe = synth.engine_drift(x, 2.0 ** -10, 1)
    ld, w13d, wdd = logits.to(G.DEV), w13.to(G.DEV), wd.to(G.DEV)
    sym = nv.QatMoE(w13d, wdd, topk, T, fake=True, sym=True)
    asym = nv.QatMoE(w13d, wdd, topk, T, fake=True)
    bf16 = nv.QatMoE(w13d, wdd, topk, T, fake=False)
    roll = nv.RolloutMoE(w13d, wdd, None, None, topk, T)
    run = lambda lay, xx: lay.forward(xx.to(G.DEV), ld).clone()
    y_sym, y_asym, y_roll = run(sym, x), run(asym, x), run(roll, x)
    y16, y16e, y_rolle = run(bf16, x), run(bf16, xe), run(roll, xe)
    for lay in (sym, asym, bf16, roll):
        G.status_ok(lay.dev_status)
    n = lambda t: float(t.double().norm())
    ny = n(y_roll)
    ref = _chains.trainer(synth.u16(x), logits.numpy(), w13, wd, topk, fake=True, sym=True)
    d_ref = np.linalg.norm(y_sym.cpu().double().numpy() - ref)
    assert d_ref <= 1e-2 * np.linalg.norm(ref), d_ref
    d_sym0, d_asym = n(y_roll - y_sym), n(y_roll - y_asym)
    assert d_sym0 <= 1e-2 * ny and d_sym0 < 0.2 * d_asym, (d_sym0, d_asym)
    d_eta, d_sym = n(y16e - y16), n(y_rolle - y_sym)
    assert d_sym > 5 * d_eta > 0, (d_sym, d_eta)
    print("sym-vs-oracle %.3g  sym-vs-rollout %.3g  asym %.3g  eta %.3g  sym(eta) %.3g  |Y| %.3g"
          % (d_ref, d_sym0, d_asym, d_eta, d_sym, ny))
