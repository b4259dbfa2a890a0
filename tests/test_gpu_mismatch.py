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
