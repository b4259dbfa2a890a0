"""Pin of the oracle's layer-mismatch chains (QUADS §3.1 Eq. 11, Fig. 4b): on a
small MoE layer whose activations carry outlier channels, the forward mismatch
dY = ||Y_infer - Y_train|| against a W4A4 rollout must shrink when the trainer
fake-quantizes its weights (W4A16 QAT removes the weight term of Eq. 11, §3.2)
and shrink again when the rollout adds the RAC residual on the selected
channels (Eq. 20-22 remove part of the activation term).  A sign error in the
correction, a dropped fake-quant or a transposed operand breaks the order."""
import numpy as np
import torch

import oracle
import synth
from tests import _chains


def small_moe(seed=0, T=64, E=4, H=256, I=256, n_out=4):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, H), generator=g, dtype=torch.float64)
    out_ch = torch.randperm(H, generator=g)[:n_out]
    x[:, out_ch] *= 40
    logits = torch.randn((T, E), generator=g)
    w13 = (torch.randn((E, 2 * I, H), generator=g) * 0.02).to(torch.bfloat16)
    wd = (torch.randn((E, H, I), generator=g) * 0.02).to(torch.bfloat16)
    return x.to(torch.bfloat16), logits, w13, wd


def test_mismatch_order_no_qat_qat_rac():
    x, logits, w13, wd = small_moe()
    xu = x.contiguous().view(torch.int16).numpy().view(np.uint16)
    S13 = oracle.select_channels(oracle.channel_scores_sq(xu), 32)
    Sd = np.arange(0, 256, 16, dtype=np.int32)
    l = logits.numpy()
    y16 = _chains.trainer(xu, l, w13, wd, 2, fake=False)
    y416 = _chains.trainer(xu, l, w13, wd, 2, fake=True)
    y44 = _chains.rollout(xu, l, w13, wd, 2)
    y44r = _chains.rollout(xu, l, w13, wd, 2, S13, Sd)
    d_noqat = np.linalg.norm(y44 - y16)
    d_qat = np.linalg.norm(y44 - y416)
    d_rac = np.linalg.norm(y44r - y416)
    assert d_noqat > d_qat > d_rac > 0


def test_symmetric_qat_aligns_only_without_engine_drift():
    """Symmetric W4A4 QAT (QUADS §4.3.1 Fig. 7): the learner fake-quantizes x
    and h with the rollout's own NVFP4 recipe (§3.2 Eq. 15-16 for the shared
    QDQ path), so with identical inputs (eta = 0, Eq. 8) its forward IS the
    W4A4 rollout forward -- every quantized operand is exact in BF16 and both
    chains sum in binary64.  With a drift eta of ~2^-10 relative on the
    rollout's input, the two sides quantize different activations (Table 1)
    and the E2M1 decision boundaries amplify it: the symmetric mismatch is
    many times the drift's own effect on the BF16 layer."""
    x, logits, w13, wd = small_moe()
    xu, l = synth.u16(x), logits.numpy()
    y_sym = _chains.trainer(xu, l, w13, wd, 2, fake=True, sym=True)
    y44 = _chains.rollout(xu, l, w13, wd, 2)
    assert np.array_equal(y_sym, y44)
    # a dropped activation fake-quant is not aligned
    y416 = _chains.trainer(xu, l, w13, wd, 2, fake=True)
    assert np.linalg.norm(y416 - y44) > 0.05 * np.linalg.norm(y44)
    xe = synth.u16(synth.engine_drift(x, 2.0 ** -10, 1))
    assert (xe != xu).any()
    d_eta = np.linalg.norm(_chains.trainer(xe, l, w13, wd, 2, fake=False)
                           - _chains.trainer(xu, l, w13, wd, 2, fake=False))
    d_sym = np.linalg.norm(_chains.rollout(xe, l, w13, wd, 2) - y_sym)
    assert d_sym > 5 * d_eta > 0


def test_online_selection_chain():
    """The oracle's online chain (Eq. 23-24 on this batch, for x and for h)
    picks the outlier channels of x and lowers the mismatch below plain W4A4."""
    x, logits, w13, wd = small_moe()
    xu, l = synth.u16(x), logits.numpy()
    out, S13, Sd, sc13, scd = _chains.rollout_online(xu, l, w13, wd, 2, 32, 16)
    assert _chains.valid_topk(S13, sc13, 32, rel=0) and _chains.valid_topk(Sd, scd, 16, rel=0)
    # the 4 scaled outlier channels of small_moe carry the largest errors
    big = np.argsort(np.abs(oracle.bf16_to_f32(xu)).max(0))[::-1][:4]
    assert set(big.tolist()) <= set(S13.tolist())
    y_qat = _chains.trainer(xu, l, w13, wd, 2, fake=True)
    assert np.linalg.norm(out - y_qat) < np.linalg.norm(_chains.rollout(xu, l, w13, wd, 2) - y_qat)
