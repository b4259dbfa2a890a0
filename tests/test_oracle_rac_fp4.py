"""Pins of the oracle's literal Eq. 21 residual (QUADS §3.3 Eq. 20-21): the
residual on the selected channels, r = x - Q_A(x), is NVFP4-quantized a second
time (gathered [M, k] residual, its own tensor scale).  What fixes it:

* every second-pass value is a point of the E2M1 grid times its block's E4M3
  scale times the residual's power-of-two tensor scale;
* the corrected activation Q_A(x) + Q_A(r) is never farther from x than
  Q_A(x) alone, element by element (round to nearest on a grid holding 0), and
  strictly closer in norm on outlier data -- a sign error in the correction
  or a residual taken against the wrong operand fails this;
* the second pass is the plain quantizer applied to the gathered residual, and
  it commutes with the power-of-two unit change between r and its stored form.
"""
import numpy as np

import oracle
from tests.test_oracle_quant import GRID, _rand_x


def _setup(seed=3, M=96, K=512, k=64):
    x = _rand_x(M, K, seed)
    ssq = oracle.channel_scores_sq(x)
    S = oracle.select_channels(ssq, k)
    codes, scales, resid, gs = oracle.quantize(x, S=S)
    return x, S, codes, scales, resid, gs


def test_second_pass_values_lie_on_the_scaled_grid():
    x, S, codes, scales, resid, gs = _setup()
    q, gs_r = oracle.requant_residual(resid, gs)
    assert gs_r > 0 and np.log2(gs_r) == np.round(np.log2(gs_r))
    vals = oracle.bf16_to_f32(q).astype(np.float64) * gs  # Q_A(r)
    c2, s2, _, g2 = oracle.quantize(oracle.bf16_round((oracle.bf16_to_f32(resid).astype(np.float64) * gs)
                                                      .astype(np.float32)))
    assert g2 == gs_r
    sb = np.repeat(np.array([oracle.e4m3_value(int(c)) for c in s2.reshape(-1)]).reshape(s2.shape), 16, axis=1)
    mult = np.abs(vals) / np.where(sb > 0, sb * gs_r, 1.0)
    assert np.all(np.isin(np.where(sb > 0, mult, 0.0), GRID))


def test_corrected_activation_is_never_farther_from_x():
    x, S, codes, scales, resid, gs = _setup()
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    xq = oracle.dequantize_exact(codes, scales, gs)
    r = oracle.bf16_to_f32(resid).astype(np.float64) * gs
    # r is the quantization residual on S (Eq. 20 with the sign of Eq. 22)
    assert np.allclose(r, xf[:, S] - xq[:, S], rtol=2.0 ** -8, atol=0)
    q, _ = oracle.requant_residual(resid, gs)
    qr = oracle.bf16_to_f32(q).astype(np.float64) * gs
    e0 = np.abs(xf[:, S] - xq[:, S])
    e1 = np.abs(xf[:, S] - xq[:, S] - qr)
    # Q_A(r) is the nearest scaled grid point to r (or saturated), so it is at
    # least as close to r as 0 is -- up to the BF16 rounding of r itself
    assert np.all(e1 <= e0 + 2.0 ** -8 * np.abs(r) + 1e-300)
    assert np.linalg.norm(e1) < 0.5 * np.linalg.norm(e0)
    # and the BF16 residual (Q9's form) is closer still
    assert np.linalg.norm(xf[:, S] - xq[:, S] - r) < np.linalg.norm(e1)


def test_second_pass_commutes_with_the_power_of_two_unit():
    x, S, codes, scales, resid, gs = _setup(seed=5)
    q, gs_r = oracle.requant_residual(resid, gs)
    # the quantizer applied directly to the stored residual (units of gs)
    c, s, _, g = oracle.quantize(resid)
    assert g * gs == gs_r
    assert np.array_equal(oracle.dequantize_exact(c, s, g), oracle.bf16_to_f32(q).astype(np.float64))
    # an all-zero residual stays zero
    z, _ = oracle.requant_residual(np.zeros_like(resid), gs)
    assert not z.any()


def test_layer_mismatch_order_with_the_second_pass():
    """On the small outlier MoE layer of the mismatch pins: against the W4A16
    QAT trainer, the W4A4 rollout with the second-pass (FP4) residual sits
    between plain W4A4 and the BF16-residual form -- RAC still removes most of
    the activation term, the second quantization gives a little of it back."""
    import synth
    from tests import _chains
    from tests.test_oracle_mismatch import small_moe

    x, logits, w13, wd = small_moe()
    xu, l = synth.u16(x), logits.numpy()
    S13 = oracle.select_channels(oracle.channel_scores_sq(xu), 32)
    Sd = np.arange(0, 256, 16, dtype=np.int32)
    y_qat = _chains.trainer(xu, l, w13, wd, 2, fake=True)
    d = {name: np.linalg.norm(_chains.rollout(xu, l, w13, wd, 2, **kw) - y_qat)
         for name, kw in [("w4a4", {}), ("rac", dict(S13=S13, Sd=Sd)),
                          ("rac_fp4", dict(S13=S13, Sd=Sd, fp4_resid=True))]}
    assert d["w4a4"] > 1.2 * d["rac_fp4"] and d["rac_fp4"] > d["rac"]
