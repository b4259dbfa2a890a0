"""Pins of the oracle's NVFP4 quantizer, residual and fake-quant.

What they fix, from QUADS §2.2 "FP4.", §3.2 Eq. 12 and §3.3 Eq. 20-22:
every dequantized value lies on the scaled E2M1 grid; each block's largest
element maps to +-6 whenever its scale is a normal E4M3 number; quantizing a
dequantized tensor is idempotent; sign flips and power-of-two scalings act
only on the sign bits and on gs; an all-zero tensor is all-zero codes;
every block scale is the nearest E4M3 to its target (brute force); each
element goes to the nearest point of its block's grid; the RAC residual
strictly shrinks the activation error (Eq. 22); fake-quant equals
dequantize(quantize(W)) rounded to BF16.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

GRID = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rand_x(M, K, seed, outliers=True):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((M, K))
    if outliers:
        cols = rng.choice(K, max(1, K // 64), replace=False)
        x[:, cols] *= 40
    # a few blocks with tiny dynamic range relative to the tensor (subnormal scales)
    x[0, :16] *= 1e-4
    return _bf16(x)


def _codes_unpacked(codes):
    lo = codes & 15
    hi = codes >> 4
    return np.stack([lo, hi], -1).reshape(codes.shape[0], -1)


def _scale_vals(scales):
    return np.array([oracle.e4m3_value(int(s)) for s in range(256)])[scales]


def test_grid_membership_and_amax_maps_to_six():
    x = _rand_x(64, 512, 1)
    codes, scales, _, gs = oracle.quantize(x)
    xq = oracle.dequantize_exact(codes, scales, gs)
    sv = _scale_vals(scales)
    den = np.repeat(sv, 16, axis=1) * gs
    with np.errstate(invalid="ignore", divide="ignore"):
        g = np.where(den > 0, np.abs(xq) / den, 0.0)
    # P-G: every dequantized value is +-g * sb * gs with g on the E2M1 grid
    assert np.all(np.isin(g, GRID))
    # P-A: with a normal block scale (>= 2^-6), the block's largest |x| maps to 6
    c = _codes_unpacked(codes) & 7
    xf = oracle.bf16_to_f32(x).reshape(64, -1, 16)
    amax_pos = np.abs(xf).argmax(-1)
    cb = c.reshape(64, -1, 16)
    top = np.take_along_axis(cb, amax_pos[..., None], -1)[..., 0]
    normal = sv >= 2.0 ** -6
    assert normal.sum() > 0.9 * normal.size
    assert np.all(top[normal] == 7)


def test_elements_go_to_nearest_grid_point():
    x = _rand_x(32, 256, 2)
    codes, scales, _, gs = oracle.quantize(x)
    sv = np.repeat(_scale_vals(scales), 16, axis=1)
    den = sv * gs
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    xq = oracle.dequantize_exact(codes, scales, gs)
    cand = np.concatenate([-GRID[::-1], GRID])[None, None, :] * den[..., None]
    best = np.abs(cand - xf[..., None]).min(-1)
    err = np.abs(xq - xf)
    # the element is scaled by a rounded reciprocal (one binary32 multiply), so
    # allow a relative slack of a few binary32 ulps at exact midpoints
    assert np.all(err <= best + 4 * 2.0 ** -24 * np.abs(xf) + 1e-300)


def test_block_scale_is_nearest_e4m3_brute_force():
    # P-E3 on tiny blocks: enumerate all finite non-negative E4M3 values
    x = _rand_x(4, 64, 3)
    codes, scales, _, gs = oracle.quantize(x)
    vals = np.array([oracle.e4m3_value(c) for c in range(127)], np.float64)
    xf = oracle.bf16_to_f32(x).reshape(4, -1, 16)
    p = np.float32(gs) * np.float32(6.0)
    for i in range(4):
        for b in range(xf.shape[1]):
            s = np.float32(np.abs(xf[i, b]).max()) / p  # binary32 division
            d = np.abs(vals - np.float64(s))
            cands = np.flatnonzero(d == d.min())
            if len(cands) > 1:
                cands = [c for c in cands if c % 2 == 0]
            want = cands[0] if s <= 448 else 0x7E
            assert scales[i, b] == want


def test_idempotence_with_power_of_two_scale():
    # P-I: make gs a power of two (amax 168 -> gs = 168/2688 = 2^-4), so every
    # dequantized value is exactly a BF16 number; re-quantizing it with gs held
    # fixed gives back the same codes and scales for normal-scale blocks.
    rng = np.random.default_rng(4)
    x = rng.standard_normal((16, 256))
    x *= 20
    x = np.clip(x, -160, 160)
    x[0, 0] = 168.0
    xb = _bf16(x)
    codes, scales, _, gs = oracle.quantize(xb)
    assert gs == 2.0 ** -4
    xq = oracle.dequantize_f32(codes, scales, gs)
    xqb = _bf16(xq)
    assert np.array_equal(oracle.bf16_to_f32(xqb), xq)
    codes2, scales2, _, _ = oracle.quantize(xqb, gs=gs)
    normal = np.repeat(_scale_vals(scales) >= 2.0 ** -6, 8, axis=1)
    assert np.array_equal(scales2, scales)
    assert np.array_equal(codes2[normal], codes[normal])
    # and with gs recomputed from the dequantized tensor's own amax
    codes3, scales3, _, gs3 = oracle.quantize(xqb)
    assert gs3 == gs and np.array_equal(codes3, codes2)


def test_sign_symmetry_and_power_of_two_invariance():
    x = _rand_x(16, 128, 5)
    codes, scales, _, gs = oracle.quantize(x)
    neg = x ^ np.uint16(0x8000)
    c2, s2, _, g2 = oracle.quantize(neg)
    assert g2 == gs and np.array_equal(s2, scales)
    assert np.array_equal(c2, codes ^ np.uint8(0x88))
    for n in (-3, 5):
        xs = _bf16(oracle.bf16_to_f32(x).astype(np.float64) * 2.0 ** n)
        c3, s3, _, g3 = oracle.quantize(xs)
        assert g3 == np.float32(gs * 2.0 ** n)
        assert np.array_equal(s3, scales) and np.array_equal(c3, codes)


def test_zero_tensor():
    x = np.zeros((8, 64), np.uint16)
    S = np.array([1, 7, 63], np.int32)
    codes, scales, resid, gs = oracle.quantize(x, S=S)
    assert gs == 1.0
    assert not codes.any() and not scales.any() and not resid.any()


def test_tensor_scale_is_a_power_of_two_bounding_every_block_scale():
    rng = np.random.default_rng(16)
    for a in list(np.exp(rng.uniform(-40, 40, 2000)).astype(np.float32)) + [2688.0, 168.0, 1.0, 5376.0001]:
        gs = oracle.tensor_scale(float(a))
        m, e = np.frexp(gs)
        assert m == 0.5  # a power of two
        q = np.float32(a) / np.float32(2688.0)
        # the smallest power of two not below fl(amax / 2688)
        assert gs >= q and gs / 2 < q
    assert oracle.tensor_scale(0.0) == 1.0


def test_residual_definition_and_eq22():
    x = synth.u16(synth.activations(1))
    S = np.array(sorted(np.random.default_rng(6).choice(512, 16, replace=False)), np.int32)
    codes, scales, resid, gs = oracle.quantize(x, S=S)
    xq = oracle.dequantize_f32(codes, scales, gs)
    xf = oracle.bf16_to_f32(x)
    # r = bf16(x - xq) on the channels S (Eq. 20 with the sign of -Delta X_q),
    # stored in units of gs: gs is a power of two, so this is exact here
    r = torch.from_numpy((xf[:, S] - xq[:, S]).astype(np.float32)).to(torch.bfloat16).float().numpy()
    want = torch.from_numpy((r / np.float32(gs)).astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(resid, want.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(oracle.bf16_to_f32(resid).astype(np.float64) * gs, r.astype(np.float64))
    # Eq. 22: compensating S strictly lowers the distance to X
    xt = xq.astype(np.float64).copy()
    xt[:, S] += gs * oracle.bf16_to_f32(resid)
    e_plain = np.linalg.norm(xq.astype(np.float64) - xf)
    e_rac = np.linalg.norm(xt - xf)
    assert e_rac < e_plain


def test_fake_quant_equals_dequant_of_quant():
    # P-FQ: QDQ_W uses the rollout quantizer's layout and rounding (QUADS §3.2)
    w = synth.u16(synth.dense_weight(1))
    w_hat, gs = oracle.fake_quant(w)
    codes, scales, _, gs2 = oracle.quantize(w)
    assert gs == gs2
    deq = oracle.dequantize_f32(codes, scales, gs)
    assert np.array_equal(w_hat, oracle.bf16_round(deq))
    # with a power-of-two gs nothing rounds: W_hat is exactly code * sb * gs,
    # the value the rollout GEMM multiplies (Eq. 16: zero weight mismatch)
    assert np.array_equal(oracle.bf16_to_f32(w_hat).astype(np.float64), oracle.dequantize_exact(codes, scales, gs))


def test_scale_layout_is_a_bijection_with_zero_padding():
    M, K = 200, 320  # ragged in both dimensions: 2 row tiles, 2 slices of 16 blocks (the second 4/16 full)
    rng = np.random.default_rng(8)
    sc = rng.integers(1, 255, (M, K // 16), dtype=np.uint8)
    out = oracle.scale_layout(sc, K)
    assert out.size == 2 * 2 * 2048
    assert np.count_nonzero(out) == sc.size
    assert sorted(out[out != 0].tolist()) == sorted(sc.reshape(-1).tolist())
    # 512-byte groups of 4 blocks; row r on line r%32, bytes 4*(r/32) + kb%4
    assert out[0] == sc[0, 0] and out[3] == sc[0, 3] and out[512] == sc[0, 4]
    assert out[1 * 16 + 4 * 1 + 2] == sc[33, 2]
    assert out[3 * 512 + 7 * 16 + 4 * 3 + 3] == sc[103, 15]
    assert out[2048 + 5 * 16 + 2] == sc[5, 18]      # slice 1 of row tile 0
    assert out[3 * 2048 + 3] == sc[128, 19]         # slice 1 of row tile 1
    # reading rows back through the layout gives the canonical scales
    rows = np.array([0, 5, 33, 127, 128, 199])
    assert np.array_equal(oracle.scale_rows(out, rows, K), sc[rows])
