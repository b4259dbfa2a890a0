"""Pins of the oracle's GEMMs, channel selection and MoE glue.

The W4A4 + RAC product of QUADS §3.3 Eq. 21 is checked against numpy's
matmul (a library routine) and against special cases with closed-form
answers: an exact integer case, k = 0 (plain W4A4) and S = all channels
(the W4A16 product, QUADS §3.2).  Channel selection (Eq. 23-24) is checked by
brute force over subsets; the router against numpy's stable argsort and
scipy's softmax; SwiGLU against closed-form values of silu.
"""
import itertools
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_rac_gemm_matches_numpy_matmul():
    x = synth.u16(synth.activations(1))
    w = synth.u16(synth.dense_weight(1))
    S = np.arange(0, 512, 32, dtype=np.int32)
    ca, sa, r, ga = oracle.quantize(x, S=S)
    cw, sw, _, gw = oracle.quantize(w)
    xq = oracle.dequantize_exact(ca, sa, ga)
    wq = oracle.dequantize_exact(cw, sw, gw)
    y = oracle.rac_gemm(xq, wq, r, S, ga)
    ref = xq @ wq.T + (ga * oracle.bf16_to_f32(r).astype(np.float64)) @ wq[:, S].T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_k0_is_plain_w4a4():
    x = _bf16(np.random.default_rng(1).standard_normal((16, 128)))
    w = _bf16(np.random.default_rng(2).standard_normal((32, 128)) * 0.02)
    ca, sa, _, ga = oracle.quantize(x)
    cw, sw, _, gw = oracle.quantize(w)
    xq = oracle.dequantize_exact(ca, sa, ga)
    wq = oracle.dequantize_exact(cw, sw, gw)
    y0 = oracle.rac_gemm(xq, wq)
    assert np.array_equal(y0, oracle.rac_gemm(xq, wq, np.zeros((16, 0), np.uint16), np.zeros(0, np.int32)))
    assert np.allclose(y0, xq @ wq.T, rtol=1e-12, atol=1e-14)


def test_all_channels_reproduces_w4a16():
    # P-RK: with S = every channel, X_q + r = X up to the BF16 rounding of r,
    # so the RAC product is the W4A16 product X_bf16 . W_hat^T within
    # sum_j |r_j - (x_j - xq_j)| |wq_j|.
    rng = np.random.default_rng(3)
    x = _bf16(rng.standard_normal((8, 256)) * 3)
    w = _bf16(rng.standard_normal((16, 256)) * 0.02)
    S = np.arange(256, dtype=np.int32)
    ca, sa, r, ga = oracle.quantize(x, S=S)
    cw, sw, _, gw = oracle.quantize(w)
    xq = oracle.dequantize_exact(ca, sa, ga)
    wq = oracle.dequantize_exact(cw, sw, gw)
    y = oracle.rac_gemm(xq, wq, r, S, ga)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    w4a16 = xf @ wq.T
    # error of the compensated activation, element by element
    err = np.abs(xq + ga * oracle.bf16_to_f32(r) - xf)
    bound = err @ np.abs(wq).T
    assert np.all(np.abs(y - w4a16) <= bound * (1 + 1e-9) + 1e-12)
    # the bound is much smaller than the uncompensated W4A4 error
    assert np.abs(y - w4a16).max() < 0.05 * np.abs(xq @ wq.T - w4a16).max()


def test_all_channels_exact_case():
    # With gs_a a power of two and x - xq exactly representable in BF16, the
    # RAC product equals the W4A16 product exactly (up to binary64 sums of
    # short dyadic numbers, which are exact here).
    rng = np.random.default_rng(9)
    K = 64
    xs = rng.integers(-40, 41, (4, K)) / 8.0  # multiples of 1/8, |x| <= 5
    x = _bf16(xs)
    gs = 2.0 ** -8
    S = np.arange(K, dtype=np.int32)
    ca, sa, r, _ = oracle.quantize(x, gs=gs, S=S)
    xq32 = oracle.dequantize_f32(ca, sa, gs).astype(np.float64)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    assert np.array_equal(gs * oracle.bf16_to_f32(r).astype(np.float64), xf - xq32)
    wq = rng.integers(-6, 7, (8, K)).astype(np.float64)
    y = oracle.rac_gemm(oracle.dequantize_exact(ca, sa, gs), wq, r, S, gs)
    assert np.array_equal(y, xf @ wq.T)


def test_exact_integer_gemm_case():
    # P-G1: every block scale 1.0 (E4M3 0x38) and gs = 1: the product is a sum
    # of products of grid values, all multiples of 1/4 below 36, so it is an
    # exact integer computation: compare with int64 arithmetic on 2*value.
    rng = np.random.default_rng(10)
    M, N, K = 8, 8, 256
    ca = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    cw = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    sa = np.full((M, K // 16), 0x38, np.uint8)
    sw = np.full((N, K // 16), 0x38, np.uint8)
    xq = oracle.dequantize_exact(ca, sa, 1.0)
    wq = oracle.dequantize_exact(cw, sw, 1.0)
    twice = {c: int(round(2 * oracle.e2m1_value(c))) for c in range(16)}
    lut = np.array([twice[c] for c in range(16)], np.int64)
    ia = lut[np.stack([ca & 15, ca >> 4], -1).reshape(M, K)]
    iw = lut[np.stack([cw & 15, cw >> 4], -1).reshape(N, K)]
    want = (ia @ iw.T).astype(np.float64) / 4.0
    assert np.array_equal(oracle.rac_gemm(xq, wq), want)


def test_bf16_gemm_matches_numpy():
    rng = np.random.default_rng(12)
    x = _bf16(rng.standard_normal((16, 96)))
    w = _bf16(rng.standard_normal((24, 96)) * 0.02)
    y = oracle.bf16_gemm(x, w)
    ref = oracle.bf16_to_f32(x).astype(np.float64) @ oracle.bf16_to_f32(w).astype(np.float64).T
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-15)


def test_channel_scores_match_numpy():
    x = synth.u16(synth.activations(1))
    c, s, _, gs = oracle.quantize(x)
    xq = oracle.dequantize_exact(c, s, gs)
    ref = ((xq - oracle.bf16_to_f32(x).astype(np.float64)) ** 2).sum(0)
    got = oracle.channel_scores_sq(x)
    assert np.allclose(got, ref, rtol=1e-12)
    # the seeded outlier channels carry the largest residual energy
    S = oracle.select_channels(got, 4)
    assert set(S.tolist()) == set(synth.outlier_channels(1).tolist())


@pytest.mark.parametrize("seed", range(6))
def test_select_channels_brute_force(seed):
    # P-SEL: over all k-subsets of d <= 12 channels, the selected set is the
    # unique one where every chosen score beats every unchosen one (ties: lower
    # channel index wins).  Scores are drawn from a small set to force ties.
    rng = np.random.default_rng(seed)
    d = 12
    s = rng.integers(0, 5, d).astype(np.float64)
    for k in range(0, d + 1):
        got = oracle.select_channels(s, k)
        assert list(got) == sorted(got)
        ok = []
        for sub in itertools.combinations(range(d), k):
            rest = [j for j in range(d) if j not in sub]
            if all(s[i] > s[j] or (s[i] == s[j] and i < j) for i in sub for j in rest):
                ok.append(sub)
        assert len(ok) == 1
        assert tuple(got) == ok[0]


def test_route_topk_matches_argsort_and_softmax():
    rng = np.random.default_rng(13)
    T, E, k = 64, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[0, 3] = logits[0, 5] = logits[0].max() + 1  # a tie: expert 3 first
    ids, w = oracle.route_topk(logits, k)
    ref_ids = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    assert np.array_equal(ids, ref_ids)
    assert ids[0, 0] == 3 and ids[0, 1] == 5
    p = scipy.special.softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(p, ref_ids, 1), rtol=1e-13)


def test_route_layout_invariants():
    rng = np.random.default_rng(14)
    T, E, k = 300, 8, 3
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    counts, offsets, dst = oracle.route_layout(ids, E)
    assert counts.sum() == T * k
    assert np.all(offsets % 128 == 0) and np.all(np.diff(offsets) >= counts)
    assert len(set(dst.reshape(-1).tolist())) == T * k
    for e in range(E):
        rows = np.sort(dst[ids == e])
        toks = np.nonzero((ids == e).any(1))[0]
        assert np.array_equal(rows, offsets[e] + np.arange(counts[e]))
        # within an expert, rows follow token order
        assert np.array_equal(dst[toks, np.argmax(ids[toks] == e, 1)], rows)


def test_swiglu_closed_forms():
    y = np.array([[0.0, 1.0, -1.0, 30.0, 2.0, 3.0, 0.5, 1.0]])
    h = oracle.swiglu(y, 4)
    silu1 = 1.0 / (1.0 + math.exp(-1.0))
    assert h[0, 0] == 0.0
    assert h[0, 1] == pytest.approx(silu1 * 3.0, rel=1e-15)
    assert h[0, 2] == pytest.approx(-(1 - silu1) * 0.5, rel=1e-15)  # silu(-1) = -(1 - sigmoid(1))
    assert h[0, 3] == pytest.approx(30.0, rel=1e-12)  # silu(30) ~ 30


def test_combine_matches_einsum():
    rng = np.random.default_rng(15)
    y = rng.standard_normal((40, 8))
    rows = rng.permutation(40)[:30].reshape(10, 3).astype(np.int32)
    w = rng.random((10, 3))
    out = oracle.combine(y, rows, w)
    assert np.allclose(out, np.einsum("ts,tsh->th", w, y[rows]), rtol=1e-14)
