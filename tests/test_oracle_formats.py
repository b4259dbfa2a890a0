"""Pins of the oracle's number formats against what the paper and libraries fix.

QUADS §2.2 "FP4." fixes the E2M1 value set and the 16-element E4M3 block
scale; "FP8." fixes E4M3's field widths and its maximum 448.  Each encoder is
checked against an independent formulation: brute-force nearest search over
the value set, or torch's own float8_e4m3fn / bfloat16 casts.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _grid():
    with open(os.path.join(GOLDEN, "e2m1_grid.txt")) as f:
        lines = [l for l in f if l.strip() and not l.startswith("#")]
    return [float(v) for v in lines[0].split()]


def _facts():
    d = {}
    with open(os.path.join(GOLDEN, "e4m3_facts.txt")) as f:
        for l in f:
            if l.strip() and not l.startswith("#"):
                k, v = l.split()
                d[k] = float(v)
    return d


def test_e2m1_decoder_is_the_page_value_set():
    grid = _grid()
    assert [oracle.e2m1_value(c) for c in range(8)] == grid
    for c in range(8):
        assert oracle.e2m1_value(c | 8) == -grid[c]
    # -0 decodes to a zero with the sign bit set
    assert np.signbit(oracle.e2m1_value(8))


def _e2m1_brute(v, grid):
    """nearest grid magnitude, ties to the even code index, saturate at 6"""
    a = abs(v)
    d = [abs(a - g) for g in grid]
    best = min(d)
    cands = [i for i in range(8) if d[i] == best]
    if len(cands) > 1:
        cands = [i for i in cands if i % 2 == 0]
    code = cands[0]
    return code | (8 if np.signbit(v) else 0)


def test_e2m1_encoder_brute_force_all_bf16_values():
    grid = _grid()
    pats = np.arange(65536, dtype=np.uint32)
    vals = (pats << 16).view(np.float32)
    vals = vals[np.isfinite(vals)]
    # the grid only matters within [-8, 8]; scale a copy so every bf16 mantissa
    # pattern lands in the interesting range too
    sel = np.concatenate([vals, np.ldexp(vals[np.abs(vals) > 0], 0)])
    sel = sel[np.abs(sel) < 16]
    got = oracle.e2m1_encode(sel)
    want = np.array([_e2m1_brute(float(v), grid) for v in sel], np.uint8)
    assert np.array_equal(got, want)
    # saturation: everything above 6 is 6 (code 7), sign kept
    big = np.array([6.0001, 7.0, 100.0, 1e30, np.inf, -7.0, -np.inf], np.float32)
    assert list(oracle.e2m1_encode(big)) == [7, 7, 7, 7, 7, 15, 15]


def test_e2m1_tie_cases():
    # every midpoint of the grid goes to the neighbour with the even code
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    want = [0, 2, 2, 4, 4, 6, 6]  # 0, 1, 1, 2, 2, 4, 4
    assert list(oracle.e2m1_encode(ties)) == want
    assert list(oracle.e2m1_encode(-ties)) == [w | 8 for w in want]


def test_e4m3_decoder_matches_torch_and_page_max():
    facts = _facts()
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if np.isnan(ref[c]):
            assert np.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
    finite = [oracle.e4m3_value(c) for c in range(127)]
    assert max(finite) == facts["max_magnitude"] == 448.0
    assert np.isnan(oracle.e4m3_value(0x7F))
    # field widths: 16 exponent codes x 8 mantissa codes per sign
    assert facts["exponent_bits"] == 4 and facts["mantissa_bits"] == 3


def test_e4m3_encoder_exhaustive_round_trip_and_midpoints():
    vals = np.array([oracle.e4m3_value(c) for c in range(127)], np.float64)
    # encode(decode(c)) == c for every finite non-negative code (0x00 .. 0x7E)
    assert list(oracle.e4m3_encode(vals.astype(np.float32))) == list(range(127))
    # midpoints between neighbours go to the even code
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (vals[:-1] + vals[1:]) / 2)  # exact
    got = oracle.e4m3_encode(mids)
    for i, g in enumerate(got):
        lo, hi = i, i + 1
        assert g == (lo if lo % 2 == 0 else hi), (i, g)
    # saturation at the page's maximum
    sat = np.array([448.0, 449.0, 464.0, 480.0, 1e9, np.inf], np.float32)
    assert list(oracle.e4m3_encode(sat)) == [0x7E] * 6


def test_e4m3_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.uniform(0, 448, 200000),
        np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448), 200000)),
    ]).astype(np.float32)
    got = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_e4m3_encoder_brute_force_nearest():
    # P-E3: enumerate every non-negative finite E4M3 value; the chosen code is
    # the nearest one, ties to the even code.
    vals = np.array([oracle.e4m3_value(c) for c in range(127)], np.float64)
    rng = np.random.default_rng(3)
    v = np.exp(rng.uniform(np.log(2.0 ** -11), np.log(440), 20000)).astype(np.float32)
    got = oracle.e4m3_encode(v)
    for x, g in zip(v.astype(np.float64), got):
        d = np.abs(vals - x)
        cands = np.flatnonzero(d == d.min())
        if len(cands) > 1:
            cands = [c for c in cands if c % 2 == 0]
        assert g == cands[0]


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 2 ** 32, 400000, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    # add exact ties: bf16 value + half an ulp
    base = (rng.integers(0, 2 ** 16, 10000).astype(np.uint32) << 16) | 0x8000
    t = base.view(np.float32)
    v = np.concatenate([v, t[np.isfinite(t)]])
    got = oracle.bf16_round(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
