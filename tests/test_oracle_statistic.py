"""Pins of the oracle's row statistic (reading R2): ms = RN32(mean(x^2)), the
exact mean of the squares rounded once to fp32, and r = RN32(1/sqrt(v)).

* ms against exact rational arithmetic (Python Fractions: the exact sum of the
  squares divided by D, rounded by nearest-value search with ties to even) on
  random rows of every dtype, with magnitudes spread over many binades;
* ms against hand-derived ties, near-ties, overflow, subnormal and non-finite
  rows (tests/golden/statistic_ties.txt);
* ms of one element equals the IEEE product x*x of numpy's float32 (fp32
  rows), and of a row of equal values equals that square;
* the inverse root against an exact integer test of correct rounding, for
  every fp32 value in [1, 4) (every binade pair: v * 4^k only scales the
  result by 2^-k) and for samples across the whole range.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from _cases import BOUNDARY_VARIANTS, boundary_tensor
from _exact import round_to_fp32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "statistic_ties.txt")
STORAGE = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def storage(values, dtype):
    """Raw storage (numpy) of float values that the dtype holds exactly."""
    t = torch.tensor(values, dtype=torch.float64).to(STORAGE[dtype])
    assert torch.equal(t.double(), torch.tensor(values, dtype=torch.float64)) or \
        any(not np.isfinite(v) for v in values), "value not exact in the dtype"
    if dtype == "fp32":
        return t.numpy().copy()
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def exact_ms(values):
    """RN32(sum x^2 / D) by exact rational arithmetic (NaN / inf rules of the
    reading: a NaN gives NaN, otherwise an infinity gives +inf)."""
    if any(np.isnan(v) for v in values):
        return np.float32(np.nan)
    if any(np.isinf(v) for v in values):
        return np.float32(np.inf)
    q = sum(Fraction(float(v)) ** 2 for v in values) / len(values)
    if q >= Fraction(2) ** 128 - Fraction(2) ** 103:  # RN overflow threshold
        return np.float32(np.inf)
    return np.array([round_to_fp32(q)], dtype=np.uint32).view(np.float32)[0]


def same(a, b):
    a, b = np.float32(a), np.float32(b)
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return a.view(np.uint32) == b.view(np.uint32)


def parse_golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        dtype, xs, want = (c.strip() for c in line.split("|"))
        x = [float.fromhex(v) if v not in ("inf", "-inf", "nan") else float(v)
             for v in (s.strip() for s in xs.split(","))]
        w = float(want) if want in ("inf", "nan") else float.fromhex(want)
        cases.append((dtype, x, w))
    return cases


@pytest.mark.parametrize("case", parse_golden(), ids=lambda c: f"{c[0]}-{len(c[1])}")
def test_mean_square_golden(orc, case):
    dtype, x, want = case
    got = orc.row_mean_square(storage(x, dtype), len(x), dtype)
    assert same(got, want), f"{dtype} {x}: oracle {got!r} expected {want!r}"


def test_golden_agrees_with_exact_rationals():
    """The hand-derived values themselves, against the rational evaluation."""
    for dtype, x, want in parse_golden():
        assert same(exact_ms(x), want), (dtype, x, want)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("D", [1, 2, 3, 7, 64, 127, 3077])
def test_mean_square_matches_exact_rationals(orc, dtype, D):
    rng = np.random.default_rng(1000 + D + 7 * len(dtype))
    spread = {"bf16": 40, "fp16": 4, "fp32": 60}[dtype]
    for trial in range(6 if D > 1000 else 24):
        v = rng.standard_normal(D)
        if trial % 2:  # magnitudes spread over many binades
            v = v * np.exp2(rng.uniform(-spread, spread, D))
        t = torch.tensor(v).to(STORAGE[dtype])
        vals = t.double().numpy()
        raw = storage(vals.tolist(), dtype)
        got = orc.row_mean_square(raw, D, dtype)
        want = exact_ms(vals.tolist())
        assert same(got, want), f"{dtype} D={D} trial {trial}: {got!r} vs {want!r}"


def test_one_element_is_the_ieee_square(orc):
    """D = 1 with fp32 storage: RN32(x^2) is numpy's float32 product."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(4000) * np.exp2(rng.uniform(-70, 70, 4000))).astype(np.float32)
    for v in x:
        got = orc.row_mean_square(np.array([v], dtype=np.float32), 1, "fp32")
        with np.errstate(over="ignore"):
            want = np.float32(v) * np.float32(v)
        assert same(got, want), v


def test_equal_values_give_their_square(orc):
    """A row of D copies of x has mean x^2 exactly (bf16: x^2 exact in fp32)."""
    for D in (3, 5, 12, 4097):
        for v in (0.7265625, -3.0, 1.5e-5, 1234.0):
            t = torch.full((D,), v, dtype=torch.bfloat16)
            x2 = np.float32(t[0].item()) * np.float32(t[0].item())
            raw = t.view(torch.int16).numpy().view(np.uint16).copy()
            assert same(orc.row_mean_square(raw, D, "bf16"), x2)


def test_mean_square_is_order_independent(orc):
    rng = np.random.default_rng(9)
    v = rng.standard_normal(777) * np.exp2(rng.uniform(-30, 30, 777))
    t = torch.tensor(v).to(torch.bfloat16)
    ref = orc.row_mean_square(t.view(torch.int16).numpy().view(np.uint16).copy(), 777, "bf16")
    for _ in range(5):
        p = t[torch.from_numpy(rng.permutation(777))]
        got = orc.row_mean_square(p.view(torch.int16).numpy().view(np.uint16).copy(), 777, "bf16")
        assert same(got, ref)


def _sig_exp(b):
    """positive normal fp32 bit patterns -> (M in [2^23, 2^24), e): value M * 2^e"""
    b = b.astype(np.int64)
    return (b & 0x7FFFFF) | 0x800000, ((b >> 23) & 0xFF) - 150


def _sign_mid_sq_v_minus_one(fb, vb):
    """sign of m^2 * v - 1, m the midpoint between the fp32 value of pattern fb
    and the next one up, exactly (integers)."""
    M, e = _sig_exp(fb)
    Mv, ev = _sig_exp(vb)
    P2 = (2 * M + 1) ** 2                      # m = (2M + 1) * 2^(e-1); < 2^50
    k = -(2 * e - 2 + ev)                      # compare P2 * Mv with 2^k
    hi, lo = P2 * (Mv >> 12), P2 * (Mv & 0xFFF)  # P2 * Mv = hi * 2^12 + lo
    approx = (hi.astype(np.float64) * 4096.0 + lo) / np.ldexp(1.0, k)
    out = np.sign(approx - 1.0).astype(np.int64)
    for i in np.nonzero(np.abs(approx - 1.0) < 1e-9)[0]:  # decide near ties exactly
        z = int(hi[i]) * 4096 + int(lo[i])
        t = 1 << int(k[i])
        out[i] = (z > t) - (z < t)
    return out


def _check_correctly_rounded(orc, vb):
    v = vb.astype(np.uint32).view(np.float32)
    r = orc.inverse_root(v)
    rb = r.view(np.uint32).astype(np.int64)
    above = _sign_mid_sq_v_minus_one(rb, vb)      # must be > 0: r below the midpoint above
    below = _sign_mid_sq_v_minus_one(rb - 1, vb)  # must be < 0: r above the midpoint below
    bad = np.nonzero((above <= 0) | (below >= 0))[0]
    assert bad.size == 0, f"not correctly rounded at v = {v[bad[:5]]}"


def test_inverse_root_correctly_rounded_exhaustive(orc):
    """Every fp32 v in [1, 4): 2^24 values, in chunks."""
    start, end, step = 0x3F800000, 0x40800000, 1 << 21
    for a in range(start, end, step):
        _check_correctly_rounded(orc, np.arange(a, a + step, dtype=np.int64))


def test_inverse_root_across_the_range(orc):
    rng = np.random.default_rng(3)
    # normal fp32 values whose inverse root is a normal fp32 value
    vb = rng.integers(0x00800000, 0x7F000000, 200000, dtype=np.int64)
    _check_correctly_rounded(orc, vb)
    assert same(orc.inverse_root([0.0])[0], np.inf)
    assert same(orc.inverse_root([np.inf])[0], 0.0)
    assert np.isnan(orc.inverse_root([np.nan])[0])
    assert same(orc.inverse_root([4.0])[0], 0.5)
    # subnormal v: 1/sqrt(v * 2^64) = 2^-32 / sqrt(v), an exact scaling
    sub = np.arange(1, 0x800000, 4099, dtype=np.uint32).view(np.float32)
    scaled = orc.inverse_root(sub * np.float32(2.0 ** 64))
    assert np.array_equal(orc.inverse_root(sub), scaled * np.float32(2.0 ** 32))


def test_rms_inverse_composes_the_steps(orc):
    rng = np.random.default_rng(11)
    for D in (5, 300):
        t = torch.tensor(rng.standard_normal(D)).to(torch.bfloat16)
        raw = t.view(torch.int16).numpy().view(np.uint16).copy()
        ms = np.float32(orc.row_mean_square(raw, D, "bf16"))
        v = ms + np.float32(1e-6)
        assert same(orc.row_rms_inverse(raw, D, 1e-6, "bf16"), orc.inverse_root([v])[0])


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_boundary_rows_have_the_intended_mean(orc, dtype):
    """The rows the GPU tests build on the statistic's rounding boundaries:
    the oracle's mean against the hand-derived one, and the exact rational
    mean against the same."""
    for D in (64, 3077, 4096):
        for scale_exp in ((0, 6) if dtype == "fp16" else (0, 20, -30)):
            x, names = boundary_tensor(1, 8, D, dtype, seed=D + scale_exp, scale_exp=scale_exp)
            for i, name in enumerate(names):
                want = np.float32(BOUNDARY_VARIANTS[name][2] * 4.0 ** scale_exp)
                vals = x[0, i].double().numpy()
                assert same(exact_ms(vals.tolist()), want), (dtype, D, name)
                raw = storage(vals.tolist(), dtype)
                assert same(orc.row_mean_square(raw, D, dtype), want), (dtype, D, name, scale_exp)
