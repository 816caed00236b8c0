"""Pins for the oracle's adaLN modulation
    out = rms_norm(x, eps) * (1 + scale) + shift,
with the weightless RMSNorm x / sqrt(mean(x^2) + eps) over each row of D
(prhub summary of sglang PR #34172, sections "implementation breakdown" item 2
and "key source snippet").

Error bound used below (u = 2^-24).  The oracle rounds, in fp32: the mean
square (u/2), mean + eps (u/2), the inverse root (u/2, from the correctly
rounded double), n = x*r (u/2), 1 + scale (u/2), t = n*(1+scale) (u/2) and
y = t + shift (u/2 of |y|).  Summed, the pre-rounding result y_pre obeys
    |y_pre - y_exact| <= 3u*|t| + u*|y|    (t = x*r*(1+scale), exact values),
so the stored dtype value is the correctly rounded y_exact unless y_exact lies
within that distance of a rounding boundary.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from _cases import bits, mod_inputs, oracle_mod, same_bits
from _exact import (round_to, sqrt_fraction, ulp_distance, value_of, words)
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES

DTYPES = ["bf16", "fp16", "fp32"]
LAYOUTS = ["full", "bcast"]
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = Fraction(1, 1 << 24)
EPS32 = float(np.float32(1e-6))


def _check_against_exact(out_word, y_exact: Fraction, t_exact: Fraction, dtype):
    """The oracle's stored value vs the exact result, under the bound above."""
    bound = 3 * U * abs(t_exact) + U * abs(y_exact) + Fraction(1, 1 << 140)
    if dtype == "fp32":
        assert abs(value_of(out_word, "fp32") - y_exact) <= bound + U * abs(y_exact)
        return 0
    want = round_to(y_exact, dtype)
    if out_word == want:
        return 0
    assert ulp_distance(out_word, want, dtype) == 1
    mid = (value_of(out_word, dtype) + value_of(want, dtype)) / 2
    assert abs(y_exact - mid) <= bound, "differs from the exact rounding away from a boundary"
    return 1


@pytest.mark.parametrize("layout", LAYOUTS)
def test_zero_modulation_gives_unit_mean_square(orc, layout):
    """scale = shift = 0: out = x * r, so mean(out^2) = ms / (ms + eps) for the
    row's mean square ms -- within 1e-5 (fp32 output), including rows whose
    magnitudes are spread over 10^-2 .. 10^2."""
    x, sc, sh = mod_inputs(2, 40, 256, "fp32", layout, row_spread=True)
    out = oracle_mod(orc, x, torch.zeros_like(sc), torch.zeros_like(sh), "fp32", layout)
    x64 = x.double().reshape(-1, 256).numpy()
    ms = np.mean(x64 * x64, axis=1)
    got = np.mean(out.double().reshape(-1, 256).numpy() ** 2, axis=1)
    np.testing.assert_allclose(got, ms / (ms + EPS32), rtol=0, atol=1e-5)
    big = ms >= 0.1
    assert big.any()
    np.testing.assert_allclose(got[big], 1.0, rtol=0, atol=1e-5)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_scale_minus_one_gives_shift(orc, dtype, layout):
    x, sc, sh = mod_inputs(2, 9, 77, dtype, layout)
    out = oracle_mod(orc, x, torch.full_like(sc, -1.0), sh, dtype, layout)
    assert same_bits(out, sh.expand(2, 9, 77).contiguous())


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("k", [-3, 5])
def test_power_of_two_scaling_invariance(orc, dtype, k):
    """eps = 0: scaling a row by 2^k is exact through the square, the mean,
    the root and the products, so the output is bitwise unchanged."""
    x, sc, sh = mod_inputs(1, 12, 96, dtype, "bcast")
    a = oracle_mod(orc, x, sc, sh, dtype, "bcast", eps=0.0)
    xs = (x.double() * 2.0 ** k).to(x.dtype)
    assert torch.equal(xs.double(), x.double() * 2.0 ** k)
    b = oracle_mod(orc, xs, sc, sh, dtype, "bcast", eps=0.0)
    assert same_bits(a, b)
    # with eps > 0 the statistic is not scale-free: the check has teeth
    c = oracle_mod(orc, (x.double() * 2.0 ** -12).to(x.dtype), sc, sh, dtype, "bcast",
                   eps=1e-6)
    assert not same_bits(a, c)


@pytest.mark.parametrize("c", [1.0, 0.75, 3e-3, 1e-3, 2.5e-4, 40.0])
def test_constant_row_closed_form(orc, c):
    """x = c on the whole row, scale = shift = 0: out = c / sqrt(c^2 + eps).
    (For c near sqrt(eps) this separates eps inside the root from other
    placements of eps.)"""
    D = 64
    x = torch.full((1, 3, D), c, dtype=torch.float32)
    z = torch.zeros((1, 1, D), dtype=torch.float32)
    out = oracle_mod(orc, x, z, z, "fp32", "bcast", eps=EPS32)
    cq = Fraction(float(np.float32(c)))
    exact = cq / sqrt_fraction(cq * cq + Fraction(EPS32))
    for w in words(out):
        assert abs(value_of(w, "fp32") - exact) <= 3 * U * abs(exact)
    for dtype in ("bf16", "fp16"):
        xd = x.to(TORCH_DTYPES[dtype])
        cq = Fraction(float(xd.double()[0, 0, 0]))
        exact = cq / sqrt_fraction(cq * cq + Fraction(EPS32))
        outd = oracle_mod(orc, xd, z.to(xd.dtype), z.to(xd.dtype), dtype, "bcast", eps=EPS32)
        for w in words(outd):
            _check_against_exact(w, exact, exact, dtype)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_against_torch_rms_norm_float64(orc, dtype, layout):
    """Library pin: torch.nn.functional.rms_norm in float64, then
    * (1 + scale) + shift in float64, treated as exact (its error, ~1e-16
    relative, is far below the bound)."""
    B, L, D = 2, 24, 320
    x, sc, sh = mod_inputs(B, L, D, dtype, layout, row_spread=True)
    out = oracle_mod(orc, x, sc, sh, dtype, layout, eps=EPS32)
    n64 = F.rms_norm(x.double(), (D,), eps=EPS32)
    t64 = n64 * (1.0 + sc.double())
    y64 = (t64 + sh.double()).expand(B, L, D).reshape(-1).tolist()
    t64 = t64.expand(B, L, D).reshape(-1).tolist()
    boundary = 0
    for w, y, t in zip(words(out), y64, t64):
        boundary += _check_against_exact(w, Fraction(y), Fraction(t), dtype)
    assert boundary <= len(y64) // 100  # boundary cases are rare


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 2, 3), (2, 3, 8), (2, 2, 31), (1, 2, 129)])
def test_exact_rational_bruteforce(orc, dtype, layout, shape):
    """Exact rationals (root to 80 digits) on tiny shapes, under the bound."""
    B, L, D = shape
    x, sc, sh = mod_inputs(B, L, D, dtype, layout, tag=("bf", shape))
    out = oracle_mod(orc, x, sc, sh, dtype, layout, eps=EPS32)
    xw, sw, hw, ow = words(x), words(sc), words(sh), words(out)
    eps = Fraction(EPS32)
    for r in range(B * L):
        mrow = r if layout == "full" else r // L
        xs = [value_of(xw[r * D + d], dtype) for d in range(D)]
        ms = sum(v * v for v in xs) / D
        rinv = 1 / sqrt_fraction(ms + eps)
        for d in range(D):
            s = value_of(sw[mrow * D + d], dtype)
            h = value_of(hw[mrow * D + d], dtype)
            t = xs[d] * rinv * (1 + s)
            _check_against_exact(ow[r * D + d], t + h, t, dtype)


def _golden_rows(name):
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        yield [s.strip() for s in line.split("|")]


def test_worked_examples_golden(orc):
    n = 0
    for eps, xs, scs, shs, exps in _golden_rows("modulate_worked.txt"):
        vec = lambda s: [float(v) for v in s.split(",")]
        x = torch.tensor([[vec(xs)]], dtype=torch.float64).to(torch.bfloat16)
        sc = torch.tensor([[vec(scs)]], dtype=torch.float64).to(torch.bfloat16)
        sh = torch.tensor([[vec(shs)]], dtype=torch.float64).to(torch.bfloat16)
        for t, s in ((x, xs), (sc, scs), (sh, shs)):
            assert t.double().reshape(-1).tolist() == vec(s)
        out = oracle_mod(orc, x, sc, sh, "bf16", "full", eps=float(eps))
        assert out.double().reshape(-1).tolist() == vec(exps), (xs, exps)
        n += 1
    assert n >= 4


def test_t_output_is_the_pre_shift_value(orc):
    x, sc, sh = mod_inputs(1, 5, 48, "bf16", "bcast")
    out, t = oracle_mod(orc, x, sc, sh, "bf16", "bcast", with_t=True)
    y = (t + sh.float()).to(torch.bfloat16)  # one fp32 add, then one rounding
    assert same_bits(out, y)


@pytest.mark.parametrize("dtype", DTYPES)
def test_bcast_equals_expanded_and_batches(orc, dtype):
    x, sc, sh = mod_inputs(3, 7, 45, dtype, "bcast")
    a = oracle_mod(orc, x, sc, sh, dtype, "bcast")
    b = oracle_mod(orc, x, sc.expand(3, 7, 45).contiguous(), sh.expand(3, 7, 45).contiguous(),
                   dtype, "full")
    assert same_bits(a, b)
    perm = torch.tensor([1, 2, 0])
    c = oracle_mod(orc, x[perm].contiguous(), sc[perm].contiguous(), sh[perm].contiguous(),
                   dtype, "bcast")
    assert same_bits(a[perm].contiguous(), c)


def test_rows_threads_agree(orc):
    x, sc, sh = mod_inputs(2, 21, 100, "bf16", "bcast")
    full = oracle_mod(orc, x, sc, sh, "bf16", "bcast")
    assert same_bits(full, oracle_mod(orc, x, sc, sh, "bf16", "bcast", threads=4))
    rows = [41, 0, 20, 21]
    part = oracle_mod(orc, x, sc, sh, "bf16", "bcast", rows=rows).reshape(42, 100)
    for r in rows:
        assert same_bits(part[r], full.reshape(42, 100)[r])


def test_degenerate_rows(orc):
    """A zero row with eps = 0 divides 0 by 0: NaN, as IEEE arithmetic gives.
    With eps > 0 the zero row normalises to 0 and the output is the shift."""
    x = torch.zeros((1, 2, 8), dtype=torch.float32)
    sc = torch.full((1, 1, 8), 0.5)
    sh = torch.full((1, 1, 8), 0.25)
    assert torch.isnan(oracle_mod(orc, x, sc, sh, "fp32", "bcast", eps=0.0)).all()
    assert torch.equal(oracle_mod(orc, x, sc, sh, "fp32", "bcast", eps=1e-6),
                       torch.full((1, 2, 8), 0.25))
