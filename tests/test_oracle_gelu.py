"""Pins for the oracle's tanh-GELU (FFN activation of the LTX-2 blocks,
prhub summary of sglang PR #34172, "implementation breakdown" item 3):
gelu(x) = 0.5 * x * (1 + tanh(sqrt(2/pi) * (x + 0.044715 * x^3))), in double,
rounded once to the dtype.

Pins: the single rounding of a double (brute force on exact rationals,
including a case that a naive double -> float -> bf16 conversion gets wrong);
torch's own float64 GELU; the identity gelu(x) - gelu(-x) = x; closed forms at
0 and for large |x|.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from _exact import round_to, value_of
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES, draw, seed_for

DTYPES = ["bf16", "fp16", "fp32"]


def _gelu(orc, x, dtype):
    out = torch.empty_like(x)
    orc.gelu_tanh(out, x, dtype)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_double_rounding_by_brute_force(orc, dtype):
    rng = np.random.default_rng(11)
    lim = 3e38 if dtype == "bf16" else 6e4
    v = rng.standard_normal(3000) * np.exp(rng.uniform(-20, 20, 3000))
    v = v[np.abs(v) < lim]
    got = orc.round_double(v, dtype)
    for x, g in zip(v.tolist(), got.tolist()):
        assert round_to(Fraction(x), dtype) == g, (x, hex(g))


def test_round_to_odd_avoids_double_rounding(orc):
    """1 + 2^-8 + 2^-30 lies just above the bf16 tie between 1 and 1 + 2^-7;
    a float intermediate rounded to nearest is exactly the tie (2^-30 is below
    half an fp32 ulp) and would then round to 1.  The correct result is
    1 + 2^-7."""
    v = 1 + 2.0 ** -8 + 2.0 ** -30
    assert float(np.float32(v)) == 1 + 2.0 ** -8
    bits = int(orc.round_double([v], "bf16")[0])
    assert value_of(bits, "bf16") == 1 + Fraction(1, 128)
    bits = int(orc.round_double([-v], "bf16")[0])
    assert value_of(bits, "bf16") == -(1 + Fraction(1, 128))
    # exactly on the tie: to even
    assert value_of(int(orc.round_double([1 + 2.0 ** -8], "bf16")[0]), "bf16") == 1


@pytest.mark.parametrize("dtype", DTYPES)
def test_against_torch_float64(orc, dtype):
    """torch's float64 GELU (same formula; its double evaluation differs from
    the oracle's by ~1e-16 relative): equal after rounding, except where the
    float64 value lies within 1e-13 (relative) of the midpoint between two
    neighbours -- then one ulp apart."""
    from _exact import ulp_distance, words
    x = draw("act", (64, 257), seed_for("gelu", dtype), dtype) * 3
    x = x.clamp_min(-4.0).to(TORCH_DTYPES[dtype])  # where the tanh form is well conditioned
    got = words(_gelu(orc, x, dtype))
    ref = F.gelu(x.double(), approximate="tanh").reshape(-1).tolist()
    near = 0
    for g, v in zip(got, ref):
        want = round_to(Fraction(v), dtype)
        if g != want and ulp_distance(g, want, dtype) != 0:  # (+0 and -0 are equal)
            assert ulp_distance(g, want, dtype) == 1
            mid = (value_of(g, dtype) + value_of(want, dtype)) / 2
            assert abs(Fraction(v) - mid) <= abs(Fraction(v)) * Fraction(1, 10 ** 13)
            near += 1
    assert near <= len(ref) // 1000


def _gelu_decimal(v: float) -> Fraction:
    """gelu(v) to 50 digits: v / (1 + exp(-2z)) in decimal arithmetic
    (1 + tanh(z) = 2 / (1 + exp(-2z)))."""
    from decimal import Decimal, localcontext
    with localcontext() as ctx:
        ctx.prec = 50
        x = Decimal(v)
        k = (Decimal(2) / Decimal("3.14159265358979323846264338327950288419716939937510")).sqrt()
        z = k * (x + Decimal("0.044715") * x * x * x)
        return Fraction(x / (1 + (-2 * z).exp()))


@pytest.mark.parametrize("dtype", DTYPES)
def test_against_50_digit_evaluation(orc, dtype):
    """All x, including the negative tail: the oracle's rounded value equals
    the correctly rounded 50-digit value (up to near-ties, as above)."""
    from _exact import ulp_distance, words
    vals = np.concatenate([np.linspace(-12, 6, 400), np.random.default_rng(3).normal(0, 3, 400)])
    x = torch.tensor(vals, dtype=torch.float64).to(TORCH_DTYPES[dtype])
    got = words(_gelu(orc, x, dtype))
    for g, v in zip(got, x.double().tolist()):
        exact = _gelu_decimal(v)
        want = round_to(exact, dtype)
        if g != want and ulp_distance(g, want, dtype) != 0:
            assert ulp_distance(g, want, dtype) == 1, (v, g, want)
            mid = (value_of(g, dtype) + value_of(want, dtype)) / 2
            assert abs(exact - mid) <= abs(exact) * Fraction(1, 10 ** 13)


@pytest.mark.parametrize("dtype", DTYPES)
def test_odd_identity(orc, dtype):
    """gelu(x) - gelu(-x) = x exactly; after the two roundings the difference
    is within half an ulp of each result."""
    x = (draw("act", (4096,), seed_for("gelu-odd", dtype), dtype).float() * 4).to(TORCH_DTYPES[dtype])
    a = _gelu(orc, x, dtype).double()
    b = _gelu(orc, -x, dtype).double()
    mant = {"bf16": 8, "fp16": 11, "fp32": 24}[dtype]

    def half_ulp(v):
        e = torch.floor(torch.log2(v.abs().clamp_min(1e-30)))
        return torch.pow(2.0, e - mant)
    assert torch.all((a - b - x.double()).abs() <= half_ulp(a) + half_ulp(b) + 1e-30)


@pytest.mark.parametrize("dtype", DTYPES)
def test_closed_forms(orc, dtype):
    t = TORCH_DTYPES[dtype]
    x = torch.tensor([0.0, 12.0, 30.0, -40.0], dtype=t)
    y = _gelu(orc, x, dtype).double().tolist()
    assert y[0] == 0.0
    assert y[1] == 12.0 and y[2] == 30.0  # tanh(z) = 1 to double precision
    assert y[3] == 0.0  # 0.5 * x * (1 + tanh(z)) underflows to (-)0
    # 1: 0.5 * (1 + tanh(sqrt(2/pi) * 1.044715))
    one = 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * 1.044715))
    y1 = _gelu(orc, torch.tensor([1.0], dtype=t), dtype).double().item()
    assert abs(y1 - one) <= {"bf16": 2 ** -8, "fp16": 2 ** -11, "fp32": 2 ** -24}[dtype]
