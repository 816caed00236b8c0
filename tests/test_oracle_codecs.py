"""Pins for the oracle's dtype codecs (bf16 / fp16 <-> fp32).

The codecs are pinned three ways: against the IEEE-754 definition (exact
values of every bit pattern, brute-force nearest-value search), against
library conversions (torch's bf16, numpy's float16), and against the
hand-derived tie cases in tests/golden/rounding_ties.txt.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from _exact import bf16_value, fp16_value, round_to

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _all_patterns():
    return np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)


def _special_f32():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65520.0, 65536.0, 1e-8, 5.96e-8, 6.1e-5,
            3.4028235e38, -3.4028235e38, np.inf, -np.inf, 1e-40, -1e-45, 2.0 ** -133,
            2.0 ** -134, 2.0 ** -24, 2.0 ** -25, 2.0 ** -14]
    return np.array(vals, dtype=np.float32)


def _random_f32(n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    # more samples near 1 and in the fp16 subnormal range, where ties are dense
    near = rng.integers(0x3F000000, 0x40000000, size=n // 4, dtype=np.uint64).astype(np.uint32)
    small = rng.integers(0x33000000, 0x38800000, size=n // 4, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([bits, near, small]).view(np.float32)


def test_bf16_decode_every_pattern(orc):
    pats = _all_patterns()
    got = orc.decode(pats, "bf16")
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    # and against the exact value of the format definition (finite patterns)
    for b in list(range(0, 0x7F80, 97)) + [0x7F7F, 0x0001, 0x8001, 0xFF7F]:
        assert Fraction(float(got[b])) == bf16_value(b)


def test_fp16_decode_every_pattern(orc):
    pats = _all_patterns()
    got = orc.decode(pats, "fp16")
    ref = pats.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    for b in list(range(0, 0x7C00, 89)) + [0x7BFF, 0x0001, 0x03FF, 0x0400, 0xFBFF]:
        assert Fraction(float(got[b])) == fp16_value(b)


def test_bf16_encode_matches_torch(orc):
    x = np.concatenate([_special_f32(), _random_f32(1 << 20, 1)])
    got = orc.encode(x, "bf16")
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(orc.decode(got[nan], "bf16")))  # NaN stays NaN


def test_fp16_encode_matches_numpy(orc):
    x = np.concatenate([_special_f32(), _random_f32(1 << 20, 2)])
    got = orc.encode(x, "fp16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(orc.decode(got[nan], "fp16")))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_encode_is_nearest_by_brute_force(orc, dtype):
    """Brute force: the nearest value of the format (ties to even pattern),
    found by search over every finite value, equals the oracle's rounding."""
    x = _random_f32(4000, 3)
    lim = 3.38e38 if dtype == "bf16" else 65504.0
    x = x[np.isfinite(x) & (np.abs(x) < lim)]
    got = orc.encode(x, dtype)
    for v, g in zip(x.tolist(), got.tolist()):
        assert round_to(Fraction(v), dtype) == g, (v, hex(g))


def _golden_rows(name):
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        yield [s.strip() for s in line.split("|")]


def test_rounding_ties_golden(orc):
    n = 0
    for dtype, inp, exp, why in _golden_rows("rounding_ties.txt"):
        v = float(eval(inp, {"__builtins__": {}}))
        assert Fraction(float(np.float32(v))) == Fraction(v), inp
        bits = int(orc.encode(np.array([v], np.float32), dtype)[0])
        value = orc.decode(np.array([bits], np.uint16), dtype)[0]
        if exp == "inf":
            assert np.isinf(value) and value > 0, (inp, why)
        else:
            e = eval(exp, {"__builtins__": {}})
            assert Fraction(float(value)) == Fraction(e), (dtype, inp, exp, why, value)
        n += 1
    assert n >= 20
