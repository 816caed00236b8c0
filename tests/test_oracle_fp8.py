"""Pins for the oracle's OCP E4M3 codec and its FP8-output modulation.

The codec: every one of the 256 codes decoded against the format definition
(written out independently here) and against torch.float8_e4m3fn; encoding
of random fp32 values against a brute-force search for the nearest of the
127 non-negative finite values (ties to the even code), against torch's
conversion for in-range values, and hand-derived ties
(tests/golden/e4m3_ties.txt).  The FP8 modulation: the quantised value of
the fp32 modulation of the same inputs, converted by torch; saturation; the
fused op's residual unchanged.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from _cases import mod_inputs, rga_inputs
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ties.txt")


def _definition(code: int):
    """Value of an E4M3 code from the format definition (None for NaN)."""
    s = -1 if code & 0x80 else 1
    e, m = (code >> 3) & 15, code & 7
    if e == 15 and m == 7:
        return None
    if e == 0:
        return s * Fraction(m, 2 ** 9)
    return s * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def test_decode_all_codes(orc):
    got = orc.e4m3_decode(range(256))
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        want = _definition(c)
        if want is None:
            assert math.isnan(got[c]) and math.isnan(ref[c]), c
        else:
            assert Fraction(float(got[c])) == want, c
            assert Fraction(float(ref[c])) == want, c
            if want == 0:
                assert math.copysign(1, got[c]) == (-1 if c & 0x80 else 1)


_POS = [(c, _definition(c)) for c in range(127)]  # non-negative finite, increasing


def _nearest(v: float) -> int:
    """Code of the E4M3 value nearest to v (ties to the even code), with
    saturation at 448, by brute force over all non-negative finite codes."""
    a = abs(Fraction(v))
    sign = 0x80 if math.copysign(1, v) < 0 else 0
    if a >= 448:
        return sign | 0x7E
    best = min(_POS, key=lambda cv: (abs(cv[1] - a), cv[0] & 1))
    return sign | best[0]


def test_encode_brute_force(orc):
    rng = np.random.default_rng(8)
    v = np.concatenate([rng.uniform(-500, 500, 1500), rng.normal(0, 1, 1500),
                        rng.normal(0, 0.02, 1000), rng.normal(0, 2e-3, 500)]).astype(np.float32)
    got = orc.e4m3_encode(v)
    for x, g in zip(v.tolist(), got.tolist()):
        assert g == _nearest(x), (x, g, _nearest(x))


def test_encode_against_torch(orc):
    rng = np.random.default_rng(9)
    v = np.concatenate([rng.uniform(-447.9, 447.9, 20000),
                        rng.normal(0, 0.05, 20000)]).astype(np.float32)
    got = orc.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)


def test_encode_special_values(orc):
    got = orc.e4m3_encode([float("inf"), float("-inf"), float("nan"), 0.0, -0.0])
    assert got.tolist()[:2] == [0x7E, 0xFE]
    assert got[2] & 0x7F == 0x7F
    assert got.tolist()[3:] == [0x00, 0x80]


def _golden():
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            inp, exp, _ = (c.strip() for c in line.split("|"))
            yield float(eval(inp)), Fraction(eval(exp)) if "e" not in exp else Fraction(exp)


def test_ties_golden(orc):
    for inp, exp in _golden():
        code = int(orc.e4m3_encode([inp])[0])
        assert _definition(code) == exp, (inp, code)


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("quant_scale", [1.0, 0.005, 3.0])
def test_modulate_fp8_is_quantised_fp32_modulation(orc, dtype, quant_scale):
    """q = e4m3(fl(y * fl(1/s))): y from the oracle's fp32 modulation of the
    same input values (exact widening), the product and the conversion by
    torch; values that saturate are +-448."""
    B, L, D = 2, 9, 96
    x, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="fp8")
    out = torch.empty((B, L, D), dtype=torch.uint8)
    orc.rmsnorm_modulate_fp8(out, x, sc, sh, B, L, D, 1e-6, dtype, "bcast", quant_scale)
    y = torch.empty((B, L, D), dtype=torch.float32)
    orc.rmsnorm_modulate(y, x.float(), sc.float(), sh.float(), B, L, D, 1e-6, "fp32", "bcast")
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(quant_scale, dtype=torch.float32)
    q = y * inv
    sat = q.abs() >= 448
    want = q.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(out[~sat], want[~sat])
    assert torch.all(out[sat] & 0x7F == 0x7E)
    if quant_scale == 0.005:
        assert bool(sat.any())  # the saturating case is exercised


@pytest.mark.parametrize("layouts", [("bcast", "bcast"), ("full", "full")])
def test_fused_fp8(orc, layouts):
    glay, mlay = layouts
    B, L, D, dtype = 2, 5, 64, "bf16"
    h, u, g = rga_inputs(B, L, D, dtype, glay, tag="fp8f")
    _, sc, sh = mod_inputs(B, L, D, dtype, mlay, tag="fp8f")
    res = torch.empty_like(h)
    out = torch.empty((B, L, D), dtype=torch.uint8)
    orc.gate_add_rmsnorm_modulate_fp8(res, out, h, u, g, sc, sh, B, L, D, 1e-6, dtype, glay,
                                      mlay, 0.5)
    res2, mod2 = torch.empty_like(h), torch.empty_like(h)
    orc.gate_add_rmsnorm_modulate(res2, mod2, h, u, g, sc, sh, B, L, D, 1e-6, dtype, glay, mlay)
    assert torch.equal(res.view(torch.int16), res2.view(torch.int16))
    out2 = torch.empty((B, L, D), dtype=torch.uint8)
    orc.rmsnorm_modulate_fp8(out2, res, sc, sh, B, L, D, 1e-6, dtype, mlay, 0.5)
    assert torch.equal(out, out2)  # fused = residual gate, then the FP8 modulation
