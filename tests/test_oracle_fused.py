"""Pins for the oracle's fused op: residual gate then modulation of the stored
residual, in one pass.

The fused op has no separate definition on the pages beyond the two
operations it joins (the residual gate, sglang PR #29361, Motivation; the
modulation, prhub summary of sglang PR #34172, "key source snippet"), so it is
pinned as their composition -- whose parts are pinned in the other oracle
test files -- plus exact brute force on tiny shapes.
"""
import numpy as np
import pytest
import torch

from _cases import mod_inputs, oracle_fused, oracle_mod, oracle_rga, rga_inputs, same_bits
from _exact import round_to, sqrt_fraction, ulp_distance, value_of, words

DTYPES = ["bf16", "fp16", "fp32"]
COMBOS = [("bcast", "bcast"), ("full", "bcast"), ("bcast", "full"), ("full", "full")]
EPS32 = float(np.float32(1e-6))


def _inputs(B, L, D, dtype, gl, ml, tag="fused"):
    h, u, g = rga_inputs(B, L, D, dtype, gl, tag=tag)
    _, sc, sh = mod_inputs(B, L, D, dtype, ml, tag=tag)
    return h, u, g, sc, sh


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("gl,ml", COMBOS)
def test_fused_is_composition(orc, dtype, gl, ml):
    h, u, g, sc, sh = _inputs(2, 13, 96, dtype, gl, ml)
    res, mod = oracle_fused(orc, h, u, g, sc, sh, dtype, gl, ml)
    r2 = oracle_rga(orc, h, u, g, dtype, gl)
    m2 = oracle_mod(orc, r2, sc, sh, dtype, ml)
    assert same_bits(res, r2)
    assert same_bits(mod, m2)


def test_modulation_reads_the_rounded_residual(orc):
    """The RMS is taken over the residual as stored (bf16), not over the fp32
    sum: feeding the fp32 sums to the modulation gives a different result on
    some elements, so the composition pin above can tell the two apart."""
    h, u, g, sc, sh = _inputs(1, 64, 128, "bf16", "bcast", "bcast")
    _, mod = oracle_fused(orc, h, u, g, sc, sh, "bf16", "bcast", "bcast")
    s32 = (h.float() + u.float() * g.float()).contiguous()  # unrounded sums
    m32 = oracle_mod(orc, s32, sc.float(), sh.float(), "fp32", "bcast").to(torch.bfloat16)
    assert not same_bits(mod, m32)


@pytest.mark.parametrize("dtype", DTYPES)
def test_inplace_residual(orc, dtype):
    h, u, g, sc, sh = _inputs(2, 9, 64, dtype, "bcast", "bcast")
    res, mod = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast")
    hh = h.clone()
    res2, mod2 = oracle_fused(orc, hh, u, g, sc, sh, dtype, "bcast", "bcast", residual_out=hh)
    assert same_bits(hh, res) and same_bits(mod2, mod)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("shape", [(1, 2, 3), (2, 2, 16), (1, 3, 33)])
def test_exact_bruteforce(orc, dtype, shape):
    """Residual: the exact h + u*g rounded once (the fp32 steps are exact for
    these magnitudes, which the test checks).  Modulated output: the exact
    modulation of that rounded residual, within the bound of
    test_oracle_modulate (3u|t| + u|y|) of a rounding boundary."""
    from fractions import Fraction
    U = Fraction(1, 1 << 24)
    B, L, D = shape
    h, u, g, sc, sh = _inputs(B, L, D, dtype, "bcast", "bcast", tag=("bf", shape))
    res, mod = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast", eps=EPS32)
    hw, uw, gw, sw, shw = words(h), words(u), words(g), words(sc), words(sh)
    rw, mw = words(res), words(mod)
    for r in range(B * L):
        b = r // L
        xs = []
        for d in range(D):
            q = value_of(hw[r * D + d], dtype) + value_of(uw[r * D + d], dtype) * value_of(gw[b * D + d], dtype)
            assert rw[r * D + d] == round_to(q, dtype)
            xs.append(value_of(rw[r * D + d], dtype))
        rinv = 1 / sqrt_fraction(sum(v * v for v in xs) / D + Fraction(EPS32))
        for d in range(D):
            t = xs[d] * rinv * (1 + value_of(sw[b * D + d], dtype))
            y = t + value_of(shw[b * D + d], dtype)
            want = round_to(y, dtype)
            got = mw[r * D + d]
            if got != want:
                assert ulp_distance(got, want, dtype) == 1
                mid = (value_of(got, dtype) + value_of(want, dtype)) / 2
                assert abs(y - mid) <= 3 * U * abs(t) + U * abs(y)


def test_threads_and_rows_agree(orc):
    h, u, g, sc, sh = _inputs(2, 17, 80, "bf16", "bcast", "bcast")
    res, mod = oracle_fused(orc, h, u, g, sc, sh, "bf16", "bcast", "bcast")
    res2, mod2 = oracle_fused(orc, h, u, g, sc, sh, "bf16", "bcast", "bcast", threads=3)
    assert same_bits(res, res2) and same_bits(mod, mod2)
    rows = [0, 33, 17, 16]
    res3, mod3 = oracle_fused(orc, h, u, g, sc, sh, "bf16", "bcast", "bcast", rows=rows)
    for r in rows:
        assert same_bits(res3.reshape(34, 80)[r], res.reshape(34, 80)[r])
        assert same_bits(mod3.reshape(34, 80)[r], mod.reshape(34, 80)[r])
