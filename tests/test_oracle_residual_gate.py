"""Pins for the oracle's residual gate  out = hidden + update * gate
(sglang PR #29361, section Motivation; full [B, L, D] or [B, 1, D] gate).

Each pin is fixed by something other than the oracle: invariants (gate 0,
broadcast = expanded full gate, batch permutation), library routines (torch's
own dtype add and multiply for gate 1 and hidden 0), hand-derived worked
examples, and exact rational brute force on tiny shapes.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from _cases import bits, oracle_rga, rga_inputs, same_bits
from _exact import round_to, round_to_fp32, ulp_at, ulp_distance, value_of, words
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES

DTYPES = ["bf16", "fp16", "fp32"]
LAYOUTS = ["full", "bcast"]
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_gate_zero_returns_hidden(orc, dtype, layout):
    h, u, g = rga_inputs(2, 5, 37, dtype, layout)
    out = oracle_rga(orc, h, u, torch.zeros_like(g), dtype, layout)
    assert same_bits(out, h)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", LAYOUTS)
def test_gate_one_is_library_add(orc, dtype, layout):
    """gate = 1 makes the product exact, so out = one rounding of h + u, which
    is what torch's own add in the storage dtype computes."""
    h, u, g = rga_inputs(2, 7, 129, dtype, layout)
    out = oracle_rga(orc, h, u, torch.ones_like(g), dtype, layout)
    assert same_bits(out, h + u)


@pytest.mark.parametrize("dtype", DTYPES)
def test_hidden_zero_is_library_mul(orc, dtype):
    """hidden = 0: out = one rounding of update * gate (torch's dtype multiply)."""
    h, u, g = rga_inputs(1, 9, 65, dtype, "full")
    out = oracle_rga(orc, torch.zeros_like(h), u, g, dtype, "full")
    assert same_bits(out, u * g)


@pytest.mark.parametrize("dtype", DTYPES)
def test_bcast_equals_expanded_full_gate(orc, dtype):
    h, u, g = rga_inputs(3, 11, 40, dtype, "bcast")
    a = oracle_rga(orc, h, u, g, dtype, "bcast")
    b = oracle_rga(orc, h, u, g.expand(3, 11, 40).contiguous(), dtype, "full")
    assert same_bits(a, b)


def test_bcast_batch_permutation(orc):
    """Each batch uses its own [1, D] gate row: permuting the batches of all
    inputs permutes the batches of the output."""
    h, u, g = rga_inputs(4, 6, 33, "bf16", "bcast")
    perm = torch.tensor([2, 0, 3, 1])
    a = oracle_rga(orc, h, u, g, "bf16", "bcast")
    b = oracle_rga(orc, h[perm].contiguous(), u[perm].contiguous(), g[perm].contiguous(),
                   "bf16", "bcast")
    assert same_bits(a[perm].contiguous(), b)
    # and the gate really differs between batches (the check has teeth)
    c = oracle_rga(orc, h, u, g[[0, 0, 0, 0]].contiguous(), "bf16", "bcast")
    assert not same_bits(a, c)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 2, 3), (2, 3, 7), (2, 5, 9), (1, 3, 31),
                                   (2, 2, 127)])
def test_exact_rational_bruteforce(orc, dtype, layout, shape):
    """For every element: (a) the oracle equals the definition p = fl32(u*g),
    s = fl32(h + p), out = rnd_dtype(s), each rounding found by brute-force
    nearest-value search on exact rationals; (b) it is within 1 ulp of the
    exact real h + u*g rounded once (bf16/fp16; for fp32, within the
    two-rounding bound), and equal to it whenever the fp32 steps were exact."""
    B, L, D = shape
    h, u, g = rga_inputs(B, L, D, dtype, layout, tag=("bf", shape))
    # widen the magnitude range so that fp32 sums are sometimes inexact
    h = (h.float() * torch.tensor([1.0, 2.0 ** 9, 2.0 ** -9]).repeat(D)[:D]).to(h.dtype)
    out = oracle_rga(orc, h, u, g, dtype, layout)
    hw, uw, gw, ow = words(h), words(u), words(g), words(out)
    for r in range(B * L):
        grow = r if layout == "full" else r // L
        for d in range(D):
            i = r * D + d
            hv, uv, gv = (value_of(hw[i], dtype), value_of(uw[i], dtype),
                          value_of(gw[grow * D + d], dtype))
            p = value_of(round_to_fp32(uv * gv), "fp32")
            s = value_of(round_to_fp32(hv + p), "fp32")
            want = round_to(s, dtype) if dtype != "fp32" else round_to_fp32(s)
            assert ow[i] == want, (r, d)
            q = hv + uv * gv
            single = round_to(q, dtype) if dtype != "fp32" else round_to_fp32(q)
            steps_exact = (p == uv * gv) and (s == hv + p)
            if steps_exact:
                assert ow[i] == single
            elif dtype == "fp32":
                # two fp32 roundings: |out - q| <= ulp(p)/2 + ulp(s)/2
                err = abs(value_of(ow[i], "fp32") - q)
                assert err <= (ulp_at(p, "fp32") + ulp_at(s, "fp32")) / 2
            else:
                # bf16/fp16: the product is exact in fp32, so only the fp32 sum
                # and the final narrowing round: at most one ulp of the dtype
                assert ulp_distance(ow[i], single, dtype) <= 1


def _golden_rows(name):
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        yield [s.strip() for s in line.split("|")]


def test_worked_examples_golden(orc):
    n = 0
    for dtype, hs, us, gs, exps, why in _golden_rows("residual_gate_worked.txt"):
        ev = lambda s: float(eval(s, {"__builtins__": {}}))
        t = TORCH_DTYPES[dtype]
        h = torch.tensor([[[ev(hs)]]], dtype=torch.float64).to(t)
        u = torch.tensor([[[ev(us)]]], dtype=torch.float64).to(t)
        g = torch.tensor([[[ev(gs)]]], dtype=torch.float64).to(t)
        for v, s in ((h, hs), (u, us), (g, gs)):  # inputs must be exact in dtype
            assert Fraction(float(v.double())) == Fraction(ev(s)), (dtype, s)
        out = oracle_rga(orc, h, u, g, dtype, "full")
        assert Fraction(float(out.double())) == Fraction(ev(exps)), (dtype, hs, us, gs, why)
        n += 1
    assert n >= 14


def test_row_selection_matches_full(orc):
    h, u, g = rga_inputs(2, 9, 50, "bf16", "bcast")
    full = oracle_rga(orc, h, u, g, "bf16", "bcast")
    rows = [17, 0, 9, 8, 3]
    sel = oracle_rga(orc, h, u, g, "bf16", "bcast", rows=rows,
                     out=torch.zeros_like(h))
    flat_full, flat_sel = full.reshape(18, 50), sel.reshape(18, 50)
    for r in range(18):
        if r in rows:
            assert same_bits(flat_sel[r], flat_full[r])
        else:
            assert np.all(bits(flat_sel[r]) == 0)  # untouched


@pytest.mark.parametrize("dtype", DTYPES)
def test_threads_and_inplace_agree(orc, dtype):
    h, u, g = rga_inputs(2, 33, 70, dtype, "bcast")
    one = oracle_rga(orc, h, u, g, dtype, "bcast")
    many = oracle_rga(orc, h, u, g, dtype, "bcast", threads=5)
    assert same_bits(one, many)
    hh = h.clone()
    oracle_rga(orc, hh, u, g, dtype, "bcast", out=hh)  # out aliases hidden
    assert same_bits(hh, one)


def test_bad_arguments_rejected(orc):
    h, u, g = rga_inputs(1, 2, 3, "bf16", "full")
    out = torch.empty_like(h)
    with pytest.raises(ValueError):
        orc.residual_gate_add(out, h, u, g, 1, 2, -3, "bf16", "full")
    with pytest.raises(ValueError):
        orc.residual_gate_add(out, h, u, g, 1, 2, 3, "bf16", "full", rows=[2])
    with pytest.raises(ValueError):
        orc.residual_gate_add(out, None, u, g, 1, 2, 3, "bf16", "full")
    # empty problems are fine and write nothing
    orc.residual_gate_add(None, None, None, None, 0, 5, 7, "bf16", "full")


def test_signed_zero_of_an_underflowing_product(orc):
    """Multiply, then add (reading R1): a product of bf16 subnormals below
    fp32's range rounds to a signed zero first, and +0 + (-0) = +0 in
    round-to-nearest; a fused multiply-add would keep the sign of the exact
    product and give -0.  With hidden = -0 the sum of two negative zeros is
    -0 either way."""
    tiny = 2.0 ** -133  # the smallest bf16 subnormal
    cases = [(0.0, tiny, -tiny, 0x0000), (-0.0, tiny, -tiny, 0x8000),
             (0.0, -tiny, -tiny, 0x0000), (-0.0, tiny, tiny, 0x0000),
             (0.0, 0.0, -1.0, 0x0000)]
    for hv, uv, gv, want in cases:
        h, u, g = (torch.tensor([[[v]]], dtype=torch.float32).to(torch.bfloat16)
                   for v in (hv, uv, gv))
        out = oracle_rga(orc, h, u, g, "bf16", "full")
        assert int(out.view(torch.int16).item()) & 0xFFFF == want, (hv, uv, gv)
