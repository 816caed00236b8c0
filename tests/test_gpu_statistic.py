"""GPU parity of the row statistic ms = RN32(mean(x^2)) on rows built to sit
on, or next to, its rounding boundaries, and on rows whose squares overflow
fp32, fall below its normal range or are not finite -- through every kernel
that computes it: the staged kernel (16-byte aligned rows), the phased kernel
(odd pitch), the register kernel (8-byte rows and sub-views off a 16-byte
boundary), the two-pass kernel (long rows), the fused op and the grouped
launch.  Criterion: bit-exact against the oracle.

Boundary rows (tests/_cases.py, boundary_tensor): the squares sum to exactly
D * (1 + k * 2^-24), a midpoint between two fp32 means (k odd), or just above
or below one; every row a seeded permutation, optionally scaled by 2^j (the
squares by 4^j: the same boundaries).  eps = 0 and shift = -2^j, scale = 0 expose r in
the output: an element x = 2^j gives y = 2^j r - 2^j exactly.  Which of
these rows need the exact path depends on the pair's bound; ties always do.

Every test here runs with the exact row statistic (dit_set_statistic); the
last one repeats the boundary rows with the fast statistic under its own
criterion.
"""
import zlib

import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import boundary_tensor, oracle_fused, oracle_mod
from _gpu import assert_bit_exact, ensure_built, modulation_stats, offset_copy
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.fixture(autouse=True)
def _exact_statistic():
    with dit.statistic("exact"):
        yield


def exposing_vectors(B, D, dtype, scale_exp=0, full_L=None):
    shape = (B, full_L if full_L else 1, D)
    sc = torch.zeros(shape, dtype=TORCH_DTYPES[dtype])
    sh = torch.full(shape, -(2.0 ** scale_exp), dtype=TORCH_DTYPES[dtype])
    return sc, sh


CASES = [  # (B, L, D, dtype) -- the kernel each reaches
    (1, 24, 1024, "bf16"), (2, 12, 2048, "bf16"), (1, 16, 3072, "bf16"),
    (1, 16, 4096, "bf16"), (2, 8, 4608, "bf16"), (1, 16, 4096, "fp16"),
    (1, 12, 2048, "fp32"), (1, 8, 4096, "fp32"),                       # staged
    (1, 16, 3077, "bf16"), (1, 16, 3077, "fp16"), (1, 9, 3077, "fp32"),  # phased
    (1, 16, 3076, "bf16"), (2, 5, 3080, "fp16"),                       # 8-byte rows
    (1, 8, 20000, "bf16"), (1, 4, 9000, "fp32"),                       # two-pass
    (3, 5, 64, "bf16"), (1, 8, 8192, "bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_modulation_on_rounding_boundaries(orc, case):
    B, L, D, dtype = case
    for scale_exp in ((0, 6) if dtype == "fp16" else (0, 20, -30)):
        seed = zlib.crc32(repr(case).encode()) % 1000 + scale_exp
        x, _ = boundary_tensor(B, L, D, dtype, seed=seed, scale_exp=scale_exp)
        sc, sh = exposing_vectors(B, D, dtype, scale_exp)
        out = dit.rmsnorm_modulate(x.cuda(), sc.cuda(), sh.cuda(), 0.0)
        torch.cuda.synchronize()
        ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", 0.0, with_t=True)
        modulation_stats(out, ref, t.numpy(), dtype, f"{case} 2^{scale_exp}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_boundaries_off_a_16_byte_boundary(orc, dtype):
    """A sub-view starting one element past an allocation boundary: the
    register kernel with narrow accesses."""
    B, L, D = 1, 12, 2048
    x, _ = boundary_tensor(B, L, D, dtype, seed=77)
    sc, sh = exposing_vectors(B, D, dtype)
    xd, scd, shd = offset_copy(x, 1), offset_copy(sc, 3), offset_copy(sh, 1)
    out = dit.rmsnorm_modulate(xd, scd, shd, 0.0)
    torch.cuda.synchronize()
    ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", 0.0, with_t=True)
    modulation_stats(out.cpu(), ref, t.numpy(), dtype, "sub-view")


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("D", [4096, 3077, 20000])
def test_fused_on_rounding_boundaries(orc, dtype, D):
    """hidden = boundary rows, update = 0, gate = 0: the residual is hidden
    and the modulated output that of the boundary rows, full scale/shift."""
    if dtype == "fp32" and D == 20000:
        D = 9000
    B, L = 1, 8
    h, _ = boundary_tensor(B, L, D, dtype, seed=D + 5)
    u = torch.zeros_like(h)
    g = torch.zeros((B, 1, D), dtype=h.dtype)
    sc, sh = exposing_vectors(B, D, dtype, full_L=L)
    res, mod = dit.gate_add_rmsnorm_modulate(h.cuda(), u.cuda(), g.cuda(), sc.cuda(), sh.cuda(),
                                             0.0)
    torch.cuda.synchronize()
    rr, rm, t = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "full", 0.0, with_t=True)
    assert_bit_exact(res, rr, "residual")
    modulation_stats(mod, rm, t.numpy(), dtype, f"fused D={D}")


def test_grouped_on_rounding_boundaries(orc):
    probs, refs = [], []
    for D, seed in ((4096, 1), (2048, 2)):
        x, _ = boundary_tensor(1, 12, D, "bf16", seed=seed)
        sc, sh = exposing_vectors(1, D, "bf16")
        probs.append((x.cuda(), sc.cuda(), sh.cuda()))
        refs.append(oracle_mod(orc, x, sc, sh, "bf16", "bcast", 0.0, with_t=True))
    outs = dit.rmsnorm_modulate_grouped(probs, 0.0)
    torch.cuda.synchronize()
    for o, (r, t) in zip(outs, refs):
        modulation_stats(o, r, t.numpy(), "bf16", "grouped")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [4096, 3077, 20000])
def test_squares_beyond_fp32_range(orc, dtype, D):
    """Rows whose squares overflow fp32 (one element 3e19, or 2^64, next to
    ordinary values: the mean stays finite), rows of only +inf, rows whose
    squares are fp32 subnormals or round to zero."""
    B, L = 1, 8
    rng = np.random.default_rng(D)
    rows = rng.standard_normal((L, D))
    rows[0, 5] = 3e19
    rows[1, :] = np.inf
    rows[2, 7] = 2.0 ** 64
    rows[2, 8] = -(2.0 ** 64)
    rows[3] = rng.standard_normal(D) * 2.0 ** -70   # squares near 2^-140: subnormal
    rows[4] = rng.standard_normal(D) * 2.0 ** -80   # squares round to zero
    rows[5] *= 2.0 ** 60                             # mean near 2^120
    rows[6, 0] = np.inf
    x = torch.tensor(rows[None], dtype=torch.float64).to(TORCH_DTYPES[dtype])
    sc = torch.tensor(rng.normal(0, 0.1, (B, 1, D))).to(x.dtype)
    sh = torch.tensor(rng.normal(0, 0.1, (B, 1, D))).to(x.dtype)
    for eps in (0.0, 1e-6):
        out = dit.rmsnorm_modulate(x.cuda(), sc.cuda(), sh.cuda(), eps)
        torch.cuda.synchronize()
        ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", eps, with_t=True)
        modulation_stats(out, ref, t.numpy(), dtype, f"D={D} eps={eps}")
        o = out.cpu().float()
        assert torch.isfinite(o[0, 0]).all() and torch.isfinite(o[0, 2]).all()
        assert torch.isnan(o[0, 1]).all()


@pytest.mark.parametrize("case", CASES[::3], ids=lambda c: "x".join(map(str, c)))
def test_fast_statistic_on_rounding_boundaries(orc, case):
    """The same rows with the fast statistic: its criterion, not bit-exact."""
    B, L, D, dtype = case
    x, _ = boundary_tensor(B, L, D, dtype, seed=11)
    sc, sh = exposing_vectors(B, D, dtype)
    with dit.statistic("fast"):
        assert dit.get_statistic() == "fast"
        out = dit.rmsnorm_modulate(x.cuda(), sc.cuda(), sh.cuda(), 0.0)
        torch.cuda.synchronize()
    ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", 0.0, with_t=True)
    modulation_stats(out, ref, t.numpy(), dtype, f"fast {case}", exact=False)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [4096, 3077, 20000])
def test_fast_statistic_outside_its_range(orc, dtype, D):
    """The fast statistic on rows whose fp32 sum of squares leaves
    [2^-100, 2^100]: a square that overflows (3e19, 2^64: the mean stays
    finite), rows of +inf or holding one, a mean near 2^120, squares near
    2^-120 and squares that round to zero.  The kernels sum such rows again
    scaled by 2^-64 or 2^64; every element must meet the fast criterion,
    NaN exactly where the oracle has NaN.  (A mean square in fp32's
    subnormal range with eps = 0 is left out: there the fast statistic may
    be one subnormal step of ms off, which the fp32 criterion does not
    allow.)"""
    B, L = 1, 8
    rng = np.random.default_rng(D + 1)
    rows = rng.standard_normal((L, D))
    rows[0, 5] = 3e19
    rows[1, :] = np.inf
    rows[2, 7] = 2.0 ** 64
    rows[2, 8] = -(2.0 ** 64)
    rows[3] *= 2.0 ** -60   # squares near 2^-120: the sum below 2^-100
    rows[4] *= 2.0 ** -80   # squares round to zero
    rows[5] *= 2.0 ** 60    # mean near 2^120
    rows[6, 0] = np.inf
    x = torch.tensor(rows[None], dtype=torch.float64).to(TORCH_DTYPES[dtype])
    sc = torch.tensor(rng.normal(0, 0.1, (B, 1, D))).to(x.dtype)
    sh = torch.tensor(rng.normal(0, 0.1, (B, 1, D))).to(x.dtype)
    with dit.statistic("fast"):
        for eps in (0.0, 1e-6):
            out = dit.rmsnorm_modulate(x.cuda(), sc.cuda(), sh.cuda(), eps)
            u = torch.zeros_like(x)
            g = torch.zeros((B, 1, D), dtype=x.dtype)
            res, mod = dit.gate_add_rmsnorm_modulate(x.cuda(), u.cuda(), g.cuda(), sc.cuda(),
                                                     sh.cuda(), eps)
            torch.cuda.synchronize()
            ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", eps, with_t=True)
            modulation_stats(out, ref, t.numpy(), dtype, f"fast D={D} eps={eps}", exact=False)
            modulation_stats(mod, ref, t.numpy(), dtype, f"fast fused D={D} eps={eps}",
                             exact=False)
            o = out.cpu().float()
            assert torch.isfinite(o[0, 0]).all() and torch.isfinite(o[0, 2]).all()
            assert torch.isnan(o[0, 1]).all()
