"""GPU parity of the tanh-GELU (dit_gelu_tanh) against the oracle's
double-precision value rounded once.

Criterion: bf16/fp16 -- at most 1 ulp (the fp32 evaluation with the fast
intrinsics is within ~1e-4 relative, so only values near a rounding boundary
move); fp32 -- |gpu - oracle| <= (8 + 8|z|) * 2^-24 * |y| (z's three fp32
roundings are amplified by |2z| inside exp(-2|z|); expf and the division add a
few ulps), plus one subnormal spacing (2^-149): the final rounding of a
result in the subnormal range is absolute, not relative.
"""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _gpu import ensure_built, offset_copy, ulp_distance, values
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES, draw, seed_for

pytestmark = pytest.mark.gpu
DTYPES = ["bf16", "fp16", "fp32"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def oracle_gelu(orc, x, dtype):
    out = torch.empty_like(x)
    orc.gelu_tanh(out, x.contiguous(), dtype)
    return out


def check(gpu, ref, x, dtype, what=""):
    g, r = values(gpu), values(ref)
    assert np.array_equal(np.isnan(g), np.isnan(r)), what
    ok = ~np.isnan(r)
    if dtype == "fp32":
        xv = values(x)[ok]
        z = np.sqrt(2 / np.pi) * (xv + 0.044715 * xv ** 3)
        bound = (8 + 8 * np.abs(z)) * 2.0 ** -24 * np.abs(r[ok]) + 2.0 ** -149
        with np.errstate(invalid="ignore"):  # inf - inf where both are inf
            bad = ~(np.abs(g[ok] - r[ok]) <= bound) & ~(g[ok] == r[ok])
    else:
        bad = ulp_distance(gpu, ref)[ok] > 1
    idx = np.nonzero(bad)[0]
    assert idx.size == 0, f"{what}: {idx.size} bad, first x={values(x)[ok][idx[:4]]} gpu={g[ok][idx[:4]]} oracle={r[ok][idx[:4]]}"
    return int(np.count_nonzero(ulp_distance(gpu, ref)[ok]))


@pytest.mark.parametrize("n", [1, 7, 8, 15, 16, 17, 4095, 100003])
@pytest.mark.parametrize("dtype", DTYPES)
def test_gelu(orc, dtype, n):
    x = (draw("act", (n,), seed_for("gelu", n, dtype), dtype).float() * 4).to(TORCH_DTYPES[dtype])
    out = dit.gelu_tanh(x.cuda())
    torch.cuda.synchronize()
    check(out.cpu(), oracle_gelu(orc, x, dtype), x, dtype, f"{dtype} n={n}")


@pytest.mark.parametrize("offsets", [(1, 1), (1, 0), (3, 2)])
@pytest.mark.parametrize("dtype", DTYPES)
def test_gelu_misaligned_and_in_place(orc, dtype, offsets):
    x = (draw("act", (3, 1001), seed_for("gelu-mis", dtype), dtype).float() * 5).to(TORCH_DTYPES[dtype])
    ref = oracle_gelu(orc, x, dtype)
    xo = offset_copy(x.cuda(), offsets[0])
    out = offset_copy(torch.zeros_like(x).cuda(), offsets[1])
    dit.gelu_tanh(xo, out=out)
    torch.cuda.synchronize()
    check(out.cpu(), ref, x, dtype, "misaligned")
    dit.gelu_tanh(xo, out=xo)  # in place
    torch.cuda.synchronize()
    check(xo.cpu(), ref, x, dtype, "in place")


@pytest.mark.parametrize("dtype", DTYPES)
def test_gelu_special_values(orc, dtype):
    big = {"bf16": 3e38, "fp16": 6e4, "fp32": 3e38}[dtype]
    vals = [0.0, -0.0, float("inf"), float("-inf"), float("nan"), big, -big, 1e-30, -1e-30,
            -5.0, -8.0, -9.5, -10.5, -12.0, 6.0, 12.0]
    x = torch.tensor(vals, dtype=torch.float64).to(TORCH_DTYPES[dtype])
    out = dit.gelu_tanh(x.cuda())
    torch.cuda.synchronize()
    check(out.cpu(), oracle_gelu(orc, x, dtype), x, dtype, "special")


@pytest.mark.parametrize("dtype", DTYPES)
def test_gelu_negative_tail(orc, dtype):
    """x in [-12, -3]: results shrink through the dtype's subnormal range to
    zero (e^(-2|z|) is below 2^-126 from x ~ -9.4 on)."""
    x = torch.linspace(-12.0, -3.0, 20001, dtype=torch.float64).to(TORCH_DTYPES[dtype])
    out = dit.gelu_tanh(x.cuda())
    torch.cuda.synchronize()
    check(out.cpu(), oracle_gelu(orc, x, dtype), x, dtype, "tail")


def test_gelu_ffn_full_size_sampled(orc):
    """The feed-forward activation of the largest shape, [1, 32640, 16384]
    bf16 (4 x 4096 hidden): whole tensor on the GPU, 2^20 sampled elements
    against the oracle, and the odd identity on the whole tensor."""
    x = draw("act", (1, 32640, 16384), seed_for("gelu-ffn"), "bf16", "cuda")
    out = dit.gelu_tanh(x)
    torch.cuda.synchronize()
    g = torch.Generator(device="cuda").manual_seed(5)
    idx = torch.randint(0, x.numel(), (1 << 20,), device="cuda", generator=g)
    xs = x.reshape(-1)[idx].cpu()
    nz = check(out.reshape(-1)[idx].cpu(), oracle_gelu(orc, xs, "bf16"), xs, "bf16", "ffn")
    assert nz <= xs.numel() // 100
    # gelu(x) - gelu(-x) = x on every element, within the two roundings
    neg = dit.gelu_tanh(-x)
    torch.cuda.synchronize()
    d = (out.float() - neg.float() - x.float()).abs()
    tol = (out.float().abs() + neg.float().abs()) * 2.0 ** -8 + 1e-30
    assert bool((d <= tol).all())
