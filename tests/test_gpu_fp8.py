"""GPU parity of the E4M3-output modulation and fused op against the oracle.

Criterion under the exact row statistic (dit_set_statistic): bit-exact
codes.  The statistic is the same fp32 value on both sides (single roundings
of exact values), the fp32 modulation value y is formed by the same IEEE
operations, then scaled by fl(1/s) and rounded once to E4M3 (nearest even,
saturating).  Under the fast statistic (the default) y is within a few fp32
ulps of the oracle's, far below one E4M3 step (2^-3 relative), so each code is
the oracle's or the next one over in the ordered codes; where the final add
cancels (|y| << |t|) a code may instead be within one E4M3 spacing of
max(|t|, |y|) / s.  Either way NaN codes match NaN codes and the residual of
the fused op is bit-exact.
"""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import mod_inputs, rga_inputs
from _gpu import assert_bit_exact, ensure_built
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES, draw, seed_for

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _codes(t):
    return t.view(torch.uint8).cpu().numpy().reshape(-1).astype(np.int32)


def _ordinal(c):
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _value(c):
    e, m = (c >> 3) & 15, c & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * 2.0 ** (e.astype(np.float64) - 10))
    return np.where(c & 0x80, -v, v)


def _spacing(a):
    """E4M3 spacing at magnitude a (2^-9 below 2^-6, 2^(E-3) in [2^E, 2^(E+1)))."""
    a = np.maximum(np.abs(a), 2.0 ** -6)
    return 2.0 ** (np.floor(np.log2(a)) - 3)


def check_fp8(gpu, ref, t, inv, what=""):
    """The criterion of the library's current row statistic; returns (codes
    not bit-exact, codes admitted by the cancellation rule)."""
    exact = dit.get_statistic() == "exact"
    g, r = _codes(gpu), _codes(ref)
    nan_g, nan_r = (g & 0x7F) == 0x7F, (r & 0x7F) == 0x7F
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN codes differ"
    ok = ~nan_r
    g, r = g[ok], r[ok]
    step = np.abs(_ordinal(g) - _ordinal(r))
    if exact:
        fallback = np.zeros(step.shape, bool)
        bad = step != 0
    else:
        tt = np.abs(t.numpy().reshape(-1)[ok].astype(np.float64)) * inv
        scale = np.maximum(tt, np.abs(_value(r)))
        fallback = (step > 1) & (np.abs(_value(g) - _value(r)) <= _spacing(scale))
        bad = (step > 1) & ~fallback
    idx = np.nonzero(bad)[0]
    assert idx.size == 0, (f"{what}: {idx.size} codes off, first {g[idx[:5]]} vs "
                           f"{r[idx[:5]]} (t {t.numpy().reshape(-1)[ok][idx[:5]]})")
    return int(np.count_nonzero(step)), int(np.count_nonzero(fallback))


def _oracle_mod8(orc, x, sc, sh, dtype, lay, qs, eps=EPS):
    B, L, D = x.shape
    out = torch.empty((B, L, D), dtype=torch.uint8)
    t = torch.empty((B, L, D), dtype=torch.float32)
    orc.rmsnorm_modulate_fp8(out, x, sc, sh, B, L, D, eps, dtype, lay, qs, t_out=t)
    return out, t


def _oracle_fused8(orc, h, u, g, sc, sh, dtype, glay, mlay, qs, eps=EPS):
    B, L, D = h.shape
    res = torch.empty_like(h)
    out = torch.empty((B, L, D), dtype=torch.uint8)
    t = torch.empty((B, L, D), dtype=torch.float32)
    orc.gate_add_rmsnorm_modulate_fp8(res, out, h, u, g, sc, sh, B, L, D, eps, dtype, glay,
                                      mlay, qs, t_out=t)
    return res, out, t


def _inv(qs):
    return float(np.float32(1.0) / np.float32(qs))


def _qs(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


SHAPES = [(1, 5, 64), (2, 37, 2048), (1, 9, 3072), (1, 33, 4096), (2, 6, 8192)]


@pytest.mark.parametrize("qs", [1.0, 0.005, 3.0])
@pytest.mark.parametrize("layout", ["bcast", "full"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_modulate_fp8(orc, statistic, dtype, layout, qs):
    for B, L, D in SHAPES:
        if dtype == "fp32" and D > 4096:
            continue
        x, sc, sh = mod_inputs(B, L, D, dtype, layout, tag="fp8")
        out = dit.rmsnorm_modulate_fp8(x.cuda(), sc.cuda(), sh.cuda(), _qs(qs), EPS)
        torch.cuda.synchronize()
        ref, t = _oracle_mod8(orc, x, sc, sh, dtype, layout, qs)
        check_fp8(out, ref, t, _inv(qs), f"{dtype} {layout} {qs} {(B, L, D)}")


@pytest.mark.parametrize("layouts", [("bcast", "bcast"), ("full", "bcast"), ("bcast", "full"),
                                     ("full", "full")])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_fused_fp8(orc, statistic, dtype, layouts):
    glay, mlay = layouts
    for B, L, D in SHAPES[:4]:
        h, u, g = rga_inputs(B, L, D, dtype, glay, tag="fp8f")
        _, sc, sh = mod_inputs(B, L, D, dtype, mlay, tag="fp8f")
        r, q = dit.gate_add_rmsnorm_modulate_fp8(h.cuda(), u.cuda(), g.cuda(), sc.cuda(),
                                                 sh.cuda(), _qs(0.25), EPS)
        torch.cuda.synchronize()
        res, ref, t = _oracle_fused8(orc, h, u, g, sc, sh, dtype, glay, mlay, 0.25)
        assert_bit_exact(r.cpu(), res, f"{dtype} residual")
        check_fp8(q, ref, t, 4.0, f"{dtype} {layouts} {(B, L, D)}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_fp8_bit_exact_when_the_statistic_is_exact(orc, dtype):
    """Rows of one multiset of multiples of 1/16 and eps = 1 - mean(x^2): the
    inverse root is exactly 1 on both sides, so every code must match."""
    B, L, D = 2, 21, 1024
    rng = np.random.default_rng(17)
    base = rng.integers(-15, 16, size=D) / 16.0
    rows = np.stack([rng.permutation(base) for _ in range(B * L)]).reshape(B, L, D)
    eps = 1.0 - float(np.mean(base * base))
    x = torch.tensor(rows, dtype=torch.float64).to(TORCH_DTYPES[dtype])
    _, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="fp8exact")
    for qs in (1.0, 0.01, 0.3):
        out = dit.rmsnorm_modulate_fp8(x.cuda(), sc.cuda(), sh.cuda(), _qs(qs), eps)
        torch.cuda.synchronize()
        ref, _ = _oracle_mod8(orc, x, sc, sh, dtype, "bcast", qs, eps)
        assert np.array_equal(_codes(out), _codes(ref)), (dtype, qs)


def test_fp8_special_values(orc):
    """A row holding NaN quantises to NaN codes throughout; saturation to
    +-448; outputs as uint8 or float8_e4m3fn views of the same codes."""
    B, L, D, dtype = 1, 4, 256, "bf16"
    x, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="fp8special")
    x[0, 1, 7] = float("nan")
    out8 = torch.empty((B, L, D), dtype=torch.uint8, device="cuda")
    dit.rmsnorm_modulate_fp8(x.cuda(), sc.cuda(), sh.cuda(), _qs(1e-3), EPS, out=out8)
    torch.cuda.synchronize()
    ref, t = _oracle_mod8(orc, x, sc, sh, dtype, "bcast", 1e-3)
    check_fp8(out8, ref, t, _inv(1e-3), "special")
    codes = _codes(out8).reshape(B, L, D)
    assert np.all((codes[0, 1] & 0x7F) == 0x7F)
    assert np.count_nonzero((codes[0, 0] & 0x7F) == 0x7E) > 0  # saturated
    f8 = dit.rmsnorm_modulate_fp8(x.cuda(), sc.cuda(), sh.cuda(), _qs(1e-3), EPS)
    torch.cuda.synchronize()
    if hasattr(torch, "float8_e4m3fn"):
        assert f8.dtype == torch.float8_e4m3fn
    assert np.array_equal(_codes(f8), _codes(out8))


def test_fp8_scale_read_on_device(orc):
    """The scale is read by the kernel: changing the device value between
    two calls changes the codes, with nothing else touched."""
    B, L, D, dtype = 1, 8, 2048, "bf16"
    x, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="fp8dev")
    xd, scd, shd = x.cuda(), sc.cuda(), sh.cuda()
    qs = _qs(1.0)
    a = dit.rmsnorm_modulate_fp8(xd, scd, shd, qs, EPS).clone()
    qs.fill_(0.5)
    b = dit.rmsnorm_modulate_fp8(xd, scd, shd, qs, EPS)
    torch.cuda.synchronize()
    ra, ta = _oracle_mod8(orc, x, sc, sh, dtype, "bcast", 1.0)
    rb, tb = _oracle_mod8(orc, x, sc, sh, dtype, "bcast", 0.5)
    check_fp8(a, ra, ta, 1.0, "scale 1")
    check_fp8(b, rb, tb, 2.0, "scale 0.5")


def test_fused_fp8_full_size_sampled(orc):
    """[1, 32640, 4096] bf16, [1, 1, D] vectors, in-place residual: 64 sampled
    rows against the oracle."""
    B, L, D, dtype = 1, 32640, 4096, "bf16"
    dev = [draw(k, shp, seed_for("fp8-full", j), dtype, "cuda")
           for j, (k, shp) in enumerate([("act", (B, L, D)), ("act", (B, L, D)),
                                         ("gate", (B, 1, D)), ("mod", (B, 1, D)),
                                         ("mod", (B, 1, D))])]
    h0 = dev[0].clone()
    r, q = dit.gate_add_rmsnorm_modulate_fp8(*dev, _qs(0.02), EPS, residual_out=dev[0])
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(4)
    idx = torch.cat([torch.tensor([0, L - 1]), torch.randint(1, L - 1, (62,), generator=g)])
    sub = [h0[:, idx.cuda()].cpu(), dev[1][:, idx.cuda()].cpu()] + [v.cpu() for v in dev[2:]]
    res, ref, t = _oracle_fused8(orc, *sub, dtype, "bcast", "bcast", 0.02)
    assert_bit_exact(r[:, idx.cuda()].cpu(), res, "residual")
    check_fp8(q[:, idx.cuda()], ref, t, _inv(0.02), "full size")
