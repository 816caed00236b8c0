"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on
seeded inputs, element by element, at sizes the oracle finishes quickly that
still span several CTAs, several column slices and ragged tails: every dtype,
both layouts, odd D (3077: no vector access), D = 3076 (8-byte access for
16-bit dtypes), long rows (two-pass kernel), misaligned sub-views, in-place
updates, empty tensors, IEEE special values, and canaries around outputs.
"""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import mod_inputs, oracle_fused, oracle_mod, oracle_rga, rga_inputs
from _gpu import (assert_bit_exact, ensure_built, guarded, modulation_stats, offset_copy)
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16", "fp32"]
SHAPES = [(1, 126, 2048), (2, 37, 3080), (1, 45, 3077), (1, 33, 3076), (2, 19, 4096),
          (1, 9, 4608), (3, 5, 7), (1, 1, 1), (1, 2, 127), (2, 3, 9000), (1, 2, 20000)]
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def cuda(*ts):
    return [t.cuda() for t in ts]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", ["full", "bcast"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_residual_gate(orc, dtype, layout, shape):
    B, L, D = shape
    h, u, g = rga_inputs(B, L, D, dtype, layout, row_spread=True)
    out, untouched = guarded(shape, TORCH_DTYPES[dtype], "cuda")
    dit.residual_gate_add(*cuda(h, u, g), out=out)
    torch.cuda.synchronize()
    assert untouched()
    assert_bit_exact(out, oracle_rga(orc, h, u, g, dtype, layout), f"{dtype} {layout} {shape}")


@pytest.mark.parametrize("layout", ["full", "bcast"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_residual_gate_in_place(orc, dtype, layout):
    B, L, D = 2, 41, 3080
    h, u, g = rga_inputs(B, L, D, dtype, layout)
    hd, ud, gd = cuda(h, u, g)
    ret = dit.residual_gate_add(hd, ud, gd, out=hd)
    torch.cuda.synchronize()
    assert ret.data_ptr() == hd.data_ptr()
    assert_bit_exact(hd, oracle_rga(orc, h, u, g, dtype, layout))


@pytest.mark.parametrize("offsets", [(1, 1, 1, 1), (1, 2, 0, 3), (0, 0, 0, 1), (3, 3, 3, 3)])
@pytest.mark.parametrize("layout", ["full", "bcast"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_residual_gate_misaligned(orc, dtype, layout, offsets):
    """Sub-views starting 1-3 elements past an allocation boundary: same or
    different misalignment per tensor (head/tail peel, narrow accesses)."""
    B, L, D = 1, 29, 2048
    h, u, g = rga_inputs(B, L, D, dtype, layout)
    ho, uo, go = (offset_copy(t.cuda(), k) for t, k in zip((h, u, g), offsets[:3]))
    out = offset_copy(torch.zeros_like(h).cuda(), offsets[3])
    dit.residual_gate_add(ho, uo, go, out=out)
    torch.cuda.synchronize()
    assert_bit_exact(out, oracle_rga(orc, h, u, g, dtype, layout))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("layout", ["bcast", "full"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_modulate(orc, statistic, dtype, layout, shape):
    B, L, D = shape
    x, sc, sh = mod_inputs(B, L, D, dtype, layout, row_spread=True)
    out, untouched = guarded(shape, TORCH_DTYPES[dtype], "cuda")
    dit.rmsnorm_modulate(*cuda(x, sc, sh), EPS, out=out)
    torch.cuda.synchronize()
    assert untouched()
    ref, t = oracle_mod(orc, x, sc, sh, dtype, layout, EPS, with_t=True)
    modulation_stats(out, ref, t.numpy(), dtype, f"{dtype} {layout} {shape}")


@pytest.mark.parametrize("offset", [1, 2, 3])
@pytest.mark.parametrize("dtype", DTYPES)
def test_modulate_misaligned(orc, statistic, dtype, offset):
    B, L, D = 2, 13, 4096
    x, sc, sh = mod_inputs(B, L, D, dtype, "bcast")
    xo = offset_copy(x.cuda(), offset)
    out = offset_copy(torch.zeros_like(x).cuda(), 0)
    dit.rmsnorm_modulate(xo, *cuda(sc, sh), EPS, out=out)
    torch.cuda.synchronize()
    ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", EPS, with_t=True)
    modulation_stats(out, ref, t.numpy(), dtype)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("gl,ml", [("bcast", "bcast"), ("full", "bcast"), ("bcast", "full"),
                                   ("full", "full")])
@pytest.mark.parametrize("dtype", DTYPES)
def test_fused(orc, statistic, dtype, gl, ml, shape):
    B, L, D = shape
    h, u, g = rga_inputs(B, L, D, dtype, gl, tag="fz", row_spread=True)
    _, sc, sh = mod_inputs(B, L, D, dtype, ml, tag="fz")
    res, ok1 = guarded(shape, TORCH_DTYPES[dtype], "cuda")
    mod, ok2 = guarded(shape, TORCH_DTYPES[dtype], "cuda")
    dit.gate_add_rmsnorm_modulate(*cuda(h, u, g, sc, sh), EPS, residual_out=res,
                                  modulated_out=mod)
    torch.cuda.synchronize()
    assert ok1() and ok2()
    rref, mref, t = oracle_fused(orc, h, u, g, sc, sh, dtype, gl, ml, EPS, with_t=True)
    assert_bit_exact(res, rref, f"residual {dtype} {gl}/{ml} {shape}")
    modulation_stats(mod, mref, t.numpy(), dtype, f"modulated {dtype} {gl}/{ml} {shape}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_fused_in_place_and_misaligned(orc, dtype):
    B, L, D = 2, 23, 3072
    h, u, g = rga_inputs(B, L, D, dtype, "bcast", tag="fzi")
    _, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="fzi")
    rref, mref, t = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast", EPS, with_t=True)
    hd = h.cuda()
    _, mod = dit.gate_add_rmsnorm_modulate(hd, *cuda(u, g, sc, sh), EPS, residual_out=hd)
    torch.cuda.synchronize()
    assert_bit_exact(hd, rref)
    modulation_stats(mod, mref, t.numpy(), dtype)
    ho = offset_copy(h.cuda(), 1)
    res, mod = dit.gate_add_rmsnorm_modulate(ho, *cuda(u, g, sc, sh), EPS, residual_out=ho)
    torch.cuda.synchronize()
    assert_bit_exact(ho, rref)
    modulation_stats(mod, mref, t.numpy(), dtype)


@pytest.mark.parametrize("shape", [(0, 5, 8), (2, 0, 8), (2, 5, 0)])
def test_empty_tensors_launch_nothing(shape):
    z = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    v = torch.empty((shape[0], 1, shape[2]), dtype=torch.bfloat16, device="cuda")
    dit.residual_gate_add(z, z.clone(), v)
    dit.rmsnorm_modulate(z, v, v.clone())
    dit.gate_add_rmsnorm_modulate(z, z.clone(), v, v.clone(), v.clone())
    torch.cuda.synchronize()


@pytest.mark.parametrize("dtype", DTYPES)
def test_special_values(orc, statistic, dtype):
    """inf, -inf, NaN, subnormals and overflow propagate as IEEE arithmetic
    says, identically on both sides (NaN payloads aside)."""
    B, L, D = 1, 4, 64
    h, u, g = rga_inputs(B, L, D, dtype, "full", tag="special")
    big = {"bf16": 3e38, "fp16": 6e4, "fp32": 3e38}[dtype]
    tiny = {"bf16": 1e-39, "fp16": 1e-7, "fp32": 1e-44}[dtype]
    hv = h.float()
    hv[0, 0, :4] = torch.tensor([float("inf"), float("-inf"), float("nan"), big])
    hv[0, 1, :3] = torch.tensor([tiny, -tiny, 0.0])
    h = hv.to(h.dtype)
    u = u.float()
    u[0, 0, 3] = big
    u = u.to(h.dtype)
    g = g.float()
    g[0, 0, 3] = 1.0
    g = g.to(h.dtype)
    out = dit.residual_gate_add(*cuda(h, u, g))
    torch.cuda.synchronize()
    ref = oracle_rga(orc, h, u, g, dtype, "full")
    o, r = out.cpu().float(), ref.float()
    assert torch.equal(torch.isnan(o), torch.isnan(r))
    m = ~torch.isnan(r)
    assert torch.equal(o[m], r[m])
    # modulation: a row holding NaN is NaN throughout (its sum of squares is
    # NaN); rows of subnormals and zeros are ordinary rows
    _, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="special")
    mo = dit.rmsnorm_modulate(*cuda(h, sc, sh), EPS)
    torch.cuda.synchronize()
    mr, t = oracle_mod(orc, h, sc, sh, dtype, "bcast", EPS, with_t=True)
    assert torch.isnan(mr[0, 0]).all()
    modulation_stats(mo, mr, t.numpy(), dtype, "special values")


@pytest.mark.parametrize("layout", ["bcast", "full"])
@pytest.mark.parametrize("dtype", DTYPES)
def test_modulation_rounding_order_bit_exact(orc, dtype, layout):
    """Every row holds the same multiset of small dyadic values, so the sum of
    squares is exact in fp32 in any order; eps = 1 - mean(x^2) makes the
    inverse root exactly 1 on both sides.  What remains -- n = x * r,
    1 + scale, n * (1 + scale), + shift, each rounded, then one rounding to the
    dtype -- must then match the oracle bit for bit (a contracted
    multiply-add, or another order, would not)."""
    B, L, D = 2, 37, 1024
    rng = np.random.default_rng(7)
    base = rng.integers(-15, 16, size=D) / 16.0  # multiples of 1/16 in [-15/16, 15/16]
    rows = np.stack([rng.permutation(base) for _ in range(B * L)]).reshape(B, L, D)
    ms = float(np.mean(base * base))
    eps = 1.0 - ms
    assert np.float32(eps) == eps and 0 <= eps  # exact in fp32
    x = torch.tensor(rows, dtype=torch.float64).to(TORCH_DTYPES[dtype])
    assert torch.equal(x.double(), torch.tensor(rows))
    _, sc, sh = mod_inputs(B, L, D, dtype, layout, tag="exactr")
    out = dit.rmsnorm_modulate(*cuda(x, sc, sh), eps)
    torch.cuda.synchronize()
    ref = oracle_mod(orc, x, sc, sh, dtype, layout, eps)
    assert_bit_exact(out, ref, f"{dtype} {layout}")
    # the fused op, with hidden = x and a zero gate, must agree as well
    z = torch.zeros((B, 1, D), dtype=x.dtype)
    res, mod = dit.gate_add_rmsnorm_modulate(*cuda(x, x, z, sc, sh), eps)
    torch.cuda.synchronize()
    assert_bit_exact(res, x)
    assert_bit_exact(mod, ref, f"fused {dtype} {layout}")


@pytest.mark.parametrize("dtype", DTYPES)
def test_zero_row_and_zero_eps(orc, dtype):
    B, L, D = 1, 3, 256
    x, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="zero")
    x[0, 1] = 0
    for eps in (0.0, EPS):
        out = dit.rmsnorm_modulate(*cuda(x, sc, sh), eps)
        torch.cuda.synchronize()
        ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", eps, with_t=True)
        modulation_stats(out, ref, t.numpy(), dtype, f"eps={eps}")


def test_side_stream(orc):
    B, L, D = 1, 300, 4096
    h, u, g = rga_inputs(B, L, D, "bf16", "bcast", tag="stream")
    hd, ud, gd = cuda(h, u, g)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = dit.residual_gate_add(hd, ud, gd)
    s.synchronize()
    assert_bit_exact(out, oracle_rga(orc, h, u, g, "bf16", "bcast"))


def test_cpu_tensors_are_rejected():
    h = torch.zeros((1, 2, 8), dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        dit.residual_gate_add(h, h, h)


@pytest.mark.parametrize("dtype", DTYPES)
def test_strided_adaln_table(orc, dtype):
    """Gate, scale and shift as [B, 1, D] rows of a [B, 9, D] adaLN table
    (batch stride 9 * D): identical bits to contiguous copies, and to the
    oracle."""
    from diffusion_transformer_elementwise_gb300.synth import draw, seed_for
    B, L, D = 3, 21, 3072
    h, u, _ = rga_inputs(B, L, D, dtype, "bcast", tag="strided")
    table = draw("mod", (B, 9, D), seed_for("strided", "table", dtype), dtype, "cuda")
    sh_v, sc_v, g_v = table[:, 3:4], table[:, 4:5], table[:, 5:6]
    assert not g_v.is_contiguous() and g_v.stride(0) == 9 * D
    hd, ud = cuda(h, u)
    out_s = dit.residual_gate_add(hd, ud, g_v)
    out_c = dit.residual_gate_add(hd, ud, g_v.contiguous())
    mod_s = dit.rmsnorm_modulate(hd, sc_v, sh_v, EPS)
    mod_c = dit.rmsnorm_modulate(hd, sc_v.contiguous(), sh_v.contiguous(), EPS)
    res_s, fm_s = dit.gate_add_rmsnorm_modulate(hd, ud, g_v, sc_v, sh_v, EPS)
    res_c, fm_c = dit.gate_add_rmsnorm_modulate(hd, ud, g_v.contiguous(), sc_v.contiguous(),
                                                sh_v.contiguous(), EPS)
    torch.cuda.synchronize()
    for a, b in ((out_s, out_c), (mod_s, mod_c), (res_s, res_c), (fm_s, fm_c)):
        assert_bit_exact(a, b)
    g, sc, sh = (v.cpu().contiguous() for v in (g_v, sc_v, sh_v))
    assert_bit_exact(out_s, oracle_rga(orc, h, u, g, dtype, "bcast"))
    ref, t = oracle_mod(orc, h, sc, sh, dtype, "bcast", EPS, with_t=True)
    modulation_stats(mod_s, ref, t.numpy(), dtype, "strided modulation")
    rref, mref, t2 = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast", EPS, with_t=True)
    assert_bit_exact(res_s, rref)
    modulation_stats(fm_s, mref, t2.numpy(), dtype, "strided fused")
    # the [B, 1, D] operands of one call must share their batch stride
    with pytest.raises(ValueError):
        dit.gate_add_rmsnorm_modulate(hd, ud, g_v, sc_v.contiguous(), sh_v, EPS)
