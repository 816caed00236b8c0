"""GPU parity of the phased kernels: rows whose byte pitch is not a
multiple of 16 (odd D, D = 2 mod 4 ...) in tensors that start on 16-byte
boundaries -- the staged CTA-per-row kernel (the residual gate, the exact
statistic, full scale/shift, rows above 8 KB) and the two-warp kernel (the
modulating ops with the fast statistic and [B,1,D] operands).  Every offset period (2, 4 and 8 rows), fewer rows than the
period, more rows than the grid (each CTA takes rows of one offset), batches
changing inside a CTA's run, rows shorter than a granule, the last row's
granule that runs past the tensors' end, rows too long for one CTA (column
slices of the residual gate; the two-pass kernel for the reducing ops),
in-place residuals, strided adaLN tables, and canaries around every output (a row's first and last granule are
shared with its neighbours and must be stored element by element).
"""
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import mod_inputs, oracle_fused, oracle_mod, oracle_rga, rga_inputs
from _gpu import assert_bit_exact, ensure_built, guarded, modulation_stats
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES, draw, seed_for

pytestmark = pytest.mark.gpu
EPS = 1e-6

# (B, L, D, dtype); the byte pitch modulo 16 sets the period of the rows'
# offsets: 6154 % 16 = 10 -> 8 rows, 6152 % 16 = 8 -> 2, 12308 % 16 = 4 -> 4
CASES = [
    (1, 45, 3077, "bf16"),     # period 8, fewer rows than CTAs
    (1, 1300, 3077, "bf16"),   # period 8, several rows per CTA
    (3, 500, 3077, "fp16"),    # batches change inside a CTA's run
    (1, 1100, 3076, "bf16"),   # period 2
    (2, 333, 3077, "fp32"),    # period 4
    (1, 700, 3078, "fp32"),    # period 2
    (1, 7, 1, "bf16"),         # 2-byte rows, fewer rows than the period
    (2, 9, 3, "fp32"),         # rows inside one granule
    (1, 40000, 13, "bf16"),    # 26-byte rows, many rows per CTA
    (2, 3001, 6, "fp16"),      # 12-byte rows, period 4, odd row count
    (1, 50, 8193, "bf16"),     # residual gate in two column slices; the
    (1, 30, 8191, "fp16"),     # reducing ops then take the two-pass kernel
    (1, 12, 20001, "bf16"),    # (a row beyond one CTA's 1024 granules)
    (1, 40, 8191, "fp32"),
    (2, 512, 3077, "bf16"),    # batches whose length is a multiple of the
    (4, 64, 1001, "fp16"),     # period: every batch starts at offset 0
]
IDS = [f"{b}x{l}x{d}-{t}" for b, l, d, t in CASES]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def cuda(*ts):
    return [t.cuda() for t in ts]


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_residual_gate_bcast(orc, case):
    B, L, D, dtype = case
    h, u, g = rga_inputs(B, L, D, dtype, "bcast", tag="ph", row_spread=True)
    out, untouched = guarded((B, L, D), TORCH_DTYPES[dtype], "cuda")
    dit.residual_gate_add(*cuda(h, u, g), out=out)
    torch.cuda.synchronize()
    assert untouched()
    assert_bit_exact(out, oracle_rga(orc, h, u, g, dtype, "bcast"), f"{case}")


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_residual_gate_in_place(orc, case):
    B, L, D, dtype = case
    h, u, g = rga_inputs(B, L, D, dtype, "bcast", tag="phi")
    hd, ud, gd = cuda(h, u, g)
    dit.residual_gate_add(hd, ud, gd, out=hd)
    torch.cuda.synchronize()
    assert_bit_exact(hd, oracle_rga(orc, h, u, g, dtype, "bcast"), f"{case}")


@pytest.mark.parametrize("layout", ["bcast", "full"])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_modulate(orc, statistic, case, layout):
    B, L, D, dtype = case
    x, sc, sh = mod_inputs(B, L, D, dtype, layout, tag="ph", row_spread=True)
    out, untouched = guarded((B, L, D), TORCH_DTYPES[dtype], "cuda")
    dit.rmsnorm_modulate(*cuda(x, sc, sh), EPS, out=out)
    torch.cuda.synchronize()
    assert untouched()
    ref, t = oracle_mod(orc, x, sc, sh, dtype, layout, EPS, with_t=True)
    modulation_stats(out, ref, t.numpy(), dtype, f"{case} {layout}")


@pytest.mark.parametrize("gl,ml", [("bcast", "bcast"), ("full", "bcast"), ("bcast", "full"),
                                   ("full", "full")])
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fused(orc, statistic, case, gl, ml):
    B, L, D, dtype = case
    h, u, g = rga_inputs(B, L, D, dtype, gl, tag="phf", row_spread=True)
    _, sc, sh = mod_inputs(B, L, D, dtype, ml, tag="phf")
    res, ok1 = guarded((B, L, D), TORCH_DTYPES[dtype], "cuda")
    mod, ok2 = guarded((B, L, D), TORCH_DTYPES[dtype], "cuda")
    dit.gate_add_rmsnorm_modulate(*cuda(h, u, g, sc, sh), EPS, residual_out=res,
                                  modulated_out=mod)
    torch.cuda.synchronize()
    assert ok1() and ok2()
    rref, mref, t = oracle_fused(orc, h, u, g, sc, sh, dtype, gl, ml, EPS, with_t=True)
    assert_bit_exact(res, rref, f"residual {case} {gl}/{ml}")
    modulation_stats(mod, mref, t.numpy(), dtype, f"modulated {case} {gl}/{ml}")


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fused_in_place(orc, case):
    """residual_out == hidden: a CTA reads the neighbours' elements of its
    shared granules while their own CTAs overwrite them; those elements are
    masked, so the result cannot depend on the race."""
    B, L, D, dtype = case
    h, u, g = rga_inputs(B, L, D, dtype, "bcast", tag="phfi")
    _, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="phfi")
    rref, mref, t = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast", EPS, with_t=True)
    hd = h.cuda()
    _, mod = dit.gate_add_rmsnorm_modulate(hd, *cuda(u, g, sc, sh), EPS, residual_out=hd)
    torch.cuda.synchronize()
    assert_bit_exact(hd, rref, f"{case}")
    modulation_stats(mod, mref, t.numpy(), dtype, f"{case}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_strided_adaln_table(orc, dtype):
    """[B, 1, D] operands as rows of a [B, 9, D] table (batch stride 9 * D):
    the phased kernel reads them element by element at the rows' offset."""
    B, L, D = 3, 400, 3077
    h, u, _ = rga_inputs(B, L, D, dtype, "bcast", tag="phs")
    table = draw("mod", (B, 9, D), seed_for("phs", "table", dtype), dtype, "cuda")
    sh_v, sc_v, g_v = table[:, 3:4], table[:, 4:5], table[:, 5:6]
    assert g_v.stride(0) == 9 * D
    hd, ud = cuda(h, u)
    out = dit.residual_gate_add(hd, ud, g_v)
    mod = dit.rmsnorm_modulate(hd, sc_v, sh_v, EPS)
    res, fm = dit.gate_add_rmsnorm_modulate(hd, ud, g_v, sc_v, sh_v, EPS)
    torch.cuda.synchronize()
    g, sc, sh = (v.cpu().contiguous() for v in (g_v, sc_v, sh_v))
    assert_bit_exact(out, oracle_rga(orc, h, u, g, dtype, "bcast"))
    ref, t = oracle_mod(orc, h, sc, sh, dtype, "bcast", EPS, with_t=True)
    modulation_stats(mod, ref, t.numpy(), dtype, "strided modulation")
    rref, mref, t2 = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast", EPS, with_t=True)
    assert_bit_exact(res, rref)
    modulation_stats(fm, mref, t2.numpy(), dtype, "strided fused")


def test_phased_kernel_is_the_one_launched():
    """Odd-D rows in aligned tensors run the staged kernel's phased
    instantiation (its last template argument true), not a narrow-access
    fallback; sub-views that start off a 16-byte boundary do not."""
    prof = pytest.importorskip("torch.profiler")
    B, L, D = 1, 64, 3077
    x, sc, sh = (t.cuda() for t in mod_inputs(B, L, D, "bf16", "bcast", tag="phk"))

    def kernels(fn):
        with prof.profile(activities=[prof.ProfilerActivity.CUDA]) as p:
            fn()
            torch.cuda.synchronize()
        names = [e.name for e in p.events() if e.device_type == torch.autograd.DeviceType.CUDA]
        if not names:
            pytest.skip("the profiler recorded no kernels here")
        return names

    def last_template_argument(name):
        head = name.split("(")[0]
        return head[head.index("<") + 1:head.rindex(">")].split(",")[-1].strip()

    names = kernels(lambda: dit.rmsnorm_modulate(x, sc, sh, EPS))
    ours = [n for n in names if "pipe_kernel" in n or "row_kernel" in n]
    assert ours and all("pipe_kernel" in n and last_template_argument(n) == "true"
                        for n in ours), ours
    buf = torch.empty(B * L * D + 1, dtype=x.dtype, device="cuda")
    xo = buf[1:].view(B, L, D)
    xo.copy_(x)
    names = kernels(lambda: dit.rmsnorm_modulate(xo, sc, sh, EPS))
    assert any("row_kernel" in n for n in names), names
