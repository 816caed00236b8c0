"""GPU parity of the kernels for rows whose pitch is not a multiple of 16
bytes (16-byte aligned tensors, rows that start 2, 4, ... 14 bytes past a
boundary; the narrow-access register kernels): widths covering every residue
of the row start modulo 16, rows shorter than 16 bytes, rows wider than one
residual-gate slice, in-place updates, full and [B, 1, D] operands, strided
vectors, and canaries around every output to catch a store outside the
rows."""
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import mod_inputs, oracle_fused, oracle_mod, oracle_rga, rga_inputs
from _gpu import assert_bit_exact, ensure_built, guarded, modulation_stats

pytestmark = pytest.mark.gpu
EPS = 1e-6
WIDTHS16 = [1, 3, 5, 7, 9, 13, 17, 33, 63, 255, 1001, 3077, 3076, 4099, 8191]
WIDTHS32 = [1, 3, 5, 7, 9, 1001, 3077, 4097]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _cases():
    for dt in ("bf16", "fp16"):
        for D in WIDTHS16:
            yield dt, D
    for D in WIDTHS32:
        yield "fp32", D


@pytest.mark.parametrize("dtype,D", list(_cases()))
def test_shifted_rows(orc, statistic, dtype, D):
    B, L = 2, 7
    for glay in ("bcast", "full"):
        h, u, g = rga_inputs(B, L, D, dtype, glay, tag="shift")
        out, untouched = guarded((B, L, D), h.dtype, "cuda")
        dit.residual_gate_add(h.cuda(), u.cuda(), g.cuda(), out=out)
        torch.cuda.synchronize()
        ref = oracle_rga(orc, h, u, g, dtype, glay)
        assert_bit_exact(out.cpu(), ref, f"rga {glay} D={D}")
        assert untouched()
        hd = h.cuda()  # in place
        dit.residual_gate_add(hd, u.cuda(), g.cuda(), out=hd)
        torch.cuda.synchronize()
        assert_bit_exact(hd.cpu(), ref, f"rga in place {glay} D={D}")
    for mlay in ("bcast", "full"):
        x, sc, sh = mod_inputs(B, L, D, dtype, mlay, tag="shift")
        out, untouched = guarded((B, L, D), x.dtype, "cuda")
        dit.rmsnorm_modulate(x.cuda(), sc.cuda(), sh.cuda(), EPS, out=out)
        torch.cuda.synchronize()
        ref, t = oracle_mod(orc, x, sc, sh, dtype, mlay, EPS, with_t=True)
        modulation_stats(out.cpu(), ref, t.numpy(), dtype, f"mod {mlay} D={D}")
        assert untouched()
    h, u, g = rga_inputs(B, L, D, dtype, "bcast", tag="shiftf")
    _, sc, sh = mod_inputs(B, L, D, dtype, "bcast", tag="shiftf")
    res, mod, t = oracle_fused(orc, h, u, g, sc, sh, dtype, "bcast", "bcast", EPS, with_t=True)
    hd = h.cuda()
    m_out, untouched = guarded((B, L, D), h.dtype, "cuda")
    dit.gate_add_rmsnorm_modulate(hd, u.cuda(), g.cuda(), sc.cuda(), sh.cuda(), EPS,
                                  residual_out=hd, modulated_out=m_out)
    torch.cuda.synchronize()
    assert_bit_exact(hd.cpu(), res, f"fused residual in place D={D}")
    modulation_stats(m_out.cpu(), mod, t.numpy(), dtype, f"fused D={D}")
    assert untouched()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_shifted_strided_vectors(orc, dtype):
    """[B, 1, D] vectors as rows of a [B, 9, D] table: their batch stride is
    not a multiple of 16 bytes either."""
    from diffusion_transformer_elementwise_gb300.synth import draw, seed_for
    B, L, D = 3, 6, 3077
    h, u, _ = rga_inputs(B, L, D, dtype, "bcast", tag="shiftv")
    table = draw("mod", (B, 9, D), seed_for("shiftv", dtype), dtype)
    shift, scale, gate = (table[:, k:k + 1, :] for k in (0, 1, 2))
    tg = table.cuda()
    r, m = dit.gate_add_rmsnorm_modulate(h.cuda(), u.cuda(), tg[:, 2:3], tg[:, 1:2], tg[:, 0:1],
                                         EPS)
    torch.cuda.synchronize()
    res, mod, t = oracle_fused(orc, h, u, gate.contiguous(), scale.contiguous(),
                               shift.contiguous(), dtype, "bcast", "bcast", EPS, with_t=True)
    assert_bit_exact(r.cpu(), res, "residual")
    modulation_stats(m.cpu(), mod, t.numpy(), dtype, "modulated")
