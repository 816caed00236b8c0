"""Row-block sharding on one GPU: every operation run on contiguous row
blocks of one problem -- the blocks replicas.row_block gives ranks of a world
of 2 or 3, each passed through the C ABI as an offset view of the full
tensors (inputs and outputs) -- must write the same bits as one call over all
rows.  This is the property the multi-GPU path rests on (rows are
independent; the RMS statistic is per row), checked under both row
statistics, at widths that reach the staged (4096), phased (3077), 8-byte
(3076) and two-pass (20000) kernels, with block boundaries that fall off a
16-byte boundary.

One exception, by design: the fast statistic's fp32 sum depends on the
kernel's summation order, and a block whose view starts off a 16-byte
boundary takes another kernel (narrower accesses) than the whole call.  The
modulated outputs of such a split are therefore checked against the oracle
under the fast statistic's criterion instead of bitwise; every residual, and
every output under the exact statistic, is compared bit for bit.
"""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import bits, mod_inputs, oracle_fused, oracle_mod, rga_inputs
from _gpu import ensure_built, modulation_stats
from diffusion_transformer_elementwise_gb300.replicas import row_block

pytestmark = pytest.mark.gpu

EPS = 1e-6
CASES = [(1001, 4096, "bf16"), (203, 3077, "bf16"), (77, 3076, "fp16"), (61, 4096, "fp32"),
         (11, 20000, "bf16")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _blocks(L, world):
    return [row_block(L, r, world) for r in range(world)]


def _same(a, b, what):
    assert np.array_equal(bits(a.cpu()), bits(b.cpu())), what


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c)))
def test_row_blocks_equal_one_call(orc, statistic, case, world):
    L, D, dtype = case
    es = 4 if dtype == "fp32" else 2
    h, u, gb = (t.cuda() for t in rga_inputs(1, L, D, dtype, "bcast", tag="split"))
    gf = rga_inputs(1, L, D, dtype, "full", tag="splitf")[2].cuda()
    _, scb, shb = (t.cuda() for t in mod_inputs(1, L, D, dtype, "bcast", tag="split"))
    _, scf, shf = (t.cuda() for t in mod_inputs(1, L, D, dtype, "full", tag="splitf"))
    qs = torch.full((1,), 0.02, dtype=torch.float32, device="cuda")
    blocks = _blocks(L, world)
    # every block's view starts on a 16-byte boundary: the same kernel as the
    # whole call (the tensors themselves are 256-byte aligned)
    aligned = all((s * D * es) % 16 == 0 for s, _ in blocks)

    def rows(t, s, e):
        return t[:, s:e] if t.shape[1] == L else t

    # name: (call, outputs, index of the modulated output or None, oracle of it)
    ops = {
        "rga_bcast": (lambda s, e, o: dit.residual_gate_add(rows(h, s, e), rows(u, s, e),
                                                             gb, out=o[0]), 1, None, None),
        "rga_full": (lambda s, e, o: dit.residual_gate_add(rows(h, s, e), rows(u, s, e),
                                                            rows(gf, s, e), out=o[0]), 1, None,
                     None),
        "mod_bcast": (lambda s, e, o: dit.rmsnorm_modulate(rows(h, s, e), scb, shb, EPS,
                                                            out=o[0]), 1, 0,
                      lambda: oracle_mod(orc, h.cpu(), scb.cpu(), shb.cpu(), dtype, "bcast",
                                         EPS, with_t=True)),
        "mod_full": (lambda s, e, o: dit.rmsnorm_modulate(rows(h, s, e), rows(scf, s, e),
                                                           rows(shf, s, e), EPS, out=o[0]), 1, 0,
                     lambda: oracle_mod(orc, h.cpu(), scf.cpu(), shf.cpu(), dtype, "full", EPS,
                                        with_t=True)),
        "fused_bcast": (lambda s, e, o: dit.gate_add_rmsnorm_modulate(
            rows(h, s, e), rows(u, s, e), gb, scb, shb, EPS, residual_out=o[0],
            modulated_out=o[1]), 2, 1,
            lambda: oracle_fused(orc, h.cpu(), u.cpu(), gb.cpu(), scb.cpu(), shb.cpu(), dtype,
                                 "bcast", "bcast", EPS, with_t=True)[1:]),
        "fused_full_full": (lambda s, e, o: dit.gate_add_rmsnorm_modulate(
            rows(h, s, e), rows(u, s, e), rows(gf, s, e), rows(scf, s, e), rows(shf, s, e), EPS,
            residual_out=o[0], modulated_out=o[1]), 2, 1,
            lambda: oracle_fused(orc, h.cpu(), u.cpu(), gf.cpu(), scf.cpu(), shf.cpu(), dtype,
                                 "full", "full", EPS, with_t=True)[1:]),
    }
    if (D * es) % 16 == 0 and D * es <= 16384:  # rows the E4M3 output takes
        ops["mod_fp8"] = (lambda s, e, o: dit.rmsnorm_modulate_fp8(rows(h, s, e), scb, shb, qs,
                                                                   EPS, out=o[0]), 1, None, None)
    for name, (call, nout, mk, ref) in ops.items():
        fp8 = name.endswith("fp8")

        def outputs():
            if fp8:
                return [torch.full((1, L, D), 0x55, dtype=torch.uint8, device="cuda")]
            return [torch.full_like(h, 3.0) for _ in range(nout)]
        whole, split = outputs(), outputs()
        call(0, L, whole)
        for s, e in blocks:
            call(s, e, [o[:, s:e] for o in split])
        torch.cuda.synchronize()
        for k in range(nout):
            what = f"{name} output {k} world {world} {case}"
            if k == mk and statistic == "fast" and not aligned:
                r, t = ref()
                modulation_stats(split[k].cpu(), r, t.numpy(), dtype, what)
            else:
                _same(split[k], whole[k], what)



# Large tensors: the two-warp kernel's tapered schedule (CTAs of several rows
# per team, then a last wave of one row per team, in every batch) against the
# same rows called in blocks small enough for its one-wave schedule.  The
# modulation runs the same kernel instantiation either way (same granules per
# lane), whose per-row arithmetic does not depend on which team takes the
# row, so its bits must agree under either statistic.  The fused op takes the
# CTA-per-row kernel on small blocks, so there its residual (exact
# arithmetic) is compared bit for bit, its modulated output bitwise under the
# exact statistic and against the oracle on sampled rows of every batch under
# the fast one.  NaN-filled outputs show any element left unwritten.
# Ragged L, several batches, two and four granules per lane.
LARGE = [(1, 60013, 1024, "bf16"), (3, 20011, 1024, "bf16"), (2, 30001, 1024, "fp32")]


@pytest.mark.parametrize("case", LARGE, ids=lambda c: "x".join(map(str, c)))
def test_large_tensor_schedule_equals_blocks(orc, statistic, case):
    B, L, D, dtype = case
    from diffusion_transformer_elementwise_gb300.synth import draw, seed_for
    h = draw("act", (B, L, D), seed_for("large", "h", *case), dtype, "cuda")
    u = draw("act", (B, L, D), seed_for("large", "u", *case), dtype, "cuda")
    g = draw("gate", (B, 1, D), seed_for("large", "g", *case), dtype, "cuda")
    sc = draw("mod", (B, 1, D), seed_for("large", "sc", *case), dtype, "cuda")
    sh = draw("mod", (B, 1, D), seed_for("large", "sh", *case), dtype, "cuda")
    block = 2048  # rows per call: far below one wave's eight rows per team
    calls = {
        "mod": (1, lambda hs, us, gs, scs, shs, o: dit.rmsnorm_modulate(hs, scs, shs, EPS,
                                                                       out=o[0])),
        "fused": (2, lambda hs, us, gs, scs, shs, o: dit.gate_add_rmsnorm_modulate(
            hs, us, gs, scs, shs, EPS, residual_out=o[0], modulated_out=o[1])),
    }
    for name, (nout, call) in calls.items():
        whole = [torch.full_like(h, float("nan")) for _ in range(nout)]
        parts = [torch.full_like(h, float("nan")) for _ in range(nout)]
        call(h, u, g, sc, sh, whole)
        for b in range(B):
            for s in range(0, L, block):
                e = min(L, s + block)
                call(h[b:b + 1, s:e], u[b:b + 1, s:e], g[b:b + 1], sc[b:b + 1], sh[b:b + 1],
                     [o[b:b + 1, s:e] for o in parts])
        torch.cuda.synchronize()
        for k in range(nout):
            what = f"{name} output {k} {case}"
            assert not torch.isnan(whole[k]).any(), what + ": unwritten elements"
            if name == "fused" and k == 1 and statistic == "fast":
                idx = torch.tensor(sorted({0, L - 1, *np.random.default_rng(
                    seed_for("large rows", *case) & 0xFFFFFFFF).choice(L, 254, replace=False)
                    .tolist()}))
                d = idx.cuda()
                rows = [t[:, d].contiguous().cpu() for t in (h, u)]
                _, ref, t = oracle_fused(orc, *rows, g.cpu(), sc.cpu(), sh.cpu(), dtype,
                                         "bcast", "bcast", EPS, with_t=True, threads=8)
                modulation_stats(whole[k][:, d].contiguous().cpu(), ref, t.numpy(), dtype, what)
            else:
                _same(whole[k], parts[k], what)
