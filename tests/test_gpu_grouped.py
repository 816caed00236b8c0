"""GPU parity of the grouped launches (dit_grouped) against the oracle.

Each problem of a grouped call must give what the oracle gives for it alone:
the residual bit-exact, the modulated output within the modulation
criterion.  Problem sets: the video and audio streams of an LTX-2 block
(hidden 4096 and 2048: prhub summary of sglang PR #34172, test section),
widths from 64 to 8192, eight problems, empty problems, strided adaLN-table
vectors, and sets that cannot share one kernel (unaligned rows, rows too long
for the staged kernel, a full gate), which take one launch per problem.
"""
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import mod_inputs, oracle_fused, oracle_mod, oracle_rga, rga_inputs
from _gpu import assert_bit_exact, ensure_built, modulation_stats
from diffusion_transformer_elementwise_gb300.synth import draw, seed_for

pytestmark = pytest.mark.gpu
EPS = 1e-6

SETS = {
    "video_audio": [(1, 37, 4096), (1, 19, 2048)],
    "video_audio_b2": [(2, 21, 4096), (2, 9, 2048)],
    "widths": [(1, 5, 1024), (1, 13, 3072), (1, 7, 8192), (1, 3, 64), (2, 4, 256)],
    "eight": [(1, 3 + 2 * i, 512 * (1 + i % 4)) for i in range(8)],
    "with_empty": [(1, 0, 4096), (1, 11, 2048), (0, 5, 1024)],
    "unaligned": [(1, 9, 4096), (1, 7, 3077)],
    "long_rows": [(1, 3, 16384), (1, 6, 2048)],
    "single": [(1, 17, 2048)],
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _fused_inputs(B, L, D, dtype, glay, mlay, tag):
    h, u, g = rga_inputs(B, L, D, dtype, glay, tag=tag)
    _, sc, sh = mod_inputs(B, L, D, dtype, mlay, tag=tag)
    return h, u, g, sc, sh


def _check_mod(gpu, ref, t, dtype, what):
    if ref.numel():
        modulation_stats(gpu.cpu(), ref, t.numpy(), dtype, what)


@pytest.mark.parametrize("gate_layout", ["bcast", "full"])
@pytest.mark.parametrize("name", list(SETS))
def test_grouped_residual_gate(orc, name, gate_layout):
    dtype = "bf16"
    cpu = [rga_inputs(B, L, D, dtype, gate_layout, tag=f"grp-rga{i}")
           for i, (B, L, D) in enumerate(SETS[name])]
    outs = dit.residual_gate_add_grouped([tuple(t.cuda() for t in p) for p in cpu])
    torch.cuda.synchronize()
    for i, ((h, u, g), o) in enumerate(zip(cpu, outs)):
        assert_bit_exact(o.cpu(), oracle_rga(orc, h, u, g, dtype, gate_layout), f"{name}[{i}]")


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("name", ["video_audio", "video_audio_b2", "widths", "eight",
                                  "with_empty", "unaligned", "long_rows", "single"])
def test_grouped_modulate(orc, statistic, name, dtype):
    shapes = SETS[name]  # fp32 rows above 4096 elements take one launch per problem
    cpu = [mod_inputs(B, L, D, dtype, "bcast", tag=f"grp-mod{i}")
           for i, (B, L, D) in enumerate(shapes)]
    outs = dit.rmsnorm_modulate_grouped([tuple(t.cuda() for t in p) for p in cpu], EPS)
    torch.cuda.synchronize()
    for i, ((x, sc, sh), o) in enumerate(zip(cpu, outs)):
        ref, t = oracle_mod(orc, x, sc, sh, dtype, "bcast", EPS, with_t=True)
        _check_mod(o, ref, t, dtype, f"{name}[{i}]")


@pytest.mark.parametrize("layouts", [("bcast", "bcast"), ("full", "bcast"), ("bcast", "full"),
                                     ("full", "full")])
@pytest.mark.parametrize("name", ["video_audio", "video_audio_b2", "widths", "eight",
                                  "with_empty", "unaligned", "long_rows"])
def test_grouped_fused(orc, statistic, name, layouts):
    dtype = "bf16"
    glay, mlay = layouts
    cpu = [_fused_inputs(B, L, D, dtype, glay, mlay, f"grp-fused{i}")
           for i, (B, L, D) in enumerate(SETS[name])]
    outs = dit.gate_add_rmsnorm_modulate_grouped([tuple(t.cuda() for t in p) for p in cpu], EPS)
    torch.cuda.synchronize()
    for i, (p, (r, m)) in enumerate(zip(cpu, outs)):
        res, mod, t = oracle_fused(orc, *p, dtype, glay, mlay, EPS, with_t=True)
        assert_bit_exact(r.cpu(), res, f"{name}[{i}] residual")
        _check_mod(m, mod, t, dtype, f"{name}[{i}] modulated")


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_grouped_fused_dtypes(orc, dtype):
    cpu = [_fused_inputs(B, L, D, dtype, "bcast", "bcast", f"grp-fdt{i}")
           for i, (B, L, D) in enumerate(SETS["video_audio_b2"])]
    outs = dit.gate_add_rmsnorm_modulate_grouped([tuple(t.cuda() for t in p) for p in cpu], EPS)
    torch.cuda.synchronize()
    for i, (p, (r, m)) in enumerate(zip(cpu, outs)):
        res, mod, t = oracle_fused(orc, *p, dtype, "bcast", "bcast", EPS, with_t=True)
        assert_bit_exact(r.cpu(), res, f"[{i}] residual")
        _check_mod(m, mod, t, dtype, f"[{i}] modulated")


def test_grouped_in_place_and_adaln_tables(orc):
    """In-place residuals and [B, 1, D] vectors read as rows of per-stream
    adaLN tables [B, 9, D] (batch stride 9 * D), as a block's site would."""
    dtype = "bf16"
    probs, cpu = [], []
    for i, (B, L, D) in enumerate(SETS["video_audio_b2"]):
        h, u, _ = rga_inputs(B, L, D, dtype, "bcast", tag=f"grp-tab{i}")
        table = draw("mod", (B, 9, D), seed_for("grp-table", i, B, D), dtype)
        shift, scale, gate = (table[:, k:k + 1, :] for k in (3, 4, 5))
        cpu.append((h.clone(), u, gate.contiguous(), scale.contiguous(), shift.contiguous()))
        tg = table.cuda()
        hd = h.cuda()
        probs.append((hd, u.cuda(), tg[:, 5:6, :], tg[:, 4:5, :], tg[:, 3:4, :], hd, None))
    outs = dit.gate_add_rmsnorm_modulate_grouped(probs, EPS)
    torch.cuda.synchronize()
    for i, (p, (r, m)) in enumerate(zip(cpu, outs)):
        assert r.data_ptr() == probs[i][0].data_ptr()
        res, mod, t = oracle_fused(orc, *p, dtype, "bcast", "bcast", EPS, with_t=True)
        assert_bit_exact(r.cpu(), res, f"[{i}] residual")
        _check_mod(m, mod, t, dtype, f"[{i}] modulated")


def test_grouped_video_equals_single_call():
    """The grouped launch gives the widest problem the same outputs as its
    single call, bit for bit -- under the exact statistic, which every kernel
    computes to the same bits (the fast statistic's sum order is the
    kernel's, and the single call may take the two-warp kernel)."""
    dtype = "bf16"
    video, audio = (_fused_inputs(B, L, D, dtype, "bcast", "bcast", f"grp-eq{i}")
                    for i, (B, L, D) in enumerate(SETS["video_audio"]))
    vg = tuple(t.cuda() for t in video)
    with dit.statistic("exact"):
        (rg, mg), _ = dit.gate_add_rmsnorm_modulate_grouped([vg, tuple(t.cuda() for t in audio)],
                                                            EPS)
        rs, ms = dit.gate_add_rmsnorm_modulate(*vg, EPS)
    torch.cuda.synchronize()
    assert torch.equal(rg.view(torch.int16), rs.view(torch.int16))
    assert torch.equal(mg.view(torch.int16), ms.view(torch.int16))


def test_grouped_full_size_video_audio_sampled(orc):
    """The largest video shape with the smallest (audio) shape in one fused
    launch: [1, 32640, 4096] + [1, 126, 2048] bf16; 64 sampled video rows and
    every audio row against the oracle."""
    dtype = "bf16"
    shapes = [(1, 32640, 4096), (1, 126, 2048)]
    dev = [tuple(draw(kind, shp, seed_for("grp-full", i, kind, j), dtype, "cuda")
                 for j, (kind, shp) in enumerate([("act", (B, L, D)), ("act", (B, L, D)),
                                                  ("gate", (B, 1, D)), ("mod", (B, 1, D)),
                                                  ("mod", (B, 1, D))]))
           for i, (B, L, D) in enumerate(shapes)]
    outs = dit.gate_add_rmsnorm_modulate_grouped(dev, EPS)
    torch.cuda.synchronize()
    g = torch.Generator().manual_seed(9)
    rows = [torch.cat([torch.tensor([0, 32639]), torch.randint(1, 32639, (62,), generator=g)]),
            torch.arange(126)]
    for i, ((h, u, gt, sc, sh), (r, m)) in enumerate(zip(dev, outs)):
        idx = rows[i].cuda()
        sub = [h[:, idx].cpu(), u[:, idx].cpu(), gt.cpu(), sc.cpu(), sh.cpu()]
        res, mod, t = oracle_fused(orc, *sub, dtype, "bcast", "bcast", EPS, with_t=True)
        assert_bit_exact(r[:, idx].cpu(), res, f"[{i}] residual")
        _check_mod(m[:, idx], mod, t, dtype, f"[{i}] modulated")
