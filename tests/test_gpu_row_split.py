"""Row-block sharding on one GPU: every operation run on contiguous row
blocks of one problem -- the blocks replicas.row_block gives ranks of a world
of 2 or 3, each passed through the C ABI as an offset view of the full
tensors (inputs and outputs) -- must write the same bits as one call over all
rows.  This is the property the multi-GPU path rests on (rows are
independent; the RMS statistic is per row), checked under both row
statistics, at widths that reach the staged (4096), phased (3077), 8-byte
(3076) and two-pass (20000) kernels, with block boundaries that fall off a
16-byte boundary."""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import bits, mod_inputs, rga_inputs
from _gpu import ensure_built
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
def test_row_blocks_equal_one_call(statistic, case, world):
    L, D, dtype = case
    h, u, gb = (t.cuda() for t in rga_inputs(1, L, D, dtype, "bcast", tag="split"))
    gf = rga_inputs(1, L, D, dtype, "full", tag="splitf")[2].cuda()
    _, scb, shb = (t.cuda() for t in mod_inputs(1, L, D, dtype, "bcast", tag="split"))
    _, scf, shf = (t.cuda() for t in mod_inputs(1, L, D, dtype, "full", tag="splitf"))
    qs = torch.full((1,), 0.02, dtype=torch.float32, device="cuda")

    def rows(t, s, e):
        return t[:, s:e] if t.shape[1] == L else t

    ops = {
        "rga_bcast": (lambda s, e, o: dit.residual_gate_add(rows(h, s, e), rows(u, s, e),
                                                             gb, out=o[0]), 1),
        "rga_full": (lambda s, e, o: dit.residual_gate_add(rows(h, s, e), rows(u, s, e),
                                                            rows(gf, s, e), out=o[0]), 1),
        "mod_bcast": (lambda s, e, o: dit.rmsnorm_modulate(rows(h, s, e), scb, shb, EPS,
                                                            out=o[0]), 1),
        "mod_full": (lambda s, e, o: dit.rmsnorm_modulate(rows(h, s, e), rows(scf, s, e),
                                                           rows(shf, s, e), EPS, out=o[0]), 1),
        "fused_bcast": (lambda s, e, o: dit.gate_add_rmsnorm_modulate(
            rows(h, s, e), rows(u, s, e), gb, scb, shb, EPS, residual_out=o[0],
            modulated_out=o[1]), 2),
        "fused_full_full": (lambda s, e, o: dit.gate_add_rmsnorm_modulate(
            rows(h, s, e), rows(u, s, e), rows(gf, s, e), rows(scf, s, e), rows(shf, s, e), EPS,
            residual_out=o[0], modulated_out=o[1]), 2),
        "mod_fp8": (lambda s, e, o: dit.rmsnorm_modulate_fp8(rows(h, s, e), scb, shb, qs, EPS,
                                                              out=o[0]), 1),
    }
    for name, (call, nout) in ops.items():
        fp8 = name.endswith("fp8")
        def outputs():
            if fp8:
                return [torch.full((1, L, D), 0x55, dtype=torch.uint8, device="cuda")]
            return [torch.full_like(h, 3.0) for _ in range(nout)]
        whole, split = outputs(), outputs()
        call(0, L, whole)
        for s, e in _blocks(L, world):
            call(s, e, [o[:, s:e] for o in split])
        torch.cuda.synchronize()
        for k in range(nout):
            _same(split[k], whole[k], f"{name} output {k} world {world} {case}")
