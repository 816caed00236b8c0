"""Every bf16 (update, gate) pair -- all 2^16 x 2^16 -- through the residual
gate on the GPU against the oracle, for a few hidden values: zero, ordinary
ones, and values near 2^-125, where a product that underflows fp32's
normal range meets a sum in the normal range (the case in which a fused
multiply-add and a multiply-then-add could differ).  The gate is a
[1, 1, 65536] row holding every bf16 value; update row i holds one bf16
value; 4096 rows per launch, 16 launches per hidden value.  Outputs must be
bit-exact, NaN matching NaN."""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _gpu import ensure_built

pytestmark = pytest.mark.gpu
ROWS = 4096


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _bf16(v: float) -> int:
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)[0]) & 0xFFFF


@pytest.mark.parametrize("h", [0.0, 1.0, -2.5, 2.0 ** -125, -3 * 2.0 ** -124, 2.0 ** -119])
def test_residual_gate_every_bf16_pair(orc, h):
    allw = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    gate = allw.view(torch.bfloat16).reshape(1, 1, 65536)
    gate_d = gate.cuda()
    hw = _bf16(h)
    hidden = torch.full((1, ROWS, 65536), hw if hw < 32768 else hw - 65536,
                        dtype=torch.int16).view(torch.bfloat16)
    hidden_d = hidden.cuda()
    out_d = torch.empty_like(hidden_d)
    ref = torch.empty_like(hidden)
    for c in range(65536 // ROWS):
        uw = allw[c * ROWS:(c + 1) * ROWS].reshape(1, ROWS, 1).expand(1, ROWS, 65536).contiguous()
        upd = uw.view(torch.bfloat16)
        dit.residual_gate_add(hidden_d, upd.cuda(), gate_d, out=out_d)
        orc.residual_gate_add(ref, hidden, upd, gate, 1, ROWS, 65536, "bf16", "bcast",
                              threads=16)
        torch.cuda.synchronize()
        g = out_d.cpu().view(torch.int16).numpy().view(np.uint16)
        r = ref.view(torch.int16).numpy().view(np.uint16)
        diff = g != r
        if diff.any():
            nan = lambda w: ((w & 0x7F80) == 0x7F80) & ((w & 0x7F) != 0)
            real = diff & ~(nan(g) & nan(r))
            idx = np.argwhere(real)
            assert idx.size == 0, (f"h={h}: {len(idx)} pairs differ, first (row, col) "
                                   f"{idx[:3].tolist()} in chunk {c}")
