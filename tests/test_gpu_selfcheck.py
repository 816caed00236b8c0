"""GPU tests of dit_selfcheck: every runtime key of the library passes its
own bit-for-bit check, and the check's inputs, its production outputs and
its reference outputs, read back from the workspace, all agree bit for bit
with the oracle (which pins the check's reference to the pages' definition
and shows that its inputs make every output unique)."""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import oracle_fused, oracle_mod, oracle_rga
from _gpu import assert_bit_exact, ensure_built
from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES

pytestmark = pytest.mark.gpu

# one width per kernel path: narrow, 16-byte aligned rows, 8- and 4-byte
# aligned rows (bf16 3076 / 3077), the largest staged rows, long rows
WIDTHS = [64, 2048, 3076, 3077, 4096, 8192, 16384]
KEYS = ([("residual_gate", g, "bcast") for g in ("bcast", "full")] +
        [("rmsnorm_modulate", "bcast", m) for m in ("bcast", "full")] +
        [("gate_add_rmsnorm_modulate", g, m) for g in ("bcast", "full")
         for m in ("bcast", "full")])
B, L = 2, 7


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("D", WIDTHS)
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
def test_every_key_passes(dtype, D):
    for op, glay, mlay in KEYS:
        assert dit.selfcheck(op, dtype, glay, mlay, D) == 0, (op, dtype, glay, mlay, D)


def _tensors(work, dtype, D):
    """The workspace's nine tensors (x, update, gate, scale, shift, out, out2,
    expected, expected2) as CPU tensors of [2, 7, D]."""
    es = 4 if dtype == "fp32" else 2
    n = B * L * D
    slot = (n * es + 255) // 256 * 256
    raw = work.cpu()
    out = []
    for i in range(9):
        t = raw[i * slot:i * slot + n * es].view(TORCH_DTYPES[dtype]).view(B, L, D)
        out.append(t.clone())
    return out


def _vec(t, layout):
    return t if layout == "full" else t.reshape(-1)[:B * D_of(t)].view(B, 1, D_of(t)).clone()


def D_of(t):
    return t.shape[-1]


@pytest.mark.parametrize("D", [64, 3077, 4096])
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("key", KEYS)
def test_workspace_agrees_with_oracle(orc, key, dtype, D):
    op, glay, mlay = key
    n, work = dit.selfcheck(op, dtype, glay, mlay, D, return_workspace=True)
    torch.cuda.synchronize()
    assert n == 0
    x, u, g, sc, sh, out, out2, exp, exp2 = _tensors(work, dtype, D)
    if op == "residual_gate":
        ref = oracle_rga(orc, x, u, _vec(g, glay), dtype, glay)
        assert_bit_exact(out, ref, "out")
        assert_bit_exact(exp, ref, "expected")
    elif op == "rmsnorm_modulate":
        assert set(np.unique(x.float().numpy()).tolist()) <= {-0.5, 0.5}
        ref = oracle_mod(orc, x, _vec(sc, mlay), _vec(sh, mlay), dtype, mlay, eps=0.75)
        assert_bit_exact(out, ref, "out")
        assert_bit_exact(exp, ref, "expected")
    else:
        res, mod = oracle_fused(orc, x, u, _vec(g, glay), _vec(sc, mlay), _vec(sh, mlay), dtype,
                                glay, mlay, eps=0.75)
        assert set(np.unique(res.float().numpy()).tolist()) <= {-0.5, 0.5}
        assert_bit_exact(out, res, "residual")
        assert_bit_exact(exp, res, "expected residual")
        assert_bit_exact(out2, mod, "modulated")
        assert_bit_exact(exp2, mod, "expected modulated")


def test_first_use_registry():
    key = ("gate_add_rmsnorm_modulate", "bf16", "bcast", "bcast", 1536)
    assert dit.ensure_checked(*key) is True
    assert dit.ensure_checked(*key) is False
    from diffusion_transformer_elementwise_gb300 import _binding
    x = torch.randn(1, 5, 2560, device="cuda").to(torch.bfloat16)
    sc = torch.zeros(1, 1, 2560, device="cuda", dtype=torch.bfloat16)
    dit.set_first_use_check(True)
    try:
        dit.rmsnorm_modulate(x, sc, sc, 1e-6)
    finally:
        dit.set_first_use_check(False)
    assert ("rmsnorm_modulate", "bf16", "bcast", "bcast", 2560,
            torch.cuda.current_device()) in _binding._checked
