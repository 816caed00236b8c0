"""Kernels that need more than 48 KB of dynamic shared memory are opted in
once per kernel and device.  Two kernels of one launcher -- the two-warp
kernel for rows whose pitch is a multiple of 16 bytes and its phased
variant, at the same granules per lane -- must each be opted in, in either
order of first use.  Each order runs in a fresh process, so that no earlier
call has opted either kernel in."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
import torch
import diffusion_transformer_elementwise_gb300 as dit
order = sys.argv[1].split(",")
for D in (int(d) for d in order):
    for op in ("mod", "fused"):
        L = 20000  # large enough for the fused op's two-warp schedule
        h = torch.randn(1, L, D, device="cuda").bfloat16()
        u = torch.randn(1, L, D, device="cuda").bfloat16()
        g = torch.randn(1, 1, D, device="cuda").bfloat16()
        sc = torch.randn(1, 1, D, device="cuda").bfloat16() * 0.1
        sh = torch.randn(1, 1, D, device="cuda").bfloat16() * 0.1
        if op == "mod":
            dit.rmsnorm_modulate(h, sc, sh)
        else:
            dit.gate_add_rmsnorm_modulate(h, u, g, sc, sh)
torch.cuda.synchronize()
print("ok")
"""


@pytest.mark.parametrize("order", ["3080,3077", "3077,3080"])
def test_both_kernels_opted_in_in_either_order(order):
    from _gpu import ensure_built
    ensure_built()
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", SCRIPT, order], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
