"""Small helpers shared by the tests: seeded inputs and oracle calls on torch
CPU tensors.  No arithmetic of the method lives here."""
from __future__ import annotations

import numpy as np
import torch

from diffusion_transformer_elementwise_gb300.synth import draw, seed_for, vector_shape


def rga_inputs(B, L, D, dtype, gate_layout, tag="rga", device="cpu", row_spread=False):
    h = draw("act", (B, L, D), seed_for(tag, "hidden", B, L, D, dtype), dtype, device,
             row_spread=row_spread)
    u = draw("act", (B, L, D), seed_for(tag, "update", B, L, D, dtype), dtype, device)
    g = draw("gate", vector_shape(B, L, D, gate_layout),
             seed_for(tag, "gate", gate_layout, B, L, D, dtype), dtype, device)
    return h, u, g


def mod_inputs(B, L, D, dtype, mod_layout, tag="mod", device="cpu", row_spread=False):
    x = draw("act", (B, L, D), seed_for(tag, "x", B, L, D, dtype), dtype, device,
             row_spread=row_spread)
    sc = draw("mod", vector_shape(B, L, D, mod_layout),
              seed_for(tag, "scale", mod_layout, B, L, D, dtype), dtype, device)
    sh = draw("mod", vector_shape(B, L, D, mod_layout),
              seed_for(tag, "shift", mod_layout, B, L, D, dtype), dtype, device)
    return x, sc, sh


def oracle_rga(orc, h, u, g, dtype, gate_layout, rows=None, threads=1, out=None):
    B, L, D = h.shape
    out = torch.empty_like(h) if out is None else out
    orc.residual_gate_add(out, h, u, g, B, L, D, dtype, gate_layout, rows=rows,
                          threads=threads)
    return out


def oracle_mod(orc, x, sc, sh, dtype, mod_layout, eps=1e-6, rows=None, with_t=False,
               threads=1):
    B, L, D = x.shape
    out = torch.empty_like(x)
    t = torch.empty(x.shape, dtype=torch.float32) if with_t else None
    orc.rmsnorm_modulate(out, x, sc, sh, B, L, D, eps, dtype, mod_layout, rows=rows,
                         t_out=t, threads=threads)
    return (out, t) if with_t else out


def oracle_fused(orc, h, u, g, sc, sh, dtype, gate_layout, mod_layout, eps=1e-6,
                 rows=None, with_t=False, threads=1, residual_out=None):
    B, L, D = h.shape
    res = torch.empty_like(h) if residual_out is None else residual_out
    mod = torch.empty_like(h)
    t = torch.empty(h.shape, dtype=torch.float32) if with_t else None
    orc.gate_add_rmsnorm_modulate(res, mod, h, u, g, sc, sh, B, L, D, eps, dtype,
                                  gate_layout, mod_layout, rows=rows, t_out=t,
                                  threads=threads)
    return (res, mod, t) if with_t else (res, mod)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw storage words of a tensor as an unsigned numpy array."""
    t = t.contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.shape == b.shape and np.array_equal(bits(a), bits(b))
