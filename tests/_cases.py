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


# ---------------------------------------------------------------------------
# rows on the rounding boundaries of the row statistic ms = RN32(mean x^2)
# ---------------------------------------------------------------------------

# name: (k, extra element, expected mean).  The squares of a row add up to
# exactly D * (1 + k * 2^-24): the mean is the midpoint between two fp32
# values (k odd).  k = 1 rounds down to 1 (even), k = 3 up to 1 + 2^-22; one
# more tiny element lifts the k = 1 mean above its midpoint (up to
# 1 + 2^-23); one 1-unit element made 2^-12 * 255/256 puts the k = 3 mean
# below its midpoint (down to 1 + 2^-23).
BOUNDARY_VARIANTS = {
    "tie_even": (1, None, 1.0),
    "tie_up": (3, None, 1.0 + 2.0 ** -22),
    "above": (1, "tiny", 1.0 + 2.0 ** -23),
    "below": (3, "short", 1.0 + 2.0 ** -23),
}


def _greedy(total, values):
    """Elements from `values` (value, weight) whose weights add to total."""
    out = []
    for v, w in values:
        n, total = divmod(total, w)
        out += [v] * n
    assert total == 0
    return out


def boundary_row(D, variant, rng, dtype, scale_exp=0):
    """One row of D values (float64, exact in `dtype`): the integer part of
    the squares' sum from elements 8, 4, 2, 1 (squares 64, 16, 4, 1), the
    rest from 2^-9 .. 2^-12 (squares 64, 16, 4, 1 units of 2^-24), in a
    seeded order with seeded signs, scaled by 2^scale_exp (the squares by
    4^scale_exp: the same boundaries)."""
    k, extra, _ = BOUNDARY_VARIANTS[variant]
    units = k * D - (1 if extra == "short" else 0)
    elems = _greedy(D, [(8.0, 64), (4.0, 16), (2.0, 4), (1.0, 1)])
    elems += _greedy(units, [(2.0 ** -9, 64), (2.0 ** -10, 16), (2.0 ** -11, 4),
                             (2.0 ** -12, 1)])
    if extra == "tiny":  # its square is far below half an ulp of the sum
        elems.append(2.0 ** -24 if dtype == "fp16" else 2.0 ** -30)
    elif extra == "short":
        elems.append(2.0 ** -12 * 255 / 256)
    assert len(elems) <= D, (D, variant, len(elems))
    row = np.zeros(D)
    row[: len(elems)] = elems
    row = rng.permutation(row) * rng.choice([-1.0, 1.0], size=D)
    return row * 2.0 ** scale_exp


def boundary_tensor(B, L, D, dtype, seed, scale_exp=0):
    """[B, L, D] of boundary rows, the variants in turn; returns the tensor
    (CPU, dtype) and the variant of each row."""
    from diffusion_transformer_elementwise_gb300.synth import TORCH_DTYPES
    rng = np.random.default_rng(seed)
    names = list(BOUNDARY_VARIANTS)
    rows = np.stack([boundary_row(D, names[i % len(names)], rng, dtype, scale_exp)
                     for i in range(B * L)]).reshape(B, L, D)
    x = torch.tensor(rows, dtype=torch.float64).to(TORCH_DTYPES[dtype])
    assert torch.equal(x.double(), torch.tensor(rows)), "row values not exact in the dtype"
    return x, [names[i % len(names)] for i in range(B * L)]
