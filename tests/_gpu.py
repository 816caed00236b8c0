"""Comparison helpers for the GPU parity tests (CUDA path vs CPU oracle).

Criteria (each stated in the repository's design notes with its derivation):

* residual gate and the fused op's residual: bit-exact;
* modulation with the exact row statistic (dit_set_statistic): bit-exact for
  every dtype -- the statistic is two single roundings of exact values on
  both sides and the rest is the same IEEE operations in the same order;
* modulation with the fast statistic (the default): bf16/fp16 every element
  bit-exact or 1 ulp away, except where the final add cancels (|t| >> |y|):
  there within one dtype ulp of max(|t|, |y|) -- the bound of a rounded sum --
  and such elements are counted; fp32 |gpu - oracle| <= 2^-18 max(|t|, |y|).
NaN outputs must be NaN at the same positions (their payload bits are not
compared).
"""
from __future__ import annotations

import numpy as np
import torch

from diffusion_transformer_elementwise_gb300.build import build


def ensure_built():
    build()


def words(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16).reshape(-1)
    return t.view(torch.int32).numpy().view(np.uint32).reshape(-1)


def values(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().reshape(-1).astype(np.float64)


def ordered(w: np.ndarray, bits: int) -> np.ndarray:
    w = w.astype(np.int64)
    sign = 1 << (bits - 1)
    return np.where(w & sign, -(w & (sign - 1)), w)


def ulp_distance(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    bits = 8 * a.element_size()
    return np.abs(ordered(words(a), bits) - ordered(words(b), bits))


def spacing(v: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the dtype's values at |v| (normal range; subnormal floor)."""
    mant = {"bf16": 8, "fp16": 11, "fp32": 24}[dtype]
    emin = {"bf16": -126, "fp16": -14, "fp32": -126}[dtype]
    _, e = np.frexp(np.abs(v))
    e = np.maximum(e - 1, emin)
    return np.ldexp(1.0, e - mant + 1)


def assert_bit_exact(gpu: torch.Tensor, ref: torch.Tensor, what=""):
    g, r = words(gpu), words(ref)
    bad = np.nonzero(g != r)[0]
    assert bad.size == 0, f"{what}: {bad.size} elements differ, first at {bad[:5]}: " \
                          f"gpu {values(gpu)[bad[:5]]} oracle {values(ref)[bad[:5]]}"


def modulation_stats(gpu: torch.Tensor, ref: torch.Tensor, t: np.ndarray, dtype: str,
                     what="", exact=None) -> dict:
    """Check the modulation criterion of the library's current row statistic
    (or of `exact` when given); return the reported statistics."""
    if exact is None:
        import diffusion_transformer_elementwise_gb300 as dit
        exact = dit.get_statistic() == "exact"
    gv, rv = values(gpu), values(ref)
    nan_g, nan_r = np.isnan(gv), np.isnan(rv)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    ok = ~nan_r
    gv, rv, tt = gv[ok], rv[ok], np.abs(t.reshape(-1)[ok].astype(np.float64))
    scale = np.maximum(tt, np.abs(rv))
    diff = np.abs(gv - rv)
    d = ulp_distance(gpu, ref)[ok]
    if exact:
        bad = d != 0
        fallback = np.zeros_like(bad)
    elif dtype == "fp32":
        bad = diff > 2.0 ** -18 * scale + 1e-38
        fallback = np.zeros_like(bad)
    else:
        within = d <= 1
        fallback = ~within & (diff <= spacing(scale, dtype))
        bad = ~within & ~fallback
    idx = np.nonzero(bad)[0]
    assert idx.size == 0, (f"{what}: {idx.size} elements outside the "
                           f"{'exact' if exact else 'fast'}-statistic criterion "
                           f"(max {int(d.max())} ulp), first {idx[:5]}: gpu {gv[idx[:5]]} "
                           f"oracle {rv[idx[:5]]} t {tt[idx[:5]]}")
    denom = np.sqrt(np.sum(rv * rv))
    pos = scale > 0
    err_u = float((diff[pos] / scale[pos]).max()) / 2.0 ** -24 if pos.any() else 0.0
    return {
        # |gpu - oracle| / max(|t|, |y|) in units of 2^-24 (the fp32
        # criterion's measure: 2^-18 is 64 of them)
        "max_err_u": err_u,
        "statistic": "exact" if exact else "fast",
        "max_ulp": int(d.max()) if d.size else 0,
        "not_bit_exact": int(np.count_nonzero(d)),
        "fallback": int(np.count_nonzero(fallback)),
        "max_abs": float(diff.max()) if diff.size else 0.0,
        "rel_l2": float(np.sqrt(np.sum(diff * diff)) / denom) if denom > 0 else 0.0,
        "n": int(d.size),
    }


def guarded(shape, dtype, device, pad=64, fill=-7.0):
    """An output tensor inside a larger buffer whose pad elements on both
    sides hold a canary; returns (view, checker)."""
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * pad,), fill, dtype=dtype, device=device)
    view = buf[pad:pad + n].view(shape)

    def untouched():
        b = buf.cpu().float()
        return bool(torch.all(b[:pad] == fill)) and bool(torch.all(b[pad + n:] == fill))

    return view, untouched


def offset_copy(t: torch.Tensor, offset_elems: int) -> torch.Tensor:
    """A copy of t on the GPU whose data starts offset_elems elements past an
    allocation boundary (to make misaligned pointers)."""
    n = t.numel()
    buf = torch.empty(n + offset_elems + 16, dtype=t.dtype, device="cuda")
    v = buf[offset_elems:offset_elems + n].view(t.shape)
    v.copy_(t)
    return v
