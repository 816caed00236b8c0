"""Seeded synthetic inputs shaped like the pages' DiT workloads.

This module draws random numbers and nothing else: it holds none of the
operations' arithmetic, so the CUDA path and the CPU oracle can both consume
its output without sharing code.  Two generators:

* host (``device="cpu"``): a counter-based SplitMix64 stream turned into
  uniform doubles (top 53 bits) and, by the Box-Muller transform, normals.
  Identical on every host; used for the small parity cases.
* device (``device="cuda..."``): torch's seeded device generator, used for the
  full-size tensors (hundreds of MB), where host generation would dominate the
  run time.

Every value is rounded once to the storage dtype by torch's conversion.

Workload recipes (shapes from sglang PR #29361, section "Speed Tests and
Profiling", B200 kernel benchmark table: ltx2_bcast_s32640_c4096,
ltx2_full_s8160_c4096, ideogram4_bcast_s4096_c4608, flux2_bcast_s4608_c3072,
ltx2_full_s126_c2048; hidden sizes 4096 video / 2048 audio from the prhub
summary of sglang PR #34172, test section):

* activations (hidden, update, x) ~ N(0, 1);
* gate ~ U(-1, 1);
* adaLN scale / shift ~ N(0, 0.1);
* "row spread": each row of hidden (or x) multiplied by 10^U(-2, 2).
"""
from __future__ import annotations

import hashlib
import math

import numpy as np
import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}

_M64 = (1 << 64) - 1
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


def seed_for(*names, base: int = 42) -> int:
    """A stable 63-bit seed from a base seed and a tuple of names."""
    text = "/".join(str(n) for n in (base,) + names).encode()
    return int.from_bytes(hashlib.blake2b(text, digest_size=8).digest(), "little") & (_M64 >> 1)


def splitmix64(counter: np.ndarray, seed: int) -> np.ndarray:
    """SplitMix64 output for each 64-bit counter value (Steele, Lea and Flood,
    "Fast splittable pseudorandom number generators", OOPSLA 2014)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & _M64) + (counter.astype(np.uint64) + np.uint64(1)) * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
        return z ^ (z >> np.uint64(31))


def uniform01(n: int, seed: int, offset: int = 0) -> np.ndarray:
    """n doubles in [0, 1) from counters offset .. offset+n-1."""
    c = np.arange(offset, offset + n, dtype=np.uint64)
    return (splitmix64(c, seed) >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))


def host_normal(shape, seed: int, std: float = 1.0) -> np.ndarray:
    """Box-Muller normals: two uniforms per sample (counters 2i and 2i+1)."""
    n = int(np.prod(shape)) if len(shape) else 1
    u = uniform01(2 * n, seed).reshape(n, 2)
    radius = np.sqrt(-2.0 * np.log1p(-u[:, 0]))  # 1 - u in (0, 1]
    z = radius * np.cos(2.0 * math.pi * u[:, 1])
    return (z * std).reshape(shape)


def host_uniform(shape, seed: int, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return (lo + (hi - lo) * uniform01(n, seed)).reshape(shape)


def draw(kind: str, shape, seed: int, dtype: str = "bf16", device="cpu",
         row_spread: bool = False) -> torch.Tensor:
    """A tensor of the named distribution, rounded once to ``dtype``.

    kind: ``"act"`` N(0, 1) | ``"gate"`` U(-1, 1) | ``"mod"`` N(0, 0.1).
    row_spread: multiply each row (last dim) by 10^U(-2, 2).
    """
    shape = tuple(int(s) for s in shape)
    dev = torch.device(device)
    if dev.type == "cpu":
        if kind == "act":
            v = host_normal(shape, seed, 1.0)
        elif kind == "mod":
            v = host_normal(shape, seed, 0.1)
        elif kind == "gate":
            v = host_uniform(shape, seed, -1.0, 1.0)
        else:
            raise ValueError(kind)
        if row_spread:
            rows = int(np.prod(shape[:-1]))
            mag = 10.0 ** host_uniform((rows,), seed ^ 0x5A5A5A5A, -2.0, 2.0)
            v = (v.reshape(rows, shape[-1]) * mag[:, None]).reshape(shape)
        return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(TORCH_DTYPES[dtype])
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    if kind == "act":
        v = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    elif kind == "mod":
        v = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).mul_(0.1)
    elif kind == "gate":
        v = torch.rand(shape, generator=g, device=dev, dtype=torch.float32).mul_(2.0).sub_(1.0)
    else:
        raise ValueError(kind)
    if row_spread:
        rows = int(np.prod(shape[:-1]))
        e = torch.rand((rows, 1), generator=g, device=dev, dtype=torch.float32).mul_(4.0).sub_(2.0)
        v = (v.reshape(rows, shape[-1]) * torch.pow(10.0, e)).reshape(shape)
    return v.to(TORCH_DTYPES[dtype]).contiguous()


def vector_shape(B, L, D, layout):
    """[B, L, D] for a full operand, [B, 1, D] for a row-broadcast one."""
    return (B, L, D) if layout == "full" else (B, 1, D)


# --------------------------------------------------------------------------
# Named workloads (shapes and layouts; draw() makes the tensors).
# --------------------------------------------------------------------------

WORKLOADS = {
    # smallest: full gate, [1,126,2048] (launch-bound on every GPU)
    "ltx2_full_s126_c2048": dict(B=1, L=126, D=2048, gate="full", mod="bcast"),
    # broadcast mid shapes
    "flux2_bcast_s4608_c3072": dict(B=1, L=4608, D=3072, gate="bcast", mod="bcast"),
    "ideogram4_bcast_s4096_c4608": dict(B=1, L=4096, D=4608, gate="bcast", mod="bcast"),
    # ragged shapes: L odd; D = 3080 (8 | D), 3076 (4 | D, 8 does not), 3077 (odd)
    "tail_s4097_c3080": dict(B=1, L=4097, D=3080, gate="bcast", mod="bcast"),
    "tail_s4097_c3076": dict(B=1, L=4097, D=3076, gate="bcast", mod="bcast"),
    "tail_s4097_c3077": dict(B=1, L=4097, D=3077, gate="bcast", mod="bcast"),
    # full-gate large shape with row magnitude spread
    "ltx2_full_s8160_c4096": dict(B=1, L=8160, D=4096, gate="full", mod="full",
                                  row_spread=True),
    # largest broadcast shape (the roofline case)
    "ltx2_bcast_s32640_c4096": dict(B=1, L=32640, D=4096, gate="bcast", mod="bcast"),
    # the block chain: B=2, 8 blocks x 3 sites
    "ltx2_chain_b2_s32640_c4096": dict(B=2, L=32640, D=4096, gate="bcast",
                                       mod="bcast", blocks=8),
}

EPS = 1e-6  # the adaLN RMSNorm epsilon of the LTX-2 blocks
