"""A synthetic DiT block chain over the three ops: the residual stream of
LTX-2-style transformer blocks with the attention and MLP replaced by
stand-in updates.

Each block carries an adaLN table of nine [B, 1, D] vectors: (shift, scale,
gate) for each of its three sites -- self-attention, prompt cross-attention,
feed-forward (prhub summary of sglang PR #34172, "implementation breakdown"
item 3: the adaLN modulation sites of LTX2TransformerBlock.forward).  The
sites run in the order sa -> ca -> ff -> next block's sa.  With x the
residual stream:

    m = rmsnorm_modulate(x; scale, shift of site 0)
    for each site j:
        u = stand-in update of site j's kind (independent of m)
        if j is not the last site:
            x, m = gate_add_rmsnorm_modulate(x, u, gate_j; scale, shift of site j+1)
        else:
            x = residual_gate_add(x, u, gate_j)

so 8 blocks = 24 sites = 1 modulation + 23 fused + 1 residual gate.  x is
updated in place.  The chain moves (2 + 23 * 4 + 3) * N * s bytes of
activations (N = B * L * D elements of s bytes) plus the small vectors.
"""
from __future__ import annotations

from ._binding import (
    gate_add_rmsnorm_modulate,
    gate_add_rmsnorm_modulate_grouped,
    residual_gate_add,
    residual_gate_add_grouped,
    rmsnorm_modulate,
    rmsnorm_modulate_grouped,
)
from .synth import draw, seed_for

SITES = ("sa", "ca", "ff")


PARTS = ("shift", "scale", "gate")


def make_inputs(B, L, D, blocks=8, dtype="bf16", device="cuda", seed_tag="chain"):
    """x [B, L, D], one stand-in update per site kind, and per block an adaLN
    table [B, 9, D] (shift, scale, gate of sa, ca, ff), all seeded.  Returns
    (x, updates, tables) where tables[blk][site] = (shift, scale, gate) are
    [B, 1, D] views into the block's table (batch stride 9 * D)."""
    x = draw("act", (B, L, D), seed_for(seed_tag, "x", B, L, D), dtype, device)
    updates = [draw("act", (B, L, D), seed_for(seed_tag, "u", k, B, L, D), dtype, device)
               for k in range(len(SITES))]
    tables = []
    for blk in range(blocks):
        table = draw("mod", (B, 3 * len(SITES), D), seed_for(seed_tag, "table", blk, B, D),
                     dtype, device)
        t = {}
        for k, site in enumerate(SITES):
            t[site] = tuple(table[:, 3 * k + i:3 * k + i + 1, :] for i in range(len(PARTS)))
        tables.append(t)
    return x, updates, tables


def site_list(blocks):
    return [(b, k) for b in range(blocks) for k in range(len(SITES))]


def run(x, updates, tables, eps=1e-6, m=None, on_site=None, stream=None):
    """Run the chain on the GPU through the C ABI.  x is updated in place;
    m (allocated if None) holds the last modulated input.  on_site(j, x, m)
    is called after site j's op is enqueued (j = -1 after the first
    modulation).  Returns (x, m)."""
    import torch
    sites = site_list(len(tables))
    if m is None:
        m = torch.empty_like(x)
    shift0, scale0, _ = tables[0][SITES[0]]
    rmsnorm_modulate(x, scale0, shift0, eps, out=m, stream=stream)
    if on_site:
        on_site(-1, x, m)
    for j, (blk, k) in enumerate(sites):
        gate = tables[blk][SITES[k]][2]
        u = updates[k]
        if j + 1 < len(sites):
            nb, nk = sites[j + 1]
            shift, scale, _ = tables[nb][SITES[nk]]
            gate_add_rmsnorm_modulate(x, u, gate, scale, shift, eps, residual_out=x,
                                      modulated_out=m, stream=stream)
        else:
            residual_gate_add(x, u, gate, out=x, stream=stream)
        if on_site:
            on_site(j, x, m)
    return x, m


def capture(x, updates, tables, eps=1e-6, m=None):
    """Record one pass of the chain (1 + 3 * blocks launches on x, m and the
    tables' buffers) in a CUDA graph.  Replaying the graph runs the same
    kernels on the same buffers -- x is updated in place on every replay --
    with no host work per launch.  Capturing runs nothing.  Returns (graph, m)."""
    import torch
    if m is None:
        m = torch.empty_like(x)
    side = torch.cuda.Stream(device=x.device)
    side.wait_stream(torch.cuda.current_stream(x.device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run(x, updates, tables, eps, m=m)
    torch.cuda.current_stream(x.device).wait_stream(side)
    return graph, m


def run_streams(streams, eps=1e-6, ms=None, grouped=True, stream=None):
    """The chain over several streams at once -- the video and audio streams
    of LTX-2 blocks, whose six adaLN sites each modulate both (prhub summary
    of sglang PR #34172, "implementation breakdown" item 3).  streams: a list
    of (x, updates, tables) as make_inputs returns, with the same number of
    blocks.  grouped=True: one grouped launch per site for all streams
    (1 + 3 * blocks launches); False: one launch per stream and site.
    Each x is updated in place; returns the list of (x, m)."""
    import torch
    blocks = len(streams[0][2])
    sites = site_list(blocks)
    if ms is None:
        ms = [torch.empty_like(x) for x, _, _ in streams]

    def vectors(tables, blk, k):
        return tables[blk][SITES[k]]

    first = []
    for (x, _, tables), m in zip(streams, ms):
        shift, scale, _ = vectors(tables, 0, 0)
        first.append((x, scale, shift, m))
    if grouped:
        rmsnorm_modulate_grouped(first, eps, stream=stream)
    else:
        for x, scale, shift, m in first:
            rmsnorm_modulate(x, scale, shift, eps, out=m, stream=stream)
    for j, (blk, k) in enumerate(sites):
        last = j + 1 == len(sites)
        calls = []
        for (x, updates, tables), m in zip(streams, ms):
            gate = vectors(tables, blk, k)[2]
            if last:
                calls.append((x, updates[k], gate, x))
            else:
                nb, nk = sites[j + 1]
                shift, scale, _ = vectors(tables, nb, nk)
                calls.append((x, updates[k], gate, scale, shift, x, m))
        if grouped:
            if last:
                residual_gate_add_grouped(calls, stream=stream)
            else:
                gate_add_rmsnorm_modulate_grouped(calls, eps, stream=stream)
        else:
            for c in calls:
                if last:
                    residual_gate_add(c[0], c[1], c[2], out=c[3], stream=stream)
                else:
                    gate_add_rmsnorm_modulate(c[0], c[1], c[2], c[3], c[4], eps, residual_out=c[5],
                                              modulated_out=c[6], stream=stream)
    return [(x, m) for (x, _, _), m in zip(streams, ms)]


def capture_streams(streams, eps=1e-6, ms=None, grouped=True):
    """run_streams recorded in a CUDA graph (nothing runs while capturing).
    Returns (graph, ms)."""
    import torch
    x0 = streams[0][0]
    if ms is None:
        ms = [torch.empty_like(x) for x, _, _ in streams]
    side = torch.cuda.Stream(device=x0.device)
    side.wait_stream(torch.cuda.current_stream(x0.device))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        run_streams(streams, eps, ms=ms, grouped=grouped)
    torch.cuda.current_stream(x0.device).wait_stream(side)
    return graph, ms


def launches(blocks: int) -> int:
    return 1 + 3 * blocks


def algorithmic_bytes(B, L, D, blocks, es):
    """Bytes the chain must move: the first modulation reads x and writes m,
    each fused site reads x and u and writes x and m, the last residual gate
    reads x and u and writes x; each op's [B, 1, D] vectors counted once."""
    n = B * L * D * es
    v = B * D * es
    sites = 3 * blocks
    first = 2 * n + 2 * v
    fused = (sites - 1) * (4 * n + 3 * v)
    last = 3 * n + v
    return first + fused + last
