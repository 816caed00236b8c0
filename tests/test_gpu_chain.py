"""The synthetic DiT block chain (8 blocks x 3 sites: 1 modulation, 23 fused
ops, 1 residual gate) on the GPU against the oracle's chain.

The residual stream x depends only on x, the stand-in updates and the gates,
and the residual gate is bit-exact, so x stays bit-exact through all 24
sites; every modulated input m is within the modulation criterion.

* full chain at B = 2, L = 32640, D = 4096 bf16, 48 sampled rows per batch,
  every site's m compared;
* a short chain (L = 64) compared on every row.
"""
import numpy as np
import pytest
import torch

from _cases import oracle_fused, oracle_mod, oracle_rga
from _gpu import assert_bit_exact, ensure_built, modulation_stats
from diffusion_transformer_elementwise_gb300 import chain
from diffusion_transformer_elementwise_gb300.synth import seed_for

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def oracle_chain(orc, x, updates, tables, dtype="bf16"):
    """The chain on CPU tensors with the oracle's ops; returns the list of m
    after each site (index 0: the first modulation) and the final x."""
    sites = chain.site_list(len(tables))
    x = x.clone()
    ms = []
    shift0, scale0, _ = tables[0][chain.SITES[0]]
    m, t = oracle_mod(orc, x, scale0, shift0, dtype, "bcast", EPS, with_t=True)
    ms.append((m, t))
    for j, (blk, k) in enumerate(sites):
        gate = tables[blk][chain.SITES[k]][2]
        u = updates[k]
        if j + 1 < len(sites):
            nb, nk = sites[j + 1]
            shift, scale, _ = tables[nb][chain.SITES[nk]]
            x, m, t = oracle_fused(orc, x, u, gate, scale, shift, dtype, "bcast", "bcast", EPS,
                                   with_t=True)
            ms.append((m, t))
        else:
            x = oracle_rga(orc, x, u, gate, dtype, "bcast")
    return ms, x


def _run(orc, B, L, D, rows):
    x, updates, tables = chain.make_inputs(B, L, D, 8, "bf16", "cuda", seed_tag=f"chain{L}")
    idx = rows.cuda()
    xs = x[:, idx, :].contiguous().cpu()
    us = [u[:, idx, :].contiguous().cpu() for u in updates]
    ts = [{s: tuple(v.cpu().contiguous() for v in tb[s]) for s in chain.SITES} for tb in tables]
    got = []

    def on_site(j, xd, md):
        if j + 1 < 24:  # the last site is a plain residual gate: m is unchanged
            got.append(md[:, idx, :].contiguous().cpu())

    chain.run(x, updates, tables, EPS, on_site=on_site)
    torch.cuda.synchronize()
    ms, xref = oracle_chain(orc, xs, us, ts)
    assert len(got) == len(ms) == 24
    assert_bit_exact(x[:, idx, :].contiguous().cpu(), xref, "final residual")
    worst = 0
    for j, (g, (m, t)) in enumerate(zip(got, ms)):
        st = modulation_stats(g, m, t.numpy(), "bf16", f"site {j}")
        worst = max(worst, st["max_ulp"])
    return worst


def test_chain_full_size_sampled(orc):
    B, L, D = 2, 32640, 4096
    rng = np.random.default_rng(seed_for("chainrows") & 0xFFFFFFFF)
    rows = torch.tensor(sorted({0, L - 1, *rng.choice(L, 46, replace=False).tolist()}))
    _run(orc, B, L, D, rows)


def test_chain_short_every_row(orc):
    B, L, D = 2, 64, 4096
    _run(orc, B, L, D, torch.arange(L))


def test_chain_graph_replay_equals_eager():
    """The chain captured in a CUDA graph and replayed twice gives, bit for
    bit, what two eager passes give (x is updated in place by each pass).
    Audio-stream shape [1, 126, 2048]: the launch-bound case a graph is for."""
    B, L, D = 1, 126, 2048
    xe, updates, tables = chain.make_inputs(B, L, D, 8, "bf16", "cuda", seed_tag="graph")
    xg = xe.clone()
    me = torch.empty_like(xe)
    for _ in range(2):
        chain.run(xe, updates, tables, EPS, m=me)
    graph, mg = chain.capture(xg, updates, tables, EPS)
    torch.cuda.synchronize()
    assert torch.equal(xg, chain.make_inputs(B, L, D, 8, "bf16", "cuda", seed_tag="graph")[0])
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(xg.view(torch.int16), xe.view(torch.int16))
    assert torch.equal(mg.view(torch.int16), me.view(torch.int16))


@pytest.mark.parametrize("graph", [False, True])
def test_video_audio_chain_grouped(orc, graph):
    """Video [1, 64, 4096] and audio [1, 126, 2048] streams through 8 blocks
    with one grouped launch per site: x bit-exact against the oracle's chain
    of each stream, the last m within the modulation criterion; and the
    grouped run equals the per-stream run on x bitwise."""
    shapes = [(1, 64, 4096), (1, 126, 2048)]
    streams = [chain.make_inputs(B, L, D, 8, "bf16", "cuda", seed_tag=f"av{i}")
               for i, (B, L, D) in enumerate(shapes)]
    ref_in = [(x.cpu(), [u.cpu() for u in us],
               [{s: tuple(v.cpu().contiguous() for v in tb[s]) for s in chain.SITES} for tb in ts])
              for x, us, ts in streams]
    sep = [(x.clone(), us, ts) for x, us, ts in streams]
    if graph:
        g, ms = chain.capture_streams(streams)
        g.replay()
        out = [(x, m) for (x, _, _), m in zip(streams, ms)]
    else:
        out = chain.run_streams(streams)
    chain.run_streams(sep, grouped=False)
    torch.cuda.synchronize()
    for i, ((x, m), (xs, us, ts), (x2, _, _)) in enumerate(zip(out, ref_in, sep)):
        ms_ref, x_ref = oracle_chain(orc, xs, us, ts)
        assert_bit_exact(x.cpu(), x_ref, f"stream {i} residual")
        assert torch.equal(x.view(torch.int16), x2.view(torch.int16))
        m_ref, t = ms_ref[-1]
        modulation_stats(m.cpu(), m_ref, t.numpy(), "bf16", f"stream {i} last m")
