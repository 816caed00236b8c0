"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times: the whole tensor runs on the GPU; the oracle recomputes a
sample of rows (first and last row of every batch plus seeded random rows),
and properties that hold at any size are checked on every element:

* residual gate: equals torch's own fp32 multiply then fp32 add, rounded to
  the dtype (two separately rounded eager kernels: the same arithmetic);
* modulation: scale = -1 gives exactly the shift everywhere;
* fused: the residual equals the residual gate, and the modulated output
  equals the modulation of that residual over the whole tensor -- bitwise
  under the exact statistic; under the fast one (whose sum order is the
  kernel's) within 2^-5 absolute, on fewer than 1% of the elements.

Shapes: sglang PR #29361, B200 kernel benchmark table (ltx2_bcast_s32640_c4096,
ltx2_full_s8160_c4096, ideogram4_bcast_s4096_c4608, flux2_bcast_s4608_c3072),
plus the ragged shapes L = 4097, D in {3076, 3077, 3080}.
"""
import numpy as np
import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import oracle_fused, oracle_mod, oracle_rga
from _gpu import assert_bit_exact, ensure_built, modulation_stats
from diffusion_transformer_elementwise_gb300.synth import draw, seed_for, vector_shape

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def sample_rows(L, k, tag):
    rng = np.random.default_rng(seed_for("rows", tag, L) & 0xFFFFFFFF)
    rest = rng.choice(np.arange(1, L - 1), size=min(k - 2, L - 2), replace=False)
    return torch.tensor(sorted({0, L - 1, *rest.tolist()}), dtype=torch.long)


def gather(t, idx, L):
    """Rows idx of every batch of a [B, L, D] tensor (a [B, 1, D] one is
    returned as is), as a contiguous CPU tensor."""
    if t.shape[1] == L and L != 1:
        return t[:, idx.to(t.device), :].contiguous().cpu()
    return t.contiguous().cpu()


def inputs(tag, B, L, D, dtype, gate_layout, mod_layout, row_spread=False):
    h = draw("act", (B, L, D), seed_for(tag, "h"), dtype, "cuda", row_spread=row_spread)
    u = draw("act", (B, L, D), seed_for(tag, "u"), dtype, "cuda")
    g = draw("gate", vector_shape(B, L, D, gate_layout), seed_for(tag, "g"), dtype, "cuda")
    sc = draw("mod", vector_shape(B, L, D, mod_layout), seed_for(tag, "sc"), dtype, "cuda")
    sh = draw("mod", vector_shape(B, L, D, mod_layout), seed_for(tag, "sh"), dtype, "cuda")
    return h, u, g, sc, sh


WORKLOADS = [
    # name, B, L, D, dtype, gate layout, mod layout, row spread
    ("ltx2_bcast_s32640_c4096", 1, 32640, 4096, "bf16", "bcast", "bcast", False),
    ("ltx2_full_s8160_c4096", 1, 8160, 4096, "bf16", "full", "full", True),
    ("ltx2_full_s8160_c4096_modbcast", 1, 8160, 4096, "bf16", "full", "bcast", True),
    ("ideogram4_bcast_s4096_c4608", 1, 4096, 4608, "bf16", "bcast", "bcast", False),
    ("flux2_bcast_s4608_c3072", 1, 4608, 3072, "bf16", "bcast", "bcast", False),
    ("flux2_bcast_s4608_c3072_fp16", 1, 4608, 3072, "fp16", "bcast", "bcast", False),
    ("flux2_bcast_s4608_c3072_fp32", 1, 4608, 3072, "fp32", "bcast", "bcast", False),
    ("ltx2_full_s126_c2048", 1, 126, 2048, "bf16", "full", "bcast", False),
] + [
    (f"tail_s4097_c{D}_{dt}", 1, 4097, D, dt, "bcast", "bcast", False)
    for D in (3080, 3076, 3077) for dt in ("bf16", "fp16", "fp32")
]


@pytest.mark.parametrize("w", WORKLOADS, ids=[w[0] for w in WORKLOADS])
def test_workload(orc, statistic, w):
    name, B, L, D, dtype, gl, ml, spread = w
    h, u, g, sc, sh = inputs(name, B, L, D, dtype, gl, ml, spread)
    idx = sample_rows(L, 48, name)
    k = len(idx)
    hs, us, gs, scs, shs = (gather(t, idx, L) for t in (h, u, g, sc, sh))

    # residual gate: sampled rows vs the oracle, every element vs torch eager fp32
    out = dit.residual_gate_add(h, u, g)
    torch.cuda.synchronize()
    assert_bit_exact(gather(out, idx, L), oracle_rga(orc, hs, us, gs, dtype, gl), name)
    eager = (h.float() + u.float() * g.float()).to(h.dtype)
    assert torch.equal(out.view(torch.int16 if out.element_size() == 2 else torch.int32),
                       eager.view(torch.int16 if out.element_size() == 2 else torch.int32))
    del eager

    # modulation of hidden: sampled rows vs the oracle
    m = dit.rmsnorm_modulate(h, sc, sh, EPS)
    torch.cuda.synchronize()
    mref, t = oracle_mod(orc, hs, scs, shs, dtype, ml, EPS, with_t=True)
    stats = modulation_stats(gather(m, idx, L), mref, t.numpy(), dtype, name)
    print(name, "modulation", stats)
    # scale = -1 gives the shift, over the whole tensor
    neg = dit.rmsnorm_modulate(h, torch.full_like(sc, -1.0), sh, EPS)
    torch.cuda.synchronize()
    assert torch.equal(neg, sh.expand(B, L, D))
    del neg

    # fused, and its consistency with the two single ops over every element
    res, mod = dit.gate_add_rmsnorm_modulate(h, u, g, sc, sh, EPS)
    torch.cuda.synchronize()
    assert torch.equal(res, out)
    m2 = dit.rmsnorm_modulate(res, sc, sh, EPS)
    torch.cuda.synchronize()
    if statistic == "exact":
        # one correctly rounded statistic: every kernel gives the same bits
        assert torch.equal(mod, m2)
    else:
        # the fast statistic's sum order is the kernel's (the fused op and the
        # modulation may take different kernels): the last bit may differ
        d = (mod.float() - m2.float()).abs()
        assert float(d.max()) <= 2.0 ** -5, float(d.max())
        assert int((d > 0).sum()) <= mod.numel() // 100
    rref, mref2, t2 = oracle_fused(orc, hs, us, gs, scs, shs, dtype, gl, ml, EPS, with_t=True)
    assert_bit_exact(gather(res, idx, L), rref)
    print(name, "fused", modulation_stats(gather(mod, idx, L), mref2, t2.numpy(), dtype, name))
    assert k >= 2


def test_in_place_largest_broadcast(orc):
    """The in-place variant on [1, 32640, 4096] bf16 (out = hidden)."""
    B, L, D = 1, 32640, 4096
    h, u, g, _, _ = inputs("inplace32640", B, L, D, "bf16", "bcast", "bcast")
    idx = sample_rows(L, 48, "inplace32640")
    hs, us, gs = gather(h, idx, L), gather(u, idx, L), gather(g, idx, L)
    ref_full = dit.residual_gate_add(h, u, g)
    dit.residual_gate_add(h, u, g, out=h)
    torch.cuda.synchronize()
    assert torch.equal(h, ref_full)
    assert_bit_exact(gather(h, idx, L), oracle_rga(orc, hs, us, gs, "bf16", "bcast"))
