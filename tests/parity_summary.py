"""Per-workload parity summary of the modulating operations (run on a GPU).

For every workload of the benchmark's recipe -- the shapes of sglang PR
#29361's B200 kernel benchmark table, the ragged L = 4097 rows, the
[1,8160,4096] full-gate shape with per-token or broadcast modulation, and the
8-block DiT chain at [2,32640,4096] -- and under each row statistic ("fast",
the default, and "exact"), the modulation and the fused op run over the
whole tensor on the GPU and the oracle recomputes sampled rows.  Printed per
(workload, op, statistic), as a Markdown table: elements compared, elements
not bit-exact, the largest distance in dtype ulps, the elements admitted only
by the cancellation rule (the fast statistic's criterion: within one dtype
ulp of max(|t|, |y|)), the largest |gpu - oracle| / max(|t|, |y|) in units
of u = 2^-24 (the measure of the fp32 criterion, whose bound 2^-18 is 64 u;
ulp counts mean little for fp32 values near zero), max |gpu - oracle| and
the relative L2 error.  Every
comparison also asserts its statistic's criterion (tests/_gpu.py).

    python tests/parity_summary.py [--rows N] [--out FILE]
"""
import argparse
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import diffusion_transformer_elementwise_gb300 as dit  # noqa: E402
import oracle  # noqa: E402
from _cases import oracle_fused, oracle_mod  # noqa: E402
from _gpu import modulation_stats  # noqa: E402
from diffusion_transformer_elementwise_gb300 import chain  # noqa: E402
from diffusion_transformer_elementwise_gb300.synth import seed_for  # noqa: E402
from test_gpu_fullsize import WORKLOADS, gather, inputs, sample_rows  # noqa: E402

EPS = 1e-6


def workload_rows(orc, w, nrows):
    name, B, L, D, dtype, gl, ml, spread = w
    h, u, g, sc, sh = inputs(name, B, L, D, dtype, gl, ml, spread)
    idx = sample_rows(L, nrows, name)
    hs, us, gs, scs, shs = (gather(t, idx, L) for t in (h, u, g, sc, sh))
    out = []
    m = dit.rmsnorm_modulate(h, sc, sh, EPS)
    torch.cuda.synchronize()
    mref, t = oracle_mod(orc, hs, scs, shs, dtype, ml, EPS, with_t=True, threads=8)
    out.append(("modulate_" + ml, modulation_stats(gather(m, idx, L), mref, t.numpy(), dtype,
                                                   name)))
    del m
    res, mod = dit.gate_add_rmsnorm_modulate(h, u, g, sc, sh, EPS)
    torch.cuda.synchronize()
    _, mref2, t2 = oracle_fused(orc, hs, us, gs, scs, shs, dtype, gl, ml, EPS, with_t=True,
                                threads=8)
    out.append((f"fused_{gl}_{ml}", modulation_stats(gather(mod, idx, L), mref2, t2.numpy(),
                                                     dtype, name)))
    return out


def chain_rows(orc, nrows):
    """Every site's modulated input of the 8-block chain on sampled rows."""
    from test_gpu_chain import oracle_chain
    B, L, D = 2, 32640, 4096
    x, updates, tables = chain.make_inputs(B, L, D, 8, "bf16", "cuda", seed_tag=f"chain{L}")
    rng = np.random.default_rng(seed_for("chainrows") & 0xFFFFFFFF)
    idx = torch.tensor(sorted({0, L - 1, *rng.choice(L, nrows - 2, replace=False).tolist()}))
    d = idx.cuda()
    xs = x[:, d, :].contiguous().cpu()
    us = [v[:, d, :].contiguous().cpu() for v in updates]
    ts = [{s: tuple(v.cpu().contiguous() for v in tb[s]) for s in chain.SITES} for tb in tables]
    got = []

    def on_site(j, xd, md):
        if j + 1 < 24:
            got.append(md[:, d, :].contiguous().cpu())

    chain.run(x, updates, tables, EPS, on_site=on_site)
    torch.cuda.synchronize()
    ms, _ = oracle_chain(orc, xs, us, ts)
    total = {"max_ulp": 0, "not_bit_exact": 0, "fallback": 0, "max_abs": 0.0, "n": 0,
             "rel_l2_max": 0.0, "max_err_u": 0.0}
    for j, (g, (m, t)) in enumerate(zip(got, ms)):
        st = modulation_stats(g, m, t.numpy(), "bf16", f"site {j}")
        total["max_ulp"] = max(total["max_ulp"], st["max_ulp"])
        total["not_bit_exact"] += st["not_bit_exact"]
        total["fallback"] += st["fallback"]
        total["max_abs"] = max(total["max_abs"], st["max_abs"])
        total["max_err_u"] = max(total["max_err_u"], st["max_err_u"])
        total["rel_l2_max"] = max(total["rel_l2_max"], st["rel_l2"])
        total["n"] += st["n"]
    total["rel_l2"] = total.pop("rel_l2_max")
    return [("chain: 24 modulated inputs", total)]


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--rows", type=int, default=512, help="sampled rows per workload")
    p.add_argument("--out", default=None, help="also write the table to this file")
    args = p.parse_args()
    dit.build()
    oracle.build()
    torch.cuda.set_device(0)
    lines = ["| workload | op | dtype | statistic | elements | not bit-exact | max ulp | "
             "cancellation rule | max err / max(\\|t\\|,\\|y\\|) (u) | max abs | rel L2 |",
             "|---|---|---|---|---|---|---|---|---|---|---|"]
    for stat in ("fast", "exact"):
        with dit.statistic(stat):
            jobs = [(w[0], w[4], lambda w=w: workload_rows(oracle, w, args.rows))
                    for w in WORKLOADS]
            jobs.append(("chain_b2_s32640_c4096", "bf16", lambda: chain_rows(oracle, 64)))
            for name, dtype, job in jobs:
                for op, st in job():
                    lines.append(f"| {name} | {op} | {dtype} | {stat} | {st['n']} | "
                                 f"{st['not_bit_exact']} | {st['max_ulp']} | {st['fallback']} | "
                                 f"{st['max_err_u']:.2f} | {st['max_abs']:.3g} | "
                                 f"{st['rel_l2']:.3g} |")
                    print(lines[-1], flush=True)
    if args.out:
        with open(args.out, "w") as f:
            f.write("\n".join(lines) + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
