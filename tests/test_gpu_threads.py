"""Entry points called from several host threads at once (each on its own
stream): the per-device caches (SM count, shared-memory limit, resident
CTAs, shared-memory opt-in) are filled concurrently on first use, and every
result must still match the oracle.  Shapes include rings above the 48 KB
default (full scale/shift at D = 8192), so the opt-in races too."""
import threading

import pytest
import torch

import diffusion_transformer_elementwise_gb300 as dit
from _cases import mod_inputs, oracle_fused, rga_inputs
from _gpu import assert_bit_exact, ensure_built, modulation_stats

pytestmark = pytest.mark.gpu
EPS = 1e-6
SHAPES = [(1, 33, 8192, "full", "full"), (2, 17, 4096, "bcast", "bcast"), (1, 9, 3077, "bcast", "full"),
          (1, 64, 2048, "full", "bcast")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def test_concurrent_host_threads(orc):
    cases = []
    for i, (B, L, D, gl, ml) in enumerate(SHAPES):
        h, u, g = rga_inputs(B, L, D, "bf16", gl, tag=f"thr{i}")
        _, sc, sh = mod_inputs(B, L, D, "bf16", ml, tag=f"thr{i}")
        cases.append(((h, u, g, sc, sh), gl, ml, oracle_fused(orc, h, u, g, sc, sh, "bf16", gl, ml,
                                                               EPS, with_t=True)))
    results, errors = [None] * len(cases), []
    start = threading.Barrier(len(cases))

    def work(i):
        try:
            (h, u, g, sc, sh), _, _, _ = cases[i]
            dev = [t.cuda() for t in (h, u, g, sc, sh)]
            stream = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(stream):
                for _ in range(20):
                    r, m = dit.gate_add_rmsnorm_modulate(*dev, EPS)
            stream.synchronize()
            results[i] = (r.cpu(), m.cpu())
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(cases))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (_, gl, ml, (res, mod, t)), (r, m) in zip(cases, results):
        assert_bit_exact(r, res, f"{gl}/{ml} residual")
        modulation_stats(m, mod, t.numpy(), "bf16", f"{gl}/{ml} modulated")
