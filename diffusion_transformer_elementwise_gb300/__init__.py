"""GB300 (sm_103a) kernels for the memory-bound elementwise hot path of
LTX-2-style video diffusion transformers.

* :func:`residual_gate_add` -- ``hidden + update * gate`` (full or [B, 1, D] gate)
* :func:`rmsnorm_modulate` -- ``rms_norm(x, eps) * (1 + scale) + shift``
* :func:`gate_add_rmsnorm_modulate` -- both in one pass
* :func:`rmsnorm_modulate_fp8`, :func:`gate_add_rmsnorm_modulate_fp8` -- the
  modulated output quantised to FP8 (OCP E4M3) with a per-tensor scale
* :func:`gelu_tanh` -- the feed-forward's tanh-GELU
* ``*_grouped`` -- the first three over several problems (e.g. the video and
  audio streams of a block) in one launch
* :func:`selfcheck` / :func:`ensure_checked` -- bit-for-bit check of one
  runtime key (op, dtype, layouts, D) on the GPU
* :func:`set_statistic` / :func:`statistic` -- the modulation's row
  statistic: "fast" (default) or "exact" (correctly rounded, bit-exact)

Each call is one kernel of ``libdit_elementwise.so`` (C ABI in
``include/dit_elementwise.h``), launched on the current torch stream.  Build
the library with :func:`build`; without it every call raises.
"""
from ._binding import (  # noqa: F401
    DitError,
    ensure_checked,
    gate_add_rmsnorm_modulate,
    gate_add_rmsnorm_modulate_fp8,
    gate_add_rmsnorm_modulate_grouped,
    gelu_tanh,
    library,
    residual_gate_add,
    residual_gate_add_grouped,
    rmsnorm_modulate,
    rmsnorm_modulate_fp8,
    rmsnorm_modulate_grouped,
    get_statistic,
    selfcheck,
    set_first_use_check,
    set_statistic,
    statistic,
)
from .build import build  # noqa: F401
