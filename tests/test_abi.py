"""The C ABI without a GPU: the library loads, exports every function that
include/dit_elementwise.h declares, and rejects bad arguments with the
documented status before touching the device.  Pointers here are plain
integers that are never dereferenced: validation happens on the host."""
import ctypes
import os
import re

import pytest

from diffusion_transformer_elementwise_gb300 import library
from diffusion_transformer_elementwise_gb300.build import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "dit_elementwise.h")

(OK, NULLP, SHAPE, DTYPE, LAYOUT, ALIAS, EPS, LAUNCH, MISALIGNED, NODEV, BADOP, WORKSPACE,
 BADSTAT) = range(13)
BF16, FP16, FP32 = 0, 1, 2
FULL, BCAST = 0, 1


@pytest.fixture(scope="module")
def lib():
    build()
    return library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dit_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"dit_residual_gate_add", "dit_rmsnorm_modulate",
            "dit_gate_add_rmsnorm_modulate", "dit_status_string",
            "dit_abi_version"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_status_strings(lib):
    m = re.search(r"#define DIT_ABI_VERSION (\d+)", open(HEADER).read())
    assert lib.dit_abi_version() == int(m.group(1))
    seen = set()
    for code in range(13):
        s = lib.dit_status_string(code).decode()
        assert s.startswith("DIT_") and s not in seen
        seen.add(s)
    assert lib.dit_status_string(99).decode() == "unknown dit_status"


A = 1 << 20  # fake, well-separated, 256-byte aligned "device" addresses
H, U, G, O, O2, S, SH = (A * k for k in range(1, 8))


def rga(lib, out=O, h=H, u=U, g=G, B=1, L=4, D=8, dt=BF16, lay=FULL):
    return lib.dit_residual_gate_add(out, h, u, g, B, L, D, dt, lay, None)


def mod(lib, out=O, x=H, s=S, sh=SH, B=1, L=4, D=8, eps=1e-6, dt=BF16, lay=BCAST):
    return lib.dit_rmsnorm_modulate(out, x, s, sh, B, L, D, eps, dt, lay, None)


def fused(lib, r=O, m=O2, h=H, u=U, g=G, s=S, sh=SH, B=1, L=4, D=8, eps=1e-6, dt=BF16,
          gl=BCAST, ml=BCAST):
    return lib.dit_gate_add_rmsnorm_modulate(r, m, h, u, g, s, sh, B, L, D, eps, dt, gl, ml,
                                             None)


def test_bad_dtype_layout_shape(lib):
    assert rga(lib, dt=3) == DTYPE
    assert rga(lib, lay=2) == LAYOUT
    assert mod(lib, lay=-1) == LAYOUT
    assert fused(lib, ml=7) == LAYOUT
    assert rga(lib, D=-1) == SHAPE
    assert mod(lib, B=-2) == SHAPE
    assert fused(lib, B=1 << 40, L=1 << 40, D=4) == SHAPE  # overflows int64
    assert rga(lib, B=1 << 31, L=1 << 31, D=1 << 2, dt=FP32) == SHAPE  # bytes overflow


def test_bad_eps(lib):
    for eps in (-1e-6, float("inf"), float("nan")):
        assert mod(lib, eps=eps) == EPS
        assert fused(lib, eps=eps) == EPS
    assert mod(lib, eps=0.0) != EPS


def test_empty_problems_need_no_pointers_and_no_device(lib):
    assert rga(lib, out=None, h=None, u=None, g=None, L=0) == OK
    assert mod(lib, out=None, x=None, s=None, sh=None, D=0) == OK
    assert fused(lib, r=None, m=None, h=None, u=None, g=None, s=None, sh=None, B=0) == OK


def test_null_pointers(lib):
    assert rga(lib, g=None) == NULLP
    assert mod(lib, sh=None) == NULLP
    assert fused(lib, m=None) == NULLP


def test_misaligned(lib):
    assert rga(lib, u=U + 1) == MISALIGNED
    assert mod(lib, x=H + 2, dt=FP32) == MISALIGNED
    assert fused(lib, sh=SH + 3) == MISALIGNED
    # 2-byte aligned bf16 pointers are accepted (they pass validation and only
    # then fail for want of a device here)
    assert rga(lib, u=U + 2) in (NODEV, LAUNCH, OK)


def test_aliasing_rules(lib):
    n = 1 * 4 * 8 * 2
    assert rga(lib, out=H) in (NODEV, LAUNCH, OK)         # in place: allowed
    assert rga(lib, out=H + 2) == ALIAS                   # partial overlap with hidden
    assert rga(lib, out=U + n - 2) == ALIAS               # overlaps update's last element
    assert rga(lib, out=U + n) not in (ALIAS,)            # adjacent, no overlap
    assert rga(lib, out=G, lay=BCAST) == ALIAS
    assert mod(lib, out=H) == ALIAS                       # modulation is not in place
    assert mod(lib, out=S + 8) == ALIAS                   # inside the [1,1,8] scale
    assert fused(lib, r=H) in (NODEV, LAUNCH, OK)         # residual in place: allowed
    assert fused(lib, m=H) == ALIAS
    assert fused(lib, r=O, m=O) == ALIAS
    assert fused(lib, r=S) == ALIAS
    assert fused(lib, m=G + 4) == ALIAS


def test_valid_call_without_device_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert rga(lib) == NODEV
    assert mod(lib) == NODEV
    assert fused(lib) == NODEV


def test_strided_vectors_validation(lib):
    """vec_stride: >= D when B > 1; the strided span counts for aliasing."""
    f = lib.dit_gate_add_rmsnorm_modulate_strided
    B, L, D = 2, 4, 8
    args = lambda r=O, m=O2, g=G, vs=9 * D: (r, m, H, U, g, S, SH, B, L, D, 1e-6, BF16, BCAST,
                                              BCAST, vs, None)
    assert f(*args(vs=D - 1)) == SHAPE
    assert f(*args(vs=D)) in (NODEV, LAUNCH, OK)
    assert f(*args(vs=9 * D)) in (NODEV, LAUNCH, OK)
    # an output inside the gap of a strided operand's span is an alias
    assert f(*args(r=G + 2 * D * 2)) == ALIAS
    assert lib.dit_rmsnorm_modulate_strided(O, H, S, SH, B, L, D, 1e-6, BF16, BCAST, 3, None) == SHAPE
    assert lib.dit_residual_gate_add_strided(O, H, U, G, 1, L, D, BF16, BCAST, 0, None) in (NODEV, LAUNCH, OK)
    # full layouts ignore the stride
    assert lib.dit_residual_gate_add_strided(O, H, U, G, B, L, D, BF16, FULL, 0, None) in (NODEV, LAUNCH, OK)


def test_gelu_validation(lib):
    f = lib.dit_gelu_tanh
    assert f(O, H, -1, BF16, None) == SHAPE
    assert f(O, H, 10, 5, None) == DTYPE
    assert f(None, None, 0, BF16, None) == OK
    assert f(None, H, 10, BF16, None) == NULLP
    assert f(O + 1, H, 10, BF16, None) == MISALIGNED
    assert f(H + 4, H, 10, BF16, None) == ALIAS          # partial overlap
    assert f(H, H, 10, BF16, None) in (NODEV, LAUNCH, OK)  # in place


def test_grouped_validation(lib):
    from diffusion_transformer_elementwise_gb300._binding import Problem
    f = lib.dit_grouped
    RGA, MOD, FUSED = 0, 1, 2

    def probs(*ps):
        return (Problem * max(1, len(ps)))(*ps)

    n4, n2 = 4 * 8 * 2, 3 * 4 * 2  # bytes of [1,4,8] and [1,3,4] bf16
    video = Problem(O, O2, H, U, G, S, SH, 1, 4, 8, 8)
    audio = Problem(O + 4096, O2 + 4096, H + 4096, U + 4096, G + 4096, S + 4096, SH + 4096,
                    1, 3, 4, 4)
    assert f(3, probs(video), 1, 1e-6, BF16, BCAST, BCAST, None) == BADOP
    assert f(-1, probs(video), 1, 1e-6, BF16, BCAST, BCAST, None) == BADOP
    assert f(RGA, probs(video), 9, 1e-6, BF16, BCAST, BCAST, None) == BADOP
    assert f(RGA, probs(video), -1, 1e-6, BF16, BCAST, BCAST, None) == BADOP
    assert f(RGA, None, 2, 1e-6, BF16, BCAST, BCAST, None) == NULLP
    assert f(RGA, None, 0, 1e-6, BF16, BCAST, BCAST, None) == OK
    assert f(FUSED, probs(video, audio), 2, -1.0, BF16, BCAST, BCAST, None) == EPS
    assert f(FUSED, probs(video, audio), 2, 1e-6, 7, BCAST, BCAST, None) == DTYPE
    assert f(FUSED, probs(video, audio), 2, 1e-6, BF16, 5, BCAST, None) == LAYOUT
    # the single-call checks, per problem: the first failing problem's status
    bad = Problem(O, O2, H, U, G, S, SH, 1, -4, 8, 8)
    assert f(FUSED, probs(video, bad), 2, 1e-6, BF16, BCAST, BCAST, None) == SHAPE
    assert f(FUSED, probs(Problem(O, None, H, U, G, S, SH, 1, 4, 8, 8)), 1, 1e-6, BF16,
             BCAST, BCAST, None) == NULLP
    assert f(RGA, probs(Problem(O, None, H, U, G, None, None, 1, 4, 8, 8)), 1, 1e-6, BF16,
             BCAST, BCAST, None) in (NODEV, LAUNCH, OK)  # out2, scale, shift unused
    # across problems: no output may overlap another problem's tensors
    clash = Problem(H + 2, O2 + 4096, H + 4096, U + 4096, G + 4096, S + 4096, SH + 4096,
                    1, 3, 4, 4)  # writes into video's hidden
    assert f(FUSED, probs(video, clash), 2, 1e-6, BF16, BCAST, BCAST, None) == ALIAS
    clash2 = Problem(O + 4096, O2 + 8, H + 4096, U + 4096, G + 4096, S + 4096, SH + 4096,
                     1, 3, 4, 4)  # its modulated output inside video's
    assert f(FUSED, probs(video, clash2), 2, 1e-6, BF16, BCAST, BCAST, None) == ALIAS
    # reading the same tensor from two problems is fine (e.g. a shared gate)
    share = Problem(O + 4096, O2 + 4096, H + 4096, U + 4096, G, S, SH, 1, 3, 4, 4)
    assert f(FUSED, probs(video, share), 2, 1e-6, BF16, BCAST, BCAST, None) in (NODEV, LAUNCH, OK)
    # empty problems need no pointers
    empty = Problem(None, None, None, None, None, None, None, 0, 3, 4, 4)
    assert f(MOD, probs(empty, empty), 2, 1e-6, BF16, BCAST, BCAST, None) == OK
    import torch
    if not torch.cuda.is_available():
        assert f(FUSED, probs(video, audio), 2, 1e-6, BF16, BCAST, BCAST, None) == NODEV


def test_selfcheck_validation(lib):
    f, wb = lib.dit_selfcheck, lib.dit_selfcheck_workspace_bytes
    RGA, MOD, FUSED = 0, 1, 2
    # nine tensors of 14 * D elements rounded up to 256 bytes, then 256 bytes
    assert wb(RGA, BF16, 4096) == 9 * 14 * 4096 * 2 + 256
    assert wb(FUSED, FP32, 3) == 9 * 256 + 256
    assert wb(MOD, FP16, 3077) == 9 * ((14 * 3077 * 2 + 255) // 256 * 256) + 256
    assert wb(3, BF16, 64) == -1 and wb(MOD, 9, 64) == -1 and wb(MOD, BF16, 0) == -1
    assert wb(MOD, BF16, 1 << 60) == -1
    W, CNT = A * 64, A * 1024
    n = wb(FUSED, BF16, 64)
    assert f(7, BF16, BCAST, BCAST, 64, W, n, CNT, None) == BADOP
    assert f(FUSED, 5, BCAST, BCAST, 64, W, n, CNT, None) == DTYPE
    assert f(FUSED, BF16, 2, BCAST, 64, W, n, CNT, None) == LAYOUT
    assert f(FUSED, BF16, BCAST, BCAST, 0, W, n, CNT, None) == SHAPE
    assert f(FUSED, BF16, BCAST, BCAST, -5, W, n, CNT, None) == SHAPE
    assert f(FUSED, BF16, BCAST, BCAST, 64, W, n, None, None) == NULLP
    assert f(FUSED, BF16, BCAST, BCAST, 64, W, n, CNT + 2, None) == MISALIGNED
    assert f(FUSED, BF16, BCAST, BCAST, 64, None, n, CNT, None) == WORKSPACE
    assert f(FUSED, BF16, BCAST, BCAST, 64, W + 16, n, CNT, None) == WORKSPACE
    assert f(FUSED, BF16, BCAST, BCAST, 64, W, n - 1, CNT, None) == WORKSPACE
    assert f(FUSED, BF16, BCAST, BCAST, 64, W, n, W + 512, None) == ALIAS
    import torch
    if not torch.cuda.is_available():
        assert f(FUSED, BF16, BCAST, BCAST, 64, W, n, CNT, None) == NODEV


def test_fp8_validation(lib):
    """E4M3-output calls: the staged kernel's rules (16-byte aligned inputs and
    rows, output aligned to its per-granule store, rows of at most 16 KB),
    the quantisation scale as a device pointer, and one byte per output
    element in the aliasing checks."""
    f, g = lib.dit_rmsnorm_modulate_fp8, lib.dit_gate_add_rmsnorm_modulate_fp8
    Q = A * 9
    B, L, D = 1, 4, 64

    def mod8(out=O, x=H, s=S, sh=SH, D=D, dt=BF16, lay=BCAST, vs=None, q=Q, eps=1e-6):
        return f(out, x, s, sh, B, L, D, eps, dt, lay, D if vs is None else vs, q, None)

    def fused8(r=O2, out=O, h=H, u=U, gt=G, s=S, sh=SH, D=D, dt=BF16, q=Q):
        return g(r, out, h, u, gt, s, sh, B, L, D, 1e-6, dt, BCAST, BCAST, D, q, None)

    ok = (NODEV, LAUNCH, OK)
    assert mod8() in ok and fused8() in ok
    assert mod8(q=None) == NULLP and fused8(q=None) == NULLP
    assert mod8(q=Q + 2) == MISALIGNED
    assert mod8(x=H + 2) == MISALIGNED           # element-aligned, not 16-byte aligned
    assert fused8(r=O2 + 8) == MISALIGNED
    assert mod8(D=60) == MISALIGNED              # rows of 120 bytes
    assert mod8(D=60, dt=FP32) in ok             # 240 bytes = 15 * 16
    assert mod8(D=62, dt=FP32) == MISALIGNED     # 248 bytes
    assert mod8(out=O + 8) in ok                 # 8-byte aligned E4M3 output for 16-bit input
    assert mod8(out=O + 4) == MISALIGNED
    assert mod8(out=O + 4, dt=FP32) in ok        # 4-byte stores for fp32 input
    assert mod8(D=8192) in ok and mod8(D=8200) == SHAPE
    assert mod8(D=4096, dt=FP32) in ok and mod8(D=4104, dt=FP32) == SHAPE
    assert mod8(eps=-1.0) == EPS
    assert mod8(out=H + B * L * D * 2 - 16) == ALIAS   # inside x
    assert mod8(out=Q - 32) == ALIAS                    # covers the scale word
    assert mod8(out=H - B * L * D) in ok                # ends right where x begins
    assert fused8(out=O2 + 64) == ALIAS                 # inside the residual
    assert fused8(r=H) in ok                            # residual in place
    assert f(None, None, None, None, 0, L, D, 1e-6, BF16, BCAST, D, None, None) == OK


def test_statistic_mode(lib):
    """dit_set_statistic / dit_get_statistic: fast (0) by default, exact (1)
    on request, anything else rejected with the mode left as it was."""
    import diffusion_transformer_elementwise_gb300 as dit
    assert lib.dit_get_statistic() == 0
    assert lib.dit_set_statistic(1) == OK and lib.dit_get_statistic() == 1
    assert lib.dit_set_statistic(2) == BADSTAT and lib.dit_get_statistic() == 1
    assert lib.dit_set_statistic(-1) == BADSTAT
    assert lib.dit_set_statistic(0) == OK and lib.dit_get_statistic() == 0
    with dit.statistic("exact"):
        assert dit.get_statistic() == "exact"
    assert dit.get_statistic() == "fast"
    with pytest.raises(ValueError):
        dit.set_statistic("approximate")


def test_modulating_row_limit(lib):
    """Rows longer than 2^24 elements are rejected by the modulating ops."""
    G1 = 1 << 30
    D = (1 << 24) + 1
    assert mod(lib, out=G1, x=2 * G1, s=3 * G1, sh=4 * G1, D=D, L=1) == SHAPE
    assert fused(lib, r=G1, m=2 * G1, h=3 * G1, u=4 * G1, g=5 * G1, s=6 * G1, sh=7 * G1, D=D,
                 L=1) == SHAPE
