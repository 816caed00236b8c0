"""dit_selfcheck_static: the runtime-key self-check for callers that cannot
allocate device memory (device memory held by a framework's caching
allocator, or a loop that must not call cudaMalloc/cudaFree).  Its workspace
is a 4 MiB static device array inside the library.

The GPU test calls it through the C ABI twice in a row per key and checks
that its result -- the mismatch count -- equals that of dit_selfcheck with a
caller-provided workspace (zero on both).  This file is collected last."""
import ctypes

import pytest
import torch

from diffusion_transformer_elementwise_gb300 import library
from diffusion_transformer_elementwise_gb300.build import build

OK, WORKSPACE, NODEV, SHAPE, NULLP = 0, 11, 9, 2, 1
BF16, FP16, FP32 = 0, 1, 2
FULL, BCAST = 0, 1
RGA, MOD, FUSED = 0, 1, 2
LIMIT = 4 << 20


def _lib():
    build()
    lib = library()
    f = lib.dit_selfcheck_static
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.argtypes = [ci, ci, ci, ci, i64, vp, vp]
    f.restype = ci
    lib.dit_selfcheck_workspace_bytes.argtypes = [ci, ci, i64]
    lib.dit_selfcheck_workspace_bytes.restype = i64
    return lib


def test_static_limit_and_validation():
    """Keys beyond the static array are refused before any device work, and
    the other argument checks are those of dit_selfcheck."""
    lib = _lib()
    f = lib.dit_selfcheck_static
    assert lib.dit_selfcheck_workspace_bytes(FUSED, FP32, 16384) > LIMIT
    assert lib.dit_selfcheck_workspace_bytes(FUSED, FP32, 8192) <= LIMIT
    assert lib.dit_selfcheck_workspace_bytes(FUSED, BF16, 16384) <= LIMIT
    cnt = 1 << 24  # never dereferenced: every call below returns before a launch
    assert f(FUSED, FP32, BCAST, BCAST, 16384, cnt, None) == WORKSPACE
    assert f(MOD, BF16, BCAST, BCAST, 0, cnt, None) == SHAPE
    assert f(MOD, BF16, BCAST, BCAST, 64, None, None) == NULLP
    if not torch.cuda.is_available():
        assert f(MOD, BF16, BCAST, BCAST, 64, cnt, None) == NODEV


KEYS = [(RGA, BCAST, BCAST), (RGA, FULL, BCAST), (MOD, BCAST, BCAST), (MOD, BCAST, FULL),
        (FUSED, BCAST, BCAST), (FUSED, FULL, FULL)]


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,D", [(BF16, 4096), (BF16, 3077), (FP16, 2048), (FP32, 4096),
                                     (BF16, 16384), (FP32, 8192)])
def test_static_equals_workspace_entry_two_calls(dtype, D):
    lib = _lib()
    dev = torch.cuda.current_device()
    stream = torch.cuda.current_stream().cuda_stream
    count = torch.full((2,), 7, dtype=torch.int32, device="cuda")
    for op, glay, mlay in KEYS:
        nbytes = lib.dit_selfcheck_workspace_bytes(op, dtype, D)
        ws = torch.empty(nbytes + 256, dtype=torch.uint8, device="cuda")
        wp = ws.data_ptr() + (-ws.data_ptr()) % 256
        for call in range(2):
            st = lib.dit_selfcheck_static(op, dtype, glay, mlay, D, count.data_ptr(), stream)
            assert st == OK, (op, dtype, D, call, st)
            st = lib.dit_selfcheck(op, dtype, glay, mlay, D, wp, nbytes, count.data_ptr() + 4,
                                   stream)
            assert st == OK
            torch.cuda.synchronize(dev)
            static_n, ws_n = count.tolist()
            assert static_n == ws_n == 0, (op, glay, mlay, dtype, D, call, static_n, ws_n)
            count.fill_(7)  # each call must reset the counter itself
