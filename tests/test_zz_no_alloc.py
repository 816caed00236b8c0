"""dit_selfcheck_static: the runtime-key self-check for callers that cannot
allocate device memory (device memory held by a framework's caching
allocator, or a loop that must not call cudaMalloc/cudaFree).  Its workspace
is a 4 MiB static device array inside the library.

The GPU tests call it through the C ABI: twice in a row per key, its result --
the mismatch count -- must equal that of dit_selfcheck with a caller-provided
workspace (zero on both); then the static array is read back
(dit_selfcheck_static_workspace) and the outputs the check left in it are
compared bit for bit with the CPU oracle run on the inputs it left there; and
the device's free memory (cudaMemGetInfo) must be the same before and after a
call.  This file is collected last."""
import ctypes

import numpy as np
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
    lib.dit_selfcheck_static_workspace.argtypes = [ctypes.POINTER(vp), ctypes.POINTER(i64)]
    lib.dit_selfcheck_static_workspace.restype = ci
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
        p, n = ctypes.c_void_p(1), ctypes.c_int64(1)
        assert lib.dit_selfcheck_static_workspace(ctypes.byref(p), ctypes.byref(n)) == NODEV
        assert not p.value and n.value == 0
    assert lib.dit_selfcheck_static_workspace(None, None) == NULLP


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


class _DeviceBytes:
    """A byte range of device memory, for torch.as_tensor (no copy)."""

    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1",
                                         "data": (ptr, False), "version": 3, "strides": None}


def _static_array(lib):
    p, n = ctypes.c_void_p(), ctypes.c_int64()
    assert lib.dit_selfcheck_static_workspace(ctypes.byref(p), ctypes.byref(n)) == OK
    assert n.value == LIMIT and p.value and p.value % 256 == 0
    return torch.as_tensor(_DeviceBytes(p.value, n.value), device="cuda")


TORCH_DT = {BF16: torch.bfloat16, FP16: torch.float16, FP32: torch.float32}
NAME_DT = {BF16: "bf16", FP16: "fp16", FP32: "fp32"}


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,D", [(BF16, 4096), (BF16, 3077), (FP16, 2048), (FP32, 1000)])
def test_static_array_read_back_against_the_oracle(orc, dtype, D):
    """What the check left in the static array -- its inputs and the
    library's outputs -- read back and recomputed by the oracle."""
    from _cases import bits
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    count = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    B, L, es = 2, 7, TORCH_DT[dtype].itemsize
    slot = -(-(B * L * D * es) // 256) * 256
    n = B * L * D
    for op, glay, mlay in KEYS:
        st = lib.dit_selfcheck_static(op, dtype, glay, mlay, D, count.data_ptr(), stream)
        assert st == OK
        torch.cuda.synchronize()
        assert count.item() == 0
        raw = _static_array(lib).cpu()

        def tensor(k, full=True):
            m = n if full else B * D
            t = raw[k * slot: k * slot + m * es].view(TORCH_DT[dtype])
            return t.reshape(B, L, D) if full else t.reshape(B, 1, D)

        dt = NAME_DT[dtype]
        gl, ml = ("full" if glay == FULL else "bcast"), ("full" if mlay == FULL else "bcast")
        if op == RGA:
            ref = torch.empty(B, L, D, dtype=TORCH_DT[dtype])
            orc.residual_gate_add(ref, tensor(0), tensor(1), tensor(2, glay == FULL), B, L, D,
                                  dt, gl)
            assert np.array_equal(bits(tensor(5)), bits(ref)), (op, dt, D)
        elif op == MOD:
            ref = torch.empty(B, L, D, dtype=TORCH_DT[dtype])
            orc.rmsnorm_modulate(ref, tensor(0), tensor(3, mlay == FULL), tensor(4, mlay == FULL),
                                 B, L, D, 0.75, dt, ml)
            assert np.array_equal(bits(tensor(5)), bits(ref)), (op, dt, D)
        else:
            res = torch.empty(B, L, D, dtype=TORCH_DT[dtype])
            mod = torch.empty(B, L, D, dtype=TORCH_DT[dtype])
            orc.gate_add_rmsnorm_modulate(res, mod, tensor(0), tensor(1),
                                          tensor(2, glay == FULL), tensor(3, mlay == FULL),
                                          tensor(4, mlay == FULL), B, L, D, 0.75, dt, gl, ml)
            assert np.array_equal(bits(tensor(5)), bits(res)), (op, dt, D, "residual")
            assert np.array_equal(bits(tensor(6)), bits(mod)), (op, dt, D, "modulated")


@pytest.mark.gpu
def test_static_call_allocates_no_device_memory():
    """cudaMemGetInfo's free bytes are the same before and after a call (the
    first call of the process may load the library's device code, so one
    call runs before the measurement)."""
    lib = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    count = torch.zeros((1,), dtype=torch.int32, device="cuda")
    assert lib.dit_selfcheck_static(FUSED, BF16, BCAST, BCAST, 4096, count.data_ptr(),
                                    stream) == OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for op, glay, mlay in KEYS:
        assert lib.dit_selfcheck_static(op, BF16, glay, mlay, 4096, count.data_ptr(),
                                        stream) == OK
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, (op, free0 - free1)
    assert count.item() == 0
