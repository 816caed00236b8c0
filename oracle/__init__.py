"""Plain CPU oracle for the DiT elementwise hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it shares no code with it: the C source here (dit_oracle.c) has
its own header, its own codecs and its own build step.

Operations (see dit_oracle.h for the passages each one follows):

* :func:`residual_gate_add` -- ``out = hidden + update * gate`` (sglang PR
  #29361, section Motivation), full ``[B, L, D]`` or ``[B, 1, D]`` gate.
* :func:`rmsnorm_modulate` -- ``rms_norm(x, eps) * (1 + scale) + shift``
  (prhub summary of sglang PR #34172, section "key source snippet"), with a
  weightless RMSNorm per row over D.
* :func:`gate_add_rmsnorm_modulate` -- both, the RMS taken over the stored
  (rounded) residual.
* :func:`gelu_tanh` -- the FFN's tanh-approximated GELU (prhub summary of
  sglang PR #34172, "implementation breakdown" item 3), in double, rounded
  once.
* :func:`rmsnorm_modulate_fp8`, :func:`gate_add_rmsnorm_modulate_fp8` -- the
  modulated output quantised to OCP E4M3 with a per-tensor scale (the
  RMSNorm + FP8 quantisation family named among the prhub summary's related
  PRs); :func:`e4m3_decode`, :func:`e4m3_encode` -- the E4M3 codec.

Arrays are numpy arrays or CPU torch tensors, contiguous, holding the raw
storage of the dtype: 16-bit words for bf16 and fp16, ``float32`` for fp32.
Outputs are written in place.

Every function is pinned in ``tests/test_oracle_*.py`` against values fixed by
the mathematics (closed forms, invariants, exact rational brute force on tiny
inputs) and by library routines (torch and numpy dtype conversions, torch's
``rms_norm`` in float64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dit_oracle.c")
_HDR = os.path.join(_HERE, "dit_oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}
LAYOUTS = {"full": 0, "bcast": 1}
ELEM_SIZE = {"bf16": 2, "fp16": 2, "fp32": 4}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` from ``dit_oracle.c`` with gcc (no fast-math,
    no FMA contraction).  Returns the library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(_HDR))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC,
           "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    """ctypes handle of an oracle library with its signatures declared."""
    lib = ctypes.CDLL(path)
    i64, vp, fp = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
    ci = ctypes.c_int
    lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_bf16_to_f32.restype = fp
    lib.orc_f32_to_bf16.argtypes = [fp]
    lib.orc_f32_to_bf16.restype = ctypes.c_uint16
    lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f32.restype = fp
    lib.orc_f32_to_f16.argtypes = [fp]
    lib.orc_f32_to_f16.restype = ctypes.c_uint16
    lib.orc_decode_array.argtypes = [vp, vp, i64, ci]
    lib.orc_decode_array.restype = None
    lib.orc_encode_array.argtypes = [vp, vp, i64, ci]
    lib.orc_encode_array.restype = None
    lib.orc_rmsnorm_modulate.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64,
                                         fp, ci, ci, vp, i64]
    lib.orc_rmsnorm_modulate.restype = ci
    lib.orc_gate_add_rmsnorm_modulate.argtypes = [
        vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, fp, ci, ci, ci, vp, i64]
    lib.orc_gate_add_rmsnorm_modulate.restype = ci
    lib.orc_gelu_tanh.argtypes = [vp, vp, i64, ci]
    lib.orc_gelu_tanh.restype = ci
    lib.orc_store_double.argtypes = [vp, i64, ctypes.c_double, ci]
    lib.orc_store_double.restype = None
    lib.orc_row_rms_inverse.argtypes = [vp, i64, fp, ci]
    lib.orc_row_rms_inverse.restype = fp
    lib.orc_row_mean_square.argtypes = [vp, i64, ci]
    lib.orc_row_mean_square.restype = fp
    lib.orc_inverse_root_array.argtypes = [vp, vp, i64]
    lib.orc_inverse_root_array.restype = None
    lib.orc_residual_gate_add_mt.argtypes = [ci, vp, vp, vp, vp, i64, i64,
                                             i64, ci, ci, vp, i64]
    lib.orc_residual_gate_add_mt.restype = ci
    lib.orc_rmsnorm_modulate_mt.argtypes = [ci, vp, vp, vp, vp, i64, i64,
                                            i64, fp, ci, ci, vp, i64]
    lib.orc_rmsnorm_modulate_mt.restype = ci
    lib.orc_gate_add_rmsnorm_modulate_mt.argtypes = [
        ci, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, fp, ci, ci, ci, vp, i64]
    lib.orc_gate_add_rmsnorm_modulate_mt.restype = ci
    lib.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_f32.restype = fp
    lib.orc_f32_to_e4m3.argtypes = [fp]
    lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
    lib.orc_rmsnorm_modulate_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, fp, ci, ci,
                                             fp, vp, i64]
    lib.orc_rmsnorm_modulate_fp8.restype = ci
    lib.orc_gate_add_rmsnorm_modulate_fp8.argtypes = [
        vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, fp, ci, ci, ci, fp, vp, i64]
    lib.orc_gate_add_rmsnorm_modulate_fp8.restype = ci
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _ptr(a):
    """Address of a contiguous numpy array or CPU torch tensor (None -> NULL)."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):  # torch tensor
        if a.device.type != "cpu" or not a.is_contiguous():
            raise ValueError("oracle inputs must be contiguous CPU tensors")
        return a.data_ptr() or None
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle inputs must be C-contiguous arrays")
    return a.ctypes.data or None


def _rows(rows):
    """(pointer, count, keep-alive) for an optional row selection."""
    if rows is None:
        return None, 0, None
    import numpy as np
    arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return (arr.ctypes.data if arr.size else None), int(arr.size), arr


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad argument")


def decode(src, dtype):
    """fp32 values of an array of dtype storage (numpy float32 result)."""
    import numpy as np
    n = int(src.numel() if hasattr(src, "numel") else src.size)
    dst = np.empty(n, dtype=np.float32)
    _load().orc_decode_array(_ptr(dst), _ptr(src), n, DTYPES[dtype])
    return dst


def encode(src_f32, dtype):
    """Storage words of fp32 values rounded once to dtype (numpy uint16 for
    bf16/fp16, float32 for fp32)."""
    import numpy as np
    src = np.ascontiguousarray(np.asarray(src_f32, dtype=np.float32)).ravel()
    dst = np.empty(src.size, dtype=np.float32 if dtype == "fp32" else np.uint16)
    _load().orc_encode_array(_ptr(dst), _ptr(src), src.size, DTYPES[dtype])
    return dst


def residual_gate_add(out, hidden, update, gate, B, L, D, dtype="bf16",
                      gate_layout="full", rows=None, threads=1):
    rp, n, keep = _rows(rows)
    rc = _load().orc_residual_gate_add_mt(int(threads), _ptr(out), _ptr(hidden),
                                          _ptr(update), _ptr(gate), B, L, D,
                                          DTYPES[dtype], LAYOUTS[gate_layout], rp, n)
    del keep
    _check(rc, "residual_gate_add")


def rmsnorm_modulate(out, x, scale, shift, B, L, D, eps=1e-6, dtype="bf16",
                     mod_layout="bcast", rows=None, t_out=None, threads=1):
    rp, n, keep = _rows(rows)
    lib = _load()
    if t_out is not None:
        rc = lib.orc_rmsnorm_modulate(_ptr(out), _ptr(t_out), _ptr(x), _ptr(scale),
                                      _ptr(shift), B, L, D, float(eps),
                                      DTYPES[dtype], LAYOUTS[mod_layout], rp, n)
    else:
        rc = lib.orc_rmsnorm_modulate_mt(int(threads), _ptr(out), _ptr(x),
                                         _ptr(scale), _ptr(shift), B, L, D,
                                         float(eps), DTYPES[dtype],
                                         LAYOUTS[mod_layout], rp, n)
    del keep
    _check(rc, "rmsnorm_modulate")


def gate_add_rmsnorm_modulate(residual_out, modulated_out, hidden, update, gate,
                              scale, shift, B, L, D, eps=1e-6, dtype="bf16",
                              gate_layout="bcast", mod_layout="bcast", rows=None,
                              t_out=None, threads=1):
    rp, n, keep = _rows(rows)
    lib = _load()
    if t_out is not None:
        rc = lib.orc_gate_add_rmsnorm_modulate(
            _ptr(residual_out), _ptr(modulated_out), _ptr(t_out), _ptr(hidden),
            _ptr(update), _ptr(gate), _ptr(scale), _ptr(shift), B, L, D,
            float(eps), DTYPES[dtype], LAYOUTS[gate_layout], LAYOUTS[mod_layout],
            rp, n)
    else:
        rc = lib.orc_gate_add_rmsnorm_modulate_mt(
            int(threads), _ptr(residual_out), _ptr(modulated_out), _ptr(hidden),
            _ptr(update), _ptr(gate), _ptr(scale), _ptr(shift), B, L, D,
            float(eps), DTYPES[dtype], LAYOUTS[gate_layout], LAYOUTS[mod_layout],
            rp, n)
    del keep
    _check(rc, "gate_add_rmsnorm_modulate")


def gelu_tanh(out, x, dtype="bf16"):
    """out = gelu(x) with the tanh approximation, evaluated in double and
    rounded once to dtype."""
    n = int(x.numel() if hasattr(x, "numel") else x.size)
    _check(_load().orc_gelu_tanh(_ptr(out), _ptr(x), n, DTYPES[dtype]), "gelu_tanh")


def e4m3_decode(codes):
    """fp32 values (numpy) of E4M3 codes (any iterable of 0..255)."""
    import numpy as np
    lib = _load()
    return np.array([lib.orc_e4m3_to_f32(int(c)) for c in codes], dtype=np.float32)


def e4m3_encode(values):
    """E4M3 codes (numpy uint8) of fp32 values, each rounded once."""
    import numpy as np
    lib = _load()
    v = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.orc_f32_to_e4m3(float(x)) for x in v.tolist()], dtype=np.uint8)


def rmsnorm_modulate_fp8(out, x, scale, shift, B, L, D, eps=1e-6, dtype="bf16",
                         mod_layout="bcast", quant_scale=1.0, rows=None, t_out=None):
    """out (uint8, one E4M3 code per element) = e4m3(fl(y * fl(1 / quant_scale)))
    of the fp32 modulation value y."""
    rp, n, keep = _rows(rows)
    rc = _load().orc_rmsnorm_modulate_fp8(_ptr(out), _ptr(t_out), _ptr(x), _ptr(scale),
                                          _ptr(shift), B, L, D, float(eps), DTYPES[dtype],
                                          LAYOUTS[mod_layout], float(quant_scale), rp, n)
    del keep
    _check(rc, "rmsnorm_modulate_fp8")


def gate_add_rmsnorm_modulate_fp8(residual_out, out, hidden, update, gate, scale, shift,
                                  B, L, D, eps=1e-6, dtype="bf16", gate_layout="bcast",
                                  mod_layout="bcast", quant_scale=1.0, rows=None,
                                  t_out=None):
    rp, n, keep = _rows(rows)
    rc = _load().orc_gate_add_rmsnorm_modulate_fp8(
        _ptr(residual_out), _ptr(out), _ptr(t_out), _ptr(hidden), _ptr(update), _ptr(gate),
        _ptr(scale), _ptr(shift), B, L, D, float(eps), DTYPES[dtype], LAYOUTS[gate_layout],
        LAYOUTS[mod_layout], float(quant_scale), rp, n)
    del keep
    _check(rc, "gate_add_rmsnorm_modulate_fp8")


def round_double(values, dtype):
    """Storage words of doubles rounded once to dtype."""
    import numpy as np
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64)).ravel()
    dst = np.empty(v.size, dtype=np.float32 if dtype == "fp32" else np.uint16)
    lib = _load()
    for i, x in enumerate(v.tolist()):
        lib.orc_store_double(_ptr(dst), i, x, DTYPES[dtype])
    return dst


def row_rms_inverse(x_row, D, eps=1e-6, dtype="bf16") -> float:
    return _load().orc_row_rms_inverse(_ptr(x_row), D, float(eps), DTYPES[dtype])


def row_mean_square(x_row, D, dtype="bf16") -> float:
    """ms = RN32(mean(x^2)) of one row: the exact mean rounded once to fp32."""
    return _load().orc_row_mean_square(_ptr(x_row), D, DTYPES[dtype])


def inverse_root(v):
    """RN32(1 / sqrt(v)) of fp32 values (numpy float32 result), the
    statistic's inverse-root step."""
    import numpy as np
    src = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).ravel()
    dst = np.empty_like(src)
    _load().orc_inverse_root_array(_ptr(src), _ptr(dst), src.size)
    return dst


def variant(lib_path: str):
    """A namespace with this module's functions bound to another build of the
    oracle source (used by the tests that plant mistakes in a copy of it)."""
    import sys
    import types
    ns = types.ModuleType("oracle_variant")
    src = sys.modules[__name__]
    lib = _bind(lib_path)
    for name in ("decode", "encode", "residual_gate_add", "rmsnorm_modulate",
                 "gate_add_rmsnorm_modulate", "row_rms_inverse", "row_mean_square",
                 "inverse_root", "gelu_tanh", "round_double",
                 "e4m3_decode", "e4m3_encode", "rmsnorm_modulate_fp8",
                 "gate_add_rmsnorm_modulate_fp8"):
        fn = getattr(src, name)
        g = dict(fn.__globals__)
        g["_load"] = lambda lib=lib: lib
        setattr(ns, name, types.FunctionType(fn.__code__, g, name, fn.__defaults__))
    for name in ("DTYPES", "LAYOUTS", "ELEM_SIZE"):
        setattr(ns, name, getattr(src, name))
    return ns
