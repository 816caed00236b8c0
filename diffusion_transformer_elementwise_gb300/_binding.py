"""ctypes binding of libdit_elementwise.so (include/dit_elementwise.h).

Argument marshalling only: every function checks that its tensors are
contiguous CUDA tensors of one dtype (a [B, 1, D] gate, scale or shift may be
a view with contiguous rows and any batch stride, e.g. a row of an adaLN
table), passes their addresses, sizes, dtype, layouts, the vectors' batch
stride and the current torch stream to the C ABI, and raises
:class:`DitError` on a non-OK status.  There is no other code path: without
the built library, or with CPU tensors, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB

DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
FULL, ROW_BCAST = 0, 1

_lock = threading.Lock()
_lib = None


class Problem(ctypes.Structure):
    """dit_problem of include/dit_elementwise.h."""
    _fields_ = [("out", ctypes.c_void_p), ("out2", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("update", ctypes.c_void_p), ("gate", ctypes.c_void_p),
                ("scale", ctypes.c_void_p), ("shift", ctypes.c_void_p),
                ("B", ctypes.c_int64), ("L", ctypes.c_int64), ("D", ctypes.c_int64),
                ("vec_stride", ctypes.c_int64)]


OP_RESIDUAL_GATE, OP_RMSNORM_MODULATE, OP_GATE_ADD_RMSNORM_MODULATE = 0, 1, 2
MAX_GROUP = 8


class DitError(RuntimeError):
    """A dit_* call returned a status other than DIT_OK."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def library() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(
                    f"{LIB} is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` "
                    "(nvcc for sm_103a); there is no fallback path")
            lib = ctypes.CDLL(LIB)
            vp, i64, ci, cf = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.dit_abi_version.argtypes = []
            lib.dit_abi_version.restype = ci
            lib.dit_status_string.argtypes = [ci]
            lib.dit_status_string.restype = ctypes.c_char_p
            lib.dit_residual_gate_add.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci, vp]
            lib.dit_residual_gate_add.restype = ci
            lib.dit_rmsnorm_modulate.argtypes = [vp, vp, vp, vp, i64, i64, i64, cf, ci, ci, vp]
            lib.dit_rmsnorm_modulate.restype = ci
            lib.dit_gate_add_rmsnorm_modulate.argtypes = [
                vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, cf, ci, ci, ci, vp]
            lib.dit_gate_add_rmsnorm_modulate.restype = ci
            lib.dit_gelu_tanh.argtypes = [vp, vp, i64, ci, vp]
            lib.dit_gelu_tanh.restype = ci
            lib.dit_residual_gate_add_strided.argtypes = [vp, vp, vp, vp, i64, i64, i64, ci, ci,
                                                          i64, vp]
            lib.dit_residual_gate_add_strided.restype = ci
            lib.dit_rmsnorm_modulate_strided.argtypes = [vp, vp, vp, vp, i64, i64, i64, cf, ci,
                                                         ci, i64, vp]
            lib.dit_rmsnorm_modulate_strided.restype = ci
            lib.dit_gate_add_rmsnorm_modulate_strided.argtypes = [
                vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, cf, ci, ci, ci, i64, vp]
            lib.dit_gate_add_rmsnorm_modulate_strided.restype = ci
            lib.dit_grouped.argtypes = [ci, ctypes.POINTER(Problem), ci, cf, ci, ci, ci, vp]
            lib.dit_grouped.restype = ci
            lib.dit_rmsnorm_modulate_fp8.argtypes = [vp, vp, vp, vp, i64, i64, i64, cf, ci, ci,
                                                     i64, vp, vp]
            lib.dit_rmsnorm_modulate_fp8.restype = ci
            lib.dit_gate_add_rmsnorm_modulate_fp8.argtypes = [
                vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, cf, ci, ci, ci, i64, vp, vp]
            lib.dit_gate_add_rmsnorm_modulate_fp8.restype = ci
            lib.dit_selfcheck_workspace_bytes.argtypes = [ci, ci, i64]
            lib.dit_selfcheck_workspace_bytes.restype = i64
            lib.dit_selfcheck.argtypes = [ci, ci, ci, ci, i64, vp, i64, vp, vp]
            lib.dit_selfcheck.restype = ci
            lib.dit_set_statistic.argtypes = [ci]
            lib.dit_set_statistic.restype = ci
            lib.dit_get_statistic.argtypes = []
            lib.dit_get_statistic.restype = ci
            _lib = lib
    return _lib


def check(status: int, what: str) -> None:
    if status != 0:
        msg = library().dit_status_string(status).decode()
        raise DitError(status, f"{what}: {msg}")


STATISTICS = {"fast": 0, "exact": 1}


def set_statistic(kind: str) -> None:
    """The row statistic of the modulating operations for the whole process
    (dit_set_statistic): "fast" (default) or "exact"."""
    if kind not in STATISTICS:
        raise ValueError(f"statistic must be one of {sorted(STATISTICS)}")
    check(library().dit_set_statistic(STATISTICS[kind]), "set_statistic")


def get_statistic() -> str:
    code = library().dit_get_statistic()
    return {v: k for k, v in STATISTICS.items()}[code]


class statistic:
    """Context manager: the given row statistic inside the block, the
    previous one restored after it (calls are read when made)."""

    def __init__(self, kind: str):
        self.kind = kind
        self.prev = None

    def __enter__(self):
        self.prev = get_statistic()
        set_statistic(self.kind)
        return self

    def __exit__(self, *exc):
        set_statistic(self.prev)
        return False


def _shape3(t: torch.Tensor, name: str):
    if t.dim() != 3:
        raise ValueError(f"{name} must be [B, L, D], got {tuple(t.shape)}")
    return tuple(int(s) for s in t.shape)


def _cuda(*tensors):
    """Checks the tensors; returns the index of their (common) CUDA device."""
    dev = None
    for name, t in tensors:
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor (there is no CPU path)")
        vector = name in ("gate", "scale", "shift")
        if not t.is_contiguous() and not (vector and _strided_vector(t)):
            raise ValueError(f"{name} must be contiguous" +
                             (" (or a [B, 1, D] view with contiguous rows)" if vector else ""))
        if dev is None:
            dev = t.get_device()
        elif t.get_device() != dev:
            raise ValueError(f"{name} is on cuda:{t.get_device()}, expected cuda:{dev}")
    return dev


def _dtype(ref: torch.Tensor, *others) -> int:
    if ref.dtype not in DTYPE_CODES:
        raise TypeError(f"unsupported dtype {ref.dtype}: bf16, fp16 or fp32")
    for name, t in others:
        if t.dtype != ref.dtype:
            raise TypeError(f"{name} is {t.dtype}, expected {ref.dtype}")
    return DTYPE_CODES[ref.dtype]


def _strided_vector(t: torch.Tensor) -> bool:
    """A [B, 1, D] view whose rows are contiguous (e.g. rows of an adaLN
    table [B, 9, D]): passed with a batch stride."""
    return t.dim() == 3 and t.shape[1] == 1 and (t.shape[2] <= 1 or t.stride(2) == 1)


def _vector_stride(D: int, *vectors) -> int:
    """The common batch stride (elements) of the [B, 1, D] operands."""
    strides = {int(t.stride(0)) for t in vectors if t.shape[0] > 1}
    if len(strides) > 1:
        raise ValueError("the [B, 1, D] operands of one call must share their batch stride")
    return strides.pop() if strides else D


def layout_of(t: torch.Tensor, B: int, L: int, D: int, name: str) -> int:
    """FULL for [B, L, D], ROW_BCAST for [B, 1, D]."""
    shape = tuple(t.shape)
    if shape == (B, L, D) and (L != 1 or t.is_contiguous()):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return FULL
    if shape == (B, 1, D):
        return ROW_BCAST
    raise ValueError(f"{name} must be [{B}, {L}, {D}] or [{B}, 1, {D}], got {shape}")


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(dev: int, stream) -> int:
    """The cudaStream_t to launch on: `stream` (a torch.cuda.Stream or a raw
    handle), else torch's current stream of device `dev`."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(dev)
        stream = torch.cuda.current_stream(dev)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _launch(dev: int, fn, *args) -> int:
    """Calls the C entry point with `dev` as the current CUDA device."""
    if torch.cuda.current_device() == dev:
        return fn(*args)
    with torch.cuda.device(dev):
        return fn(*args)


def residual_gate_add(hidden, update, gate, out=None, stream=None):
    """out = hidden + update * gate; gate [B, L, D] or [B, 1, D].  Pass
    out=hidden for the in-place update.  Returns out."""
    B, L, D = _shape3(hidden, "hidden")
    if out is None:
        out = torch.empty_like(hidden)
    dev = _cuda(("hidden", hidden), ("update", update), ("gate", gate), ("out", out))
    dt = _dtype(hidden, ("update", update), ("gate", gate), ("out", out))
    if tuple(update.shape) != (B, L, D) or tuple(out.shape) != (B, L, D):
        raise ValueError("update and out must have the shape of hidden")
    lay = layout_of(gate, B, L, D, "gate")
    vs = _vector_stride(D, gate) if lay == ROW_BCAST else D
    if _first_use:
        _first_use_check("residual_gate", hidden.dtype, lay, ROW_BCAST, D, dev)
    st = _launch(dev, library().dit_residual_gate_add_strided, out.data_ptr(), hidden.data_ptr(),
                 update.data_ptr(), gate.data_ptr(), B, L, D, dt, lay, vs, _stream(dev, stream))
    check(st, "dit_residual_gate_add")
    return out


def rmsnorm_modulate(x, scale, shift, eps=1e-6, out=None, stream=None):
    """out = rms_norm(x, eps) * (1 + scale) + shift; scale/shift [B, L, D] or
    [B, 1, D] (the same layout for both).  Returns out."""
    B, L, D = _shape3(x, "x")
    if out is None:
        out = torch.empty_like(x)
    dev = _cuda(("x", x), ("scale", scale), ("shift", shift), ("out", out))
    dt = _dtype(x, ("scale", scale), ("shift", shift), ("out", out))
    if tuple(out.shape) != (B, L, D):
        raise ValueError("out must have the shape of x")
    lay = layout_of(scale, B, L, D, "scale")
    if layout_of(shift, B, L, D, "shift") != lay:
        raise ValueError("scale and shift must have the same layout")
    vs = _vector_stride(D, scale, shift) if lay == ROW_BCAST else D
    if _first_use:
        _first_use_check("rmsnorm_modulate", x.dtype, ROW_BCAST, lay, D, dev)
    st = _launch(dev, library().dit_rmsnorm_modulate_strided, out.data_ptr(), x.data_ptr(),
                 scale.data_ptr(), shift.data_ptr(), B, L, D, float(eps), dt, lay, vs,
                 _stream(dev, stream))
    check(st, "dit_rmsnorm_modulate")
    return out


def gate_add_rmsnorm_modulate(hidden, update, gate, scale, shift, eps=1e-6,
                              residual_out=None, modulated_out=None, stream=None):
    """residual_out = hidden + update * gate; modulated_out =
    rms_norm(residual_out, eps) * (1 + scale) + shift, in one pass.  Pass
    residual_out=hidden to update the residual in place.  Returns
    (residual_out, modulated_out)."""
    B, L, D = _shape3(hidden, "hidden")
    if residual_out is None:
        residual_out = torch.empty_like(hidden)
    if modulated_out is None:
        modulated_out = torch.empty_like(hidden)
    dev = _cuda(("hidden", hidden), ("update", update), ("gate", gate), ("scale", scale),
                ("shift", shift), ("residual_out", residual_out),
                ("modulated_out", modulated_out))
    dt = _dtype(hidden, ("update", update), ("gate", gate), ("scale", scale),
                ("shift", shift), ("residual_out", residual_out),
                ("modulated_out", modulated_out))
    for name, t in (("update", update), ("residual_out", residual_out),
                    ("modulated_out", modulated_out)):
        if tuple(t.shape) != (B, L, D):
            raise ValueError(f"{name} must have the shape of hidden")
    glay = layout_of(gate, B, L, D, "gate")
    mlay = layout_of(scale, B, L, D, "scale")
    if layout_of(shift, B, L, D, "shift") != mlay:
        raise ValueError("scale and shift must have the same layout")
    vecs = ([gate] if glay == ROW_BCAST else []) + ([scale, shift] if mlay == ROW_BCAST else [])
    vs = _vector_stride(D, *vecs)
    if _first_use:
        _first_use_check("gate_add_rmsnorm_modulate", hidden.dtype, glay, mlay, D, dev)
    st = _launch(dev, library().dit_gate_add_rmsnorm_modulate_strided,
                 residual_out.data_ptr(), modulated_out.data_ptr(), hidden.data_ptr(),
                 update.data_ptr(), gate.data_ptr(), scale.data_ptr(), shift.data_ptr(), B, L, D,
                 float(eps), dt, glay, mlay, vs, _stream(dev, stream))
    check(st, "dit_gate_add_rmsnorm_modulate")
    return residual_out, modulated_out


def gelu_tanh(x, out=None, stream=None):
    """out = 0.5 * x * (1 + tanh(sqrt(2/pi) * (x + 0.044715 * x^3))),
    elementwise over a contiguous tensor of any shape.  Pass out=x for the
    in-place form.  Returns out."""
    if out is None:
        out = torch.empty_like(x)
    dev = _cuda(("x", x), ("out", out))
    dt = _dtype(x, ("out", out))
    if out.shape != x.shape:
        raise ValueError("out must have the shape of x")
    st = _launch(dev, library().dit_gelu_tanh, out.data_ptr(), x.data_ptr(), x.numel(), dt,
                 _stream(dev, stream))
    check(st, "dit_gelu_tanh")
    return out


# ---------------------------------------------------------------------------
# grouped launches (dit_grouped): one operation over several problems
# ---------------------------------------------------------------------------

def _group_call(op, problems, eps, dt, glay, mlay, dev, stream, what):
    if len(problems) > MAX_GROUP:
        raise ValueError(f"at most {MAX_GROUP} problems per grouped call")
    arr = (Problem * max(1, len(problems)))(*problems)
    st = _launch(dev, library().dit_grouped, op, arr, len(problems), float(eps), dt, glay, mlay,
                 _stream(dev, stream))
    check(st, what)


def _either(layout, L, B, D, vs):
    """None where both layouts read the same memory (one row per batch and
    contiguous vectors), so the problem takes the group's layout."""
    return None if L == 1 and (B <= 1 or vs == D) else layout


def _common(values, what):
    vals = set(v for v in values if v is not None)
    if not vals:
        return FULL
    if len(vals) > 1:
        raise ValueError(f"the problems of one grouped call must share their {what}")
    return vals.pop()


def residual_gate_add_grouped(problems, stream=None):
    """out = hidden + update * gate for each (hidden, update, gate[, out]) of
    `problems` (out None or missing: allocated; out=hidden: in place), in one
    launch when the problems allow it (dit_grouped).  All problems share the
    dtype and the gate layout.  Returns the list of outputs."""
    if not problems:
        return []
    descs, outs, devs, dts, lays = [], [], [], [], []
    for hidden, update, gate, *rest in problems:
        out = rest[0] if rest and rest[0] is not None else torch.empty_like(hidden)
        B, L, D = _shape3(hidden, "hidden")
        devs.append(_cuda(("hidden", hidden), ("update", update), ("gate", gate), ("out", out)))
        dts.append(_dtype(hidden, ("update", update), ("gate", gate), ("out", out)))
        if tuple(update.shape) != (B, L, D) or tuple(out.shape) != (B, L, D):
            raise ValueError("update and out must have the shape of hidden")
        lay = layout_of(gate, B, L, D, "gate")
        vs = _vector_stride(D, gate) if lay == ROW_BCAST else D
        lays.append(_either(lay, L, B, D, vs))
        descs.append(Problem(out.data_ptr(), None, hidden.data_ptr(), update.data_ptr(),
                             gate.data_ptr(), None, None, B, L, D, vs))
        outs.append(out)
    dev, dt, lay = _common(devs, "device"), _common(dts, "dtype"), _common(lays, "gate layout")
    _group_call(OP_RESIDUAL_GATE, descs, 0.0, dt, lay, FULL, dev, stream,
                "dit_grouped(residual gate)")
    return outs


def rmsnorm_modulate_grouped(problems, eps=1e-6, stream=None):
    """out = rms_norm(x, eps) * (1 + scale) + shift for each
    (x, scale, shift[, out]) of `problems`, in one launch when the problems
    allow it (dit_grouped).  All problems share the dtype and the layout of
    scale/shift.  Returns the list of outputs."""
    if not problems:
        return []
    descs, outs, devs, dts, lays = [], [], [], [], []
    for x, scale, shift, *rest in problems:
        out = rest[0] if rest and rest[0] is not None else torch.empty_like(x)
        B, L, D = _shape3(x, "x")
        devs.append(_cuda(("x", x), ("scale", scale), ("shift", shift), ("out", out)))
        dts.append(_dtype(x, ("scale", scale), ("shift", shift), ("out", out)))
        if tuple(out.shape) != (B, L, D):
            raise ValueError("out must have the shape of x")
        lay = layout_of(scale, B, L, D, "scale")
        if layout_of(shift, B, L, D, "shift") != lay:
            raise ValueError("scale and shift must have the same layout")
        vs = _vector_stride(D, scale, shift) if lay == ROW_BCAST else D
        lays.append(_either(lay, L, B, D, vs))
        descs.append(Problem(out.data_ptr(), None, x.data_ptr(), None, None, scale.data_ptr(),
                             shift.data_ptr(), B, L, D, vs))
        outs.append(out)
    dev, dt, lay = _common(devs, "device"), _common(dts, "dtype"), _common(lays, "scale layout")
    _group_call(OP_RMSNORM_MODULATE, descs, eps, dt, FULL, lay, dev, stream,
                "dit_grouped(modulation)")
    return outs


def gate_add_rmsnorm_modulate_grouped(problems, eps=1e-6, stream=None):
    """The fused op for each (hidden, update, gate, scale, shift[,
    residual_out[, modulated_out]]) of `problems`, in one launch when the
    problems allow it (dit_grouped).  All problems share the dtype, the gate
    layout and the scale/shift layout.  Returns the list of
    (residual_out, modulated_out)."""
    if not problems:
        return []
    descs, outs, devs, dts, glays, mlays = [], [], [], [], [], []
    for hidden, update, gate, scale, shift, *rest in problems:
        r = rest[0] if len(rest) > 0 and rest[0] is not None else torch.empty_like(hidden)
        m = rest[1] if len(rest) > 1 and rest[1] is not None else torch.empty_like(hidden)
        B, L, D = _shape3(hidden, "hidden")
        devs.append(_cuda(("hidden", hidden), ("update", update), ("gate", gate),
                          ("scale", scale), ("shift", shift), ("residual_out", r),
                          ("modulated_out", m)))
        dts.append(_dtype(hidden, ("update", update), ("gate", gate), ("scale", scale),
                          ("shift", shift), ("residual_out", r), ("modulated_out", m)))
        for name, t in (("update", update), ("residual_out", r), ("modulated_out", m)):
            if tuple(t.shape) != (B, L, D):
                raise ValueError(f"{name} must have the shape of hidden")
        glay = layout_of(gate, B, L, D, "gate")
        mlay = layout_of(scale, B, L, D, "scale")
        if layout_of(shift, B, L, D, "shift") != mlay:
            raise ValueError("scale and shift must have the same layout")
        vecs = ([gate] if glay == ROW_BCAST else []) + ([scale, shift] if mlay == ROW_BCAST else [])
        vs = _vector_stride(D, *vecs)
        glays.append(_either(glay, L, B, D, vs))
        mlays.append(_either(mlay, L, B, D, vs))
        descs.append(Problem(r.data_ptr(), m.data_ptr(), hidden.data_ptr(), update.data_ptr(),
                             gate.data_ptr(), scale.data_ptr(), shift.data_ptr(), B, L, D, vs))
        outs.append((r, m))
    dev, dt = _common(devs, "device"), _common(dts, "dtype")
    glay, mlay = _common(glays, "gate layout"), _common(mlays, "scale layout")
    _group_call(OP_GATE_ADD_RMSNORM_MODULATE, descs, eps, dt, glay, mlay, dev, stream,
                "dit_grouped(fused)")
    return outs


# ---------------------------------------------------------------------------
# self-check of runtime keys (dit_selfcheck)
# ---------------------------------------------------------------------------

OPS = {"residual_gate": OP_RESIDUAL_GATE, "rmsnorm_modulate": OP_RMSNORM_MODULATE,
       "gate_add_rmsnorm_modulate": OP_GATE_ADD_RMSNORM_MODULATE}
LAYOUTS = {"full": FULL, "bcast": ROW_BCAST}
_NAMES = {torch.bfloat16: "bf16", torch.float16: "fp16", torch.float32: "fp32"}
_CODES = {"bf16": 0, "fp16": 1, "fp32": 2}


def selfcheck(op, dtype, gate_layout="bcast", mod_layout="bcast", D=4096, device=None,
              stream=None, return_workspace=False):
    """Run dit_selfcheck for the key (op, dtype, gate_layout, mod_layout, D)
    on a [2, 7, D] problem and return the number of output words that differ
    from their one correct value (0: the key's path computes the
    definition).  Synchronises the stream to read the count.  op: a key of
    OPS; dtype: "bf16", "fp16" or "fp32" (or a torch dtype); layouts: "full"
    or "bcast".  return_workspace=True also returns the workspace (a uint8
    device tensor laid out as include/dit_elementwise.h states)."""
    opc = OPS[op] if isinstance(op, str) else int(op)
    dt = _CODES[_NAMES.get(dtype, dtype)]
    dev = torch.cuda.current_device() if device is None else torch.device(device).index
    nbytes = library().dit_selfcheck_workspace_bytes(opc, dt, int(D))
    if nbytes < 0:
        raise ValueError(f"no self-check for op={op!r} dtype={dtype!r} D={D}")
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=f"cuda:{dev}")
    off = (-ws.data_ptr()) % 256
    work = ws[off:off + nbytes]
    count = torch.zeros(1, dtype=torch.int32, device=f"cuda:{dev}")
    st = _launch(dev, library().dit_selfcheck, opc, dt, LAYOUTS[gate_layout],
                 LAYOUTS[mod_layout], int(D), work.data_ptr(), nbytes, count.data_ptr(),
                 _stream(dev, stream))
    check(st, "dit_selfcheck")
    n = int(count.item())
    return (n, work) if return_workspace else n


_checked: set = set()
_first_use = False


def ensure_checked(op, dtype, gate_layout="bcast", mod_layout="bcast", D=4096, device=None):
    """Self-check the key once per process (the pages' first-use guard,
    without a fallback).  Raises DitError with status -1 if any output word
    differs (the key is then not recorded); returns True if the check ran
    now, False if the key had passed before.  The check covers the kernel
    the library picks for 256-byte aligned tensors of row width D."""
    dt = _NAMES.get(dtype, dtype)
    dev = torch.cuda.current_device() if device is None else torch.device(device).index
    key = (op, dt, gate_layout, mod_layout, int(D), dev)
    if key in _checked:
        return False
    n = selfcheck(op, dt, gate_layout, mod_layout, D, device=dev)
    if n:
        raise DitError(-1, f"self-check failed for {key}: {n} output words differ")
    _checked.add(key)
    return True


def set_first_use_check(enabled: bool) -> None:
    """When enabled, the first call of each runtime key (op, dtype, layouts,
    D, device) through residual_gate_add, rmsnorm_modulate and
    gate_add_rmsnorm_modulate runs ensure_checked first (one synchronisation
    per new key).  Off by default."""
    global _first_use
    _first_use = bool(enabled)


def _first_use_check(op, dtype, glay, mlay, D, dev):
    if _first_use:
        names = {FULL: "full", ROW_BCAST: "bcast"}
        ensure_checked(op, dtype, names[glay], names[mlay], D, device=dev)


# ---------------------------------------------------------------------------
# modulated output in FP8 (OCP E4M3)
# ---------------------------------------------------------------------------

_FP8 = getattr(torch, "float8_e4m3fn", None)


def _fp8_out(out, like, name="out"):
    """The E4M3 output tensor: float8_e4m3fn (allocated if None) or uint8."""
    if out is None:
        return torch.empty(like.shape, dtype=_FP8 or torch.uint8, device=like.device)
    if out.dtype not in tuple(t for t in (_FP8, torch.uint8) if t is not None):
        raise TypeError(f"{name} must be float8_e4m3fn or uint8, got {out.dtype}")
    if tuple(out.shape) != tuple(like.shape):
        raise ValueError(f"{name} must have the shape {tuple(like.shape)}")
    return out


def _quant_scale(qs, dev):
    if (not isinstance(qs, torch.Tensor) or not qs.is_cuda or qs.dtype != torch.float32
            or qs.numel() != 1 or qs.get_device() != dev):
        raise TypeError("quant_scale must be a one-element float32 CUDA tensor on the "
                        "tensors' device (read by the kernel)")
    return qs


def rmsnorm_modulate_fp8(x, scale, shift, quant_scale, eps=1e-6, out=None, stream=None):
    """out = e4m3(fl(y * fl(1 / quant_scale))) with y = rms_norm(x, eps) *
    (1 + scale) + shift in fp32 (dit_rmsnorm_modulate_fp8): OCP E4M3,
    nearest-even, saturating at +-448.  quant_scale: one-element float32
    CUDA tensor.  Returns out (float8_e4m3fn, or the uint8 tensor given)."""
    B, L, D = _shape3(x, "x")
    out = _fp8_out(out, x)
    dev = _cuda(("x", x), ("scale", scale), ("shift", shift), ("out", out))
    dt = _dtype(x, ("scale", scale), ("shift", shift))
    lay = layout_of(scale, B, L, D, "scale")
    if layout_of(shift, B, L, D, "shift") != lay:
        raise ValueError("scale and shift must have the same layout")
    vs = _vector_stride(D, scale, shift) if lay == ROW_BCAST else D
    qs = _quant_scale(quant_scale, dev)
    st = _launch(dev, library().dit_rmsnorm_modulate_fp8, out.data_ptr(), x.data_ptr(),
                 scale.data_ptr(), shift.data_ptr(), B, L, D, float(eps), dt, lay, vs,
                 qs.data_ptr(), _stream(dev, stream))
    check(st, "dit_rmsnorm_modulate_fp8")
    return out


def gate_add_rmsnorm_modulate_fp8(hidden, update, gate, scale, shift, quant_scale, eps=1e-6,
                                  residual_out=None, out=None, stream=None):
    """residual_out = hidden + update * gate (dtype of hidden); out = the E4M3
    modulation of residual_out (dit_gate_add_rmsnorm_modulate_fp8).  Returns
    (residual_out, out)."""
    B, L, D = _shape3(hidden, "hidden")
    if residual_out is None:
        residual_out = torch.empty_like(hidden)
    out = _fp8_out(out, hidden)
    dev = _cuda(("hidden", hidden), ("update", update), ("gate", gate), ("scale", scale),
                ("shift", shift), ("residual_out", residual_out), ("out", out))
    dt = _dtype(hidden, ("update", update), ("gate", gate), ("scale", scale), ("shift", shift),
                ("residual_out", residual_out))
    for name, t in (("update", update), ("residual_out", residual_out)):
        if tuple(t.shape) != (B, L, D):
            raise ValueError(f"{name} must have the shape of hidden")
    glay = layout_of(gate, B, L, D, "gate")
    mlay = layout_of(scale, B, L, D, "scale")
    if layout_of(shift, B, L, D, "shift") != mlay:
        raise ValueError("scale and shift must have the same layout")
    vecs = ([gate] if glay == ROW_BCAST else []) + ([scale, shift] if mlay == ROW_BCAST else [])
    vs = _vector_stride(D, *vecs)
    qs = _quant_scale(quant_scale, dev)
    st = _launch(dev, library().dit_gate_add_rmsnorm_modulate_fp8, residual_out.data_ptr(),
                 out.data_ptr(), hidden.data_ptr(), update.data_ptr(), gate.data_ptr(),
                 scale.data_ptr(), shift.data_ptr(), B, L, D, float(eps), dt, glay, mlay, vs,
                 qs.data_ptr(), _stream(dev, stream))
    check(st, "dit_gate_add_rmsnorm_modulate_fp8")
    return residual_out, out
