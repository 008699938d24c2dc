"""GB300-native forward pass of ONNX recurrent layers (LSTM, GRU, RNN).

A thin Python binding over the C ABI in ``include/rk.h`` (``librk.so``, built
in-tree by ``build()``).  The functions ``rk_create``, ``rk_encode``, ... carry
the C names and only marshal arguments; every step of a layer runs in the
library's CUDA kernels.  ``RecurrentLayer`` is a convenience wrapper that takes
torch CUDA tensors (torch supplies device memory and streams only).

There is no CPU path: if the library is missing the binding raises.
"""
from __future__ import annotations

import ctypes
import os
import struct
from dataclasses import dataclass, field
from typing import Optional, Sequence

from ._build import LIB as _LIB_PATH, build  # noqa: F401

__all__ = [
    "build", "load", "Problem", "RecurrentLayer", "RkError",
    "rk_create", "rk_destroy", "rk_encode", "rk_encode_host", "rk_validate", "rk_xw_length",
    "rk_state_length", "rk_status_poll", "rk_set_wait_limit", "rk_last_error", "rk_launch_count",
    "rk_describe_plan", "rk_version", "rk_selftest_timeout", "rk_set_profiling", "rk_last_timings",
    "rk_encode_noalloc", "rk_validate_lengths", "RK_OK", "RK_ERR_SHAPE", "RK_ERR_UNSUPPORTED", "RK_ERR_CUDA", "RK_ERR_TIMEOUT", "RK_ERR_OOM", "RK_ERR_ARG",
    "RK_FORCE_SIMT_PROJECTION", "RK_FORCE_GRID_STEP", "RK_FORCE_GENERAL_STEP", "RK_FORCE_SIMT_STEP",
    "RK_SEPARATE_PROJECTION", "RK_PREFER_TENSOR_STEP", "EXPORTED_SYMBOLS",
]

RK_OK, RK_ERR_SHAPE, RK_ERR_UNSUPPORTED, RK_ERR_CUDA, RK_ERR_TIMEOUT, RK_ERR_OOM, RK_ERR_ARG = range(7)
RK_FORCE_SIMT_PROJECTION = 1
RK_FORCE_GRID_STEP = 2
RK_FORCE_GENERAL_STEP = 4
RK_FORCE_SIMT_STEP = 8
RK_SEPARATE_PROJECTION = 16
RK_PREFER_TENSOR_STEP = 32
CELLS = {"lstm": 0, "gru": 1, "rnn": 2}
DIRECTIONS = {"forward": 0, "reverse": 1, "bidirectional": 2}
DTYPES = {"f32": 0, "float32": 0, "f16": 1, "float16": 1, "half": 1, "bf16": 2, "bfloat16": 2}
ACTIVATIONS = {
    "sigmoid": 0, "tanh": 1, "relu": 2, "affine": 3, "leakyrelu": 4, "thresholdedrelu": 5,
    "scaledtanh": 6, "hardsigmoid": 7, "elu": 8, "softsign": 9, "softplus": 10,
}
GATES = {"lstm": 4, "gru": 3, "rnn": 1}
ACTS_PER_DIR = {"lstm": 3, "gru": 2, "rnn": 1}

EXPORTED_SYMBOLS = [
    "rk_version", "rk_create", "rk_destroy", "rk_xw_length", "rk_state_length", "rk_validate",
    "rk_encode", "rk_encode_host", "rk_status_poll", "rk_set_wait_limit", "rk_last_error",
    "rk_launch_count", "rk_describe_plan", "rk_selftest_timeout", "rk_set_profiling", "rk_last_timings",
    "rk_encode_noalloc", "rk_validate_lengths",
]


class RkError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"rk error {code}: {message}")
        self.code = code
        self.message = message


class rk_activation(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("alpha", ctypes.c_float), ("beta", ctypes.c_float)]


class rk_problem(ctypes.Structure):
    _fields_ = [
        ("cell", ctypes.c_int32), ("direction", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("layout", ctypes.c_int32),
        ("seq", ctypes.c_int64), ("batch", ctypes.c_int64), ("input", ctypes.c_int64),
        ("hidden", ctypes.c_int64),
        ("clip", ctypes.c_float), ("input_forget", ctypes.c_int32),
        ("linear_before_reset", ctypes.c_int32), ("num_acts", ctypes.c_int32),
        ("act", rk_activation * 6), ("max_length", ctypes.c_int64),
    ]


class rk_tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("offset", ctypes.c_int64), ("length", ctypes.c_int64)]


_OPERAND_NAMES = ["X", "W", "R", "B", "sequence_lens", "initial_h", "initial_c", "P", "Y", "Y_h", "Y_c"]


class rk_operands(ctypes.Structure):
    _fields_ = [(n, rk_tensor) for n in _OPERAND_NAMES]


_OPERAND_INDEX = {n: i for i, n in enumerate(_OPERAND_NAMES)}
# rk_operands as raw bytes: (pointer, offset, length) per operand, packed in
# one call instead of a ctypes object per operand (the binding's per-layer
# host cost)
_OPERANDS_PACK = struct.Struct("=" + "Qqq" * len(_OPERAND_NAMES))
assert _OPERANDS_PACK.size == ctypes.sizeof(rk_operands)


def _pack_operands(entries) -> rk_operands:
    """rk_operands from (name, pointer, element offset, length) entries."""
    vals = [0] * (3 * len(_OPERAND_NAMES))
    for name, ptr, off, n in entries:
        i = _OPERAND_INDEX.get(name)
        if i is None:
            raise KeyError(name)
        vals[3 * i], vals[3 * i + 1], vals[3 * i + 2] = ptr, off, n
    return rk_operands.from_buffer_copy(_OPERANDS_PACK.pack(*vals))


class rk_scratch(ctypes.Structure):
    _fields_ = [("xw", ctypes.c_void_p), ("xw_offset", ctypes.c_int64), ("xw_length", ctypes.c_int64),
                ("state", ctypes.c_void_p), ("state_offset", ctypes.c_int64),
                ("state_length", ctypes.c_int64)]


_lib = None


def load(path: Optional[str] = None):
    """Load librk.so (built by ``build()``).  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or _LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"librk.so not built ({path} missing): run onnx_lstm_gru_gb300.build() first; "
                           "there is no CPU fallback")
    lib = ctypes.CDLL(path)
    H = ctypes.c_void_p
    P = ctypes.POINTER(rk_problem)
    O = ctypes.POINTER(rk_operands)
    sig = {
        "rk_version": (ctypes.c_int32, []),
        "rk_create": (ctypes.c_int32, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint32]),
        "rk_destroy": (ctypes.c_int32, [H]),
        "rk_xw_length": (ctypes.c_int64, [P]),
        "rk_state_length": (ctypes.c_int64, [P]),
        "rk_validate": (ctypes.c_int32, [H, P, O]),
        "rk_encode": (ctypes.c_int32, [H, P, O, ctypes.POINTER(rk_scratch), ctypes.c_void_p]),
        "rk_encode_host": (ctypes.c_int32, [H, P, O, ctypes.c_void_p]),
        "rk_status_poll": (ctypes.c_int32, [H, ctypes.c_void_p]),
        "rk_set_wait_limit": (ctypes.c_int32, [H, ctypes.c_int64]),
        "rk_last_error": (ctypes.c_char_p, [H]),
        "rk_launch_count": (ctypes.c_uint64, [H]),
        "rk_describe_plan": (ctypes.c_int32, [H, P, ctypes.c_char_p, ctypes.c_int64]),
        "rk_selftest_timeout": (ctypes.c_int32, [H, ctypes.c_void_p, ctypes.c_int64]),
        "rk_set_profiling": (ctypes.c_int32, [H, ctypes.c_int32]),
        "rk_encode_noalloc": (ctypes.c_int32, [H, P, O, ctypes.c_void_p]),
        "rk_validate_lengths": (ctypes.c_int32, [H, P, ctypes.POINTER(ctypes.c_int32), ctypes.c_int64]),
        "rk_last_timings": (ctypes.c_int32, [H, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


# ---- thin wrappers with the C names (argument marshalling only) ----------------------------

def rk_version() -> int:
    return load().rk_version()


def rk_create(flags: int = 0) -> int:
    h = ctypes.c_void_p()
    st = load().rk_create(ctypes.byref(h), flags)
    if st != RK_OK:
        raise RkError(st, "rk_create failed")
    return h.value


def rk_destroy(handle: int) -> int:
    return load().rk_destroy(handle)


def rk_xw_length(problem: rk_problem) -> int:
    return load().rk_xw_length(ctypes.byref(problem))


def rk_state_length(problem: rk_problem) -> int:
    return load().rk_state_length(ctypes.byref(problem))


def rk_validate(handle: int, problem: rk_problem, ops: rk_operands) -> int:
    return load().rk_validate(handle, ctypes.byref(problem), ctypes.byref(ops))


def rk_validate_lengths(handle: int, problem: rk_problem, lens) -> int:
    """Host check of sequence_lens (a sequence of ints or an int32 array)."""
    import numpy as np
    a = np.ascontiguousarray(np.asarray(lens, dtype=np.int32))
    return load().rk_validate_lengths(handle, ctypes.byref(problem),
                                      a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), a.size)


def rk_encode(handle: int, problem: rk_problem, ops: rk_operands, scratch: Optional[rk_scratch],
              stream: int) -> int:
    return load().rk_encode(handle, ctypes.byref(problem), ctypes.byref(ops),
                            ctypes.byref(scratch) if scratch is not None else None, stream)


def rk_encode_noalloc(handle: int, problem: rk_problem, ops: rk_operands, stream: int) -> int:
    """rk_encode with the scratch in the library's fixed 16 MiB device array:
    for callers that cannot allocate device memory.  No allocation happens."""
    return load().rk_encode_noalloc(handle, ctypes.byref(problem), ctypes.byref(ops), stream)


def rk_encode_host(handle: int, problem: rk_problem, ops: rk_operands, stream: int) -> int:
    return load().rk_encode_host(handle, ctypes.byref(problem), ctypes.byref(ops), stream)


def rk_status_poll(handle: int, stream: int) -> int:
    return load().rk_status_poll(handle, stream)


def rk_set_wait_limit(handle: int, limit_ns: int) -> int:
    return load().rk_set_wait_limit(handle, limit_ns)


def rk_last_error(handle: int) -> str:
    return load().rk_last_error(handle).decode()


def rk_launch_count(handle: int) -> int:
    return load().rk_launch_count(handle)


def rk_selftest_timeout(handle: int, stream: int, timeout_ns: int) -> int:
    return load().rk_selftest_timeout(handle, stream, timeout_ns)


def rk_set_profiling(handle: int, enabled: bool) -> int:
    return load().rk_set_profiling(handle, 1 if enabled else 0)


def rk_last_timings(handle: int):
    """(projection_ms, step_ms) of the most recent encode; raises on error."""
    a, b = ctypes.c_float(), ctypes.c_float()
    st = load().rk_last_timings(handle, ctypes.byref(a), ctypes.byref(b))
    if st != RK_OK:
        raise RkError(st, rk_last_error(handle))
    return a.value, b.value


def rk_describe_plan(handle: int, problem: rk_problem) -> str:
    buf = ctypes.create_string_buffer(512)
    st = load().rk_describe_plan(handle, ctypes.byref(problem), buf, 512)
    if st != RK_OK:
        raise RkError(st, rk_last_error(handle))
    return buf.value.decode()


# ---- problem description ---------------------------------------------------------------------

@dataclass
class Problem:
    """A recurrent layer (mirrors rk_problem).  ``activations`` is None for the
    ONNX defaults, else a list of (name, alpha, beta), direction-major."""
    cell: str
    seq: int
    batch: int
    input: int
    hidden: int
    direction: str = "forward"
    dtype: str = "f32"
    layout: int = 0
    clip: float = 0.0
    input_forget: int = 0
    linear_before_reset: int = 0
    activations: Optional[Sequence] = None
    max_length: int = 0

    @property
    def num_directions(self) -> int:
        return 2 if self.direction == "bidirectional" else 1

    @property
    def gates(self) -> int:
        return GATES[self.cell]

    def to_c(self) -> rk_problem:
        p = rk_problem()
        p.cell = CELLS[self.cell]
        p.direction = DIRECTIONS[self.direction]
        p.dtype = DTYPES[self.dtype]
        p.layout = int(self.layout)
        p.seq, p.batch, p.input, p.hidden = int(self.seq), int(self.batch), int(self.input), int(self.hidden)
        p.clip = float(self.clip or 0.0)
        p.input_forget = int(self.input_forget)
        p.linear_before_reset = int(self.linear_before_reset)
        acts = list(self.activations or [])
        p.num_acts = len(acts)
        for i, (n, a, b) in enumerate(acts):
            p.act[i].kind = ACTIVATIONS[str(n).lower()]
            p.act[i].alpha = float(a)
            p.act[i].beta = float(b)
        p.max_length = int(self.max_length)
        return p

    def shapes(self) -> dict:
        D, G, S, N, I, H = self.num_directions, self.gates, self.seq, self.batch, self.input, self.hidden
        st = (D, N, H) if self.layout == 0 else (N, D, H)
        return {
            "X": (S, N, I) if self.layout == 0 else (N, S, I),
            "W": (D, G * H, I), "R": (D, G * H, H), "B": (D, 2 * G * H), "sequence_lens": (N,),
            "initial_h": st, "initial_c": st, "P": (D, 3 * H),
            "Y": (S, D, N, H) if self.layout == 0 else (N, S, D, H), "Y_h": st, "Y_c": st,
        }


def torch_dtype(dtype: str):
    """The torch element type of a problem's tensors (all but sequence_lens)."""
    import torch
    return (torch.float32, torch.float16, torch.bfloat16)[DTYPES[dtype]]


def operands_from_tensors(_dtype=None, **tensors) -> rk_operands:
    """rk_operands from torch tensors (device memory, contiguous).  A value may
    be a tensor or a (tensor, element_offset) pair; the tensor is then the
    whole buffer and the operand starts ``element_offset`` elements in.  With
    _dtype given, every tensor but sequence_lens (int32) must have it."""
    import torch
    entries = []
    for name, v in tensors.items():
        if name not in _OPERAND_INDEX:
            raise KeyError(name)
        if v is None:
            continue
        t, off = (v[0], int(v[1])) if isinstance(v, tuple) else (v, 0)
        if t is None:
            continue
        if _dtype is not None:
            need = torch.int32 if name == "sequence_lens" else _dtype
            if t.dtype != need:
                raise TypeError(f"{name}: expected {need}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError("operands must be contiguous")
        entries.append((name, t.data_ptr(), off, t.numel()))
    return _pack_operands(entries)


class RecurrentLayer:
    """Owns an rk handle.  ``encode`` enqueues a layer on the current torch
    stream (or ``stream``) for caller-allocated torch CUDA tensors; ``forward``
    allocates the outputs.  No CPU path exists."""

    def __init__(self, flags: int = 0):
        load()
        self.handle = rk_create(flags)

    def close(self):
        if getattr(self, "handle", None):
            rk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st: int):
        if st != RK_OK:
            raise RkError(st, rk_last_error(self.handle))

    def plan(self, problem: Problem) -> str:
        return rk_describe_plan(self.handle, problem.to_c())

    def launches(self) -> int:
        return rk_launch_count(self.handle)

    def set_wait_limit(self, ns: int):
        self._check(rk_set_wait_limit(self.handle, int(ns)))

    def poll(self, stream=None):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        self._check(rk_status_poll(self.handle, s.cuda_stream))

    def encode(self, problem: Problem, stream=None, scratch: Optional[rk_scratch] = None, **tensors):
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        ops = operands_from_tensors(torch_dtype(problem.dtype), **tensors)
        self._check(rk_encode(self.handle, problem.to_c(), ops, scratch, s.cuda_stream))

    def encode_host(self, problem: Problem, stream=None, **arrays):
        """Host-buffer entry point: numpy arrays (or CPU tensors) in and out;
        the library copies to and from the device and synchronises."""
        import numpy as np
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        entries = []
        for name, a in arrays.items():
            if a is None:
                continue
            if isinstance(a, torch.Tensor):
                if a.is_cuda or not a.is_contiguous():
                    raise ValueError(f"{name}: host tensors must be contiguous CPU tensors")
                ptr, n = a.data_ptr(), a.numel()
            else:
                if not (isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"]):
                    raise ValueError(f"{name}: host arrays must be C-contiguous numpy arrays")
                ptr, n = a.ctypes.data, a.size
            entries.append((name, ptr, 0, n))
        self._check(rk_encode_host(self.handle, problem.to_c(), _pack_operands(entries), s.cuda_stream))

    def forward(self, problem: Problem, X, W, R, B=None, sequence_lens=None, initial_h=None,
                initial_c=None, P=None, want=("Y", "Y_h", "Y_c"), stream=None):
        import torch
        dt = torch_dtype(problem.dtype)
        shp = problem.shapes()
        outs = {}
        for name in want:
            if name == "Y_c" and problem.cell != "lstm":
                continue
            outs[name] = torch.empty(shp[name], dtype=dt, device=X.device)
        self.encode(problem, stream=stream, X=X, W=W, R=R, B=B, sequence_lens=sequence_lens,
                    initial_h=initial_h, initial_c=initial_c, P=P, **outs)
        return outs
