"""CPU oracle of the ONNX recurrent layer forward pass (double precision).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library in ``onnx_lstm_gru_gb300`` and imports nothing
from it; the library never imports this package.

The arithmetic lives in ``rk_oracle.c`` (plain C, single-threaded, every value
a double, sums in increasing index order), which follows the web page
"Recurrent layers" (sections "How a layer runs", "Arithmetic and determinism"
and "Semantics") and takes the eleven activation formulas from the ONNX
operator definitions, since the page only names them.  This module compiles it
with gcc, widens inputs exactly to float64 and marshals arguments.

Pins (tests/test_oracle_pins.py) tie it to things other than itself: the
Getting-started Gemm example of the pages, closed forms at hidden size 1,
torch.nn.LSTM / GRU / RNN in float64 on the CPU for the default activations,
torch.nn.functional for the activations, and invariants (reverse vs
time-reversed forward, bidirectional vs its two halves, zeroing past the
length, layout 1 vs layout 0).

Problem descriptions are duck-typed: any object (or dict) with the fields
``cell`` ('lstm'|'gru'|'rnn'), ``direction`` ('forward'|'reverse'|
'bidirectional'), ``layout``, ``seq``, ``batch``, ``input``, ``hidden``,
``clip``, ``input_forget``, ``linear_before_reset`` and ``activations``
(None for the ONNX defaults, else a list of (name, alpha, beta) per slot,
direction-major).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rk_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

CELLS = {"lstm": 0, "gru": 1, "rnn": 2}
DIRECTIONS = {"forward": 0, "reverse": 1, "bidirectional": 2}
ACTIVATIONS = {
    "sigmoid": 0, "tanh": 1, "relu": 2, "affine": 3, "leakyrelu": 4,
    "thresholdedrelu": 5, "scaledtanh": 6, "hardsigmoid": 7, "elu": 8,
    "softsign": 9, "softplus": 10,
}
GATES = {"lstm": 4, "gru": 3, "rnn": 1}
ACTS_PER_DIR = {"lstm": 3, "gru": 2, "rnn": 1}
DEFAULT_ACTS = {
    "lstm": [("sigmoid", 0.0, 0.0), ("tanh", 0.0, 0.0), ("tanh", 0.0, 0.0)],
    "gru": [("sigmoid", 0.0, 0.0), ("tanh", 0.0, 0.0)],
    "rnn": [("tanh", 0.0, 0.0)],
}


class _Problem(ctypes.Structure):
    _fields_ = [
        ("cell", ctypes.c_int32), ("direction", ctypes.c_int32), ("layout", ctypes.c_int32),
        ("seq", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("input", ctypes.c_int64), ("hidden", ctypes.c_int64),
        ("clip", ctypes.c_double),
        ("input_forget", ctypes.c_int32), ("linear_before_reset", ctypes.c_int32),
        ("act_kind", ctypes.c_int32 * 6),
        ("act_alpha", ctypes.c_double * 6), ("act_beta", ctypes.c_double * 6),
    ]


def build(force: bool = False) -> str:
    """Compile rk_oracle.c into _build/liboracle.so with gcc (no fast-math,
    no FMA contraction, portable flags) and return the path."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        os.makedirs(_BUILD_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.rko_activation.restype = ctypes.c_double
        lib.rko_activation.argtypes = [ctypes.c_int32, ctypes.c_double, ctypes.c_double, ctypes.c_double]
        lib.rko_projection.restype = None
        lib.rko_projection.argtypes = [ctypes.c_int64] * 4 + [dp, dp, dp]
        lib.rko_layer.restype = ctypes.c_int
        lib.rko_layer.argtypes = [ctypes.POINTER(_Problem), dp, dp, dp, dp,
                                  ctypes.POINTER(ctypes.c_int32), dp, dp, dp, dp, dp, dp]
        _lib = lib
    return _lib


def _get(spec, name, default=None):
    if isinstance(spec, dict):
        return spec.get(name, default)
    return getattr(spec, name, default)


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a), dtype=np.float64)


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def activation(name: str, alpha: float, beta: float, x: float) -> float:
    """One ONNX activation, evaluated by the oracle in double."""
    return _load().rko_activation(ACTIVATIONS[name.lower()], alpha, beta, float(x))


def projection(X, W):
    """Xw[d] = X . W[d]^T.  X [M, K], W [D, N, K] (or [N, K]); returns float64
    [D, M, N] (or [M, N] when W is 2-D)."""
    X = _f64(X)
    W = _f64(W)
    squeeze = W.ndim == 2
    if squeeze:
        W = W[None]
    D, N, K = W.shape
    M = X.shape[0]
    assert X.shape == (M, K)
    out = np.zeros((D, M, N), dtype=np.float64)
    _load().rko_projection(D, M, N, K, _ptr(X), _ptr(W), _ptr(out))
    return out[0] if squeeze else out


def resolved_activations(spec):
    cell = _get(spec, "cell")
    D = 2 if _get(spec, "direction") == "bidirectional" else 1
    acts = _get(spec, "activations")
    if not acts:
        acts = DEFAULT_ACTS[cell] * D
    if len(acts) != ACTS_PER_DIR[cell] * D:
        raise ValueError(f"{cell}: expected {ACTS_PER_DIR[cell] * D} activations, got {len(acts)}")
    return [(str(n).lower(), float(a), float(b)) for (n, a, b) in acts]


def layer(spec, X, W, R, B=None, sequence_lens=None, initial_h=None, initial_c=None, P=None):
    """Run the whole layer in double.  Returns dict(Y=..., Y_h=..., Y_c=...)
    (Y_c only for an LSTM), float64 numpy arrays in the layout of ``spec``."""
    cell = _get(spec, "cell")
    direction = _get(spec, "direction")
    layout = int(_get(spec, "layout", 0))
    S, NB = int(_get(spec, "seq")), int(_get(spec, "batch"))
    I, H = int(_get(spec, "input")), int(_get(spec, "hidden"))
    D = 2 if direction == "bidirectional" else 1
    G = GATES[cell]
    prob = _Problem()
    prob.cell = CELLS[cell]
    prob.direction = DIRECTIONS[direction]
    prob.layout = layout
    prob.seq, prob.batch, prob.input, prob.hidden = S, NB, I, H
    clip = _get(spec, "clip", 0.0)
    prob.clip = float(clip) if clip is not None else 0.0
    prob.input_forget = int(bool(_get(spec, "input_forget", 0)))
    prob.linear_before_reset = int(bool(_get(spec, "linear_before_reset", 0)))
    for i, (n, a, b) in enumerate(resolved_activations(spec)):
        prob.act_kind[i] = ACTIVATIONS[n]
        prob.act_alpha[i] = a
        prob.act_beta[i] = b

    Xd = _f64(X).reshape(-1)
    Wd = _f64(W).reshape(-1)
    Rd = _f64(R).reshape(-1)
    assert Xd.size == S * NB * I and Wd.size == D * G * H * I and Rd.size == D * G * H * H
    Bd = _f64(B).reshape(-1) if B is not None else None
    Pd = _f64(P).reshape(-1) if P is not None else None
    hd = _f64(initial_h).reshape(-1) if initial_h is not None else None
    cd = _f64(initial_c).reshape(-1) if initial_c is not None else None
    lens = None
    if sequence_lens is not None:
        lens = np.ascontiguousarray(np.asarray(sequence_lens), dtype=np.int32).reshape(-1)
        assert lens.size == NB
    if layout == 0:
        yshape, sshape = (S, D, NB, H), (D, NB, H)
    else:
        yshape, sshape = (NB, S, D, H), (NB, D, H)
    Y = np.zeros(yshape, dtype=np.float64)
    Yh = np.zeros(sshape, dtype=np.float64)
    Yc = np.zeros(sshape, dtype=np.float64) if cell == "lstm" else None
    rc = _load().rko_layer(
        ctypes.byref(prob), _ptr(Xd), _ptr(Wd), _ptr(Rd), _ptr(Bd),
        lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if lens is not None else None,
        _ptr(hd), _ptr(cd), _ptr(Pd), _ptr(Y), _ptr(Yh), _ptr(Yc))
    if rc != 0:
        raise MemoryError("oracle: out of host memory")
    out = {"Y": Y, "Y_h": Yh}
    if Yc is not None:
        out["Y_c"] = Yc
    return out
