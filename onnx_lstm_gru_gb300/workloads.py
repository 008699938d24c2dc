"""Named workloads and seeded synthetic inputs for tests and benchmarks.

This module only describes layers and draws random arrays; it holds none of
the layer's arithmetic.  Inputs are drawn with numpy's PCG64
(``numpy.random.default_rng(seed)``) in float64, in the order X, W, R, B, P,
initial_h, initial_c, sequence_lens (each only when the workload has it), and
then cast to the tensor dtype: float32 and float16 by numpy's
round-to-nearest-even; bfloat16 (which numpy lacks) by rounding to float32
first and then to the 8-bit significand, nearest-even on the float32 bits,
the result kept as float32 arrays whose values are all bfloat16 numbers.  "N(0, s)"
means standard deviation s.  The same arrays feed the CUDA library and the
oracle.

The named workloads are the layer shapes the recurrent-layers page measures
and tests (its bidirectional LSTM 80 x 1 x 256 float32 and the recognizer's
second shape, 48 x 8 x 192 x 96), plus larger layers for the grid and
tensor-core paths.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

from . import Problem


@dataclass
class Workload:
    name: str
    problem: Problem
    seed: int
    x: tuple                 # ("normal", sd) or ("uniform", a)  -> U(-a, a)
    weights: tuple           # W, R, B distribution
    p: Optional[tuple] = None
    init_h: Optional[tuple] = None
    init_c: Optional[tuple] = None
    lens: Optional[str] = None    # None: no sequence_lens; "full": all = seq; "uniform": U{1..seq}
    outputs: tuple = ("Y", "Y_h", "Y_c")


def _draw(rng, dist, shape):
    kind, a = dist
    if kind == "normal":
        return rng.normal(0.0, a, shape)
    if kind == "uniform":
        return rng.uniform(-a, a, shape)
    raise ValueError(kind)


WORKLOADS = {
    "lstm_fwd_s8_b1_i16_h16_f32": Workload(
        "lstm_fwd_s8_b1_i16_h16_f32",
        Problem("lstm", seq=8, batch=1, input=16, hidden=16, direction="forward", dtype="f32", layout=0),
        seed=0, x=("uniform", 0.5), weights=("uniform", 0.5)),
    "bilstm_s80_b1_i256_h256_f32": Workload(
        "bilstm_s80_b1_i256_h256_f32",
        Problem("lstm", seq=80, batch=1, input=256, hidden=256, direction="bidirectional", dtype="f32", layout=0),
        seed=1, x=("normal", 1.0), weights=("uniform", 1.0 / 16), init_h=("normal", 0.1), init_c=("normal", 0.1)),
    "bigru_s128_b8_i512_h512_f16_lbr0": Workload(
        "bigru_s128_b8_i512_h512_f16_lbr0",
        Problem("gru", seq=128, batch=8, input=512, hidden=512, direction="bidirectional", dtype="f16", layout=1,
                linear_before_reset=0),
        seed=2, x=("normal", 1.0), weights=("uniform", 0.044), init_h=("normal", 0.5), lens="uniform",
        outputs=("Y", "Y_h")),
    "bigru_s128_b8_i512_h512_f16_lbr1": Workload(
        "bigru_s128_b8_i512_h512_f16_lbr1",
        Problem("gru", seq=128, batch=8, input=512, hidden=512, direction="bidirectional", dtype="f16", layout=1,
                linear_before_reset=1),
        seed=2, x=("normal", 1.0), weights=("uniform", 0.044), init_h=("normal", 0.5), lens="uniform",
        outputs=("Y", "Y_h")),
    "revlstm_peep_clip_s200_b4_i128_h1024_f32": Workload(
        "revlstm_peep_clip_s200_b4_i128_h1024_f32",
        Problem("lstm", seq=200, batch=4, input=128, hidden=1024, direction="reverse", dtype="f32", layout=0,
                clip=3.0, input_forget=1,
                activations=[("hardsigmoid", 0.2, 0.5), ("scaledtanh", 1.0, 1.0), ("softsign", 0.0, 0.0)]),
        seed=3, x=("normal", 1.0), weights=("uniform", 0.03), p=("uniform", 0.1)),
    "bilstm_s512_b64_i1024_h1024_f16": Workload(
        "bilstm_s512_b64_i1024_h1024_f16",
        Problem("lstm", seq=512, batch=64, input=1024, hidden=1024, direction="bidirectional", dtype="f16",
                layout=0),
        seed=4, x=("normal", 1.0), weights=("uniform", 0.03), lens="full"),
    # the recognizer's second shape (bidirectional LSTM over 48 columns of 8
    # text lines of varying width, 192 features, 96 units), float32 and Half
    "bilstm_s48_b8_i192_h96_f32": Workload(
        "bilstm_s48_b8_i192_h96_f32",
        Problem("lstm", seq=48, batch=8, input=192, hidden=96, direction="bidirectional", dtype="f32", layout=0),
        seed=5, x=("normal", 1.0), weights=("uniform", 0.1), init_h=("normal", 0.1), init_c=("normal", 0.1),
        lens="uniform"),
    # bfloat16 variants of the largest layer and of the recognizer's shape
    "bilstm_s512_b64_i1024_h1024_bf16": Workload(
        "bilstm_s512_b64_i1024_h1024_bf16",
        Problem("lstm", seq=512, batch=64, input=1024, hidden=1024, direction="bidirectional", dtype="bf16",
                layout=0),
        seed=7, x=("normal", 1.0), weights=("uniform", 0.03), lens="full"),
    "bilstm_s48_b8_i192_h96_bf16": Workload(
        "bilstm_s48_b8_i192_h96_bf16",
        Problem("lstm", seq=48, batch=8, input=192, hidden=96, direction="bidirectional", dtype="bf16", layout=0),
        seed=8, x=("normal", 1.0), weights=("uniform", 0.1), init_h=("normal", 0.1), init_c=("normal", 0.1),
        lens="uniform"),
    "bilstm_s48_b8_i192_h96_f16": Workload(
        "bilstm_s48_b8_i192_h96_f16",
        Problem("lstm", seq=48, batch=8, input=192, hidden=96, direction="bidirectional", dtype="f16", layout=0),
        seed=6, x=("normal", 1.0), weights=("uniform", 0.1), init_h=("normal", 0.1), init_c=("normal", 0.1),
        lens="uniform"),
}

# the headline workload: the pages' bidirectional LSTM layer
HEADLINE = "bilstm_s80_b1_i256_h256_f32"


def round_bf16(a) -> np.ndarray:
    """float32 array of the bfloat16 numbers nearest (ties to even) to the
    float32 rounding of ``a`` (finite values)."""
    u = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def cast(a, dtype: str) -> np.ndarray:
    """Values in the tensor dtype: float32, float16, or float32 holding bfloat16 numbers."""
    if dtype in ("f32", "float32"):
        return np.asarray(a).astype(np.float32)
    if dtype in ("bf16", "bfloat16"):
        return round_bf16(a)
    return np.asarray(a).astype(np.float16)


def make_inputs(w: Workload, problem: Optional[Problem] = None) -> dict:
    """Draw the workload's inputs (numpy arrays in the tensor dtype, see
    ``cast``; lengths int32).  ``problem`` may override sizes for scaled-down
    variants."""
    pr = problem or w.problem
    rng = np.random.default_rng(w.seed)
    shp = pr.shapes()
    out = {}
    out["X"] = cast(_draw(rng, w.x, shp["X"]), pr.dtype)
    out["W"] = cast(_draw(rng, w.weights, shp["W"]), pr.dtype)
    out["R"] = cast(_draw(rng, w.weights, shp["R"]), pr.dtype)
    out["B"] = cast(_draw(rng, w.weights, shp["B"]), pr.dtype)
    if w.p is not None and pr.cell == "lstm":
        out["P"] = cast(_draw(rng, w.p, shp["P"]), pr.dtype)
    if w.init_h is not None:
        out["initial_h"] = cast(_draw(rng, w.init_h, shp["initial_h"]), pr.dtype)
    if w.init_c is not None and pr.cell == "lstm":
        out["initial_c"] = cast(_draw(rng, w.init_c, shp["initial_c"]), pr.dtype)
    if w.lens == "full":
        out["sequence_lens"] = np.full((pr.batch,), pr.seq, dtype=np.int32)
    elif w.lens == "uniform":
        out["sequence_lens"] = rng.integers(1, pr.seq + 1, size=pr.batch).astype(np.int32)
    return out


def algorithmic_flops(pr: Problem, lens=None) -> float:
    """Projection 2*S*N*I*G*H*D (every step, as the method forms it) plus
    recurrence 2*(sum of lengths)*G*H*H*D."""
    D, G = pr.num_directions, pr.gates
    total_len = pr.seq * pr.batch if lens is None else int(np.clip(np.asarray(lens), 0, pr.seq).sum())
    return 2.0 * pr.seq * pr.batch * pr.input * G * pr.hidden * D + 2.0 * total_len * G * pr.hidden * pr.hidden * D


def compulsory_bytes(pr: Problem, present: dict) -> float:
    """Inputs read once plus requested outputs written once (no scratch)."""
    eb = 4 if pr.dtype in ("f32", "float32") else 2
    shp = pr.shapes()
    total = 0
    for name, v in present.items():
        n = int(np.prod(shp[name]))
        total += n * (4 if name == "sequence_lens" else eb)
    return float(total)
