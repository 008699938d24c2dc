"""Host-side tests of the C ABI: no GPU needed, no compute call made.

The library must load, export every function include/rk.h declares, and reject
bad problems and operands on the host with an error that names the cell and
the argument (the recurrent-layers page: "Sizes, offsets and shapes are checked
in safe arithmetic before anything is recorded").
"""
import ctypes
import os
import re

import numpy as np
import pytest

import onnx_lstm_gru_gb300 as rk
from onnx_lstm_gru_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    rk.build()
    return rk.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "rk.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rk_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(rk.EXPORTED_SYMBOLS) == names
    assert rk.rk_version() == 100


class Host:
    """Fake device buffers: only pointer values and lengths matter to validation."""

    def __init__(self, problem):
        self.problem = problem
        self.bufs = {}

    def ops(self, **override):
        shp = self.problem.shapes()
        ops = rk.rk_operands()
        names = ["X", "W", "R", "B", "Y", "Y_h"]
        if self.problem.cell == "lstm":
            names += ["Y_c"]
        for n in names:
            size = int(np.prod(shp[n]))
            setattr(ops, n, rk.rk_tensor(0x10000 + 0x100000 * len(self.bufs), 0, size))
            self.bufs[n] = size
        for n, v in override.items():
            setattr(ops, n, v)
        return ops


@pytest.fixture
def handle(lib):
    h = rk.rk_create(0)
    yield h
    rk.rk_destroy(h)


def validate(h, problem, ops):
    st = rk.rk_validate(h, problem.to_c(), ops)
    return st, rk.rk_last_error(h)


def test_valid_problems_pass(handle):
    for w in workloads.WORKLOADS.values():
        st, msg = validate(handle, w.problem, Host(w.problem).ops())
        assert st == rk.RK_OK, (w.name, msg)


def test_offset_past_buffer_names_cell_and_argument(handle):
    p = rk.Problem("lstm", seq=4, batch=2, input=3, hidden=512, direction="bidirectional")
    host = Host(p)
    bad = rk.rk_tensor(0x9000, 7, 2 * 2 * 512 + 6)  # offset 7 + 2048 > 2054
    st, msg = validate(handle, p, host.ops(initial_h=bad))
    assert st == rk.RK_ERR_SHAPE
    assert msg.startswith("LSTM: initial_h:") and "offset 7" in msg and "2048" in msg
    st, msg = validate(handle, p, host.ops(X=rk.rk_tensor(0x9000, -1, 10 ** 6)))
    assert st == rk.RK_ERR_SHAPE and "LSTM: X: negative offset" in msg
    st, msg = validate(handle, p, host.ops(W=rk.rk_tensor(None, 0, 0)))
    assert st == rk.RK_ERR_SHAPE and "W: required" in msg


@pytest.mark.parametrize("cell,field,msg", [
    ("gru", "P", "GRU: P: peepholes exist only for an LSTM"),
    ("rnn", "initial_c", "RNN: initial_c: exists only for an LSTM"),
    ("gru", "Y_c", "GRU: Y_c: exists only for an LSTM"),
])
def test_lstm_only_operands_rejected(handle, cell, field, msg):
    p = rk.Problem(cell, seq=2, batch=1, input=2, hidden=4)
    ops = Host(p).ops(**{field: rk.rk_tensor(0x5000, 0, 10 ** 6)})
    st, m = validate(handle, p, ops)
    assert st == rk.RK_ERR_SHAPE and m == msg


def test_options_illegal_for_cell(handle):
    st, m = validate(handle, rk.Problem("gru", 2, 1, 2, 4, input_forget=1), Host(rk.Problem("gru", 2, 1, 2, 4)).ops())
    assert st == rk.RK_ERR_SHAPE and m.startswith("GRU: input_forget")
    st, m = validate(handle, rk.Problem("lstm", 2, 1, 2, 4, linear_before_reset=1),
                     Host(rk.Problem("lstm", 2, 1, 2, 4)).ops())
    assert st == rk.RK_ERR_SHAPE and m.startswith("LSTM: linear_before_reset")
    p = rk.Problem("rnn", 2, 1, 2, 4, activations=[("tanh", 0, 0), ("relu", 0, 0)])
    st, m = validate(handle, p, Host(p).ops())
    assert st == rk.RK_ERR_SHAPE and "activations: expected 0 or 1, got 2" in m
    p = rk.Problem("rnn", 2, 1, 2, 4)
    c = p.to_c()
    c.num_acts = 1
    c.act[0].kind = 11
    st = rk.rk_validate(handle, c, Host(p).ops())
    assert st == rk.RK_ERR_SHAPE and "unknown kind 11" in rk.rk_last_error(handle)
    for bad in [dict(layout=2), dict(seq=-1), dict(max_length=5), dict(dtype=3), dict(dtype=-1)]:
        q = rk.Problem("lstm", 2, 1, 2, 4)
        cq = q.to_c()
        for k, v in bad.items():
            setattr(cq, k, v)
        assert rk.rk_validate(handle, cq, Host(q).ops()) == rk.RK_ERR_SHAPE
    # max_length below seq needs sequence_lens
    q = rk.Problem("lstm", 5, 1, 2, 4, max_length=3)
    assert validate(handle, q, Host(q).ops())[0] == rk.RK_ERR_SHAPE
    ops = Host(q).ops(sequence_lens=rk.rk_tensor(0x7000, 0, 1))
    assert validate(handle, q, ops)[0] == rk.RK_OK


def test_overflow_is_caught_in_64bit(handle):
    p = rk.Problem("lstm", seq=2 ** 31 - 1, batch=2 ** 31 - 1, input=2 ** 31 - 1, hidden=4)
    st = rk.rk_validate(handle, p.to_c(), rk.rk_operands())
    assert st == rk.RK_ERR_SHAPE and "overflow" in rk.rk_last_error(handle)
    assert rk.rk_xw_length(p.to_c()) == -1


def test_null_arguments():
    lib = rk.load()
    assert lib.rk_validate(None, None, None) == rk.RK_ERR_ARG
    h = rk.rk_create(0)
    try:
        assert lib.rk_validate(h, None, None) == rk.RK_ERR_ARG
        p = rk.Problem("lstm", 2, 1, 2, 4)
        assert lib.rk_validate(h, ctypes.byref(p.to_c()), None) == rk.RK_ERR_ARG
        assert rk.rk_set_wait_limit(h, 0) == rk.RK_ERR_ARG
        assert rk.rk_launch_count(h) == 0
        assert rk.rk_status_poll(h, 0) == rk.RK_OK  # nothing ran yet
    finally:
        rk.rk_destroy(h)
    assert lib.rk_destroy(None) == rk.RK_OK


def test_host_length_check(handle):
    """rk_validate_lengths: every length in [0, seq] (and [0, max_length]
    when set), one per batch row; messages name the cell, row and value."""
    p = rk.Problem("gru", seq=10, batch=4, input=3, hidden=8)
    assert rk.rk_validate_lengths(handle, p.to_c(), [10, 0, 3, 7]) == rk.RK_OK
    assert rk.rk_validate_lengths(handle, p.to_c(), [10, -1, 3, 7]) == rk.RK_ERR_SHAPE
    assert "GRU: sequence_lens[1] = -1 outside [0, 10]" in rk.rk_last_error(handle)
    assert rk.rk_validate_lengths(handle, p.to_c(), [10, 2, 11, 7]) == rk.RK_ERR_SHAPE
    assert "sequence_lens[2] = 11" in rk.rk_last_error(handle)
    assert rk.rk_validate_lengths(handle, p.to_c(), [1, 2, 3]) == rk.RK_ERR_SHAPE
    assert "3 values for batch 4" in rk.rk_last_error(handle)
    q = rk.Problem("lstm", seq=10, batch=2, input=3, hidden=8, max_length=6)
    assert rk.rk_validate_lengths(handle, q.to_c(), [6, 0]) == rk.RK_OK
    assert rk.rk_validate_lengths(handle, q.to_c(), [7, 0]) == rk.RK_ERR_SHAPE
    assert "(max_length)" in rk.rk_last_error(handle)
    bad = rk.Problem("lstm", seq=10, batch=2, input=3, hidden=8, max_length=11)
    assert rk.rk_validate_lengths(handle, bad.to_c(), [1, 1]) == rk.RK_ERR_SHAPE  # the problem itself
    lib = rk.load()
    assert lib.rk_validate_lengths(None, ctypes.byref(p.to_c()), None, 0) == rk.RK_ERR_ARG
    assert lib.rk_validate_lengths(handle, ctypes.byref(p.to_c()), None, 4) == rk.RK_ERR_ARG
    assert rk.rk_validate_lengths(handle, rk.Problem("rnn", seq=5, batch=0, input=1, hidden=2).to_c(), []) == rk.RK_OK


def test_operand_table_packing():
    """The binding packs rk_operands in one call: every field lands where the
    C struct has it, tuples carry an element offset, dtypes are checked."""
    import torch
    t = {n: torch.zeros(3 + i, dtype=torch.int32 if n == "sequence_lens" else torch.float32)
         for i, n in enumerate(rk._OPERAND_NAMES)}
    ops = rk.operands_from_tensors(torch.float32, **{n: ((v, 2) if n == "R" else v) for n, v in t.items()})
    for i, n in enumerate(rk._OPERAND_NAMES):
        f = getattr(ops, n)
        assert f.ptr == t[n].data_ptr() and f.length == 3 + i and f.offset == (2 if n == "R" else 0), n
    partial = rk.operands_from_tensors(X=t["X"], Y_c=None)
    assert partial.X.ptr == t["X"].data_ptr() and partial.W.ptr is None and partial.Y_c.ptr is None
    with pytest.raises(TypeError):
        rk.operands_from_tensors(torch.float16, X=t["X"])
    with pytest.raises(KeyError):
        rk.operands_from_tensors(Q=t["X"])
    with pytest.raises(ValueError):
        rk.operands_from_tensors(X=torch.zeros(4, 4).t())


def test_scratch_lengths():
    p = rk.Problem("lstm", seq=80, batch=1, input=256, hidden=256, direction="bidirectional")
    assert rk.rk_xw_length(p.to_c()) == 2 * 80 * 1 * 4 * 256
    # header, team counters (64 per direction and group of 64 batch rows),
    # the double-buffered h, r.h or the 16-bit copies of h
    assert rk.rk_state_length(p.to_c()) == 256 + 2 * 64 + 2 * 2 * 1 * 256 + 2 * (1 + 128) * 256
    g = rk.Problem("gru", seq=0, batch=8, input=5, hidden=100)
    assert rk.rk_xw_length(g.to_c()) == 0
    assert rk.rk_state_length(g.to_c()) == 256 + 64 + 2 * 1 * 8 * 128 + 1 * (8 + 128) * 128
    w = rk.Problem("rnn", seq=3, batch=65, input=5, hidden=100)
    assert rk.rk_state_length(w.to_c()) == 256 + 2 * 64 + 2 * 1 * 65 * 128 + 1 * (65 + 128) * 128


def test_plans_without_device(handle):
    """With no GPU the planner assumes a GB300 (152 SMs, 227 KB shared memory
    per block) and skips the occupancy check."""
    plans = {name: rk.rk_describe_plan(handle, w.problem.to_c()) for name, w in workloads.WORKLOADS.items()}
    assert "step=fast" in plans["lstm_fwd_s8_b1_i16_h16_f32"]
    assert "step=fast" in plans["bilstm_s80_b1_i256_h256_f32"] and "ctas=16" in plans["bilstm_s80_b1_i256_h256_f32"]
    # small batches of Half layers, GRU linear_before_reset = 0 included, run the
    # small-batch tensor-core kernel (16 rows of h per direction: nb=8, 16 CTAs of 32 units)
    assert "step=tensor" in plans["bigru_s128_b8_i512_h512_f16_lbr0"] and "J=32" in plans["bigru_s128_b8_i512_h512_f16_lbr0"]
    h4 = rk.rk_create(rk.RK_FORCE_SIMT_STEP)
    try:
        lbr0 = workloads.WORKLOADS["bigru_s128_b8_i512_h512_f16_lbr0"].problem.to_c()
        assert "step=cluster" in rk.rk_describe_plan(h4, lbr0)  # 16 clusters of 16 would not fit at once
    finally:
        rk.rk_destroy(h4)
    assert "step=grid" in plans["revlstm_peep_clip_s200_b4_i128_h1024_f32"]
    # the projection runs on the SMs the 128 recurrence CTAs leave idle
    assert "proj=fused step=tensor" in plans["bilstm_s512_b64_i1024_h1024_f16"]
    assert "step=tensor" in plans["bigru_s128_b8_i512_h512_f16_lbr1"]
    # bfloat16 layers take the same kernels as Half ones
    assert plans["bilstm_s512_b64_i1024_h1024_bf16"] == plans["bilstm_s512_b64_i1024_h1024_f16"]
    assert plans["bilstm_s48_b8_i192_h96_bf16"] == plans["bilstm_s48_b8_i192_h96_f16"]
    # the register-resident SIMT kernel wherever all its clusters fit (here 16
    # rows x 2 directions x 4 CTAs), the tensor-core kernel only when asked
    assert "step=fast" in plans["bilstm_s48_b8_i192_h96_f16"] and "ctas=4" in plans["bilstm_s48_b8_i192_h96_f16"]
    h5 = rk.rk_create(rk.RK_PREFER_TENSOR_STEP)
    try:
        rec = workloads.WORKLOADS["bilstm_s48_b8_i192_h96_bf16"].problem.to_c()
        assert "step=tensor" in rk.rk_describe_plan(h5, rec) and "J=32" in rk.rk_describe_plan(h5, rec)
        # float32 layers never take the tensor cores
        assert "step=fast" in rk.rk_describe_plan(h5, workloads.WORKLOADS["bilstm_s48_b8_i192_h96_f32"].problem.to_c())
    finally:
        rk.rk_destroy(h5)
    for name, text in plans.items():
        smem = int(re.search(r"smem=(\d+)", text).group(1))
        assert smem <= 232448 - 1024, (name, text)
    empty = rk.Problem("lstm", seq=3, batch=0, input=2, hidden=4)
    assert rk.rk_describe_plan(handle, empty.to_c()) == "noop"
    c2 = workloads.WORKLOADS["bilstm_s80_b1_i256_h256_f32"].problem.to_c()
    c5 = workloads.WORKLOADS["bilstm_s512_b64_i1024_h1024_f16"].problem.to_c()
    h3 = rk.rk_create(rk.RK_FORCE_SIMT_STEP | rk.RK_FORCE_SIMT_PROJECTION)
    try:
        assert "proj=simt step=grid" in rk.rk_describe_plan(h3, c5)
    finally:
        rk.rk_destroy(h3)
    for flags, want in [(rk.RK_FORCE_GRID_STEP, "step=grid"), (rk.RK_FORCE_GENERAL_STEP, "step=cluster")]:
        h2 = rk.rk_create(flags)
        try:
            assert want in rk.rk_describe_plan(h2, c2), flags
        finally:
            rk.rk_destroy(h2)


def test_bfloat16_inputs_round_like_torch():
    """The generator's bfloat16 rounding (float32 first, then nearest-even on
    the float32 bits) gives torch's own float32 -> bfloat16 conversion, ties
    included, and every bfloat16 workload input is a bfloat16 number."""
    import torch
    rng = np.random.default_rng(11)
    a = rng.normal(size=20000) * np.exp(rng.uniform(-30, 30, 20000))
    # exact ties between two bfloat16 neighbours, both parities, and signed zeros
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3 * 2.0 ** -9 + 1, 0.0, -0.0, 1e30, -1e-30])
    for v in (a, ties):
        want = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).float().numpy()
        got = workloads.round_bf16(v)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert workloads.round_bf16([1 + 2.0 ** -8])[0] == 1.0           # tie to even (down)
    assert workloads.round_bf16([1 + 3 * 2.0 ** -8])[0] == 1 + 2.0 ** -6  # tie to even (up)
    for name in ("bilstm_s48_b8_i192_h96_bf16",):
        for k, v in workloads.make_inputs(workloads.WORKLOADS[name]).items():
            if k != "sequence_lens":
                assert v.dtype == np.float32 and np.all((v.view(np.uint32) & 0xFFFF) == 0), k


def test_workload_inputs_are_seeded_and_shaped():
    w = workloads.WORKLOADS["bigru_s128_b8_i512_h512_f16_lbr0"]
    a = workloads.make_inputs(w)
    b = workloads.make_inputs(w)
    for k in a:
        assert np.array_equal(a[k], b[k])
        assert a[k].shape == w.problem.shapes()[k]
    assert a["X"].dtype == np.float16 and a["sequence_lens"].dtype == np.int32
    assert a["sequence_lens"].min() >= 1 and a["sequence_lens"].max() <= 128
    w2 = workloads.WORKLOADS["bigru_s128_b8_i512_h512_f16_lbr1"]
    assert np.array_equal(workloads.make_inputs(w2)["R"], a["R"])  # both GRU runs share inputs
