"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Every case compares Y, Y_h and Y_c element by element on the same seeded
inputs: |gpu - oracle| <= tol or <= tol * |oracle| with tol 1e-4 for float32
and 5e-3 for Half tensors (float32 accumulation and state, outputs rounded to
half).  bfloat16 tensors get 2e-2: the Half tolerance times the ratio of the
two types' unit roundoffs (2^-9 / 2^-11 = 4), since the two errors that
matter scale with it -- the rounding of every output, and on the tensor
cores the rounding of h before the recurrent product (the Gemm page's own
bounds grow by the same factor, 2e-3 to 8e-3).  Positions past a row's length must be exactly 0, bytes around every
output (sentinels) must be untouched, and two runs must give the same bits.

The test matrix follows the one the recurrent-layers page lists: every cell x
direction x layout with option sets (bias, lengths including 0, initial state,
peepholes, clip, input_forget, linear_before_reset), every activation in every
slot of both directions, odd offsets with sentinels around every output, empty
sequence and batch, hidden sizes that do not divide the tiles, batches above
eight, and both step kernels (cluster and grid).  The named workloads run at
full size; the largest one is checked on sampled batch rows (rows are
independent, so the oracle can run on those rows alone).
"""
import numpy as np
import pytest
import torch

import onnx_lstm_gru_gb300 as rk
import oracle
from onnx_lstm_gru_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 5e-3, "bf16": 2e-2}
SENTINEL = -776.0  # exactly representable in float32, binary16 and bfloat16


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rk.build()
    rk.load()
    yield
    torch.cuda.synchronize()


_layers = {}


def layer(flags=0):
    if flags not in _layers:
        _layers[flags] = rk.RecurrentLayer(flags)
    return _layers[flags]


def torch_dtype(pr):
    return rk.torch_dtype(pr.dtype)


def to_device(arr, offset, dtype):
    """Place arr at element `offset` inside a larger device buffer."""
    flat = torch.from_numpy(np.ascontiguousarray(arr).reshape(-1))
    if dtype is not None:
        flat = flat.to(dtype)
    if offset == 0:
        return flat.cuda()
    buf = torch.full((flat.numel() + offset + 3,), 7.0 if flat.is_floating_point() else 7, dtype=flat.dtype)
    buf[offset:offset + flat.numel()] = flat
    return (buf.cuda(), offset)


def run_gpu(pr, inputs, outputs=("Y", "Y_h", "Y_c"), in_off=0, out_off=0, flags=0, scratch=None):
    dt = torch_dtype(pr)
    shp = pr.shapes()
    args = {}
    for k, v in inputs.items():
        args[k] = to_device(v, in_off, None if k == "sequence_lens" else dt)
    outs = {}
    pad = max(out_off, 8)
    for name in outputs:
        if name == "Y_c" and pr.cell != "lstm":
            continue
        n = int(np.prod(shp[name]))
        buf = torch.full((n + 2 * pad,), SENTINEL, dtype=dt, device="cuda")
        outs[name] = (buf, pad, n)
        args[name] = (buf, pad)
    L = layer(flags)
    L.encode(pr, scratch=scratch, **args)
    torch.cuda.synchronize()
    L.poll()
    res = {}
    for name, (buf, off, n) in outs.items():
        host = buf.float().cpu().numpy().astype(np.float64)
        assert np.all(host[:off] == SENTINEL) and np.all(host[off + n:] == SENTINEL), f"{name}: sentinel overwritten"
        res[name] = host[off:off + n].reshape(shp[name])
        res[name + "_raw"] = buf[off:off + n].clone()
    return res


def spec_of(pr):
    return dict(cell=pr.cell, direction=pr.direction, layout=pr.layout, seq=pr.seq, batch=pr.batch,
                input=pr.input, hidden=pr.hidden, clip=pr.clip, input_forget=pr.input_forget,
                linear_before_reset=pr.linear_before_reset,
                activations=list(pr.activations) if pr.activations else None)


def run_oracle(pr, inputs):
    args = {k: (v.astype(np.float64) if k != "sequence_lens" else v) for k, v in inputs.items()}
    return oracle.layer(spec_of(pr), **args)


def past_length_mask(pr, lens):
    """True at Y positions t >= len (or t >= max_length) of their row."""
    S, N, D, H = pr.seq, pr.batch, pr.num_directions, pr.hidden
    L = np.full(N, S) if lens is None else np.clip(lens, 0, S)
    t = np.arange(S)[:, None]
    m = t >= L[None, :]                              # [S, N]
    m = np.broadcast_to(m[:, None, :, None], (S, D, N, H))
    return m if pr.layout == 0 else m.transpose(2, 0, 1, 3)


def compare(pr, got, ref, lens=None):
    tol = TOL[pr.dtype]
    for name in ref:
        if name not in got:
            continue
        g, r = got[name], ref[name]
        assert g.shape == r.shape, name
        nan_g, nan_r = np.isnan(g), np.isnan(r)
        assert np.array_equal(nan_g, nan_r), f"{name}: NaN positions differ"
        d = np.abs(g - r)[~nan_r]
        rr = np.abs(r)[~nan_r]
        ok = (d <= tol) | (d <= tol * rr)
        if not ok.all():
            i = np.argmax(np.where(ok, 0, d))
            raise AssertionError(f"{name}: {int((~ok).sum())} of {ok.size} elements off; worst |d|={d.flat[i]:.3g} "
                                 f"at ref={r[~nan_r].flat[i]:.6g}")
    if "Y" in got and pr.seq > 0:
        m = past_length_mask(pr, lens)
        assert np.all(got["Y"][m] == 0.0), "Y must be exactly 0 past the length"


def rand_inputs(pr, seed, lens=None, init=True, peep=False, bias=True, scale=0.5):
    rng = np.random.default_rng(seed)
    shp = pr.shapes()
    def dt(v):
        return workloads.cast(v, pr.dtype)
    # bfloat16 keeps 8 significant bits, and the tensor-core steps round h to
    # it before every recurrent product, so that error grows by the
    # recurrence's gain each step.  Uniform R of scale a has gain about
    # a * sqrt(H / 3); above 1 (large H at the default scales) the layer is
    # chaotic and no fixed tolerance holds, so bfloat16 cases cap R's scale
    # at sqrt(3 / H) (gain at most 1).
    rscale = min(scale, float(np.sqrt(3.0 / max(pr.hidden, 1)))) if pr.dtype == "bf16" else scale
    a = {"X": dt(rng.uniform(-1, 1, shp["X"])),
         "W": dt(rng.uniform(-scale, scale, shp["W"])),
         "R": dt(rng.uniform(-rscale, rscale, shp["R"]))}
    if bias:
        a["B"] = dt(rng.uniform(-scale, scale, shp["B"]))
    if peep and pr.cell == "lstm":
        a["P"] = dt(rng.uniform(-scale, scale, shp["P"]))
    if init:
        a["initial_h"] = dt(rng.uniform(-1, 1, shp["initial_h"]))
        if pr.cell == "lstm":
            a["initial_c"] = dt(rng.uniform(-1, 1, shp["initial_c"]))
    if lens is not None:
        a["sequence_lens"] = np.asarray(lens, dtype=np.int32)
    return a


# ------------------------------------------------------------------ the named workloads

LARGE = ["bilstm_s512_b64_i1024_h1024_f16", "bilstm_s512_b64_i1024_h1024_bf16"]


@pytest.mark.parametrize("name", [n for n in workloads.WORKLOADS if n not in LARGE])
def test_workload_full_size(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_inputs(w)
    got = run_gpu(w.problem, inp, outputs=w.outputs)
    ref = run_oracle(w.problem, inp)
    compare(w.problem, got, ref, inp.get("sequence_lens"))
    again = run_gpu(w.problem, inp, outputs=w.outputs)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], again[k]), f"{k}: two runs differ"


@pytest.mark.parametrize("name", LARGE)
def test_large_workload_sampled_rows(name):
    """bi-LSTM 512 x 64 x 1024 x 1024 (Half, bfloat16), run whole on the GPU;
    batch rows 0, 29 and 63 re-run through the oracle alone (rows are
    independent)."""
    w = workloads.WORKLOADS[name]
    pr = w.problem
    inp = workloads.make_inputs(w)
    got = run_gpu(pr, inp)
    rows = [0, 29, 63]
    sub = rk.Problem(pr.cell, seq=pr.seq, batch=len(rows), input=pr.input, hidden=pr.hidden,
                     direction=pr.direction, dtype=pr.dtype, layout=pr.layout)
    sinp = dict(inp)
    sinp["X"] = inp["X"][:, rows]
    sinp["sequence_lens"] = inp["sequence_lens"][rows]
    ref = run_oracle(sub, sinp)
    gsub = {"Y": got["Y"][:, :, rows], "Y_h": got["Y_h"][:, rows], "Y_c": got["Y_c"][:, rows]}
    compare(sub, gsub, ref, sinp["sequence_lens"])
    assert np.all(np.isfinite(got["Y"]))


# ------------------------------------------------------------------ the option matrix

CASES = []
for cell in ("lstm", "gru", "rnn"):
    for direction in ("forward", "reverse", "bidirectional"):
        for layout in (0, 1):
            for opts in ("plain", "full"):
                CASES.append((cell, direction, layout, opts))


KERNELS = {"fast": 0, "cluster": rk.RK_FORCE_GENERAL_STEP, "grid": rk.RK_FORCE_GRID_STEP}
# the tensor-core step kernels ahead of the register-resident SIMT kernel,
# which the planner prefers wherever all its clusters fit the GPU
TC = rk.RK_PREFER_TENSOR_STEP


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("cell,direction,layout,opts", CASES)
def test_option_matrix(cell, direction, layout, opts, kernel):
    S, N, I, H = 7, 3, 5, 40
    kw = {}
    lens = None
    if opts == "full":
        lens = [7, 0, 4]
        kw = dict(clip=0.9)
        if cell == "lstm":
            kw["input_forget"] = 1
    pr = rk.Problem(cell, seq=S, batch=N, input=I, hidden=H, direction=direction, layout=layout, **kw)
    for lbr in ((0, 1) if cell == "gru" else (0,)):
        pr.linear_before_reset = lbr
        inp = rand_inputs(pr, seed=100 + len(cell) + layout, lens=lens, init=opts == "full",
                          peep=opts == "full", bias=opts == "full")
        got = run_gpu(pr, inp, flags=KERNELS[kernel])
        ref = run_oracle(pr, inp)
        compare(pr, got, ref, lens)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("cell,direction", [(c, d) for c in ("lstm", "gru", "rnn")
                                            for d in ("forward", "reverse", "bidirectional")])
def test_bfloat16_option_matrix(cell, direction, kernel):
    """bfloat16 tensors on the SIMT step kernels (bfloat16 R in registers or
    shared memory, widened exactly; float32 products and state): every cell
    and direction with lengths, initial state, peepholes, clip and
    input_forget, both layouts."""
    for layout in (0, 1):
        kw = dict(clip=0.9)
        if cell == "lstm":
            kw["input_forget"] = 1
        pr = rk.Problem(cell, seq=7, batch=3, input=5, hidden=40, direction=direction, layout=layout, dtype="bf16",
                        **kw)
        lens = [7, 0, 4]
        for lbr in ((0, 1) if cell == "gru" else (0,)):
            pr.linear_before_reset = lbr
            inp = rand_inputs(pr, seed=200 + len(cell) + layout, lens=lens, peep=True)
            compare(pr, run_gpu(pr, inp, flags=KERNELS[kernel] | rk.RK_FORCE_SIMT_STEP), run_oracle(pr, inp), lens)


ALL_ACTS = [("sigmoid", 0, 0), ("tanh", 0, 0), ("relu", 0, 0), ("affine", 0.7, -0.2), ("leakyrelu", 0.15, 0),
            ("thresholdedrelu", 0.3, 0), ("scaledtanh", 1.3, 0.6), ("hardsigmoid", 0.25, 0.45), ("elu", 0.8, 0),
            ("softsign", 0, 0), ("softplus", 0, 0)]


@pytest.mark.parametrize("cell", ["lstm", "gru", "rnn"])
@pytest.mark.parametrize("act", ALL_ACTS, ids=[a[0] for a in ALL_ACTS])
def test_every_activation_in_every_slot(cell, act):
    A = {"lstm": 3, "gru": 2, "rnn": 1}[cell]
    defaults = {"lstm": [("sigmoid", 0, 0), ("tanh", 0, 0), ("tanh", 0, 0)],
                "gru": [("sigmoid", 0, 0), ("tanh", 0, 0)], "rnn": [("tanh", 0, 0)]}[cell] * 2
    for slot in range(2 * A):
        acts = list(defaults)
        acts[slot] = act
        pr = rk.Problem(cell, seq=5, batch=2, input=3, hidden=12, direction="bidirectional",
                        activations=acts, clip=4.0)
        inp = rand_inputs(pr, seed=7 + slot, lens=[5, 3], peep=True)
        got = run_gpu(pr, inp)
        compare(pr, got, run_oracle(pr, inp), [5, 3])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_odd_offsets_and_sentinels(dtype):
    pr = rk.Problem("lstm", seq=6, batch=3, input=7, hidden=36, direction="bidirectional", dtype=dtype, layout=1)
    inp = rand_inputs(pr, seed=3, lens=[6, 2, 5], peep=True)
    got = run_gpu(pr, inp, in_off=3, out_off=5)
    compare(pr, got, run_oracle(pr, inp), [6, 2, 5])


def test_empty_sequence_and_batch():
    pr = rk.Problem("lstm", seq=0, batch=3, input=4, hidden=20, direction="bidirectional")
    inp = rand_inputs(pr, seed=5)
    got = run_gpu(pr, inp, outputs=("Y_h", "Y_c"))
    np.testing.assert_array_equal(got["Y_h"], inp["initial_h"].astype(np.float64))
    np.testing.assert_array_equal(got["Y_c"], inp["initial_c"].astype(np.float64))
    pr0 = rk.Problem("gru", seq=5, batch=0, input=4, hidden=20)
    before = layer().launches()
    run_gpu(pr0, rand_inputs(pr0, seed=6, init=False))  # sentinels checked inside
    assert layer().launches() == before  # Batch = 0 records nothing


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("H,N", [(100, 11), (37, 9), (130, 2), (513, 1), (250, 3)])
def test_ragged_hidden_and_large_batch(H, N, kernel):
    for lbr in (0, 1):
        pr = rk.Problem("gru", seq=6, batch=N, input=9, hidden=H, direction="bidirectional", linear_before_reset=lbr)
        lens = list(np.random.default_rng(H).integers(0, 7, N))
        inp = rand_inputs(pr, seed=H + N, lens=lens, scale=0.2)
        compare(pr, run_gpu(pr, inp, flags=KERNELS[kernel]), run_oracle(pr, inp), lens)


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_kernels_agree_on_lstm_with_every_option(kernel, dtype):
    pr = rk.Problem("lstm", seq=9, batch=2, input=70, hidden=96, direction="bidirectional", dtype=dtype, layout=1,
                    clip=2.5, input_forget=1,
                    activations=[("hardsigmoid", 0.2, 0.5), ("scaledtanh", 1.0, 1.0), ("softsign", 0, 0)] * 2)
    inp = rand_inputs(pr, seed=31, lens=[9, 4], peep=True, scale=0.3)
    compare(pr, run_gpu(pr, inp, flags=KERNELS[kernel]), run_oracle(pr, inp), [9, 4])


def test_max_length_shortens_loop():
    pr = rk.Problem("lstm", seq=9, batch=3, input=4, hidden=24, direction="bidirectional", max_length=5)
    inp = rand_inputs(pr, seed=9, lens=[5, 2, 0])
    compare(pr, run_gpu(pr, inp), run_oracle(pr, inp), [5, 2, 0])


def test_nan_passes_through_clip():
    pr = rk.Problem("rnn", seq=1, batch=2, input=1, hidden=1, activations=[("affine", 1.0, 0.0)], clip=1.0)
    inp = {"X": np.array([np.nan, 0.5], dtype=np.float32).reshape(1, 2, 1),
           "W": np.ones((1, 1, 1), np.float32), "R": np.zeros((1, 1, 1), np.float32)}
    got = run_gpu(pr, inp, outputs=("Y",))
    assert np.isnan(got["Y"][0, 0, 0, 0]) and got["Y"][0, 0, 1, 0] == 0.5


def test_getting_started_rows_exact():
    """RNN with Affine(1, 0), R = 0: Y is the projection, the pages' example rows."""
    A = np.arange(1, 9, dtype=np.float32).reshape(4, 1, 2)
    Bm = np.array([[1, 0, 2], [0, 1, 3]], dtype=np.float32)
    for dtype in ("f32", "f16", "bf16"):  # small integers: exact in all three types
        pr = rk.Problem("rnn", seq=4, batch=1, input=2, hidden=3, activations=[("affine", 1.0, 0.0)], dtype=dtype)
        inp = {"X": workloads.cast(A, dtype), "W": workloads.cast(Bm.T.copy()[None], dtype),
               "R": workloads.cast(np.zeros((1, 3, 3)), dtype)}
        got = run_gpu(pr, inp, outputs=("Y",))
        np.testing.assert_array_equal(got["Y"].reshape(4, 3), [[1, 2, 8], [3, 4, 18], [5, 6, 28], [7, 8, 38]])


# ------------------------------------------------------------------ boundary behaviour

@pytest.mark.parametrize("flags,per_layer", [(0, 2), (rk.RK_FORCE_GENERAL_STEP, 2), (rk.RK_FORCE_GRID_STEP, 2)])
def test_launches_do_not_grow_with_seq(flags, per_layer):
    """The projection plus one persistent step kernel per layer, whatever the
    sequence length."""
    L = layer(flags)
    for S in (4, 64):
        pr = rk.Problem("lstm", seq=S, batch=1, input=8, hidden=32)
        inp = rand_inputs(pr, seed=S)
        before = L.launches()
        run_gpu(pr, inp, flags=flags)
        assert L.launches() - before == per_layer


def test_caller_scratch_in_one_arena_is_bitwise_equal():
    w = workloads.WORKLOADS["bilstm_s80_b1_i256_h256_f32"]
    inp = workloads.make_inputs(w)
    base = run_gpu(w.problem, inp)
    c = w.problem.to_c()
    nx, ns = rk.rk_xw_length(c), rk.rk_state_length(c)
    arena = torch.empty(nx + ns + 64, dtype=torch.float32, device="cuda")
    sc = rk.rk_scratch(arena.data_ptr(), 17, nx + 17, arena.data_ptr(), nx + 40, nx + ns + 64)
    got = run_gpu(w.problem, inp, scratch=sc)
    for k in ("Y_raw", "Y_h_raw", "Y_c_raw"):
        assert torch.equal(base[k], got[k])


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cell", ["lstm", "gru", "rnn"])
def test_tensor_core_step_with_odd_offsets(cell, dtype):
    """Operands at odd element offsets (R not 16-byte aligned: element loads
    of the R slice; Y pieces stored element-wise) give the oracle's result
    and leave the sentinels around the outputs untouched."""
    pr = rk.Problem(cell, seq=5, batch=6, input=24, hidden=72, direction="bidirectional", dtype=dtype,
                    linear_before_reset=1 if cell == "gru" else 0)
    assert "step=tensor" in layer(TC).plan(pr)
    inp = rand_inputs(pr, seed=77, scale=0.15)
    got = run_gpu(pr, inp, in_off=3, out_off=5, flags=TC)
    compare(pr, got, run_oracle(pr, inp), None)
    # unaligned X and W take the SIMT projection: compare against it
    aligned = run_gpu(pr, inp, flags=TC | rk.RK_FORCE_SIMT_PROJECTION)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], aligned[k]), k


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cell,H,N,direction", [("lstm", 576, 16, "bidirectional"),
                                                ("gru", 640, 40, "reverse"),
                                                ("rnn", 1024, 70, "forward")])
def test_fused_projection_matches_separate(cell, H, N, direction, dtype):
    """With flag-published tensor-core teams the projection runs on the SMs
    the recurrence leaves idle, its tiles produced in the order the steps
    consume them and each step waiting for its rows' tile.  The same tile
    arithmetic as the projection's own launch: bit-identical outputs, and the
    oracle's within the tolerance of the element type."""
    pr = rk.Problem(cell, seq=6, batch=N, input=72, hidden=H, direction=direction, dtype=dtype,
                    linear_before_reset=1 if cell == "gru" else 0)
    assert "proj=fused step=tensor" in layer().plan(pr)
    assert "proj=tc step=tensor" in layer(rk.RK_SEPARATE_PROJECTION).plan(pr)
    lens = list(np.random.default_rng(N).integers(0, 7, N))
    inp = rand_inputs(pr, seed=H + N, lens=lens, scale=0.15)
    got = run_gpu(pr, inp)
    sep = run_gpu(pr, inp, flags=rk.RK_SEPARATE_PROJECTION)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], sep[k]), k
    compare(pr, got, run_oracle(pr, inp), lens)


XW_RING_CASES = [
    # (cell, S, N, H, direction, lengths): 128-row tiles of Xw per direction > 16
    ("lstm", 40, 64, 576, "bidirectional", "uniform"),   # every row 37 steps: ring
    ("gru", 60, 40, 640, "reverse", None),                # no lengths: ring
    ("rnn", 36, 72, 1024, "forward", "uniform"),
    ("lstm", 40, 64, 576, "bidirectional", "varied"),    # rows of different lengths: whole Xw
]


@pytest.mark.parametrize("cell,S,N,H,direction,lens_kind", XW_RING_CASES)
def test_fused_projection_xw_ring(cell, S, N, H, direction, lens_kind):
    """Long layers whose projection runs inside the tensor-core step launch
    keep Xw in a ring of 8 128-row tiles per direction (it stays in L2) when
    every row has the same length: a tile is overwritten only after every
    gate warp of its direction has loaded the steps that read it.  Same tile
    arithmetic as the projection's own launch: bit-identical outputs; the
    oracle's within tolerance on sampled batch rows."""
    pr = rk.Problem(cell, seq=S, batch=N, input=72, hidden=H, direction=direction, dtype="f16",
                    linear_before_reset=1 if cell == "gru" else 0)
    assert "proj=fused step=tensor" in layer().plan(pr)
    rng = np.random.default_rng(S * N + H)
    lens = None
    if lens_kind == "uniform":
        lens = [S - 3] * N
    elif lens_kind == "varied":
        lens = list(rng.integers(0, S + 1, N))
    # weights of scale 0.04: recurrent gain about 0.04 * sqrt(H / 3) < 1, so
    # 40 steps of Half rounding stay far inside the tolerance (a chaotic
    # layer would amplify them past any fixed bound)
    inp = rand_inputs(pr, seed=H + N, lens=lens, scale=0.04)
    got = run_gpu(pr, inp)
    sep = run_gpu(pr, inp, flags=rk.RK_SEPARATE_PROJECTION)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], sep[k]), k
    rows = [0, N // 3, N - 1]
    sub = rk.Problem(cell, seq=S, batch=len(rows), input=72, hidden=H, direction=direction, dtype="f16",
                     linear_before_reset=pr.linear_before_reset)
    sinp = {k: v for k, v in inp.items()}
    sinp["X"] = inp["X"][:, rows]
    if lens is not None:
        sinp["sequence_lens"] = inp["sequence_lens"][rows]
    for k in ("initial_h", "initial_c"):
        if k in sinp:
            sinp[k] = inp[k][:, rows]
    ref = run_oracle(sub, sinp)
    gsub = {"Y": got["Y"][:, :, rows], "Y_h": got["Y_h"][:, rows]}
    if "Y_c" in got:
        gsub["Y_c"] = got["Y_c"][:, rows]
    compare(sub, gsub, ref, sinp.get("sequence_lens"))


@pytest.mark.parametrize("H,N,direction,layout,opts", [(40, 4, "bidirectional", 0, "plain"),
                                                     (96, 9, "reverse", 1, "full"),
                                                     (200, 16, "forward", 0, "full"),
                                                     (512, 8, "bidirectional", 1, "plain")])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tensor_core_gru_lbr0(H, N, direction, layout, opts, dtype):
    """GRU with linear_before_reset = 0 on the small-batch tensor-core kernel:
    two products per step, r (.) h_prev rounded to the 16-bit type and
    exchanged inside the cluster before the candidate's product.  Matches
    the oracle within the type's tolerance and the SIMT cluster kernel."""
    kw = dict(clip=1.5) if opts == "full" else {}
    if opts == "full":
        D = 2 if direction == "bidirectional" else 1
        kw["activations"] = [("hardsigmoid", 0.2, 0.5), ("softsign", 0, 0)] * D
    pr = rk.Problem("gru", seq=9, batch=N, input=24, hidden=H, direction=direction, dtype=dtype, layout=layout,
                    linear_before_reset=0, **kw)
    plan = layer(TC).plan(pr)
    assert "step=tensor" in plan and "J=32" in plan
    lens = list(np.random.default_rng(H).integers(0, 10, N))
    inp = rand_inputs(pr, seed=H + 7 * N, lens=lens, scale=0.2)
    got = run_gpu(pr, inp, flags=TC)
    compare(pr, got, run_oracle(pr, inp), lens)
    simt = run_gpu(pr, inp, flags=rk.RK_FORCE_SIMT_STEP)
    compare(pr, got, {k: v for k, v in simt.items() if not k.endswith("_raw")}, lens)
    again = run_gpu(pr, inp, flags=TC)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], again[k]), f"{k}: two runs differ"


@pytest.mark.parametrize("H,N,direction,layout,opts", [(40, 4, "bidirectional", 0, "plain"),
                                                     (200, 9, "reverse", 1, "full"),
                                                     (512, 16, "bidirectional", 0, "full"),
                                                     (512, 8, "forward", 1, "plain")])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tensor_core_rnn_stacked_quarters(H, N, direction, layout, opts, dtype):
    """RNN on the small-batch tensor-core kernel, whose one gate is multiplied
    with its four k quarters stacked into the MMA rows (whole and partly
    empty quarters): matches the oracle within the type's tolerance and the
    SIMT cluster kernel, and two runs give the same bits."""
    kw = dict(clip=1.5) if opts == "full" else {}
    if opts == "full":
        D = 2 if direction == "bidirectional" else 1
        kw["activations"] = [("softsign", 0, 0)] * D
    pr = rk.Problem("rnn", seq=9, batch=N, input=24, hidden=H, direction=direction, dtype=dtype, layout=layout, **kw)
    plan = layer(TC).plan(pr)
    assert "variant=small" in plan, plan
    lens = list(np.random.default_rng(H + N).integers(0, 10, N))
    inp = rand_inputs(pr, seed=H + 5 * N, lens=lens, scale=0.2)
    got = run_gpu(pr, inp, flags=TC)
    compare(pr, got, run_oracle(pr, inp), lens)
    simt = run_gpu(pr, inp, flags=rk.RK_FORCE_SIMT_STEP)
    compare(pr, got, {k: v for k, v in simt.items() if not k.endswith("_raw")}, lens)
    again = run_gpu(pr, inp, flags=TC)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], again[k]), f"{k}: two runs differ"


@pytest.mark.parametrize("H,N", [(40, 5), (96, 130)])
def test_tensor_core_step_ignores_stale_scratch(H, N):
    """The tensor-core step kernel reads its Half h copies in whole 64-wide k
    blocks and batch blocks; parts no CTA owns must not leak stale scratch.
    Caller scratch filled with NaN bytes gives the same bits as fresh scratch."""
    pr = rk.Problem("lstm", seq=6, batch=N, input=16, hidden=H, direction="bidirectional", dtype="f16")
    assert "step=tensor" in layer(TC).plan(pr)
    inp = rand_inputs(pr, seed=H * N, scale=0.15)
    base = run_gpu(pr, inp, flags=TC)
    c = pr.to_c()
    nx, ns = rk.rk_xw_length(c), rk.rk_state_length(c)
    arena = torch.full((nx + ns + 64,), float("nan"), dtype=torch.float32, device="cuda")
    sc = rk.rk_scratch(arena.data_ptr(), 0, nx, arena.data_ptr(), nx + 4, nx + ns + 64)
    got = run_gpu(pr, inp, scratch=sc, flags=TC)
    for k in ("Y_raw", "Y_h_raw", "Y_c_raw"):
        assert torch.equal(base[k], got[k]), k
    assert np.isfinite(got["Y"]).all()


def test_host_buffer_entry_matches_device_entry():
    w = workloads.WORKLOADS["bigru_s128_b8_i512_h512_f16_lbr0"]
    pr = w.problem
    inp = workloads.make_inputs(w)
    dev = run_gpu(pr, inp, outputs=("Y", "Y_h"))
    shp = pr.shapes()
    Y = np.zeros(shp["Y"], np.float16)
    Yh = np.zeros(shp["Y_h"], np.float16)
    layer().encode_host(pr, Y=Y, Y_h=Yh, **inp)
    np.testing.assert_array_equal(Y.astype(np.float64), dev["Y"])
    np.testing.assert_array_equal(Yh.astype(np.float64), dev["Y_h"])


def test_host_buffer_entry_bfloat16():
    """bfloat16 host buffers (CPU tensors: numpy has no bfloat16) through the
    host entry point give the device entry point's bits."""
    w = workloads.WORKLOADS["bilstm_s48_b8_i192_h96_bf16"]
    pr = w.problem
    inp = workloads.make_inputs(w)
    dev = run_gpu(pr, inp)
    host_in = {k: (torch.from_numpy(v) if k == "sequence_lens" else torch.from_numpy(v).to(torch.bfloat16))
               for k, v in inp.items()}
    shp = pr.shapes()
    outs = {n: torch.zeros(shp[n], dtype=torch.bfloat16) for n in ("Y", "Y_h", "Y_c")}
    layer().encode_host(pr, **outs, **host_in)
    for n, t in outs.items():
        assert torch.equal(t.reshape(-1), dev[n + "_raw"].cpu()), n


@pytest.mark.parametrize("name,flags", [("bilstm_s80_b1_i256_h256_f32", 0),
                                        ("revlstm_peep_clip_s200_b4_i128_h1024_f32", 0),
                                        ("bilstm_s48_b8_i192_h96_f16", 0),
                                        ("bilstm_s48_b8_i192_h96_bf16", TC),
                                        ("bigru_s128_b8_i512_h512_f16_lbr0", 0)])
@pytest.mark.parametrize("mode", ["pinned", "pageable", "mixed"])
def test_host_entry_pinned_buffers_in_place(name, flags, mode):
    """The host entry reads page-locked inputs other than X and W, and
    writes page-locked outputs, in place through the device's mapping of
    that memory, and copies the rest: all pinned, all pageable and a mix give
    the device entry's bits on the register-resident, grid, small-batch and
    row-team tensor-core kernels, and the kernels' writes stay inside each
    output (sentinels around it)."""
    w = workloads.WORKLOADS[name]
    pr = w.problem
    inp = workloads.make_inputs(w)
    dt = torch_dtype(pr)
    want = run_gpu(pr, inp, flags=flags)

    def place(t, i):
        pinned = mode == "pinned" or (mode == "mixed" and i % 2 == 0)
        return t.pin_memory() if pinned else t

    ins = {k: place(torch.from_numpy(v) if k == "sequence_lens" else torch.from_numpy(v).to(dt), i)
           for i, (k, v) in enumerate(sorted(inp.items()))}
    shp = pr.shapes()
    names = [n for n in ("Y", "Y_h", "Y_c") if not (n == "Y_c" and pr.cell != "lstm")]
    bufs, outs = {}, {}
    for i, n in enumerate(names):
        m = int(np.prod(shp[n]))
        bufs[n] = place(torch.full((m + 16,), SENTINEL, dtype=dt), i + 1)
        outs[n] = bufs[n][8:8 + m]
    for _ in range(2):
        layer(flags).encode_host(pr, **ins, **outs)
        for n in names:
            b = bufs[n]
            assert torch.all(b[:8] == SENTINEL) and torch.all(b[-8:] == SENTINEL), f"{n}: sentinel overwritten"
            assert torch.equal(b[8:-8], want[n + "_raw"].cpu()), n
    layer(flags).poll()


def test_host_entry_planner_memory_round_robin():
    """One handle encodes six different layers twice in turn through the host
    entry (more problems than the handle remembers plans for, so plans are
    both recalled and recomputed), on a stream of its own with pinned host
    buffers: every result has the device entry's bits on a fresh handle."""
    cases = [
        (rk.Problem("lstm", seq=9, batch=3, input=5, hidden=24), dict(peep=True)),
        (rk.Problem("gru", direction="bidirectional", seq=7, batch=2, input=8, hidden=40, linear_before_reset=1), {}),
        (rk.Problem("rnn", direction="reverse", seq=11, batch=5, input=3, hidden=17), {}),
        (rk.Problem("gru", direction="bidirectional", seq=6, batch=4, input=16, hidden=64, dtype="f16"), {}),
        (rk.Problem("lstm", direction="bidirectional", seq=5, batch=2, input=8, hidden=32, dtype="bf16",
                    clip=2.0), {}),
        (rk.Problem("lstm", seq=4, batch=9, input=6, hidden=300), dict(lens=[4, 1, 3, 0, 2, 4, 4, 1, 2])),
    ]
    L = rk.RecurrentLayer()
    stream = torch.cuda.Stream()
    want, ins = [], []
    for i, (pr, kw) in enumerate(cases):
        inp = rand_inputs(pr, seed=40 + i, **kw)
        fresh = rk.RecurrentLayer()
        dt = torch_dtype(pr)
        shp = pr.shapes()
        args = {k: (torch.from_numpy(v).cuda() if k == "sequence_lens" else torch.from_numpy(v).to(dt).cuda())
                for k, v in inp.items()}
        outs = {n: torch.zeros(shp[n], dtype=dt, device="cuda") for n in ("Y", "Y_h")}
        fresh.encode(pr, **args, **outs)
        torch.cuda.synchronize()
        fresh.poll()
        fresh.close()
        want.append({n: t.cpu() for n, t in outs.items()})
        ins.append({k: (torch.from_numpy(v) if k == "sequence_lens" else torch.from_numpy(v).to(dt)).pin_memory()
                    for k, v in inp.items()})
    for rnd in range(2):
        for i, (pr, _) in enumerate(cases):
            shp = pr.shapes()
            outs = {n: torch.full(shp[n], 9.0, dtype=torch_dtype(pr)).pin_memory() for n in ("Y", "Y_h")}
            L.encode_host(pr, stream=stream, **ins[i], **outs)
            for n, t in outs.items():
                assert torch.equal(t, want[i][n]), (rnd, i, n)
    L.poll()
    L.close()


def test_bounded_wait_gives_up_and_context_survives():
    L = rk.RecurrentLayer()
    s = torch.cuda.current_stream()
    assert rk.rk_selftest_timeout(L.handle, s.cuda_stream, 200_000) == rk.RK_OK
    assert rk.rk_status_poll(L.handle, s.cuda_stream) == rk.RK_ERR_TIMEOUT
    assert rk.rk_status_poll(L.handle, s.cuda_stream) == rk.RK_OK  # cleared
    # the context is still usable
    pr = rk.Problem("rnn", seq=3, batch=2, input=2, hidden=8)
    inp = rand_inputs(pr, seed=1)
    L.encode(pr, X=torch.from_numpy(inp["X"]).cuda(), W=torch.from_numpy(inp["W"]).cuda(),
             R=torch.from_numpy(inp["R"]).cuda(), B=torch.from_numpy(inp["B"]).cuda())
    L.poll()
    L.close()


def test_validation_error_launches_nothing():
    L = layer()
    pr = rk.Problem("gru", seq=3, batch=2, input=2, hidden=8)
    X = torch.zeros(3 * 2 * 2, device="cuda")
    before = L.launches()
    with pytest.raises(rk.RkError) as e:
        L.encode(pr, X=X, W=torch.zeros(3 * 8 * 2, device="cuda"), R=torch.zeros(5, device="cuda"))
    assert e.value.code == rk.RK_ERR_SHAPE and "GRU: R:" in e.value.message
    assert L.launches() == before


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("S,N,I,H", [(75, 4, 200, 600), (1, 1, 8, 16), (130, 1, 1024, 256)])
def test_16bit_projection_tensor_cores(S, N, I, H, dtype):
    """An RNN with Affine(1, 0), R = 0 and no bias outputs its projection:
    Y[t] = x_t . W^T.  Half and bfloat16 inputs take the tcgen05 projection;
    the result matches the oracle's projection and the SIMT projection (same
    float32 products of 16-bit values, different summation order)."""
    pr = rk.Problem("rnn", seq=S, batch=N, input=I, hidden=H, direction="bidirectional", dtype=dtype,
                    activations=[("affine", 1.0, 0.0)] * 2)
    plan = layer().plan(pr)
    assert "proj=tc" in plan or "proj=fused" in plan  # both the tcgen05 projection
    rng = np.random.default_rng(S + I)
    inp = {"X": workloads.cast(rng.uniform(-1, 1, (S, N, I)), dtype),
           "W": workloads.cast(rng.uniform(-0.1, 0.1, (2, H, I)), dtype),
           "R": workloads.cast(np.zeros((2, H, H)), dtype)}
    got = run_gpu(pr, inp, outputs=("Y",))
    want = oracle.projection(inp["X"].astype(np.float64).reshape(S * N, I), inp["W"].astype(np.float64))
    ref = {"Y": want.reshape(2, S, N, H).transpose(1, 0, 2, 3)}
    compare(pr, got, ref)
    simt = run_gpu(pr, inp, outputs=("Y",), flags=rk.RK_FORCE_SIMT_PROJECTION)
    compare(pr, got, {"Y": simt["Y"]})


TC_STEP_CASES = [
    ("lstm", 40, 5, "bidirectional", 0, "plain"),
    ("lstm", 96, 130, "reverse", 1, "full"),
    ("gru", 64, 9, "forward", 0, "full"),
    ("rnn", 48, 17, "bidirectional", 1, "plain"),
    ("lstm", 256, 64, "bidirectional", 0, "plain"),
    # more than 16 CTAs of 32 units: teams published by global flags
    ("lstm", 576, 16, "bidirectional", 1, "plain"),
    ("gru", 544, 33, "reverse", 0, "full"),
]


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("cell,H,N,direction,layout,opts", TC_STEP_CASES)
def test_tensor_core_step_kernel(cell, H, N, direction, layout, opts, dtype):
    """16-bit layers (Half, bfloat16) with a batch of 4 or more run R . h on
    the tensor cores (h rounded to the 16-bit type for the product, state
    float32); results match the oracle within the type's tolerance and the
    SIMT step kernel."""
    kw = dict(clip=1.5) if opts == "full" else {}
    if opts == "full" and cell == "lstm":
        kw["input_forget"] = 1
    if opts == "full":
        A = {"lstm": 3, "gru": 2, "rnn": 1}[cell]
        D = 2 if direction == "bidirectional" else 1
        kw["activations"] = ([("hardsigmoid", 0.2, 0.5), ("softsign", 0, 0), ("tanh", 0, 0)][:A]) * D
    pr = rk.Problem(cell, seq=7, batch=N, input=24, hidden=H, direction=direction, dtype=dtype, layout=layout,
                    linear_before_reset=1 if cell == "gru" else 0, **kw)
    assert "step=tensor" in layer(TC).plan(pr)
    lens = list(np.random.default_rng(N).integers(0, 8, N))
    inp = rand_inputs(pr, seed=H + N, lens=lens, peep=(opts == "full"), scale=0.15)
    got = run_gpu(pr, inp, flags=TC)
    compare(pr, got, run_oracle(pr, inp), lens)
    simt = run_gpu(pr, inp, flags=rk.RK_FORCE_SIMT_STEP)
    compare(pr, got, {k: v for k, v in simt.items() if not k.endswith("_raw")}, lens)
    again = run_gpu(pr, inp, flags=TC)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], again[k]), f"{k}: two runs differ"


# ------------------------------------------------------------------ lengths out of range and an empty input

# Every step-kernel family, each as (flags, cell / size overrides, the plan
# text that proves which kernel ran).  The recurrent-layers page ("Semantics")
# runs a length above Seq as Seq, a length of 0 as no step (Y_h = Y_c = 0);
# a negative length is read as 0.  The kernels clamp the lengths they read on
# the device, so every family is given all of these at once.
FAMILIES = {
    "fast": (0, dict(N=6, H=40), "step=fast"),
    "cluster": (rk.RK_FORCE_GENERAL_STEP, dict(N=6, H=40), "step=cluster"),
    "grid": (rk.RK_FORCE_GRID_STEP, dict(N=6, H=40), "step=grid"),
    "tensor_small": (TC, dict(N=9, H=96), "variant=small"),
    "tensor_cluster": (TC, dict(N=40, H=128), "variant=cluster"),
    "tensor_pairs": (TC | rk.RK_SEPARATE_PROJECTION, dict(N=16, H=576), "variant=pairs"),
    "tensor_rows": (TC | rk.RK_SEPARATE_PROJECTION, dict(N=130, H=96), "variant=rows"),
    "tensor_fused": (TC, dict(N=16, H=576), "proj=fused step=tensor"),
}
FAMILY_DTYPES = {"fast": ("f32", "f16"), "cluster": ("f32", "f16"), "grid": ("f32", "bf16")}
TENSOR_ONLY_CELLS = ("lstm", "gru1", "rnn")  # GRU lbr 0 with many rows runs on the SIMT cluster kernel


def _family_cases():
    out = []
    for fam in FAMILIES:
        dts = FAMILY_DTYPES.get(fam, ("f16",))
        cells = ("lstm", "gru0", "gru1", "rnn") if fam in FAMILY_DTYPES or fam == "tensor_small" else TENSOR_ONLY_CELLS
        for dt in dts:
            for c in cells:
                out.append((fam, dt, c))
    return out


def out_of_range_lengths(S, N):
    """Negative, zero, in-range, exactly Seq and above-Seq lengths, cycled over N rows."""
    pattern = [-3, S + 4, 0, 2, S, S - 1, -1, 1, 2 * S + 9, S // 2]
    return [pattern[i % len(pattern)] for i in range(N)]


def family_scale(pr):
    # weights of scale a give a recurrent gain of about a * sqrt(H / 3); keep
    # it below 1 so the 16-bit roundings of h are not amplified past the
    # tolerance (a chaotic layer would defeat any fixed bound)
    return min(0.15, float(np.sqrt(2.0 / pr.hidden)))


def family_problem(fam, dtype, cellkey, S=7, I=24, direction="bidirectional"):
    flags, kw, want = FAMILIES[fam]
    cell = cellkey[:3] if cellkey.startswith("gru") else cellkey
    lbr = 1 if cellkey == "gru1" else 0
    pr = rk.Problem(cell, seq=S, batch=kw["N"], input=I, hidden=kw["H"], direction=direction, dtype=dtype,
                    linear_before_reset=lbr)
    return pr, flags, want


@pytest.mark.parametrize("fam,dtype,cellkey", _family_cases())
def test_out_of_range_lengths_every_kernel(fam, dtype, cellkey):
    """sequence_lens holding negative values, 0, in-range values, Seq and
    values above Seq: every step-kernel family matches the oracle (which
    clamps the same way) element by element, with Y exactly 0 past each
    clamped length and Y_h / Y_c = 0 for rows of length <= 0."""
    pr, flags, want = family_problem(fam, dtype, cellkey)
    assert want in layer(flags).plan(pr), layer(flags).plan(pr)
    lens = out_of_range_lengths(pr.seq, pr.batch)
    inp = rand_inputs(pr, seed=500 + pr.batch + pr.hidden, lens=lens, scale=family_scale(pr))
    got = run_gpu(pr, inp, flags=flags)
    compare(pr, got, run_oracle(pr, inp), lens)
    dead = np.clip(lens, 0, pr.seq) == 0
    yh = got["Y_h"] if pr.layout == 1 else got["Y_h"].transpose(1, 0, 2)  # [N, D, H]
    assert np.all(yh[dead] == 0.0), "rows of length <= 0 end with Y_h = 0"


@pytest.mark.parametrize("fam,dtype,cellkey", _family_cases())
def test_empty_input_every_kernel(fam, dtype, cellkey):
    """A layer with input size 0: X and W are empty, every xw term is the
    empty sum 0, so the recurrence runs on R, the biases and the initial
    state alone.  Matches the oracle on every step-kernel family."""
    pr, flags, want = family_problem(fam, dtype, cellkey, I=0)
    plan = layer(flags).plan(pr)
    assert want.replace("proj=fused ", "") in plan, plan
    lens = [pr.seq - (i % 3) for i in range(pr.batch)]
    inp = rand_inputs(pr, seed=600 + pr.batch + pr.hidden, lens=lens, scale=family_scale(pr))
    assert inp["X"].size == 0 and inp["W"].size == 0
    got = run_gpu(pr, inp, flags=flags)
    compare(pr, got, run_oracle(pr, inp), lens)
    assert np.all(np.isfinite(got["Y"]))


@pytest.mark.parametrize("lens_kind", ["all_above_seq", "mixed"])
def test_fused_projection_xw_ring_out_of_range_lengths(lens_kind):
    """The tensor-core launch that computes its own projection keeps Xw in an
    L2 ring only when every row has the same length after clamping: every
    length above Seq (all clamp to Seq) takes the ring, a mix of negative,
    zero and above-Seq lengths takes the whole scratch.  Both are
    bit-identical to the projection's own launch and match the oracle on
    sampled rows."""
    S, N, H = 40, 64, 576
    pr = rk.Problem("lstm", seq=S, batch=N, input=72, hidden=H, direction="bidirectional", dtype="f16")
    assert "proj=fused step=tensor" in layer().plan(pr)
    if lens_kind == "all_above_seq":
        lens = [S + 1 + (i % 5) for i in range(N)]
    else:
        lens = out_of_range_lengths(S, N)
    inp = rand_inputs(pr, seed=S + N + H, lens=lens, scale=0.04)
    got = run_gpu(pr, inp)
    sep = run_gpu(pr, inp, flags=rk.RK_SEPARATE_PROJECTION)
    for k in got:
        if k.endswith("_raw"):
            assert torch.equal(got[k], sep[k]), k
    rows = [0, 1, 2, 4, N - 1]
    sub = rk.Problem("lstm", seq=S, batch=len(rows), input=72, hidden=H, direction="bidirectional", dtype="f16")
    sinp = dict(inp)
    sinp["X"] = inp["X"][:, rows]
    sinp["sequence_lens"] = inp["sequence_lens"][rows]
    for k in ("initial_h", "initial_c"):
        sinp[k] = inp[k][:, rows]
    ref = run_oracle(sub, sinp)
    gsub = {"Y": got["Y"][:, :, rows], "Y_h": got["Y_h"][:, rows], "Y_c": got["Y_c"][:, rows]}
    compare(sub, gsub, ref, sinp["sequence_lens"])


# ------------------------------------------------------------------ small-grid projection forms

def projection_case(S, N, I, H, dtype, direction="bidirectional", seed=0, flags=rk.RK_FORCE_SIMT_PROJECTION):
    """RNN with Affine(1, 0), R = 0 and no bias: Y[t] = x_t . W^T, the
    projection alone, compared with the oracle's projection."""
    pr = rk.Problem("rnn", seq=S, batch=N, input=I, hidden=H, direction=direction, dtype=dtype,
                    activations=[("affine", 1.0, 0.0)] * (2 if direction == "bidirectional" else 1))
    D = pr.num_directions
    rng = np.random.default_rng(seed + S * 7 + I)
    inp = {"X": workloads.cast(rng.uniform(-1, 1, (S, N, I)), dtype),
           "W": workloads.cast(rng.uniform(-0.2, 0.2, (D, H, I)), dtype),
           "R": workloads.cast(np.zeros((D, H, H)), dtype)}
    got = run_gpu(pr, inp, outputs=("Y",), flags=flags)
    want = oracle.projection(inp["X"].astype(np.float64).reshape(S * N, I), inp["W"].astype(np.float64))
    ref = {"Y": want.reshape(D, S, N, H).transpose(1, 0, 2, 3)}
    compare(pr, got, ref)
    return got


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S,N,I,H", [(1, 1, 4, 3), (1, 4, 256, 100), (2, 2, 1000, 37), (3, 1, 128, 1024),
                                     (4, 1, 36, 200)])
def test_few_rows_projection(S, N, I, H, dtype):
    """At most four rows of X (S * N <= 4): the projection streams W once, a
    warp per column with its lanes on consecutive k, lane sums added in lane
    order ("Matrix multiplication (Gemm)", section "Small grids and few
    rows").  Matches the oracle's projection; two runs give the same bits."""
    a = projection_case(S, N, I, H, dtype)
    b = projection_case(S, N, I, H, dtype)
    assert torch.equal(a["Y_raw"], b["Y_raw"])


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("S,N,I,H", [(80, 1, 256, 1024), (5, 7, 512, 100), (37, 1, 264, 64), (9, 9, 256, 333)])
def test_split_k_projection(S, N, I, H, dtype):
    """A grid of tiles that cannot fill the GPU over k >= 256: k in 4 ranges
    per CTA, each output the sum of its range sums in range order (the Gemm
    page's split k, inside one launch).  Ragged rows and columns; matches the
    oracle's projection; two runs give the same bits."""
    a = projection_case(S, N, I, H, dtype)
    b = projection_case(S, N, I, H, dtype)
    assert torch.equal(a["Y_raw"], b["Y_raw"])


@pytest.mark.parametrize("cell", ["lstm", "gru", "rnn"])
def test_single_step_layers_use_few_rows_projection(cell):
    """Layers of one step and a batch of up to four (one step of a decoder):
    the whole layer through the few-rows projection matches the oracle."""
    for N in (1, 3):
        pr = rk.Problem(cell, seq=1, batch=N, input=64, hidden=48, direction="bidirectional",
                        linear_before_reset=1 if cell == "gru" else 0)
        inp = rand_inputs(pr, seed=90 + N, lens=[1] * N, peep=True)
        compare(pr, run_gpu(pr, inp), run_oracle(pr, inp), [1] * N)
