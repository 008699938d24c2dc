"""rk_encode_noalloc: the layer with its scratch in the library's fixed device
array, for callers that cannot allocate device memory (a runtime whose memory
planner owns every device allocation, a fixed device-memory budget, code that
must not pay the synchronisation cudaFree can imply).

Each case calls the entry point through the C ABI three times in a row and
checks every output against the regular entry point rk_encode on the same
inputs, within the tolerance of the parity tests (1e-4 for float32, 5e-3 for
Half, absolute or relative), and rk_encode's result against the oracle.  The
later calls check that what an earlier call left in the shared array (barrier
counters, publication flags, exchange buffers) does not leak into the next
result; across the second and third calls the device's free memory must not
change (nothing is allocated), and the status word must report no wait that
gave up.  The cases cover the float32 SIMT step kernels (register-resident,
grid) and the Half tensor-core paths (the tcgen05 projection, the small-batch
step kernel with GRU linear_before_reset 0 and 1, flag-published teams).
This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import onnx_lstm_gru_gb300 as rk
import oracle
from onnx_lstm_gru_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "f16": 5e-3, "bf16": 2e-2}

# a Half LSTM whose hidden size needs more than one cluster of 32-unit CTAs:
# the tensor-core step kernel's flag-published teams (the publication flags
# live in the shared array's header)
TEAMS = workloads.Workload(
    "noalloc_bilstm_s20_b16_i64_h576_f16",
    rk.Problem("lstm", seq=20, batch=16, input=64, hidden=576, direction="bidirectional", dtype="f16"),
    seed=11, x=("normal", 1.0), weights=("uniform", 0.04), init_h=("normal", 0.1), init_c=("normal", 0.1),
    lens="uniform")

CASES = [
    ("bilstm_s80_b1_i256_h256_f32", 0, "step=fast"),
    ("revlstm_peep_clip_s200_b4_i128_h1024_f32", 0, "step=grid"),
    ("bigru_s128_b8_i512_h512_f16_lbr0", 0, "variant=small"),
    ("bigru_s128_b8_i512_h512_f16_lbr1", 0, "variant=small"),
    ("bilstm_s48_b8_i192_h96_f16", rk.RK_PREFER_TENSOR_STEP, "variant=small"),
    (TEAMS.name, rk.RK_PREFER_TENSOR_STEP, "variant=pairs"),
]


def workload(name):
    return TEAMS if name == TEAMS.name else workloads.WORKLOADS[name]


@pytest.fixture(scope="module")
def handles():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rk.build()
    rk.load()
    hs = {}
    yield hs
    for h in hs.values():
        rk.rk_destroy(h)


def handle_for(handles, flags):
    if flags not in handles:
        handles[flags] = rk.rk_create(flags)
    return handles[flags]


def device_operands(w):
    pr = w.problem
    inp = workloads.make_inputs(w)
    dt = rk.torch_dtype(pr.dtype)
    dev = {k: (torch.from_numpy(v) if k == "sequence_lens" else torch.from_numpy(v).to(dt)).cuda()
           for k, v in inp.items()}
    shp = pr.shapes()
    outs = {n: torch.full(shp[n], -777.0, dtype=dt, device="cuda") for n in w.outputs
            if not (n == "Y_c" and pr.cell != "lstm")}
    return inp, dev, outs


def close(a, b, tol):
    a, b = torch.as_tensor(a).double().cpu(), torch.as_tensor(b).double().cpu()
    d = (a - b).abs()
    return bool(((d <= tol) | (d <= tol * b.abs())).all())


def spec_of(pr):
    return dict(cell=pr.cell, direction=pr.direction, layout=pr.layout, seq=pr.seq, batch=pr.batch,
                input=pr.input, hidden=pr.hidden, clip=pr.clip, input_forget=pr.input_forget,
                linear_before_reset=pr.linear_before_reset,
                activations=list(pr.activations) if pr.activations else None)


@pytest.mark.parametrize("name,flags,plan", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_regular_entry(handles, name, flags, plan):
    w = workload(name)
    pr = w.problem
    tol = TOL[pr.dtype]
    h = handle_for(handles, flags)
    assert plan in rk.rk_describe_plan(h, pr.to_c())
    inp, dev, ref_out = device_operands(w)
    stream = torch.cuda.current_stream().cuda_stream
    ops = rk.operands_from_tensors(**dev, **ref_out)
    assert rk.rk_encode(h, pr.to_c(), ops, None, stream) == rk.RK_OK, rk.rk_last_error(h)
    torch.cuda.synchronize()
    # rk_encode itself against the oracle (double precision, same inputs)
    want = oracle.layer(spec_of(pr), **{k: (v.astype(np.float64) if k != "sequence_lens" else v)
                                         for k, v in inp.items()})
    for n, t in ref_out.items():
        assert close(t, want[n], tol), f"rk_encode: {n} differs from the oracle"
    outs = [{n: torch.full_like(t, -777.0) for n, t in ref_out.items()} for _ in range(3)]
    free = []
    for call in range(3):
        ops = rk.operands_from_tensors(**dev, **outs[call])
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        st = rk.rk_encode_noalloc(h, pr.to_c(), ops, stream)
        assert st == rk.RK_OK, rk.rk_last_error(h)
        torch.cuda.synchronize()
        assert rk.rk_status_poll(h, stream) == rk.RK_OK, rk.rk_last_error(h)
        for n in outs[call]:
            assert close(outs[call][n], ref_out[n], tol), f"call {call + 1}: {n} differs from rk_encode"
    free.append(torch.cuda.mem_get_info()[0])
    # the first call may load kernels and take the array's address; the
    # later calls allocate nothing at all
    assert free[1] == free[2] == free[3], f"free device memory changed across calls: {free}"


def test_noalloc_rejects_layers_beyond_its_array(handles):
    h = handle_for(handles, 0)
    w = workloads.WORKLOADS["bilstm_s512_b64_i1024_h1024_f16"]
    pr = w.problem
    shp = pr.shapes()
    ops = rk.rk_operands()
    for n in ("X", "W", "R", "Y"):
        ops.__setattr__(n, rk.rk_tensor(0x1000, 0, int(np.prod(shp[n]))))
    before = rk.rk_launch_count(h)
    st = rk.rk_encode_noalloc(h, pr.to_c(), ops, torch.cuda.current_stream().cuda_stream)
    assert st == rk.RK_ERR_UNSUPPORTED
    msg = rk.rk_last_error(h)
    assert "no-alloc scratch holds 4194304 floats" in msg and "needs" in msg
    assert rk.rk_launch_count(h) == before
