"""rk_encode_noalloc: the layer with its scratch in the library's fixed device
array, for callers that cannot allocate device memory (a runtime whose memory
planner owns every device allocation, a fixed device-memory budget, code that
must not pay the synchronisation cudaFree can imply).

Each case calls the entry point through the C ABI twice in a row and checks
both outputs against the regular entry point rk_encode on the same inputs,
within the tolerance of the parity tests (1e-4, absolute or relative, float32).
The second call checks that what the first call left in the shared array
(barrier counters, exchange buffers) does not leak into the next result.
This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import onnx_lstm_gru_gb300 as rk
from onnx_lstm_gru_gb300 import workloads

pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def handle():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rk.build()
    rk.load()
    h = rk.rk_create(0)
    yield h
    rk.rk_destroy(h)


def device_operands(w):
    pr = w.problem
    inp = workloads.make_inputs(w)
    dev = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    shp = pr.shapes()
    outs = {n: torch.full(shp[n], -777.0, dtype=torch.float32, device="cuda") for n in w.outputs
            if not (n == "Y_c" and pr.cell != "lstm")}
    return dev, outs


def close(a, b):
    d = (a.double() - b.double()).abs()
    return bool(((d <= TOL) | (d <= TOL * b.double().abs())).all())


@pytest.mark.parametrize("name", ["bilstm_s80_b1_i256_h256_f32", "revlstm_peep_clip_s200_b4_i128_h1024_f32"])
def test_noalloc_matches_regular_entry_twice(handle, name):
    w = workloads.WORKLOADS[name]
    pr = w.problem
    dev, ref_out = device_operands(w)
    stream = torch.cuda.current_stream().cuda_stream
    ops = rk.operands_from_tensors(**dev, **ref_out)
    assert rk.rk_encode(handle, pr.to_c(), ops, None, stream) == rk.RK_OK, rk.rk_last_error(handle)
    torch.cuda.synchronize()
    for call in range(2):
        outs = {n: torch.full_like(t, -777.0) for n, t in ref_out.items()}
        ops = rk.operands_from_tensors(**dev, **outs)
        st = rk.rk_encode_noalloc(handle, pr.to_c(), ops, stream)
        assert st == rk.RK_OK, rk.rk_last_error(handle)
        torch.cuda.synchronize()
        for n in outs:
            assert close(outs[n], ref_out[n]), f"call {call + 1}: {n} differs from rk_encode"


def test_noalloc_rejects_layers_beyond_its_array(handle):
    w = workloads.WORKLOADS["bilstm_s512_b64_i1024_h1024_f16"]
    pr = w.problem
    shp = pr.shapes()
    ops = rk.rk_operands()
    for n in ("X", "W", "R", "Y"):
        ops.__setattr__(n, rk.rk_tensor(0x1000, 0, int(np.prod(shp[n]))))
    before = rk.rk_launch_count(handle)
    st = rk.rk_encode_noalloc(handle, pr.to_c(), ops, torch.cuda.current_stream().cuda_stream)
    assert st == rk.RK_ERR_UNSUPPORTED
    msg = rk.rk_last_error(handle)
    assert "no-alloc scratch holds 4194304 floats" in msg and "needs" in msg
    assert rk.rk_launch_count(handle) == before
