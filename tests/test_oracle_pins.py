"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties a part of the oracle to a fact fixed by the pages or by
mathematics: the pages' worked Gemm example, closed forms at hidden size 1,
torch.nn.LSTM / GRU / RNN in float64 (a library special case of the default
activations), torch.nn.functional for the activations, and invariants of the
definition (reverse vs time-reversed forward, bidirectional vs its halves,
layout 1 vs layout 0, zeroing past the sequence length, ...).  The choice is
made so that a dropped term, a wrong sign, a wrong index, a transposed
operand or a wrong gate order fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import load_golden

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def spec(cell, direction="forward", layout=0, seq=1, batch=1, input=1, hidden=1,
         clip=0.0, input_forget=0, linear_before_reset=0, activations=None):
    return dict(cell=cell, direction=direction, layout=layout, seq=seq, batch=batch,
                input=input, hidden=hidden, clip=clip, input_forget=input_forget,
                linear_before_reset=linear_before_reset, activations=activations)


def rand_inputs(rng, s, with_bias=True, with_init=True, with_p=False, lens=None, scale=0.5):
    G = oracle.GATES[s["cell"]]
    D = 2 if s["direction"] == "bidirectional" else 1
    S, NB, I, H = s["seq"], s["batch"], s["input"], s["hidden"]
    X = rng.uniform(-1, 1, (S, NB, I) if s["layout"] == 0 else (NB, S, I))
    W = rng.uniform(-scale, scale, (D, G * H, I))
    R = rng.uniform(-scale, scale, (D, G * H, H))
    B = rng.uniform(-scale, scale, (D, 2 * G * H)) if with_bias else None
    st = (D, NB, H) if s["layout"] == 0 else (NB, D, H)
    h0 = rng.uniform(-1, 1, st) if with_init else None
    c0 = rng.uniform(-1, 1, st) if (with_init and s["cell"] == "lstm") else None
    P = rng.uniform(-scale, scale, (D, 3 * H)) if with_p else None
    return dict(X=X, W=W, R=R, B=B, sequence_lens=lens, initial_h=h0, initial_c=c0, P=P)


# ---------------------------------------------------------------- projection

def test_projection_matches_getting_started_example():
    """The pages' worked example: A (4x2) times B (2x3) prints the rows
    1 2 8 / 3 4 18 / 5 6 28 / 7 8 38.  The layer's projection takes W in the
    transposed-B form, so W = B^T."""
    g = load_golden("gemm_getting_started.txt")
    out = oracle.projection(g["A"], g["B"].T.copy())
    assert np.array_equal(out, g["C"])


def test_rnn_affine_identity_reproduces_example_rows():
    """End to end: an RNN with Affine(1, 0), R = 0 and no bias outputs the
    projection itself, so Y[t] is row t of the example (exact integers)."""
    g = load_golden("gemm_getting_started.txt")
    W = g["B"].T.copy()[None]               # [1, 3, 2]
    R = np.zeros((1, 3, 3))
    for layout in (0, 1):
        for direction in ("forward", "reverse"):
            s = spec("rnn", direction=direction, layout=layout, seq=4, batch=1, input=2,
                     hidden=3, activations=[("affine", 1.0, 0.0)])
            X = g["A"].reshape(4, 1, 2) if layout == 0 else g["A"].reshape(1, 4, 2)
            out = oracle.layer(s, X, W, R)
            Y = out["Y"].reshape(4, 3)
            assert np.array_equal(Y, g["C"]), (layout, direction)
            last = g["C"][3] if direction == "forward" else g["C"][0]
            assert np.array_equal(out["Y_h"].reshape(3), last)


# ---------------------------------------------------------------- activations

X_PTS = np.array([-7.5, -2.0, -1.0, -0.3, 0.0, 0.25, 0.5, 1.0, 2.0, 9.0])


@pytest.mark.parametrize("name,alpha,beta,ref", [
    ("sigmoid", 0, 0, lambda x: torch.sigmoid(x)),
    ("tanh", 0, 0, lambda x: torch.tanh(x)),
    ("relu", 0, 0, lambda x: torch.relu(x)),
    ("leakyrelu", 0.01, 0, lambda x: torch.nn.functional.leaky_relu(x, 0.01)),
    ("leakyrelu", 0.3, 0, lambda x: torch.nn.functional.leaky_relu(x, 0.3)),
    ("thresholdedrelu", 1.0, 0, lambda x: torch.nn.functional.threshold(x, 1.0, 0.0)),
    ("thresholdedrelu", 0.2, 0, lambda x: torch.nn.functional.threshold(x, 0.2, 0.0)),
    ("hardsigmoid", 1 / 6, 0.5, lambda x: torch.nn.functional.hardsigmoid(x)),
    ("elu", 1.0, 0, lambda x: torch.nn.functional.elu(x, 1.0)),
    ("elu", 0.7, 0, lambda x: torch.nn.functional.elu(x, 0.7)),
    ("softsign", 0, 0, lambda x: torch.nn.functional.softsign(x)),
    ("softplus", 0, 0, lambda x: torch.nn.functional.softplus(x, beta=1.0, threshold=1000.0)),
])
def test_activation_matches_torch(name, alpha, beta, ref):
    x = torch.tensor(X_PTS, dtype=torch.float64)
    want = ref(x).numpy()
    got = np.array([oracle.activation(name, alpha, beta, v) for v in X_PTS])
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-15)


def test_activation_closed_forms():
    ln3 = math.log(3.0)
    # sigmoid(ln 3) = 3/4, tanh(ln 3) = (9 - 1)/(9 + 1) = 4/5
    assert oracle.activation("sigmoid", 0, 0, ln3) == pytest.approx(0.75, abs=1e-15)
    assert oracle.activation("tanh", 0, 0, ln3) == pytest.approx(0.8, abs=1e-15)
    assert oracle.activation("affine", 2.0, 0.5, 3.0) == 6.5
    assert oracle.activation("affine", -1.0, 0.0, 3.0) == -3.0
    # ScaledTanh(a, b)(x) = a * tanh(b * x): a = 2, b = 0.5 at x = 2 ln 3 gives 1.6
    assert oracle.activation("scaledtanh", 2.0, 0.5, 2 * ln3) == pytest.approx(1.6, abs=1e-15)
    # HardSigmoid(0.2, 0.5): 0 -> 0.5, 1 -> 0.7, saturates at 0 and 1
    assert oracle.activation("hardsigmoid", 0.2, 0.5, 0.0) == 0.5
    assert oracle.activation("hardsigmoid", 0.2, 0.5, 1.0) == pytest.approx(0.7, abs=1e-16)
    assert oracle.activation("hardsigmoid", 0.2, 0.5, 3.0) == 1.0
    assert oracle.activation("hardsigmoid", 0.2, 0.5, -3.0) == 0.0
    # Softplus(0) = ln 2, Softsign(1) = 1/2, Elu(-ln 2) = -alpha/2
    assert oracle.activation("softplus", 0, 0, 0.0) == pytest.approx(math.log(2.0), abs=1e-16)
    assert oracle.activation("softsign", 0, 0, 1.0) == 0.5
    assert oracle.activation("elu", 0.8, 0, -math.log(2.0)) == pytest.approx(-0.4, abs=1e-16)
    # ThresholdedRelu is strict: x == alpha gives 0
    assert oracle.activation("thresholdedrelu", 1.0, 0, 1.0) == 0.0


# ---------------------------------------------------------------- closed forms, hidden 1

def _sig(x):
    return 1.0 / (1.0 + math.exp(-x))


def test_lstm_hidden1_two_steps_with_peepholes():
    """LSTM, I = H = 1, two steps, peepholes, initial state.  The expected
    values are worked through by hand below (gate order i, o, f, c; P order
    i, o, f; i and f see the previous c, o sees the new c)."""
    wi, wo, wf, wc = 0.5, -0.25, 0.75, 1.5
    ri, ro, rf, rc = 0.2, 0.1, -0.3, 0.4
    bi, bo, bf, bc = 0.1, 0.2, 0.3, -0.1       # Wb
    ci, co, cf, cc = -0.05, 0.05, 0.15, 0.25   # Rb
    pi, po, pf = 0.6, -0.7, 0.8
    x = [1.0, -2.0]
    h, c = 0.5, -0.4
    ys = []
    for t in range(2):
        pre_i = ((wi * x[t] + ri * h) + bi) + ci + pi * c
        pre_f = ((wf * x[t] + rf * h) + bf) + cf + pf * c
        pre_c = ((wc * x[t] + rc * h) + bc) + cc
        pre_o = ((wo * x[t] + ro * h) + bo) + co
        i, f, g = _sig(pre_i), _sig(pre_f), math.tanh(pre_c)
        c = f * c + i * g
        o = _sig(pre_o + po * c)
        h = o * math.tanh(c)
        ys.append(h)
    s = spec("lstm", seq=2)
    out = oracle.layer(s, np.array(x).reshape(2, 1, 1),
                       np.array([wi, wo, wf, wc]).reshape(1, 4, 1),
                       np.array([ri, ro, rf, rc]).reshape(1, 4, 1),
                       B=np.array([bi, bo, bf, bc, ci, co, cf, cc]).reshape(1, 8),
                       initial_h=np.array([[[0.5]]]), initial_c=np.array([[[-0.4]]]),
                       P=np.array([pi, po, pf]).reshape(1, 3))
    np.testing.assert_allclose(out["Y"].reshape(2), ys, rtol=1e-14)
    assert out["Y_h"].item() == pytest.approx(ys[-1], rel=1e-14)
    assert out["Y_c"].item() == pytest.approx(c, rel=1e-14)


def test_lstm_hidden1_exact_numbers():
    """Numbers that come out exactly: with pre_i = ln 3 the input gate is 3/4,
    with pre_c = ln 3 the candidate is 4/5, so c = 3/4 * 4/5 = 3/5 (f*c = 0 from
    the zero initial state); with p_o = ln 3 / (3/5) the output gate sees ln 3
    and is 3/4, so h = 3/4 * tanh(3/5).  input_forget then makes f = 1 - i."""
    ln3 = math.log(3.0)
    s = spec("lstm")
    W = np.array([ln3, 0.0, 0.0, ln3]).reshape(1, 4, 1)
    R = np.zeros((1, 4, 1))
    P = np.array([0.0, ln3 / 0.6, 0.0]).reshape(1, 3)
    out = oracle.layer(s, np.ones((1, 1, 1)), W, R, P=P)
    assert out["Y_c"].item() == pytest.approx(0.6, abs=1e-15)
    assert out["Y_h"].item() == pytest.approx(0.75 * math.tanh(0.6), abs=1e-15)
    # input_forget: f = 1 - i = 1/4 regardless of the f row; c0 = 1 gives
    # c = 1/4 * 1 + 3/4 * 4/5 = 17/20
    s2 = spec("lstm", input_forget=1)
    W2 = np.array([ln3, 0.0, 123.0, ln3]).reshape(1, 4, 1)
    out2 = oracle.layer(s2, np.ones((1, 1, 1)), W2, R, initial_c=np.ones((1, 1, 1)))
    assert out2["Y_c"].item() == pytest.approx(0.85, abs=1e-15)


@pytest.mark.parametrize("lbr", [0, 1])
def test_gru_hidden1_closed_form(lbr):
    """GRU, I = H = 1, one step from h0 = 0.8, gate order z, r, h.  lbr = 0:
    h~ = g(((xw_h + R_h*(r*h0)) + Wb_h) + Rb_h); lbr = 1:
    h~ = g((xw_h + r*(R_h*h0 + Rb_h)) + Wb_h); h = (1 - z)*h~ + z*h0."""
    wz, wr, wh = 0.3, -0.6, 0.9
    rz, rr, rh = 0.5, 0.4, -1.2
    bz, br, bh = 0.1, 0.2, 0.3
    cz, cr, ch = -0.2, 0.1, 0.7
    x, h0 = 1.5, 0.8
    z = _sig(((wz * x + rz * h0) + bz) + cz)
    r = _sig(((wr * x + rr * h0) + br) + cr)
    if lbr == 0:
        pre_h = ((wh * x + rh * (r * h0)) + bh) + ch
    else:
        pre_h = (wh * x + r * (rh * h0 + ch)) + bh
    want = (1 - z) * math.tanh(pre_h) + z * h0
    s = spec("gru", linear_before_reset=lbr)
    out = oracle.layer(s, np.array(x).reshape(1, 1, 1), np.array([wz, wr, wh]).reshape(1, 3, 1),
                       np.array([rz, rr, rh]).reshape(1, 3, 1),
                       B=np.array([bz, br, bh, cz, cr, ch]).reshape(1, 6),
                       initial_h=np.array([[[h0]]]))
    assert out["Y_h"].item() == pytest.approx(want, rel=1e-14)
    # the two forms differ here (r != 1, Rb_h != 0): a swapped form would fail
    other = (wh * x + r * (rh * h0 + ch)) + bh if lbr == 0 else ((wh * x + rh * (r * h0)) + bh) + ch
    assert abs(math.tanh(other) - math.tanh(pre_h)) > 1e-3


def test_gru_lbr0_reset_applies_per_source_unit():
    """GRU with linear_before_reset = 0 and H = 2 (torch has no such form):
    the candidate's product is R_h . (r (.) h_prev), so unit j's sum weighs
    h_prev[k] by r[k], the reset gate of the SOURCE unit k.  Identity
    (Affine(1, 0)) activations, one step, x = 1, h0 = (1, 2), no bias,
    W_z = (1/2, 1/4), W_r = (1/2, 2), W_h = 0, R = 0 except
    R_h = [[1, 1/2], [1/4, 1]].  By hand: r (.) h0 = (1/2, 4);
    pre_h = (1/2 + 2, 1/8 + 4) = (5/2, 33/8); h = (1 - z) h~ + z h0 =
    (1/2 * 5/2 + 1/2, 3/4 * 33/8 + 1/2) = (7/4, 115/32).  Weighting by r[j]
    instead, or reading R_h transposed, changes both values."""
    s = spec("gru", hidden=2, linear_before_reset=0, activations=[("affine", 1.0, 0.0)] * 2)
    W = np.array([0.5, 0.25, 0.5, 2.0, 0.0, 0.0]).reshape(1, 6, 1)
    R = np.zeros((1, 6, 2))
    R[0, 4:6] = [[1.0, 0.5], [0.25, 1.0]]
    out = oracle.layer(s, np.ones((1, 1, 1)), W, R, initial_h=np.array([1.0, 2.0]).reshape(1, 1, 2))
    assert out["Y_h"].reshape(2).tolist() == [1.75, 115.0 / 32.0]


def test_rnn_hidden1_relu_and_clip():
    """RNN with Relu: h1 = relu(w*x1 + r*h0 + b), h2 = relu(w*x2 + r*h1 + b).
    A clip of 0.25 clamps the pre-activation before the activation."""
    w, r, wb, rb = 2.0, 0.5, 0.25, -0.5
    xs, h = [1.0, -3.0, 0.5], 1.0
    want = []
    for x in xs:
        h = max(0.0, ((w * x + r * h) + wb) + rb)
        want.append(h)
    s = spec("rnn", seq=3, activations=[("relu", 0, 0)])
    args = (np.array(xs).reshape(3, 1, 1), np.full((1, 1, 1), w), np.full((1, 1, 1), r))
    out = oracle.layer(s, *args, B=np.array([[wb, rb]]), initial_h=np.ones((1, 1, 1)))
    np.testing.assert_array_equal(out["Y"].reshape(3), want)
    s_clip = spec("rnn", seq=3, activations=[("affine", 1.0, 0.0)], clip=0.25)
    out = oracle.layer(s_clip, *args, B=np.array([[wb, rb]]), initial_h=np.ones((1, 1, 1)))
    np.testing.assert_array_equal(out["Y"].reshape(3), [0.25, -0.25, 0.25])


def test_lstm_activation_slots_by_direction():
    """Bidirectional LSTM, I = H = 1, one step from zero state, x = 1, R = 0,
    no bias, Affine activations with a different (alpha, beta) in each of the
    six slots (f, g, h of direction 0, then of direction 1).  Worked by hand
    in dyadic numbers, so exact: direction 0 with f = (1/2, 1/4), g = (2, -1),
    h = (-1, 1/2) and W = (i 1, o 1/2, f 3, c 3/4): i = 3/4, c~ = 1/2,
    c = 3/8, o = 1/2, h = 1/2 * (1/2 - 3/8) = 1/16.  Direction 1 with
    f = (1/4, 1/2), g = (-1, 1/4), h = (4, 0): i = 3/4, c~ = -1/2, c = -3/8,
    o = 5/8, h = 5/8 * (-3/2) = -15/16.  Swapping g and h, or giving one
    direction the other's slots, changes every one of these values."""
    acts = [("affine", 0.5, 0.25), ("affine", 2.0, -1.0), ("affine", -1.0, 0.5),
            ("affine", 0.25, 0.5), ("affine", -1.0, 0.25), ("affine", 4.0, 0.0)]
    s = spec("lstm", direction="bidirectional", activations=acts)
    W = np.array([1.0, 0.5, 3.0, 0.75] * 2).reshape(2, 4, 1)
    out = oracle.layer(s, np.ones((1, 1, 1)), W, np.zeros((2, 4, 1)))
    assert out["Y_c"].reshape(2).tolist() == [0.375, -0.375]
    assert out["Y_h"].reshape(2).tolist() == [0.0625, -0.9375]
    assert out["Y"].reshape(2).tolist() == [0.0625, -0.9375]


def test_gru_activation_slots_by_direction():
    """Bidirectional GRU (linear_before_reset = 1), I = H = 1, one step, x = 1,
    h0 = 1, W = (z 1, r 1, h 1/4), R = (0, 0, 1/2), no bias, Affine slots
    (f, g of direction 0, then of direction 1), worked by hand: direction 0,
    f = (1/2, 0), g = (2, 1/2): z = r = 1/2, pre_h = 1/4 + 1/2 * 1/2 = 1/2,
    h~ = 3/2, h = 1/2 * 3/2 + 1/2 * 1 = 5/4.  Direction 1, f = (1/4, 1/2),
    g = (-1, 0): z = r = 3/4, pre_h = 1/4 + 3/4 * 1/2 = 5/8, h~ = -5/8,
    h = 1/4 * -5/8 + 3/4 = 19/32."""
    acts = [("affine", 0.5, 0.0), ("affine", 2.0, 0.5), ("affine", 0.25, 0.5), ("affine", -1.0, 0.0)]
    s = spec("gru", direction="bidirectional", linear_before_reset=1, activations=acts)
    W = np.array([1.0, 1.0, 0.25] * 2).reshape(2, 3, 1)
    R = np.array([0.0, 0.0, 0.5] * 2).reshape(2, 3, 1)
    out = oracle.layer(s, np.ones((1, 1, 1)), W, R, initial_h=np.ones((2, 1, 1)))
    assert out["Y_h"].reshape(2).tolist() == [1.25, 0.59375]


def test_rnn_activation_slot_by_direction():
    """Bidirectional RNN, one slot per direction: x = 1, W = 1/4, R = 0,
    Affine(2, 0) forward gives 1/2, Affine(-1, 1/2) backward gives 1/4."""
    s = spec("rnn", direction="bidirectional", activations=[("affine", 2.0, 0.0), ("affine", -1.0, 0.5)])
    out = oracle.layer(s, np.ones((1, 1, 1)), np.full((2, 1, 1), 0.25), np.zeros((2, 1, 1)))
    assert out["Y_h"].reshape(2).tolist() == [0.5, 0.25]


# ---------------------------------------------------------------- torch special case

def _torch_module(cell, I, H, bidirectional, batch_first):
    cls = {"lstm": torch.nn.LSTM, "gru": torch.nn.GRU, "rnn": torch.nn.RNN}[cell]
    return cls(I, H, num_layers=1, bias=True, batch_first=batch_first,
               bidirectional=bidirectional).double()


# our gate order -> torch's: LSTM i,o,f,c -> i,f,g,o ; GRU z,r,h -> r,z,n
_PERM = {"lstm": [0, 2, 3, 1], "gru": [1, 0, 2], "rnn": [0]}


def _to_torch(cell, M, H):
    blocks = [M[g * H:(g + 1) * H] for g in range(len(_PERM[cell]))]
    return np.concatenate([blocks[g] for g in _PERM[cell]], axis=0)


@pytest.mark.parametrize("cell", ["lstm", "gru", "rnn"])
@pytest.mark.parametrize("direction", ["forward", "bidirectional"])
@pytest.mark.parametrize("layout", [0, 1])
def test_default_cells_match_torch_float64(cell, direction, layout):
    """torch.nn.LSTM / GRU / RNN in float64 on the CPU compute the default-
    activation cells (GRU with linear_before_reset = 1, which is torch's form)
    after the gate reorder; biases map to b_ih = Wb and b_hh = Rb."""
    rng = np.random.default_rng(7)
    S, NB, I, H = 5, 3, 4, 6
    s = spec(cell, direction=direction, layout=layout, seq=S, batch=NB, input=I, hidden=H,
             linear_before_reset=1 if cell == "gru" else 0)
    a = rand_inputs(rng, s)
    out = oracle.layer(s, **a)
    D = 2 if direction == "bidirectional" else 1
    G = oracle.GATES[cell]
    m = _torch_module(cell, I, H, D == 2, layout == 1)
    with torch.no_grad():
        for d in range(D):
            sfx = "_reverse" if d == 1 else ""
            getattr(m, "weight_ih_l0" + sfx).copy_(torch.from_numpy(_to_torch(cell, a["W"][d], H)))
            getattr(m, "weight_hh_l0" + sfx).copy_(torch.from_numpy(_to_torch(cell, a["R"][d], H)))
            getattr(m, "bias_ih_l0" + sfx).copy_(torch.from_numpy(_to_torch(cell, a["B"][d][:G * H], H)))
            getattr(m, "bias_hh_l0" + sfx).copy_(torch.from_numpy(_to_torch(cell, a["B"][d][G * H:], H)))
        h0 = a["initial_h"] if layout == 0 else a["initial_h"].transpose(1, 0, 2)
        h0 = torch.from_numpy(np.ascontiguousarray(h0))
        if cell == "lstm":
            c0 = a["initial_c"] if layout == 0 else a["initial_c"].transpose(1, 0, 2)
            y, (hn, cn) = m(torch.from_numpy(a["X"]), (h0, torch.from_numpy(np.ascontiguousarray(c0))))
        else:
            y, hn = m(torch.from_numpy(a["X"]), h0)
    y = y.numpy()
    # torch: [S, B, D*H] (batch_first: [B, S, D*H]) -> ours [S, D, B, H] / [B, S, D, H]
    if layout == 0:
        ours = out["Y"].transpose(0, 2, 1, 3).reshape(S, NB, D * H)
        ours_h = out["Y_h"]
    else:
        ours = out["Y"].reshape(NB, S, D * H)
        ours_h = out["Y_h"].transpose(1, 0, 2)
    np.testing.assert_allclose(ours, y, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ours_h, hn.numpy(), rtol=1e-12, atol=1e-13)
    if cell == "lstm":
        ours_c = out["Y_c"] if layout == 0 else out["Y_c"].transpose(1, 0, 2)
        np.testing.assert_allclose(ours_c, cn.numpy(), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("cell", ["lstm", "gru", "rnn"])
def test_reverse_equals_forward_on_time_reversed_rows(cell):
    """Row b in reverse over its first L steps equals the forward run on
    those L steps reversed in time; Y past L is zero; Y_h is Y at step 0
    (reverse) or L - 1 (forward)."""
    rng = np.random.default_rng(11)
    S, NB, I, H = 7, 3, 3, 4
    lens = np.array([7, 4, 0], dtype=np.int32)
    s_rev = spec(cell, direction="reverse", seq=S, batch=NB, input=I, hidden=H)
    a = rand_inputs(rng, s_rev, with_p=(cell == "lstm"), lens=lens)
    rev = oracle.layer(s_rev, **a)
    for b in range(NB):
        L = int(lens[b])
        if L == 0:
            assert not rev["Y"][:, 0, b].any() and not rev["Y_h"][0, b].any()
            continue
        sb = spec(cell, seq=L, batch=1, input=I, hidden=H)
        ab = dict(a)
        ab["X"] = a["X"][:L, b:b + 1][::-1].copy()
        ab["initial_h"] = a["initial_h"][:, b:b + 1]
        ab["initial_c"] = a["initial_c"][:, b:b + 1] if a["initial_c"] is not None else None
        ab["sequence_lens"] = None
        fwd = oracle.layer(sb, **ab)
        np.testing.assert_array_equal(rev["Y"][:L, 0, b], fwd["Y"][::-1, 0, 0])
        assert not rev["Y"][L:, 0, b].any()
        np.testing.assert_array_equal(rev["Y_h"][0, b], rev["Y"][0, 0, b])
        np.testing.assert_array_equal(rev["Y_h"][0, b], fwd["Y_h"][0, 0])


@pytest.mark.parametrize("cell", ["lstm", "gru", "rnn"])
def test_bidirectional_is_concatenation_of_halves(cell):
    rng = np.random.default_rng(12)
    S, NB, I, H = 6, 2, 3, 5
    lens = np.array([6, 3], dtype=np.int32)
    acts = {"lstm": [("hardsigmoid", 0.2, 0.5), ("softsign", 0, 0), ("elu", 0.9, 0),
                     ("sigmoid", 0, 0), ("tanh", 0, 0), ("softplus", 0, 0)],
            "gru": [("sigmoid", 0, 0), ("leakyrelu", 0.1, 0), ("hardsigmoid", 0.3, 0.4), ("scaledtanh", 0.9, 1.1)],
            "rnn": [("relu", 0, 0), ("thresholdedrelu", 0.1, 0)]}[cell]
    s = spec(cell, direction="bidirectional", seq=S, batch=NB, input=I, hidden=H,
             activations=acts, clip=2.0)
    a = rand_inputs(rng, s, with_p=(cell == "lstm"), lens=lens)
    both = oracle.layer(s, **a)
    A = oracle.ACTS_PER_DIR[cell]
    for d, direction in enumerate(("forward", "reverse")):
        sd = spec(cell, direction=direction, seq=S, batch=NB, input=I, hidden=H,
                  activations=acts[d * A:(d + 1) * A], clip=2.0)
        ad = {k: (v[d:d + 1] if (v is not None and k in ("W", "R", "B", "P", "initial_h", "initial_c")) else v)
              for k, v in a.items()}
        half = oracle.layer(sd, **ad)
        np.testing.assert_array_equal(both["Y"][:, d], half["Y"][:, 0])
        np.testing.assert_array_equal(both["Y_h"][d], half["Y_h"][0])


@pytest.mark.parametrize("cell", ["lstm", "gru"])
def test_layout1_is_layout0_transposed(cell):
    rng = np.random.default_rng(13)
    S, NB, I, H = 4, 3, 2, 3
    s0 = spec(cell, direction="bidirectional", layout=0, seq=S, batch=NB, input=I, hidden=H)
    a = rand_inputs(rng, s0, lens=np.array([4, 2, 1], dtype=np.int32))
    out0 = oracle.layer(s0, **a)
    s1 = dict(s0, layout=1)
    a1 = dict(a)
    a1["X"] = a["X"].transpose(1, 0, 2).copy()
    a1["initial_h"] = a["initial_h"].transpose(1, 0, 2).copy()
    if a["initial_c"] is not None:
        a1["initial_c"] = a["initial_c"].transpose(1, 0, 2).copy()
    out1 = oracle.layer(s1, **a1)
    np.testing.assert_array_equal(out1["Y"], out0["Y"].transpose(2, 0, 1, 3))
    np.testing.assert_array_equal(out1["Y_h"], out0["Y_h"].transpose(1, 0, 2))


def test_batch_rows_are_independent_and_permute():
    rng = np.random.default_rng(14)
    s = spec("lstm", seq=5, batch=4, input=3, hidden=4)
    a = rand_inputs(rng, s, with_p=True, lens=np.array([5, 1, 3, 0], dtype=np.int32))
    out = oracle.layer(s, **a)
    perm = [2, 0, 3, 1]
    ap = dict(a)
    ap["X"] = a["X"][:, perm].copy()
    ap["initial_h"] = a["initial_h"][:, perm].copy()
    ap["initial_c"] = a["initial_c"][:, perm].copy()
    ap["sequence_lens"] = a["sequence_lens"][perm].copy()
    outp = oracle.layer(s, **ap)
    np.testing.assert_array_equal(outp["Y"], out["Y"][:, :, perm])
    np.testing.assert_array_equal(outp["Y_c"], out["Y_c"][:, perm])


def test_seq0_gives_initial_state_and_len0_gives_zero():
    rng = np.random.default_rng(15)
    s = spec("lstm", seq=0, batch=2, input=3, hidden=4)
    a = rand_inputs(rng, s)
    out = oracle.layer(s, **a)
    np.testing.assert_array_equal(out["Y_h"], a["initial_h"])
    np.testing.assert_array_equal(out["Y_c"], a["initial_c"])
    s1 = spec("gru", seq=3, batch=2, input=3, hidden=4)
    a1 = rand_inputs(rng, s1, lens=np.array([0, 2], dtype=np.int32))
    out1 = oracle.layer(s1, **a1)
    assert not out1["Y_h"][0, 0].any() and out1["Y_h"][0, 1].any()
    assert not out1["Y"][:, 0, 0].any() and not out1["Y"][2, 0, 1].any()
    # lengths above seq act as seq, negative as 0
    a2 = dict(a1, sequence_lens=np.array([-5, 99], dtype=np.int32))
    out2 = oracle.layer(s1, **a2)
    a3 = dict(a1, sequence_lens=np.array([0, 3], dtype=np.int32))
    out3 = oracle.layer(s1, **a3)
    np.testing.assert_array_equal(out2["Y"], out3["Y"])


def test_out_of_range_lengths_clamp():
    """A negative length runs as 0 steps and one above seq as seq (the
    kernels read lengths unvalidated, so the oracle fixes the same reading)."""
    rng = np.random.default_rng(19)
    s = spec("lstm", direction="bidirectional", seq=5, batch=3, input=2, hidden=3)
    a = rand_inputs(rng, s, with_p=True)
    got = oracle.layer(s, **dict(a, sequence_lens=np.array([-3, 99, 2], dtype=np.int32)))
    want = oracle.layer(s, **dict(a, sequence_lens=np.array([0, 5, 2], dtype=np.int32)))
    for k in ("Y", "Y_h", "Y_c"):
        np.testing.assert_array_equal(got[k], want[k])
    assert not want["Y"][:, :, 0].any() and not want["Y_h"][:, 0].any()


def test_options():
    rng = np.random.default_rng(16)
    s = spec("lstm", seq=4, batch=2, input=3, hidden=3)
    a = rand_inputs(rng, s, with_p=True, scale=2.0)
    base = oracle.layer(s, **a)
    # a clip far above any pre-activation changes nothing
    big = oracle.layer(dict(s, clip=1e30), **a)
    np.testing.assert_array_equal(big["Y"], base["Y"])
    # a clip that bites changes the result
    small = oracle.layer(dict(s, clip=0.1), **a)
    assert np.abs(small["Y"] - base["Y"]).max() > 1e-3
    # input_forget ignores the f rows of W, R, B and P
    sf = dict(s, input_forget=1)
    f1 = oracle.layer(sf, **a)
    H = 3
    a2 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in a.items()}
    a2["W"][:, 2 * H:3 * H] = 77.0
    a2["R"][:, 2 * H:3 * H] = -55.0
    a2["B"][:, 2 * H:3 * H] = 9.0
    a2["B"][:, 4 * H + 2 * H:4 * H + 3 * H] = 9.0
    a2["P"][:, 2 * H:3 * H] = 3.0
    f2 = oracle.layer(sf, **a2)
    np.testing.assert_array_equal(f1["Y"], f2["Y"])
    assert np.abs(f1["Y"] - base["Y"]).max() > 1e-3


def test_lstm_clip_after_peepholes_exact():
    """LSTM, I = H = 1, one step, x = 1, h0 = 0, c0 = 2, clip 1/2, identity
    (Affine(1, 0)) in every slot, W = (i 1/4, o 1/4, f 1/4, c 2), R = 0, no
    bias, P = (i 1, o -4, f -1).  By hand: pre_i = 1/4 + 1 * 2 = 9/4 -> clipped
    1/2; pre_f = 1/4 - 2 -> -1/2; the candidate 2 -> 1/2 (clip covers it);
    c = -1/2 * 2 + 1/2 * 1/2 = -3/4 (the state itself is not clipped); pre_o =
    1/4 - 4 * (-3/4) = 13/4 with the new c -> 1/2; h = 1/2 * (-3/4) = -3/8.
    Clipping before the peepholes, the old c in the o peephole, an unclipped
    candidate or a clipped state each change these numbers."""
    s = spec("lstm", clip=0.5, activations=[("affine", 1.0, 0.0)] * 3)
    out = oracle.layer(s, np.ones((1, 1, 1)), np.array([0.25, 0.25, 0.25, 2.0]).reshape(1, 4, 1),
                       np.zeros((1, 4, 1)), initial_c=np.full((1, 1, 1), 2.0),
                       P=np.array([1.0, -4.0, -1.0]).reshape(1, 3))
    assert out["Y_c"].item() == -0.75
    assert out["Y_h"].item() == -0.375


def test_gru_forms_coincide_when_reset_gate_is_one():
    """With the r gate forced to 1 (a huge r bias) and Rb_h = 0 the two
    linear_before_reset forms are the same expression."""
    rng = np.random.default_rng(17)
    H = 4
    s = spec("gru", seq=5, batch=2, input=3, hidden=H)
    a = rand_inputs(rng, s)
    a["B"][:, H:2 * H] = 1e3
    a["B"][:, 3 * H + 2 * H:] = 0.0
    o0 = oracle.layer(s, **a)
    o1 = oracle.layer(dict(s, linear_before_reset=1), **a)
    np.testing.assert_array_equal(o0["Y"], o1["Y"])
    a["B"][:, H:2 * H] = 0.0
    o2 = oracle.layer(s, **a)
    assert np.abs(o2["Y"] - o0["Y"]).max() > 1e-3


def test_nan_passes_through_clip():
    s = spec("rnn", seq=1, batch=2, activations=[("affine", 1.0, 0.0)], clip=1.0)
    X = np.array([np.nan, 0.5]).reshape(1, 2, 1)
    out = oracle.layer(s, X, np.ones((1, 1, 1)), np.zeros((1, 1, 1)))
    assert math.isnan(out["Y"][0, 0, 0].item()) and out["Y"][0, 0, 1].item() == 0.5
