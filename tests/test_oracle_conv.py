"""Pins of the convolution-state oracle (oracle/conv.py) against things other
than itself: numpy.convolve over a whole sequence, the state after a
sequence, the logistic function from scipy, and a hand-worked example."""
import os

import numpy as np
import pytest

from oracle import conv as oc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "conv_scalar.txt")


def run_sequence(u_seq, weight, bias, state0, activation):
    """Step the oracle through a [T, B, C] input sequence."""
    st = state0
    outs = []
    for u in u_seq:
        st, out = oc.conv_state_step(st, u, weight, bias, activation)
        outs.append(out)
    return st, np.stack(outs)


@pytest.mark.parametrize("W", [2, 3, 4])
def test_steps_equal_causal_convolution(W):
    """From a zero state, T decode steps are the causal depthwise convolution
    of each channel's input sequence: numpy.convolve with the weight row
    reversed (convolution flips the kernel; the step is a correlation)."""
    rng = np.random.default_rng(1)
    B, C, T = 2, 5, 9
    u_seq = rng.standard_normal((T, B, C))
    weight = rng.standard_normal((C, W))
    bias = rng.standard_normal(C)
    _, outs = run_sequence(u_seq, weight, bias, np.zeros((B, C, W - 1)), activation=False)
    for b in range(B):
        for c in range(C):
            ref = np.convolve(u_seq[:, b, c], weight[c, ::-1])[:T] + bias[c]
            np.testing.assert_allclose(outs[:, b, c], ref, rtol=1e-13, atol=1e-13)


def test_state_holds_the_last_inputs_oldest_first():
    rng = np.random.default_rng(2)
    B, C, W, T = 3, 4, 4, 6
    u_seq = rng.standard_normal((T, B, C))
    st, _ = run_sequence(u_seq, rng.standard_normal((C, W)), None, rng.standard_normal((B, C, W - 1)), True)
    np.testing.assert_array_equal(st, np.moveaxis(u_seq[-(W - 1):], 0, -1))


def test_nonzero_state_is_the_history_before_the_step():
    """A step from a state equals the convolution of the concatenated history
    (state columns, then the new input), read at the last position."""
    rng = np.random.default_rng(3)
    B, C, W = 2, 3, 4
    state = rng.standard_normal((B, C, W - 1))
    u = rng.standard_normal((B, C))
    weight = rng.standard_normal((C, W))
    _, out = oc.conv_state_step(state, u, weight, None, activation=False)
    for b in range(B):
        for c in range(C):
            hist = np.concatenate([state[b, c], [u[b, c]]])
            np.testing.assert_allclose(out[b, c], np.convolve(hist, weight[c, ::-1])[W - 1], rtol=1e-13)


def test_silu_is_z_times_logistic():
    special = pytest.importorskip("scipy.special")
    z = np.linspace(-30.0, 30.0, 241)
    np.testing.assert_allclose(oc.silu(z), z * special.expit(z), rtol=1e-14, atol=1e-300)
    assert oc.silu(0.0) == 0.0


def test_activation_applies_silu_to_the_convolution():
    rng = np.random.default_rng(4)
    state, u = rng.standard_normal((2, 3, 2)), rng.standard_normal((2, 3))
    weight, bias = rng.standard_normal((3, 3)), rng.standard_normal(3)
    _, lin = oc.conv_state_step(state, u, weight, bias, activation=False)
    _, act = oc.conv_state_step(state, u, weight, bias, activation=True)
    np.testing.assert_allclose(act, oc.silu(lin), rtol=1e-15)


def test_hand_worked_example():
    """tests/golden/conv_scalar.txt: one channel, W = 3, worked by hand."""
    rows = [list(map(float, ln.split())) for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    weight = np.array([[0.5, -1.0, 2.0]])
    st = np.array([[[1.0, 2.0]]])
    for t, u, z_ref, s0, s1 in rows:
        st, z = oc.conv_state_step(st, np.array([[u]]), weight, np.array([0.25]), activation=False)
        assert z[0, 0] == z_ref, f"step {int(t)}"
        np.testing.assert_array_equal(st[0, 0], [s0, s1])


def test_split_xbc():
    out = np.arange(2 * 10).reshape(2, 10)
    x, Bm, Cm = oc.split_xbc(out, 4, 3)
    np.testing.assert_array_equal(x, out[:, :4])
    np.testing.assert_array_equal(Bm, out[:, 4:7])
    np.testing.assert_array_equal(Cm, out[:, 7:])
    with pytest.raises(ValueError):
        oc.split_xbc(out, 4, 2)
