"""Planted mistakes: each test plants one plausible error in the oracle (on the
CPU, with monkeypatch) and checks that the pins catch it, so a pin that
passes says something.  Mistakes: an off-by-one in the Mamba-2 decay
weights, a shifted ring slot, a GDN history state that drops its last entry,
GDN u stored without rounding, the wrong sign on the GDN write term, a
wrong activation and a wrong state shift in the convolution step."""
import numpy as np
import pytest

import test_oracle_conv as tc
import test_oracle_gdn as tg
import test_oracle_mamba2 as tm
from oracle import conv as oc
from oracle import gdn as og
from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def caught(pin, *args):
    """True if the pin fails under the planted mistake."""
    try:
        pin(*args)
    except AssertionError:
        return True
    return False


def test_pins_pass_unplanted():
    assert not caught(tm.test_replay_equals_recurrence, tm.SHAPES[0])
    assert not caught(tg.test_chunked_verify_random_batch)
    assert not caught(tc.test_activation_applies_silu_to_the_convolution)


def test_mamba2_decay_weight_off_by_one(monkeypatch):
    """s_j = Delta_j prod_{i >= j} a_i (one factor too many)."""
    def weights(self, b, p):
        a = [np.exp(self.A * self.ring_dt[b, :, self.slot(b, i)]) for i in range(1, p + 1)]
        abar = np.prod(a, axis=0) if a else np.ones(self.H)
        s = [self.ring_dt[b, :, self.slot(b, j)] * np.prod(a[j - 1:], axis=0) for j in range(1, p + 1)]
        return abar, s

    monkeypatch.setattr(om.Mamba2Replay, "weights", weights)
    assert caught(tm.test_replay_equals_recurrence, tm.SHAPES[0])
    assert caught(tm.test_scalar_golden_replay, 4)


def test_mamba2_ring_slot_shifted(monkeypatch):
    """The j-th entry read from slot start + j instead of start + j - 1."""
    monkeypatch.setattr(om.Mamba2Replay, "slot", lambda self, b, j: int((self.start[b] + j) % self.L))
    assert caught(tm.test_replay_equals_recurrence, tm.SHAPES[1])


def test_gdn_history_state_drops_last_entry(monkeypatch):
    orig = og.GdnReplay.state

    def state(self, b, p=None):
        if p is None:
            p = int(self.count[b])
        return orig(self, b, max(p - 1, 0))

    monkeypatch.setattr(og.GdnReplay, "state", state)
    assert caught(tg.test_chunked_verify_random_batch)


def test_gdn_u_stored_without_rounding(monkeypatch):
    monkeypatch.setattr(og, "round_storage", lambda x, dtype: np.asarray(x, np.float64))
    assert caught(tg.test_storage_rounding_bf16)


def test_gdn_correction_sign_slip(monkeypatch):
    """The rank-1 form with k negated: its write term -beta v k^T has the wrong sign."""
    orig = og.rank1_step

    def rank1_step(S, q, k, v, beta, g):
        return orig(S, q, -np.asarray(k), v, beta, g)  # the write term becomes -beta v k^T

    monkeypatch.setattr(og, "rank1_step", rank1_step)
    assert caught(tg.test_householder_equals_rank1, tg.SHAPES[0])


def test_conv_activation_wrong(monkeypatch):
    monkeypatch.setattr(oc, "silu", lambda z: np.asarray(z, np.float64) / (1.0 + np.exp(-2.0 * np.asarray(z))))
    assert caught(tc.test_silu_is_z_times_logistic)


def test_conv_state_shift_wrong(monkeypatch):
    """The state keeps the oldest columns instead of the newest."""
    orig = oc.conv_state_step

    def step(state, u, weight, bias=None, activation=True):
        new_state, out = orig(state, u, weight, bias, activation)
        st = np.asarray(state, np.float64)
        return np.concatenate([st[..., :1], new_state[..., :-1]], axis=-1) if st.shape[-1] > 1 else new_state, out

    monkeypatch.setattr(oc, "conv_state_step", step)
    assert caught(tc.test_state_holds_the_last_inputs_oldest_first)
