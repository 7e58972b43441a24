"""Recovery from a bounded wait that runs out in a precompute kernel.

Every wait inside the library's kernels is bounded; when the data wait of a
precompute kernel (two-launch decode and verify, Mamba-2 and GDN) runs out,
that block gives its sequence up: RSSM_EBIT_TIMEOUT is set, and the
streaming blocks that would change the sequence's state (its pointers, or
S_0 by a fold) skip it, so its pointers, checkpoint and committed ring
entries stay as they were; an output head is either left untouched or
written exactly as by an ordinary call.  The next ordinary call must then
match the oracle.

RSSM_WAIT_LIMIT_NS (read by the library at every call) shortens that limit:
0 makes every precompute wait count as run out at once (every sequence is
skipped), a few microseconds makes some of them run out (each sequence's
state is then either exactly an ordinary call's or left untouched).
No GPU wait is left unbounded: a block that gives up still drains its bulk
copies with the normal one-second limit before it exits.
"""
import contextlib
import os

import numpy as np
import pytest
import torch

from gpu_util import assert_close, dev, gdn_state, gdn_step_dev, host, m2_state, m2_step_dev
from oracle import gdn as og
from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

M2_SHAPE = wl.Mamba2Shape(B=8, H=32, G=8, d=64, n=128, L=16, in_dtype=wl.BF16)
GDN_SHAPE = wl.GdnShape(B=4, Hv=32, Hk=16, dk=128, dv=128, L=16, in_dtype=wl.BF16, u_dtype=wl.F32)
M2_FIELDS = ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag", "sync")
GDN_FIELDS = ("S0", "ring_u", "ring_k", "ring_g", "start", "count", "flag", "sync")

# (kind, T): T = 0 is the fused decode step; T = 4 runs the CUDA-core Mamba-2
# verify stream, T = 6 the tensor-core one; GDN verify runs on the tensor cores
CASES = [("m2", 0), ("m2", 4), ("m2", 6), ("gdn", 0), ("gdn", 4)]
CASE_ID = lambda c: f"{c[0]}-{'fused' if c[1] == 0 else f'verify{c[1]}'}"  # noqa: E731


@contextlib.contextmanager
def wait_limit(ns: str):
    old = os.environ.get("RSSM_WAIT_LIMIT_NS")
    os.environ["RSSM_WAIT_LIMIT_NS"] = ns
    try:
        yield
    finally:
        if old is None:
            del os.environ["RSSM_WAIT_LIMIT_NS"]
        else:
            os.environ["RSSM_WAIT_LIMIT_NS"] = old


class Case:
    """One seeded state and one call's inputs for a (kind, T) case."""

    def __init__(self, kind, T, seed=611):
        from ssm_decode_hybrid_gb300 import replayssm as R

        self.R, self.kind, self.T, self.seed = R, kind, T, seed
        if kind == "m2":
            self.shape = M2_SHAPE
            self.init = wl.mamba2_init(M2_SHAPE, seed, fill_max=None if T == 0 else M2_SHAPE.L - T)
            self.step = wl.mamba2_step(M2_SHAPE, seed, 0, T=T or None)
            self.fields = M2_FIELDS
            self.A = dev(self.init.A)
        else:
            self.shape = GDN_SHAPE
            self.init = wl.gdn_init(GDN_SHAPE, seed, fill_max=None if T == 0 else GDN_SHAPE.L - T)
            self.step = wl.gdn_step(GDN_SHAPE, seed, 0, T=T or None)
            self.fields = GDN_FIELDS

    def state(self):
        return m2_state(self.init) if self.kind == "m2" else gdn_state(self.init)

    def y_shape(self):
        s = self.shape
        if self.kind == "m2":
            return (s.B, s.H, s.d) if self.T == 0 else (s.B, self.T, s.H, s.d)
        return (s.B, s.Hv, s.dv) if self.T == 0 else (s.B, self.T, s.Hv, s.dv)

    def call(self, state):
        R, st = self.R, self.step
        y = torch.full(self.y_shape(), float("nan"), device="cuda")
        if self.kind == "m2":
            inp = m2_step_dev(st, self.shape.in_dtype)
            if self.T == 0:
                R.replay_decode_step_fused(state, *inp, self.A, y=y)
            else:
                R.replay_spec_verify(state, *inp, self.A, y=y)
        else:
            inp = gdn_step_dev(st, self.shape.in_dtype)
            if self.T == 0:
                R.gdn_replay_decode_fused(state, *inp, y=y)
            else:
                R.gdn_replay_verify(state, *inp, y=y)
        torch.cuda.synchronize()
        return y

    def oracle(self):
        """Outputs and final oracle after one ordinary call from the initial state."""
        i, st = self.init, self.step
        if self.kind == "m2":
            orc = om.Mamba2Replay(i.S0, i.A, i.ring_v, i.ring_k, i.ring_dt, i.start, i.count)
            if self.T == 0:
                y = orc.decode_step(st.v, st.k, st.q, st.dt)
                orc.flush()
            else:
                y = orc.spec_verify(st.v, st.k, st.q, st.dt)
        else:
            orc = og.GdnReplay(i.S0, i.ring_u, i.ring_k, i.ring_g, i.start, i.count, u_dtype=self.shape.u_dtype)
            if self.T == 0:
                y = orc.decode_step(st.q, st.k, st.v, st.beta, st.g)
                orc.flush()
            else:
                y = orc.verify(st.q, st.k, st.v, st.beta, st.g)
        return y, orc

    def committed(self, b):
        """Ring slots of sequence b's committed window at the start."""
        L = self.shape.L
        return [(int(self.init.start[b]) + j) % L for j in range(int(self.init.count[b]))]


def snapshot(state, fields):
    return {f: getattr(state, f).clone() for f in fields}


@pytest.mark.parametrize("case", CASES, ids=CASE_ID)
def test_wait_run_out_skips_every_sequence_then_recovers(case):
    c = Case(*case)
    state = c.state()
    before = snapshot(state, c.fields)
    with wait_limit("0"):
        y = c.call(state)
    assert int(host(state.err)[0]) == c.R.EBIT_TIMEOUT
    for f in c.fields:
        assert torch.equal(getattr(state, f), before[f]), f"{f} changed by a call whose sequences were all given up"
    assert bool(torch.isnan(y).all()), "outputs written for a sequence that was given up"

    # the next ordinary call, on the same workspace, matches the oracle
    state.err.zero_()
    y = c.call(state)
    y_ref, orc = c.oracle()
    assert_close(y, y_ref, what="outputs after recovery")
    np.testing.assert_array_equal(host(state.start), orc.start)
    np.testing.assert_array_equal(host(state.count), orc.count)
    np.testing.assert_array_equal(host(state.flag), orc.flag)
    assert_close(state.S0, orc.S0, what="S0 after recovery")
    assert int(host(state.err)[0]) == 0


@pytest.mark.parametrize("case", [CASES[0], CASES[4]], ids=CASE_ID)
@pytest.mark.parametrize("limit_ns", ["800", "3000"])
def test_some_waits_run_out_each_sequence_all_or_nothing(case, limit_ns):
    """With a limit of a few microseconds some precompute blocks give up and
    others finish; the blocks of one sequence may differ.  Each sequence's
    state must then be either exactly an ordinary call's or left as it was,
    and each head's outputs either untouched or exactly an ordinary call's."""
    c = Case(*case)
    ref = c.state()
    y_ref = c.call(ref)
    state = c.state()
    before = snapshot(state, c.fields)
    with wait_limit(limit_ns):
        y = c.call(state)
    err = int(host(state.err)[0])
    assert err in (0, c.R.EBIT_TIMEOUT)
    rings = [f for f in c.fields if f.startswith("ring_")]
    processed = skipped = 0
    for b in range(c.shape.B):
        same_as_ref = all(torch.equal(getattr(state, f)[b], getattr(ref, f)[b]) for f in c.fields)
        if same_as_ref:
            processed += 1
        else:
            skipped += 1
            for f in ("S0", "start", "count", "flag", "sync"):
                assert torch.equal(getattr(state, f)[b], before[f][b]), f"sequence {b} given up but {f} changed"
            # entries past the committed window may hold drafts or this step's
            # entry from the groups that finished; the committed ones may not move
            slots = torch.tensor(c.committed(b), dtype=torch.long, device="cuda")
            for f in rings:
                assert torch.equal(getattr(state, f)[b].index_select(1, slots), before[f][b].index_select(1, slots)), \
                    f"sequence {b} given up but committed {f} entries changed"
        # outputs: per head, untouched (NaN) or exactly the ordinary call's
        head_axis = 1 if c.T == 0 else 2
        yb, rb = y[b], y_ref[b]
        for h in range(yb.shape[head_axis - 1]):
            yh = yb.select(head_axis - 1, h)
            assert bool(torch.isnan(yh).all()) or torch.equal(yh, rb.select(head_axis - 1, h)), \
                f"sequence {b} head {h}: outputs neither untouched nor the ordinary call's"
    if err == 0:
        assert skipped == 0
