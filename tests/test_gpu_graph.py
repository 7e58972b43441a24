"""Speculative rounds -- verify, device commit, flush of the sequences the
verify flagged -- captured once in a CUDA graph and replayed.

"Supplementary design for CUDA Graphs": the flush decision is per-sequence
data that the kernels read at run time, and a small commit kernel moves the
buffer pointers on the device, so one captured graph serves the whole batch
whatever each sequence accepts, with no host synchronisation.  A replay must
equal the same calls made eagerly bit for bit (outputs, checkpoint, ring,
pointers), and both follow the oracle within the tolerance of the other
parity tests.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, dev, gdn_state, gdn_step_dev, host, m2_state, m2_step_dev
from oracle import gdn as og
from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def rs():
    from ssm_decode_hybrid_gb300 import replayssm

    return replayssm


def capture(fn):
    """Capture fn() into a CUDA graph on a side stream; return the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    return g


def same_state(a, b, names):
    for n in names:
        assert torch.equal(getattr(a, n), getattr(b, n)), f"{n} differs between graph replay and eager calls"


@pytest.mark.parametrize("T", [1, 4, 6])
def test_mamba2_spec_rounds_in_a_graph(T):
    R = rs()
    shape = wl.Mamba2Shape(B=24, H=8, G=2, d=64, n=128, L=16, in_dtype=wl.BF16)
    seed, rounds = 500 + T, 6
    init = wl.mamba2_init(shape, seed, fill_max=shape.L - T)
    A = dev(init.A)
    steps = [wl.mamba2_step(shape, seed, r, T=T) for r in range(rounds)]
    inp = [m2_step_dev(s, shape.in_dtype) for s in steps]
    accs = [wl.accepted_counts(shape.B, T, seed, r) for r in range(rounds)]
    acc = [dev(a, torch.int32) for a in accs]
    ys = {k: [torch.empty(shape.B, T, shape.H, shape.d, device="cuda") for _ in range(rounds)] for k in "eg"}

    def rnd(st, r, y):
        R.replay_spec_verify(st, *inp[r], A, y=y)
        R.replay_spec_commit(acc[r], st.count, T, shape.L, st.err)
        R.replay_flush(st, A)

    rnd(m2_state(init), 0, torch.empty_like(ys["e"][0]))  # sets kernel attributes outside the capture
    eager, graphed = m2_state(init), m2_state(init)
    for r in range(rounds):
        rnd(eager, r, ys["e"][r])
    g = capture(lambda: [rnd(graphed, r, ys["g"][r]) for r in range(rounds)])
    g.replay()
    torch.cuda.synchronize()
    for r in range(rounds):
        assert torch.equal(ys["g"][r], ys["e"][r]), f"round {r}: y differs"
    same_state(graphed, eager, ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag", "err"))
    assert int(host(graphed.err)[0]) == 0

    orc = om.Mamba2Replay(init.S0, init.A, init.ring_v, init.ring_k, init.ring_dt, init.start, init.count)
    for r, s in enumerate(steps):
        assert_close(ys["g"][r], orc.spec_verify(s.v, s.k, s.q, s.dt), what=f"round {r}: y vs oracle")
        orc.commit(accs[r], T)
        orc.flush()
    np.testing.assert_array_equal(host(graphed.count), orc.count)
    np.testing.assert_array_equal(host(graphed.start), orc.start)
    assert_close(graphed.S0, orc.S0, what="final S0 vs oracle")


@pytest.mark.parametrize("T", [1, 4, 6])
def test_gdn_spec_rounds_in_a_graph(T):
    R = rs()
    shape = wl.GdnShape(B=12, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16)
    seed, rounds = 600 + T, 6
    init = wl.gdn_init(shape, seed, fill_max=shape.L - T)
    steps = [wl.gdn_step(shape, seed, r, T=T) for r in range(rounds)]
    inp = [gdn_step_dev(s, shape.in_dtype) for s in steps]
    accs = [wl.accepted_counts(shape.B, T, seed, r) for r in range(rounds)]
    acc = [dev(a, torch.int32) for a in accs]
    ys = {k: [torch.empty(shape.B, T, shape.Hv, shape.dv, device="cuda") for _ in range(rounds)] for k in "eg"}

    def rnd(st, r, y):
        R.gdn_replay_verify(st, *inp[r], y=y)
        R.replay_spec_commit(acc[r], st.count, T, shape.L, st.err)
        R.gdn_replay_flush(st)

    rnd(gdn_state(init), 0, torch.empty_like(ys["e"][0]))
    eager, graphed = gdn_state(init), gdn_state(init)
    for r in range(rounds):
        rnd(eager, r, ys["e"][r])
    g = capture(lambda: [rnd(graphed, r, ys["g"][r]) for r in range(rounds)])
    g.replay()
    torch.cuda.synchronize()
    for r in range(rounds):
        assert torch.equal(ys["g"][r], ys["e"][r]), f"round {r}: y differs"
    same_state(graphed, eager, ("S0", "ring_u", "ring_k", "ring_g", "start", "count", "flag", "err"))
    assert int(host(graphed.err)[0]) == 0

    orc = og.GdnReplay(init.S0, init.ring_u, init.ring_k, init.ring_g, init.start, init.count,
                       u_dtype=shape.u_dtype)
    for r, s in enumerate(steps):
        assert_close(ys["g"][r], orc.verify(s.q, s.k, s.v, s.beta, s.g), what=f"round {r}: y vs oracle")
        orc.commit(accs[r], T)
        orc.flush()
    np.testing.assert_array_equal(host(graphed.count), orc.count)
    assert_close(graphed.S0, orc.S0, what="final S0 vs oracle")


def test_fused_decode_steps_in_a_graph():
    """Decode steps with the fused flush, replayed from a graph twice: the
    second replay continues from the state the first left (buffers fill and
    fold at run time inside the same captured launches)."""
    R = rs()
    shape = wl.Mamba2Shape(B=16, H=8, G=2, d=64, n=128, L=8, in_dtype=wl.BF16)
    seed, steps_n = 520, 5
    init = wl.mamba2_init(shape, seed)
    A = dev(init.A)
    steps = [wl.mamba2_step(shape, seed, t) for t in range(2 * steps_n)]
    inp = [m2_step_dev(s, shape.in_dtype) for s in steps]
    y = torch.empty(shape.B, shape.H, shape.d, device="cuda")
    R.replay_decode_step_fused(m2_state(init), *inp[0], A, y=y)
    eager, graphed = m2_state(init), m2_state(init)
    ys_e = []
    for t in range(2 * steps_n):
        ys_e.append(R.replay_decode_step_fused(eager, *inp[t % steps_n], A))
    ys_g = [torch.empty_like(y) for _ in range(steps_n)]
    g = capture(lambda: [R.replay_decode_step_fused(graphed, *inp[t], A, y=ys_g[t]) for t in range(steps_n)])
    orc = om.Mamba2Replay(init.S0, init.A, init.ring_v, init.ring_k, init.ring_dt, init.start, init.count)
    for rep in range(2):
        g.replay()
        torch.cuda.synchronize()
        for t in range(steps_n):
            assert torch.equal(ys_g[t], ys_e[rep * steps_n + t]), f"replay {rep} step {t}: y differs"
            s = steps[t]
            assert_close(ys_g[t], orc.decode_step(s.v, s.k, s.q, s.dt), what=f"replay {rep} step {t}: y vs oracle")
            if orc.flag.any():
                orc.flush()
    same_state(graphed, eager, ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag"))
    np.testing.assert_array_equal(host(graphed.count), orc.count)
    assert_close(graphed.S0, orc.S0, what="final S0 vs oracle")
