"""The benchmark's byte accounting follows each sequence's fill level from a
host-side trace; these CPU tests pin those traces to the oracle's own
bookkeeping (decode with the fused flush, and speculative rounds with the
early flush), so the reported GB/s counts the entries the kernels read."""
import numpy as np

import bench
from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl


def test_decode_fill_trace_matches_oracle():
    shape = wl.Mamba2Shape(B=6, H=2, G=1, d=2, n=2, L=5, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, 11)
    orc = om.Mamba2Replay(init.S0, init.A, init.ring_v, init.ring_k, init.ring_dt, init.start, init.count)
    steps = 13
    trace = bench.fill_trace(init.count, shape.L, steps)
    for t in range(steps):
        np.testing.assert_array_equal(trace[t], orc.count, err_msg=f"step {t}")
        s = wl.mamba2_step(shape, 11, t)
        orc.decode_step(s.v, s.k, s.q, s.dt)
        if orc.flag.any():  # the fused step folds a full buffer at once
            orc.flush()


def test_spec_trace_matches_oracle():
    shape = wl.Mamba2Shape(B=7, H=2, G=1, d=2, n=2, L=9, in_dtype=wl.F32)
    T, rounds = 3, 10
    init = wl.mamba2_init(shape, 12, fill_max=shape.L - T)
    orc = om.Mamba2Replay(init.S0, init.A, init.ring_v, init.ring_k, init.ring_dt, init.start, init.count)
    accs = [wl.accepted_counts(shape.B, T, 12, r) for r in range(rounds)]
    hs, folds = bench.spec_trace(init.count, accs, T, shape.L)
    for r in range(rounds):
        np.testing.assert_array_equal(hs[r], orc.count, err_msg=f"round {r}: h")
        s = wl.mamba2_step(shape, 12, r, T=T)
        orc.spec_verify(s.v, s.k, s.q, s.dt)
        orc.commit(accs[r], T)
        folded = np.where(orc.flag != 0, orc.count, -1)
        np.testing.assert_array_equal(folds[r], folded, err_msg=f"round {r}: folded entries")
        orc.flush()
    assert orc.err == 0
