"""Pins for the fp64 Mamba-2 oracle (CPU only).

The oracle is tied to things other than itself:
* a hand-worked scalar example (tests/golden/mamba2_scalar.txt);
* the page's three routes to the same numbers -- the summary recurrence, the
  history route and the output-only route -- which share no code;
* flush-anywhere and rollback-by-pointer invariants, brute-forced on tiny shapes;
* closed forms (A = 0, Delta = 0, a single token from a zero state);
* the early-flush bookkeeping, brute-forced over every (L, T, h, accepted).
"""
import itertools
import os

import numpy as np
import pytest

from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def fold_by_recurrence(init: wl.Mamba2Init, A):
    """State reached by feeding the pre-filled buffer entries through the plain
    recurrence from S_0 (q is irrelevant for the state)."""
    s = init.shape
    S = init.S0.astype(np.float64).copy()
    grp = om.head_group(s.H, s.G)
    for b in range(s.B):
        Sb = S[b:b + 1]
        for j in range(int(init.count[b])):
            sl = (init.start[b] + j) % s.L
            v = init.ring_v[b:b + 1, :, sl, :]
            k = init.ring_k[b:b + 1, :, sl, :]
            dt = init.ring_dt[b:b + 1, :, sl]
            Sb, _ = om.recurrence_step(Sb, v, k, np.zeros_like(k), dt, A)
        S[b] = Sb[0]
    return S


def make_replay(init):
    return om.Mamba2Replay(init.S0, init.A, init.ring_v, init.ring_k, init.ring_dt,
                           init.start, init.count)


# ---------------------------------------------------------------------------
# hand-worked example
# ---------------------------------------------------------------------------


def _scalar_inputs():
    ln2 = np.log(2.0)
    vkq = [(1.0, 1.0, 1.0), (2.0, 1.0, 3.0), (-1.0, 2.0, 1.0)]
    A = np.array([-1.0])
    rows = np.loadtxt(os.path.join(GOLDEN, "mamba2_scalar.txt"))
    expect = rows[:, 1] + rows[:, 2] * ln2
    return ln2, vkq, A, expect


def test_scalar_golden_recurrence():
    ln2, vkq, A, expect = _scalar_inputs()
    S = np.ones((1, 1, 1, 1))
    for t, (v, k, q) in enumerate(vkq):
        S, y = om.recurrence_step(S, np.array([[[v]]]), np.array([[[k]]]), np.array([[[q]]]),
                                  np.array([[ln2]]), A)
        assert y[0, 0, 0] == pytest.approx(expect[t], rel=1e-14, abs=1e-14)


@pytest.mark.parametrize("L", [1, 2, 3, 4])
def test_scalar_golden_replay(L):
    """Same example through the ring buffer; L = 1, 2 force flushes mid-way."""
    ln2, vkq, A, expect = _scalar_inputs()
    r = om.Mamba2Replay(np.ones((1, 1, 1, 1)), A, np.zeros((1, 1, L, 1)), np.zeros((1, 1, L, 1)),
                        np.zeros((1, 1, L)), [0], [0])
    for t, (v, k, q) in enumerate(vkq):
        y = r.decode_step(np.array([[[v]]]), np.array([[[k]]]), np.array([[[q]]]), np.array([[ln2]]))
        r.flush()
        assert y[0, 0, 0] == pytest.approx(expect[t], rel=1e-14, abs=1e-14)
    assert r.err == 0


def test_scalar_golden_snapshot_baseline():
    ln2, vkq, A, expect = _scalar_inputs()
    base = om.Mamba2SnapshotBaseline(np.ones((1, 1, 1, 1)), A, T=3)
    v = np.array([[[[x[0]]] for x in vkq]])
    k = np.array([[[[x[1]]] for x in vkq]])
    q = np.array([[[[x[2]]] for x in vkq]])
    Y = base.verify(v, k, q, np.full((1, 3, 1), ln2))
    np.testing.assert_allclose(Y[0, :, 0, 0], expect, rtol=1e-14)


# ---------------------------------------------------------------------------
# route agreement
# ---------------------------------------------------------------------------

SHAPES = [
    wl.Mamba2Shape(B=3, H=4, G=2, d=3, n=5, L=4, in_dtype=wl.F32),
    wl.Mamba2Shape(B=2, H=6, G=3, d=8, n=4, L=5, in_dtype=wl.BF16),
    wl.Mamba2Shape(B=2, H=2, G=1, d=4, n=4, L=1, in_dtype=wl.F32),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_replay_equals_recurrence(shape):
    """ReplaySSM output == plain recurrence, token for token, across flushes
    and a pre-filled, wrapped ring (page: 'does not change outputs')."""
    init = wl.mamba2_init(shape, seed=5)
    S = fold_by_recurrence(init, init.A)
    r = make_replay(init)
    for t in range(3 * shape.L + 2):
        st = wl.mamba2_step(shape, seed=5, step=t)
        S, y_ref = om.recurrence_step(S, st.v, st.k, st.q, st.dt, init.A)
        y = r.decode_step(st.v, st.k, st.q, st.dt)
        assert rel_err(y, y_ref) < 1e-12
        r.flush()
        for b in range(shape.B):
            assert rel_err(r.state(b), S[b]) < 1e-12
    assert r.err == 0


def test_history_route_equals_recurrence_states():
    """The history route (unrolled sum) reproduces every intermediate state."""
    shape = wl.Mamba2Shape(B=2, H=2, G=1, d=3, n=2, L=6, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=9, fill_max=0)
    r = make_replay(init)
    S = init.S0.astype(np.float64)
    for t in range(5):
        st = wl.mamba2_step(shape, 9, t)
        S, _ = om.recurrence_step(S, st.v, st.k, st.q, st.dt, init.A)
        r.decode_step(st.v, st.k, st.q, st.dt)
        for b in range(shape.B):
            assert rel_err(r.state(b), S[b]) < 1e-13


def test_flush_anywhere_is_a_noop_all_schedules():
    """Flushing at any step leaves every output unchanged: all 2^k schedules."""
    shape = wl.Mamba2Shape(B=2, H=2, G=1, d=3, n=4, L=8, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=11, fill_max=3)
    steps = [wl.mamba2_step(shape, 11, t) for t in range(8)]
    ref = None
    for mask in range(1 << len(steps)):
        r = make_replay(init)
        ys = []
        for t, st in enumerate(steps):
            ys.append(r.decode_step(st.v, st.k, st.q, st.dt))
            if (mask >> t) & 1:
                r.flag[:] = 1
            r.flush()
        ys = np.stack(ys)
        if ref is None:
            ref = ys
        else:
            assert rel_err(ys, ref) < 1e-12
        assert r.err == 0


def test_group_mapping_is_contiguous():
    """Heads 0,1 read group 0 and heads 2,3 read group 1 (H=4, G=2)."""
    shape = wl.Mamba2Shape(B=1, H=4, G=2, d=2, n=3, L=4, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=3, fill_max=0)
    st = wl.mamba2_step(shape, 3, 0)
    st.q[:, 0, :] = 0.0
    r = make_replay(init)
    y = r.decode_step(st.v, st.k, st.q, st.dt)
    assert np.all(y[0, :2] == 0.0)
    assert np.all(np.abs(y[0, 2:]) > 0.0)
    S, y2 = om.recurrence_step(init.S0, st.v, st.k, st.q, st.dt, init.A)
    assert np.all(y2[0, :2] == 0.0)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------


def test_closed_form_no_decay():
    """A = 0: S_t = S_0 + sum_i Delta_i v_i k_i^T."""
    shape = wl.Mamba2Shape(B=2, H=2, G=1, d=3, n=4, L=3, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=4, fill_max=0)
    A = np.zeros(shape.H)
    r = om.Mamba2Replay(init.S0, A, init.ring_v, init.ring_k, init.ring_dt, init.start, init.count)
    S = init.S0.astype(np.float64).copy()
    for t in range(7):
        st = wl.mamba2_step(shape, 4, t)
        v, k, q, dt = (x.astype(np.float64) for x in (st.v, st.k, st.q, st.dt))
        S = S + dt[:, :, None, None] * v[:, :, :, None] * k[:, [0, 0], None, :]
        y = r.decode_step(st.v, st.k, st.q, st.dt)
        r.flush()
        np.testing.assert_allclose(y, np.einsum("bhdn,bhn->bhd", S, q[:, [0, 0], :]), rtol=1e-12, atol=1e-12)


def test_closed_form_zero_step():
    """Delta = 0: a = 1 and no input enters, so y = S_0 q."""
    shape = wl.Mamba2Shape(B=1, H=2, G=2, d=3, n=4, L=2, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=6, fill_max=0)
    r = make_replay(init)
    for t in range(5):
        st = wl.mamba2_step(shape, 6, t)
        st.dt[:] = 0.0
        y = r.decode_step(st.v, st.k, st.q, st.dt)
        r.flush()
        np.testing.assert_allclose(y, np.einsum("bhdn,bhn->bhd", init.S0.astype(np.float64), st.q.astype(np.float64)), rtol=1e-13)


def test_closed_form_single_token_from_zero():
    """S_0 = 0, one token: y = Delta (k . q) v (inner-product association)."""
    shape = wl.Mamba2Shape(B=3, H=2, G=1, d=5, n=4, L=4, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=7, fill_max=0)
    init.S0[:] = 0.0
    st = wl.mamba2_step(shape, 7, 0)
    y = make_replay(init).decode_step(st.v, st.k, st.q, st.dt)
    v, k, q, dt = (x.astype(np.float64) for x in (st.v, st.k, st.q, st.dt))
    kq = np.sum(k[:, 0, :] * q[:, 0, :], axis=-1)
    np.testing.assert_allclose(y, dt[:, :, None] * kq[:, None, None] * v, rtol=1e-13)


# ---------------------------------------------------------------------------
# speculative decoding
# ---------------------------------------------------------------------------


def _spec_run(shape, T, accs, seed):
    """Run verify/commit/flush rounds and compare with the recurrence on the
    accepted prefix; returns the replay object."""
    init = wl.mamba2_init(shape, seed=seed, fill_max=shape.L - T)
    S = fold_by_recurrence(init, init.A)
    r = make_replay(init)
    for rnd, acc in enumerate(accs):
        st = wl.mamba2_step(shape, seed, rnd, T=T)
        h = r.count.copy()
        Y = r.spec_verify(st.v, st.k, st.q, st.dt)
        np.testing.assert_array_equal(r.flag, (h + 2 * T > shape.L).astype(int))
        # drafts: the recurrence continued from the committed state
        Sd = S.copy()
        for s in range(T):
            Sd, y_ref = om.recurrence_step(Sd, st.v[:, s], st.k[:, s], st.q[:, s], st.dt[:, s], init.A)
            assert rel_err(Y[:, s], y_ref) < 1e-12
        # commit: recurrence over the accepted prefix only
        a = np.asarray(acc, dtype=np.int32)
        r.commit(a, T)
        for b in range(shape.B):
            Sb = S[b:b + 1]
            for s in range(int(a[b])):
                Sb, _ = om.recurrence_step(Sb, st.v[b:b + 1, s], st.k[b:b + 1, s], st.q[b:b + 1, s],
                                           st.dt[b:b + 1, s], init.A)
            S[b] = Sb[0]
        np.testing.assert_array_equal(r.count, np.where(r.flag == 1, r.count, h + a))
        r.flush()
        assert np.all(r.count + T <= shape.L)
        for b in range(shape.B):
            assert rel_err(r.state(b), S[b]) < 1e-12
    assert r.err == 0
    return r


@pytest.mark.parametrize("T,L", [(2, 4), (2, 5), (3, 7), (1, 3)])
def test_rollback_equals_recompute_exhaustive(T, L):
    """Rollback by pointer == recomputing from the accepted prefix, for every
    sequence of accepted counts over 3 rounds."""
    shape = wl.Mamba2Shape(B=1, H=2, G=1, d=3, n=2, L=L, in_dtype=wl.F32)
    for accs in itertools.product(range(T + 1), repeat=3):
        _spec_run(shape, T, [[a] for a in accs], seed=20 + T)


def test_rollback_random_batch():
    shape = wl.Mamba2Shape(B=6, H=4, G=2, d=4, n=3, L=8, in_dtype=wl.BF16)
    T = 3
    accs = [wl.accepted_counts(shape.B, T, 31, r) for r in range(10)]
    _spec_run(shape, T, accs, seed=31)


def test_verify_window_one_equals_decode():
    """T = 1 with one accepted draft is the ordinary decode step."""
    shape = wl.Mamba2Shape(B=4, H=4, G=2, d=3, n=5, L=4, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=13)
    r1, r2 = make_replay(init), make_replay(init)
    for t in range(9):
        st = wl.mamba2_step(shape, 13, t)
        y1 = r1.decode_step(st.v, st.k, st.q, st.dt)
        f1 = r1.flag.copy()
        r1.flush()
        Y = r2.spec_verify(st.v[:, None], st.k[:, None], st.q[:, None], st.dt[:, None])
        f2 = r2.flag.copy()
        r2.commit(np.ones(shape.B, np.int32), 1)
        r2.flush()
        np.testing.assert_array_equal(f1, f2)
        assert rel_err(Y[:, 0], y1) < 1e-13
        np.testing.assert_array_equal(r1.start, r2.start)
        np.testing.assert_array_equal(r1.count, r2.count)


def test_snapshot_baseline_equals_recurrence():
    shape = wl.Mamba2Shape(B=4, H=2, G=1, d=3, n=4, L=8, in_dtype=wl.F32)
    T = 3
    init = wl.mamba2_init(shape, seed=17, fill_max=0)
    base = om.Mamba2SnapshotBaseline(init.S0, init.A, T)
    S = init.S0.astype(np.float64).copy()
    for rnd in range(6):
        st = wl.mamba2_step(shape, 17, rnd, T=T)
        Y = base.verify(st.v, st.k, st.q, st.dt)
        acc = wl.accepted_counts(shape.B, T, 17, rnd)
        Sd = S.copy()
        for s in range(T):
            Sd, y_ref = om.recurrence_step(Sd, st.v[:, s], st.k[:, s], st.q[:, s], st.dt[:, s], init.A)
            assert rel_err(Y[:, s], y_ref) < 1e-13
        base.commit(acc)
        for b in range(shape.B):
            Sb = S[b:b + 1]
            for s in range(int(acc[b])):
                Sb, _ = om.recurrence_step(Sb, st.v[b:b + 1, s], st.k[b:b + 1, s], st.q[b:b + 1, s],
                                           st.dt[b:b + 1, s], init.A)
            S[b] = Sb[0]
            assert rel_err(base.state(b), S[b]) < 1e-13


# ---------------------------------------------------------------------------
# bookkeeping brute force
# ---------------------------------------------------------------------------


def test_bookkeeping_brute_force():
    """Every (L <= 16, T <= L, h <= L - T, accepted <= T), and L = 32 with T = 4:
    flag == (h + 2T > L) and the next round starts with h' + T <= L."""
    cases = [(L, T, h, a) for L in list(range(1, 17)) + [32] for T in range(1, L + 1)
             for h in range(0, L - T + 1) for a in range(0, T + 1) if L <= 16 or T == 4]
    Ls = sorted({c[0] for c in cases})
    for L in Ls:
        cs = [c for c in cases if c[0] == L]
        B = len(cs)
        for T in sorted({c[1] for c in cs}):
            sub = [c for c in cs if c[1] == T]
            Bs = len(sub)
            h = np.array([c[2] for c in sub])
            a = np.array([c[3] for c in sub])
            r = om.Mamba2Replay(np.zeros((Bs, 1, 1, 1)), np.zeros(1), np.zeros((Bs, 1, L, 1)),
                                np.zeros((Bs, 1, L, 1)), np.zeros((Bs, 1, L)),
                                np.arange(Bs) % L, h)
            z = np.zeros((Bs, T, 1, 1))
            r.spec_verify(z, z, z, np.zeros((Bs, T, 1)))
            assert np.array_equal(r.flag, (h + 2 * T > L).astype(int))
            r.commit(a, T)
            r.flush()
            assert r.err == 0
            assert np.all(r.count + T <= L)
            exp_count = np.where(h + 2 * T > L, 0, h + a)
            assert np.array_equal(r.count, exp_count)
            exp_start = np.where(h + 2 * T > L, (np.arange(Bs) % L + h + a) % L, np.arange(Bs) % L)
            assert np.array_equal(r.start, exp_start)
        del B


def test_error_bits():
    shape = wl.Mamba2Shape(B=2, H=2, G=1, d=2, n=2, L=4, in_dtype=wl.F32)
    init = wl.mamba2_init(shape, seed=1)
    r = make_replay(init)
    r.count[:] = [4, 1]
    st = wl.mamba2_step(shape, 1, 0)
    r.decode_step(st.v, st.k, st.q, st.dt)
    assert r.err == om.ERR_COUNT_RANGE
    assert r.count[0] == 4 and r.count[1] == 2
    r.err = 0
    st = wl.mamba2_step(shape, 1, 0, T=3)
    r.count[:] = [2, 1]
    r.spec_verify(st.v, st.k, st.q, st.dt)
    assert r.err == om.ERR_WINDOW
    r.err = 0
    r.commit(np.array([4, 1]), 3)
    assert r.err == om.ERR_ACCEPTED
