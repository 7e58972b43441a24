"""Pins for the fp64 Gated DeltaNet oracle (CPU only).

* a hand-worked scalar example (tests/golden/gdn_scalar.txt);
* Householder matrix form == rank-1 correction form (two independent forms);
* replay decode (state-and-output route) == the recurrence, across flushes;
* chunked lower-triangular verify == the serial recurrence, for every
  acceptance sequence over a few rounds;
* closed forms: beta = 0; beta = 1, g = 0 with a repeated unit key (the state
  is overwritten along k); mutually orthogonal draft keys (A = 0, U = R).
"""
import itertools
import os

import numpy as np
import pytest

from oracle import gdn as og
from ssm_decode_hybrid_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def fold_by_recurrence(init: wl.GdnInit):
    """State after the pre-filled entries: S <- e^{g_j} S + u_j k_j^T from S_0."""
    s = init.shape
    kh = og.key_head(s.Hv, s.Hk)
    S = init.S0.astype(np.float64).copy()
    for b in range(s.B):
        for j in range(int(init.count[b])):
            sl = (init.start[b] + j) % s.L
            al = np.exp(init.ring_g[b, :, sl].astype(np.float64))
            u = init.ring_u[b, :, sl, :].astype(np.float64)
            k = init.ring_k[b, kh, sl, :].astype(np.float64)
            S[b] = al[:, None, None] * S[b] + u[:, :, None] * k[:, None, :]
    return S


def make_replay(init, u_dtype="f64"):
    return og.GdnReplay(init.S0, init.ring_u, init.ring_k, init.ring_g, init.start, init.count,
                        u_dtype=u_dtype)


def test_scalar_golden():
    rows = np.loadtxt(os.path.join(GOLDEN, "gdn_scalar.txt"))
    g = np.array([[-np.log(2.0)]])
    one = np.ones((1, 1, 1))
    S1 = np.full((1, 1, 1, 1), 4.0)
    S2 = S1.copy()
    r = og.GdnReplay(S1, np.zeros((1, 1, 2, 1)), np.zeros((1, 1, 2, 1)), np.zeros((1, 1, 2)), [0], [0],
                     u_dtype="f64")
    for t, (v, beta) in enumerate([(2.0, 0.5), (6.0, 0.25), (0.0, 1.0)]):
        vv = np.array([[[v]]])
        bb = np.array([[beta]])
        S1, y1 = og.householder_step(S1, one, one, vv, bb, g)
        S2, y2, u2 = og.rank1_step(S2, one, one, vv, bb, g)
        y3 = r.decode_step(one, one, vv, bb, g)
        r.flush()
        for y in (y1, y2, y3):
            assert y[0, 0, 0] == pytest.approx(rows[t, 1], abs=1e-14)
        assert u2[0, 0, 0] == pytest.approx(rows[t, 2], abs=1e-14)


SHAPES = [
    wl.GdnShape(B=2, Hv=4, Hk=2, dk=5, dv=3, L=4, in_dtype=wl.F32),
    wl.GdnShape(B=3, Hv=2, Hk=1, dk=4, dv=6, L=3, in_dtype=wl.BF16),
    wl.GdnShape(B=1, Hv=2, Hk=2, dk=3, dv=3, L=1, in_dtype=wl.F32),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_householder_equals_rank1(shape):
    init = wl.gdn_init(shape, seed=1, fill_max=0)
    S1 = init.S0.astype(np.float64)
    S2 = S1.copy()
    for t in range(6):
        st = wl.gdn_step(shape, 1, t)
        S1, y1 = og.householder_step(S1, st.q, st.k, st.v, st.beta, st.g)
        S2, y2, _ = og.rank1_step(S2, st.q, st.k, st.v, st.beta, st.g)
        assert rel_err(y1, y2) < 1e-12
        assert rel_err(S1, S2) < 1e-12


@pytest.mark.parametrize("shape", SHAPES)
def test_replay_decode_equals_recurrence(shape):
    init = wl.gdn_init(shape, seed=2)
    S = fold_by_recurrence(init)
    r = make_replay(init)
    for t in range(3 * shape.L + 2):
        st = wl.gdn_step(shape, 2, t)
        S, y_ref, _ = og.rank1_step(S, st.q, st.k, st.v, st.beta, st.g)
        y = r.decode_step(st.q, st.k, st.v, st.beta, st.g)
        assert rel_err(y, y_ref) < 1e-12
        r.flush()
        for b in range(shape.B):
            assert rel_err(r.state(b), S[b]) < 1e-12
    assert r.err == 0


def test_flush_anywhere_is_a_noop_all_schedules():
    shape = wl.GdnShape(B=2, Hv=2, Hk=1, dk=4, dv=3, L=8, in_dtype=wl.F32)
    init = wl.gdn_init(shape, seed=3, fill_max=3)
    steps = [wl.gdn_step(shape, 3, t) for t in range(7)]
    ref = None
    for mask in range(1 << len(steps)):
        r = make_replay(init)
        ys = []
        for t, st in enumerate(steps):
            ys.append(r.decode_step(st.q, st.k, st.v, st.beta, st.g))
            if (mask >> t) & 1:
                r.flag[:] = 1
            r.flush()
        ys = np.stack(ys)
        if ref is None:
            ref = ys
        else:
            assert rel_err(ys, ref) < 1e-12


def _spec_run(shape, T, accs, seed, u_dtype="f64"):
    init = wl.gdn_init(shape, seed=seed, fill_max=shape.L - T)
    S = fold_by_recurrence(init)
    r = make_replay(init, u_dtype)
    for rnd, acc in enumerate(accs):
        st = wl.gdn_step(shape, seed, rnd, T=T)
        h = r.count.copy()
        Y = r.verify(st.q, st.k, st.v, st.beta, st.g)
        np.testing.assert_array_equal(r.flag, (h + 2 * T > shape.L).astype(int))
        Sd = S.copy()
        for s in range(T):
            Sd, y_ref, _ = og.rank1_step(Sd, st.q[:, s], st.k[:, s], st.v[:, s], st.beta[:, s], st.g[:, s])
            assert rel_err(Y[:, s], y_ref) < 1e-11
        a = np.asarray(acc, dtype=np.int32)
        r.commit(a, T)
        for b in range(shape.B):
            Sb = S[b:b + 1]
            for s in range(int(a[b])):
                Sb, _, _ = og.rank1_step(Sb, st.q[b:b + 1, s], st.k[b:b + 1, s], st.v[b:b + 1, s],
                                         st.beta[b:b + 1, s], st.g[b:b + 1, s])
            S[b] = Sb[0]
        r.flush()
        assert np.all(r.count + T <= shape.L)
        for b in range(shape.B):
            assert rel_err(r.state(b), S[b]) < 1e-11
    assert r.err == 0


@pytest.mark.parametrize("T,L", [(2, 4), (3, 7), (4, 9)])
def test_chunked_verify_equals_serial_exhaustive(T, L):
    shape = wl.GdnShape(B=1, Hv=2, Hk=1, dk=4, dv=3, L=L, in_dtype=wl.F32)
    rounds = 3 if T < 4 else 2
    for accs in itertools.product(range(T + 1), repeat=rounds):
        _spec_run(shape, T, [[a] for a in accs], seed=40 + T)


def test_chunked_verify_random_batch():
    shape = wl.GdnShape(B=5, Hv=4, Hk=2, dk=6, dv=5, L=16, in_dtype=wl.BF16)
    T = 4
    _spec_run(shape, T, [wl.accepted_counts(shape.B, T, 50, r) for r in range(12)], seed=50)


def test_verify_window_one_equals_decode():
    shape = wl.GdnShape(B=3, Hv=4, Hk=2, dk=4, dv=3, L=4, in_dtype=wl.F32)
    init = wl.gdn_init(shape, seed=60)
    r1, r2 = make_replay(init), make_replay(init)
    for t in range(9):
        st = wl.gdn_step(shape, 60, t)
        y1 = r1.decode_step(st.q, st.k, st.v, st.beta, st.g)
        r1.flush()
        Y = r2.verify(st.q[:, None], st.k[:, None], st.v[:, None], st.beta[:, None], st.g[:, None])
        r2.commit(np.ones(shape.B, np.int32), 1)
        r2.flush()
        assert rel_err(Y[:, 0], y1) < 1e-13
        np.testing.assert_array_equal(r1.start, r2.start)
        np.testing.assert_array_equal(r1.count, r2.count)


def test_closed_form_beta_zero():
    """beta = 0 writes nothing: y_t = e^{g_1 + ... + g_t} S_0 q_t."""
    shape = wl.GdnShape(B=2, Hv=2, Hk=2, dk=4, dv=3, L=3, in_dtype=wl.F32)
    init = wl.gdn_init(shape, seed=7, fill_max=0)
    r = make_replay(init)
    Gsum = np.zeros((shape.B, shape.Hv))
    for t in range(7):
        st = wl.gdn_step(shape, 7, t)
        st.beta[:] = 0.0
        Gsum = Gsum + st.g
        y = r.decode_step(st.q, st.k, st.v, st.beta, st.g)
        r.flush()
        np.testing.assert_allclose(y, np.exp(Gsum)[:, :, None] * np.einsum("bhvk,bhk->bhv", init.S0.astype(np.float64), st.q.astype(np.float64)),
                                   rtol=1e-12)


def test_closed_form_overwrite_along_unit_key():
    """beta = 1, g = 0 and one unit key k repeated: (I - k k^T) is a projector,
    so y_t = S_0 (q - k (k . q)) + v_t (k . q)."""
    shape = wl.GdnShape(B=1, Hv=2, Hk=1, dk=5, dv=3, L=4, in_dtype=wl.F32)
    init = wl.gdn_init(shape, seed=8, fill_max=0)
    rng = np.random.default_rng(8)
    kvec = rng.standard_normal(shape.dk)
    kvec = kvec / np.linalg.norm(kvec)
    r = make_replay(init)
    S = init.S0.astype(np.float64)
    for t in range(6):
        st = wl.gdn_step(shape, 8, t)
        k = np.broadcast_to(kvec, st.k.shape).copy()
        st.beta[:] = 1.0
        st.g[:] = 0.0
        y = r.decode_step(st.q, k, st.v, st.beta, st.g)
        S, y2 = og.householder_step(S, st.q, k, st.v, st.beta, st.g)
        r.flush()
        q0 = st.q[0, 0].astype(np.float64)
        kq = float(kvec @ q0)
        expect = np.einsum("hvk,k->hv", init.S0[0].astype(np.float64), q0 - kvec * kq) + st.v[0].astype(np.float64) * kq
        np.testing.assert_allclose(y[0], expect, rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(y2[0], expect, rtol=1e-11, atol=1e-12)


def test_orthogonal_draft_keys_give_u_equal_r():
    """Mutually orthogonal draft keys make A = 0, so the stored u_s = R_s."""
    shape = wl.GdnShape(B=1, Hv=2, Hk=1, dk=6, dv=3, L=8, in_dtype=wl.F32)
    T = 4
    init = wl.gdn_init(shape, seed=9, fill_max=2)
    r = make_replay(init)
    st = wl.gdn_step(shape, 9, 0, T=T)
    st.k, st.q, st.v, st.beta, st.g = (x.astype(np.float64) for x in (st.k, st.q, st.v, st.beta, st.g))
    Qm, _ = np.linalg.qr(np.random.default_rng(9).standard_normal((shape.dk, shape.dk)))
    for s in range(T):
        st.k[0, s, 0] = Qm[:, s]
    h = int(r.count[0])
    Sh = r.state(0, h)
    r.verify(st.q, st.k, st.v, st.beta, st.g)
    G = np.cumsum(st.g[0].astype(np.float64), axis=0)
    for s in range(T):
        R = st.beta[0, s][:, None] * (st.v[0, s] - np.exp(G[s])[:, None] * (Sh @ st.k[0, s, 0]))
        sl = r.slot(0, h + s + 1)
        np.testing.assert_allclose(r.ring_u[0, :, sl, :], R, rtol=1e-12, atol=1e-14)


def test_snapshot_baseline_equals_recurrence():
    shape = wl.GdnShape(B=3, Hv=2, Hk=1, dk=4, dv=3, L=8, in_dtype=wl.F32)
    T = 3
    init = wl.gdn_init(shape, seed=70, fill_max=0)
    base = og.GdnSnapshotBaseline(init.S0, T)
    S = init.S0.astype(np.float64).copy()
    for rnd in range(5):
        st = wl.gdn_step(shape, 70, rnd, T=T)
        Y = base.verify(st.q, st.k, st.v, st.beta, st.g)
        Sd = S.copy()
        for s in range(T):
            Sd, y_ref = og.householder_step(Sd, st.q[:, s], st.k[:, s], st.v[:, s], st.beta[:, s], st.g[:, s])
            assert rel_err(Y[:, s], y_ref) < 1e-12
        acc = wl.accepted_counts(shape.B, T, 70, rnd)
        base.commit(acc)
        for b in range(shape.B):
            Sb = S[b:b + 1]
            for s in range(int(acc[b])):
                Sb, _ = og.householder_step(Sb, st.q[b:b + 1, s], st.k[b:b + 1, s], st.v[b:b + 1, s],
                                            st.beta[b:b + 1, s], st.g[b:b + 1, s])
            S[b] = Sb[0]
            assert rel_err(base.state(b), S[b]) < 1e-12


def test_storage_rounding_bf16():
    """bf16 storage rounds to nearest even on the 16-bit boundary."""
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -9, -3.0e-3])
    r = og.round_storage(x, "bf16")
    assert r[0] == 1.0
    assert r[1] == 1.0 + 2.0 ** -7 or r[1] == 1.0  # tie -> even mantissa
    assert r[1] == 1.0  # 1 + 2^-8 is a tie between 1 and 1 + 2^-7; even is 1
    assert r[2] == 1.0 + 2.0 ** -7
    assert abs(r[3] - x[3]) <= abs(x[3]) * 2.0 ** -8
