"""GPU parity of the Gated DeltaNet kernels against the fp64 oracle (through the C ABI).

Outputs: |gpu - ref| <= max(1e-3 |ref|, 1e-4) with the buffer's u in fp32,
max(1e-2 |ref|, 1e-3) with bf16 u or bf16 outputs.  Bookkeeping bit-exact.
"""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, dev, gdn_state, gdn_step_dev, host, take, tol_for
from oracle import gdn as og
from ssm_decode_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def rs():
    from ssm_decode_hybrid_gb300 import replayssm

    return replayssm


def oracle_replay(init, idx):
    return og.GdnReplay(take(init.S0, idx), take(init.ring_u, idx), take(init.ring_k, idx), take(init.ring_g, idx),
                        take(init.start, idx), take(init.count, idx), u_dtype=init.shape.u_dtype)


def check_pointers(state, orc, idx, what):
    np.testing.assert_array_equal(host(state.start)[idx], orc.start, err_msg=f"{what}: start")
    np.testing.assert_array_equal(host(state.count)[idx], orc.count, err_msg=f"{what}: count")
    np.testing.assert_array_equal(host(state.flag)[idx], orc.flag, err_msg=f"{what}: flag")


def run_decode(shape, seed, steps, sample=None, y_dtype=torch.float32, workspace_T=8, fused=False):
    R = rs()
    init = wl.gdn_init(shape, seed)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    state = gdn_state(init, workspace_T)
    orc = oracle_replay(init, idx)
    rtol, atol = tol_for(y_dtype)
    if shape.u_dtype == wl.BF16:
        rtol, atol = max(rtol, 1e-2), max(atol, 1e-3)
    for t in range(steps):
        st = wl.gdn_step(shape, seed, t)
        if fused:
            y = R.gdn_replay_decode_fused(state, *gdn_step_dev(st, shape.in_dtype), y_dtype=y_dtype)
        else:
            y = R.gdn_replay_decode(state, *gdn_step_dev(st, shape.in_dtype), y_dtype=y_dtype)
            flags = host(state.flag)
            R.gdn_replay_flush(state)
        y_ref = orc.decode_step(take(st.q, idx), take(st.k, idx), take(st.v, idx), take(st.beta, idx),
                                take(st.g, idx))
        if not fused:
            np.testing.assert_array_equal(flags[idx], orc.flag, err_msg=f"step {t}: flag")
        orc.flush()
        assert_close(y[idx], y_ref, rtol, atol, what=f"step {t}: y")
        check_pointers(state, orc, idx, f"step {t}")
    assert_close(state.S0[idx], orc.S0, rtol, atol, what="final S0")
    assert int(host(state.err)[0]) == 0
    assert int(host(state.sync).sum()) == 0


SHAPES = [
    wl.GdnShape(B=3, Hv=4, Hk=2, dk=16, dv=16, L=4, in_dtype=wl.F32),
    wl.GdnShape(B=4, Hv=6, Hk=3, dk=32, dv=20, L=5, in_dtype=wl.BF16),
    wl.GdnShape(B=3, Hv=4, Hk=4, dk=64, dv=68, L=7, in_dtype=wl.BF16),
    wl.GdnShape(B=4, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16),  # the GDN layer, small batch
    wl.GdnShape(B=2, Hv=2, Hk=1, dk=128, dv=136, L=1, in_dtype=wl.F32),
    wl.GdnShape(B=2, Hv=4, Hk=2, dk=128, dv=128, L=32, in_dtype=wl.BF16),  # tensor-core flush, K extent 64
    wl.GdnShape(B=3, Hv=2, Hk=2, dk=128, dv=64, L=3, in_dtype=wl.BF16, u_dtype=wl.BF16),  # bf16 u, padded K
]


WORKSPACE = [pytest.param(8, id="two-launch"), pytest.param(0, id="one-launch")]
SHAPE_ID = lambda s: f"B{s.B}Hv{s.Hv}Hk{s.Hk}dk{s.dk}dv{s.dv}L{s.L}{s.in_dtype}u{s.u_dtype}"  # noqa: E731


@pytest.mark.parametrize("workspace_T", WORKSPACE)
@pytest.mark.parametrize("shape", SHAPES, ids=SHAPE_ID)
def test_decode_parity(shape, workspace_T):
    run_decode(shape, 200, steps=2 * shape.L + 3, workspace_T=workspace_T)


FUSED_SHAPES = [
    wl.GdnShape(B=4, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16),  # the GDN layer, small batch
    wl.GdnShape(B=3, Hv=6, Hk=3, dk=64, dv=72, L=8, in_dtype=wl.BF16),  # two row blocks, ragged second
    wl.GdnShape(B=3, Hv=2, Hk=2, dk=128, dv=64, L=4, in_dtype=wl.BF16, u_dtype=wl.BF16),  # bf16 u
    wl.GdnShape(B=2, Hv=4, Hk=2, dk=32, dv=20, L=5, in_dtype=wl.BF16),  # outside the two-launch kernels
]


@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=SHAPE_ID)
def test_decode_fused_parity(shape):
    """gdn_replay_decode_fused == decode step followed by the flush."""
    run_decode(shape, 203, steps=2 * shape.L + 3, fused=True)


def test_decode_bf16_u_and_bf16_y():
    shape = wl.GdnShape(B=4, Hv=8, Hk=4, dk=128, dv=128, L=8, in_dtype=wl.BF16, u_dtype=wl.BF16)
    run_decode(shape, 201, steps=12, y_dtype=torch.bfloat16)


def test_gdn_layer_full_batch_sampled():
    """Batch 256, 32 value heads over 16 key heads, d_k = d_v = 128, L = 16."""
    run_decode(wl.GDN_LAYER, wl.SEED_GDN, steps=40, sample=[0, 77, 200, 255])


def test_baseline_parity():
    shape = wl.GdnShape(B=8, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16)
    R = rs()
    init = wl.gdn_init(shape, 202, fill_max=0)
    S = dev(init.S0)
    S_ref = init.S0.astype(np.float64)
    state = gdn_state(init)
    for t in range(24):
        st = wl.gdn_step(shape, 202, t)
        inp = gdn_step_dev(st, shape.in_dtype)
        y = R.gdn_state_update_baseline(S, *inp)
        y_rep = R.gdn_replay_decode(state, *inp)
        R.gdn_replay_flush(state)
        S_ref, y_ref, _ = og.rank1_step(S_ref, st.q, st.k, st.v, st.beta, st.g)
        assert_close(y, y_ref, what=f"baseline step {t}")
        assert_close(y_rep, y_ref, what=f"replay step {t}")
    assert_close(S, S_ref, what="baseline state")


def run_verify(shape, T, rounds, seed, sample=None, workspace_T=8, y_dtype=torch.float32):
    R = rs()
    init = wl.gdn_init(shape, seed, fill_max=shape.L - T)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    state = gdn_state(init, workspace_T)
    orc = oracle_replay(init, idx)
    rtol, atol = (1e-2, 1e-3) if shape.u_dtype == wl.BF16 else (1e-3, 1e-4)
    for r in range(rounds):
        st = wl.gdn_step(shape, seed, r, T=T)
        acc = wl.accepted_counts(shape.B, T, seed, r)
        y = R.gdn_replay_verify(state, *gdn_step_dev(st, shape.in_dtype), y_dtype=y_dtype)
        Y_ref = orc.verify(take(st.q, idx), take(st.k, idx), take(st.v, idx), take(st.beta, idx), take(st.g, idx))
        np.testing.assert_array_equal(host(state.flag)[idx], orc.flag, err_msg=f"round {r}: flag")
        yr, ya = (1e-2, 1e-3) if y_dtype == torch.bfloat16 else (rtol, atol)
        assert_close(y[idx], Y_ref, yr, ya, what=f"round {r}: y")
        R.replay_spec_commit(dev(acc, torch.int32), state.count, T, shape.L, state.err)
        orc.commit(take(acc, idx), T)
        R.gdn_replay_flush(state)
        orc.flush()
        check_pointers(state, orc, idx, f"round {r}")
    assert_close(state.S0[idx], orc.S0, rtol, atol, what="final S0")
    assert int(host(state.err)[0]) == 0


@pytest.mark.parametrize("workspace_T", WORKSPACE)
@pytest.mark.parametrize("T", [1, 2, 4, 6, 8])
def test_chunked_verify_parity(T, workspace_T):
    shape = wl.GdnShape(B=8, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16)
    run_verify(shape, T, rounds=10, seed=300 + T, workspace_T=workspace_T)


def test_chunked_verify_workspace_too_small_for_T():
    """A workspace sized for 4 drafts: T = 4 uses it, T = 6 takes the one-launch path; both match."""
    shape = wl.GdnShape(B=4, Hv=8, Hk=4, dk=64, dv=64, L=16, in_dtype=wl.BF16)
    run_verify(shape, 4, rounds=6, seed=330, workspace_T=4)
    run_verify(shape, 6, rounds=6, seed=331, workspace_T=4)


def test_chunked_verify_small_shapes():
    run_verify(wl.GdnShape(B=4, Hv=4, Hk=2, dk=16, dv=16, L=6, in_dtype=wl.F32), 3, rounds=10, seed=310)
    run_verify(wl.GdnShape(B=4, Hv=6, Hk=3, dk=64, dv=36, L=9, in_dtype=wl.BF16), 4, rounds=10, seed=311)
    run_verify(wl.GdnShape(B=3, Hv=6, Hk=3, dk=64, dv=72, L=8, in_dtype=wl.BF16), 3, rounds=8, seed=312)
    run_verify(wl.GdnShape(B=3, Hv=4, Hk=2, dk=128, dv=64, L=12, in_dtype=wl.BF16, u_dtype=wl.BF16), 2, rounds=8,
               seed=313)


@pytest.mark.parametrize("T,u_dtype,y_dtype", [(3, wl.BF16, torch.bfloat16), (7, wl.F32, torch.bfloat16),
                                               (5, wl.BF16, torch.float32)])
def test_chunked_verify_tensor_core_dtypes(T, u_dtype, y_dtype):
    """d_k = d_v = 128 with T >= 2 takes the tensor-core stream: bf16 u ring
    and bf16 outputs, four value heads per key head, a ragged window."""
    shape = wl.GdnShape(B=5, Hv=8, Hk=2, dk=128, dv=128, L=16, in_dtype=wl.BF16, u_dtype=u_dtype)
    run_verify(shape, T, rounds=8, seed=340 + T, y_dtype=y_dtype)


def test_chunked_verify_window_equal_to_ring():
    """T = L: every round starts from an empty buffer and flushes after it."""
    run_verify(wl.GdnShape(B=4, Hv=8, Hk=4, dk=128, dv=128, L=4, in_dtype=wl.BF16), 4, rounds=8, seed=350)
    run_verify(wl.GdnShape(B=3, Hv=4, Hk=2, dk=64, dv=64, L=2, in_dtype=wl.BF16), 2, rounds=8, seed=351)


def test_chunked_verify_full_batch_sampled():
    """Batch 256, T = 4, accepted ~ U{0..4}: sampled sequences."""
    run_verify(wl.GDN_LAYER, 4, rounds=16, seed=wl.SEED_GDN + 50, sample=[1, 99, 254])


@pytest.mark.parametrize("T", [1, 4])
def test_snapshot_baseline_parity(T):
    shape = wl.GdnShape(B=4, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16)
    R = rs()
    init = wl.gdn_init(shape, 320 + T, fill_max=0)
    slots = torch.zeros(shape.B, T + 1, shape.Hv, shape.dv, shape.dk, device="cuda")
    slots[:, 0] = dev(init.S0)
    cur = torch.zeros(shape.B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = og.GdnSnapshotBaseline(init.S0, T)
    for r in range(6):
        st = wl.gdn_step(shape, 320 + T, r, T=T)
        y = R.gdn_spec_verify_baseline(slots, cur, *gdn_step_dev(st, shape.in_dtype), err=err)
        Y_ref = base.verify(st.q, st.k, st.v, st.beta, st.g)
        assert_close(y, Y_ref, what=f"round {r}")
        acc = wl.accepted_counts(shape.B, T, 320 + T, r)
        R.ssm_spec_commit_baseline(dev(acc, torch.int32), cur, T, err)
        base.commit(acc)
        np.testing.assert_array_equal(host(cur), base.cur)
    for b in range(shape.B):
        assert_close(slots[b, int(base.cur[b])], base.state(b), what=f"state {b}")
    assert int(host(err)[0]) == 0


def test_tensor_core_verify_window_error_skips_the_sequence():
    """A verify window that does not fit (count + T > L) on the tensor-core
    path: the error bit is set, that sequence's outputs are left alone, the
    other sequences follow the oracle; nothing faults."""
    R = rs()
    shape = wl.GdnShape(B=3, Hv=4, Hk=2, dk=128, dv=128, L=8, in_dtype=wl.BF16)
    T = 4
    init = wl.gdn_init(shape, 360, fill_max=shape.L - T)
    init.count[:] = [2, 6, 0]  # 6 + 4 > 8
    state = gdn_state(init)
    orc = oracle_replay(init, np.array([0, 2]))
    st = wl.gdn_step(shape, 360, 0, T=T)
    y = torch.full((shape.B, T, shape.Hv, shape.dv), float("nan"), device="cuda")
    R.gdn_replay_verify(state, *gdn_step_dev(st, shape.in_dtype), y=y)
    assert R.read_error(state.err) == R.EBIT_WINDOW
    yh = host(y)
    assert np.all(np.isnan(yh[1]))
    Y_ref = orc.verify(take(st.q, [0, 2]), take(st.k, [0, 2]), take(st.v, [0, 2]), take(st.beta, [0, 2]),
                       take(st.g, [0, 2]))
    assert_close(y[[0, 2]], Y_ref, what="valid sequences")


def test_gdn_layer_fused_full_batch_sampled():
    """gdn_replay_decode_fused with the workspace (the launch pair the GDN
    benchmark times) at its own size: batch 256, Hv = 32, Hk = 16,
    d_k = d_v = 128, L = 16, random fill, 40 steps (every sequence folds at
    least twice).  Eight sampled sequences against the oracle, the first and
    last of the grid among them; every sequence's pointers against their closed
    form (the fused step folds a full buffer in place: start never moves)."""
    shape = wl.GDN_LAYER
    R = rs()
    init = wl.gdn_init(shape, wl.SEED_GDN)
    idx = np.array([0, 1, 63, 77, 128, 200, 254, 255])
    state = gdn_state(init)
    orc = oracle_replay(init, idx)
    start0, count0 = init.start.astype(np.int64), init.count.astype(np.int64)
    for t in range(40):
        st = wl.gdn_step(shape, wl.SEED_GDN, t)
        y = R.gdn_replay_decode_fused(state, *gdn_step_dev(st, shape.in_dtype))
        y_ref = orc.decode_step(take(st.q, idx), take(st.k, idx), take(st.v, idx), take(st.beta, idx),
                                take(st.g, idx))
        orc.flush()
        assert_close(y[idx], y_ref, what=f"step {t}")
        tot = count0 + t + 1
        np.testing.assert_array_equal(host(state.count), tot % shape.L, err_msg=f"step {t}: count")
        np.testing.assert_array_equal(host(state.start), start0, err_msg=f"step {t}: start")
        np.testing.assert_array_equal(host(state.flag), np.zeros(shape.B), err_msg=f"step {t}: flag")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0


def run_verify_fused(shape, T, rounds, seed, sample=None, workspace_T=8):
    """Rounds of gdn_replay_verify_fused + replay_spec_commit (no separate
    flush) against the oracle doing flush, verify, commit: outputs within
    tolerance, pointers bit-exact every round, final S_0 after a last flush."""
    R = rs()
    init = wl.gdn_init(shape, seed, fill_max=shape.L - T)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    state = gdn_state(init, workspace_T)
    orc = oracle_replay(init, idx)
    rtol, atol = (1e-2, 1e-3) if shape.u_dtype == wl.BF16 else (1e-3, 1e-4)
    for r in range(rounds):
        st = wl.gdn_step(shape, seed, r, T=T)
        acc = wl.accepted_counts(shape.B, T, seed, r)
        y = R.gdn_replay_verify_fused(state, *gdn_step_dev(st, shape.in_dtype))
        orc.flush()
        Y_ref = orc.verify(take(st.q, idx), take(st.k, idx), take(st.v, idx), take(st.beta, idx), take(st.g, idx))
        assert_close(y[idx], Y_ref, rtol, atol, what=f"round {r}: y")
        check_pointers(state, orc, idx, f"round {r}")
        R.replay_spec_commit(dev(acc, torch.int32), state.count, T, shape.L, state.err)
        orc.commit(take(acc, idx), T)
    R.gdn_replay_flush(state)
    orc.flush()
    check_pointers(state, orc, idx, "final flush")
    assert_close(state.S0[idx], orc.S0, rtol, atol, what="final S0")
    assert int(host(state.err)[0]) == 0
    assert int(host(state.sync).sum()) == 0


@pytest.mark.parametrize("workspace_T", WORKSPACE)
@pytest.mark.parametrize("T", [1, 2, 4, 6, 8])
def test_chunked_verify_fused_parity(T, workspace_T):
    """gdn_replay_verify_fused == gdn_replay_flush + gdn_replay_verify, over
    rounds whose early flushes empty windows whose slots the next drafts
    overwrite; pipelined (T >= 2), CUDA-core (T = 1) and one-launch verify."""
    shape = wl.GdnShape(B=8, Hv=8, Hk=4, dk=128, dv=128, L=16, in_dtype=wl.BF16)
    run_verify_fused(shape, T, rounds=12, seed=340 + T, workspace_T=workspace_T)


def test_chunked_verify_fused_dtypes_and_window_equal_to_ring():
    # bf16 u and bf16 keys in the flush; T = L = 4: every round flushes what it committed
    run_verify_fused(wl.GdnShape(B=4, Hv=4, Hk=2, dk=128, dv=128, L=8, in_dtype=wl.BF16, u_dtype=wl.BF16), 4,
                     rounds=10, seed=350)
    run_verify_fused(wl.GdnShape(B=5, Hv=4, Hk=4, dk=128, dv=128, L=4, in_dtype=wl.BF16), 4, rounds=8, seed=351)


def test_chunked_verify_fused_full_batch_sampled():
    """The GDN layer at its own size (B = 256, Hv = 32, Hk = 16, T = 4, L = 16),
    the pending flush, the verify and the commit, 16 rounds, eight sampled
    sequences."""
    run_verify_fused(wl.GDN_LAYER, 4, rounds=16, seed=wl.SEED_GDN + 60,
                     sample=[0, 1, 63, 128, 200, 230, 254, 255], workspace_T=4)


def test_fused_decode_output_feeds_next_step():
    """Each step's y (bf16) is the next step's v, passed as the same device
    buffer, so the next step's precompute (which may start during the previous
    S_0 stream) must read its inputs only after that grid has finished.
    Batch 64, 20 steps; the oracle gets the GPU's y as its next v."""
    R = rs()
    shape = wl.GdnShape(B=64, Hv=32, Hk=16, dk=128, dv=128, L=8, in_dtype=wl.BF16)
    seed = 271
    init = wl.gdn_init(shape, seed)
    idx = np.array([0, 1, 31, 32, 63])
    state = gdn_state(init, 1)
    orc = oracle_replay(init, idx)
    st0 = wl.gdn_step(shape, seed, 0)
    bufs = [dev(st0.v, torch.bfloat16).reshape(shape.B, shape.Hv, shape.dv),
            torch.empty(shape.B, shape.Hv, shape.dv, dtype=torch.bfloat16, device="cuda")]
    for t in range(20):
        st = wl.gdn_step(shape, seed, t)
        q, k, _, beta, g = gdn_step_dev(st, shape.in_dtype)
        v_in, y = bufs[t % 2], bufs[(t + 1) % 2]
        v_host = host(v_in.float()).reshape(np.asarray(st.v).shape)
        R.gdn_replay_decode_fused(state, q, k, v_in, beta, g, y=y)
        y_ref = orc.decode_step(take(st.q, idx), take(st.k, idx), take(v_host, idx), take(st.beta, idx),
                                take(st.g, idx))
        orc.flush()
        assert_close(y[idx], y_ref, 1e-2, 1e-3, what=f"step {t}: y")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0
