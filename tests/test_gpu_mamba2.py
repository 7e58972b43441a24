"""GPU parity of the Mamba-2 kernels against the fp64 oracle (through the C ABI).

Outputs: |gpu - ref| <= max(1e-3 |ref|, 1e-4) (fp32 y), max(1e-2 |ref|, 1e-3)
(bf16 y).  start/count/flag and the error word: bit-exact.
"""
import numpy as np
import pytest
import torch

from gpu_util import (assert_close, dev, host, m2_state, m2_step_dev, take, tol_for)
from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def rs():
    from ssm_decode_hybrid_gb300 import replayssm

    return replayssm


def oracle_replay(init, idx):
    return om.Mamba2Replay(take(init.S0, idx), init.A, take(init.ring_v, idx), take(init.ring_k, idx),
                           take(init.ring_dt, idx), take(init.start, idx), take(init.count, idx))


def check_pointers(state, orc, idx, what):
    np.testing.assert_array_equal(host(state.start)[idx], orc.start, err_msg=f"{what}: start")
    np.testing.assert_array_equal(host(state.count)[idx], orc.count, err_msg=f"{what}: count")
    np.testing.assert_array_equal(host(state.flag)[idx], orc.flag, err_msg=f"{what}: flag")


def run_decode(shape, seed, steps, sample=None, y_dtype=torch.float32, check_every=1, workspace=True):
    R = rs()
    init = wl.mamba2_init(shape, seed)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    state = m2_state(init, workspace)
    orc = oracle_replay(init, idx)
    A = dev(init.A)
    rtol, atol = tol_for(y_dtype)
    for t in range(steps):
        st = wl.mamba2_step(shape, seed, t)
        v, k, q, dt = m2_step_dev(st, shape.in_dtype)
        y = R.replay_decode_step(state, v, k, q, dt, A, y_dtype=y_dtype)
        flags_after_decode = host(state.flag)
        R.replay_flush(state, A)
        y_ref = orc.decode_step(take(st.v, idx), take(st.k, idx), take(st.q, idx), take(st.dt, idx))
        np.testing.assert_array_equal(flags_after_decode[idx], orc.flag, err_msg=f"step {t}: flag")
        orc.flush()
        if t % check_every == 0 or t == steps - 1:
            assert_close(y[idx], y_ref, rtol, atol, what=f"step {t}: y")
            check_pointers(state, orc, idx, f"step {t}")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0
    assert int(host(state.sync).sum()) == 0
    return state, orc


def test_tiny_config_parity():
    """Tiny Mamba-2 decode (batch 1, 4 heads, d = n = 16, L = 4, fp32), 32 steps."""
    run_decode(wl.TINY_MAMBA2, wl.SEED_TINY, steps=32)


SHAPES = [
    wl.Mamba2Shape(B=3, H=4, G=2, d=16, n=16, L=4, in_dtype=wl.F32),
    wl.Mamba2Shape(B=5, H=6, G=3, d=20, n=32, L=3, in_dtype=wl.BF16),
    wl.Mamba2Shape(B=4, H=8, G=2, d=68, n=64, L=7, in_dtype=wl.BF16),  # ragged rows
    wl.Mamba2Shape(B=3, H=4, G=1, d=136, n=128, L=32, in_dtype=wl.BF16),  # two row chunks + tail
    wl.Mamba2Shape(B=2, H=2, G=2, d=4, n=128, L=1, in_dtype=wl.F32),  # flush every step
    wl.Mamba2Shape(B=6, H=32, G=8, d=64, n=128, L=16, in_dtype=wl.BF16),  # the Nemotron-H layer, small batch
    wl.Mamba2Shape(B=3, H=4, G=2, d=96, n=128, L=32, in_dtype=wl.BF16),  # tensor-core flush, K extent 64
    wl.Mamba2Shape(B=2, H=2, G=1, d=32, n=128, L=5, in_dtype=wl.BF16),  # tensor-core flush, zero-padded K
]


WORKSPACE = [pytest.param(True, id="two-launch"), pytest.param(False, id="one-launch")]


@pytest.mark.parametrize("workspace", WORKSPACE)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s.B}H{s.H}G{s.G}d{s.d}n{s.n}L{s.L}{s.in_dtype}")
def test_decode_parity(shape, workspace):
    run_decode(shape, seed=123, steps=2 * shape.L + 3, workspace=workspace)


FUSED_SHAPES = [
    wl.Mamba2Shape(B=6, H=32, G=8, d=64, n=128, L=16, in_dtype=wl.BF16),
    wl.Mamba2Shape(B=5, H=8, G=4, d=32, n=64, L=8, in_dtype=wl.F32),
    wl.Mamba2Shape(B=3, H=4, G=2, d=16, n=16, L=4, in_dtype=wl.BF16),
    wl.Mamba2Shape(B=4, H=6, G=3, d=20, n=32, L=3, in_dtype=wl.BF16),  # outside the pipelined kernel
]


@pytest.mark.parametrize("workspace", WORKSPACE)
@pytest.mark.parametrize("shape", FUSED_SHAPES, ids=lambda s: f"B{s.B}H{s.H}d{s.d}n{s.n}L{s.L}{s.in_dtype}")
def test_decode_fused_parity(shape, workspace):
    """replay_decode_step_fused == decode step followed by the flush."""
    R = rs()
    seed = 321
    init = wl.mamba2_init(shape, seed)
    state = m2_state(init, workspace)
    orc = oracle_replay(init, np.arange(shape.B))
    A = dev(init.A)
    for t in range(2 * shape.L + 3):
        st = wl.mamba2_step(shape, seed, t)
        y = R.replay_decode_step_fused(state, *m2_step_dev(st, shape.in_dtype), A)
        y_ref = orc.decode_step(st.v, st.k, st.q, st.dt)
        orc.flush()
        assert_close(y, y_ref, what=f"step {t}")
        check_pointers(state, orc, np.arange(shape.B), f"step {t}")
    assert_close(state.S0, orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0
    assert int(host(state.sync).sum()) == 0


def test_decode_bf16_output():
    run_decode(wl.Mamba2Shape(B=4, H=8, G=2, d=64, n=128, L=8, in_dtype=wl.BF16), 77, steps=12,
               y_dtype=torch.bfloat16)


def test_nemotron_layer_full_batch_sampled():
    """Batch 256, 32 heads, d=64, n=128, G=8, L=16, random fill levels: 48 steps
    (three flush cycles per sequence); sampled sequences against the oracle,
    bookkeeping of every sequence against its closed form."""
    shape = wl.NEMOTRON_H_MAMBA2
    R = rs()
    init = wl.mamba2_init(shape, wl.SEED_NEMOTRON)
    idx = np.array([0, 37, 128, 255])
    state = m2_state(init)
    orc = oracle_replay(init, idx)
    A = dev(init.A)
    start0, count0 = init.start.astype(np.int64), init.count.astype(np.int64)
    for t in range(48):
        st = wl.mamba2_step(shape, wl.SEED_NEMOTRON, t)
        y = R.replay_decode_step(state, *m2_step_dev(st, shape.in_dtype), A)
        R.replay_flush(state, A)
        y_ref = orc.decode_step(take(st.v, idx), take(st.k, idx), take(st.q, idx), take(st.dt, idx))
        orc.flush()
        assert_close(y[idx], y_ref, what=f"step {t}")
        # every sequence: after t+1 steps, total = count0 + t + 1 entries went through
        tot = count0 + t + 1
        np.testing.assert_array_equal(host(state.count), tot % shape.L)
        np.testing.assert_array_equal(host(state.start), (start0 + (tot // shape.L) * shape.L) % shape.L)
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0


def test_replay_matches_baseline_kernel():
    """The replay path and the baseline kernel agree on the same inputs, and
    the baseline matches the plain recurrence."""
    shape = wl.Mamba2Shape(B=16, H=32, G=8, d=64, n=128, L=16, in_dtype=wl.BF16)
    R = rs()
    init = wl.mamba2_init(shape, 9, fill_max=0)
    state = m2_state(init)
    S = dev(init.S0)
    A = dev(init.A)
    S_ref = init.S0.astype(np.float64)
    for t in range(40):
        st = wl.mamba2_step(shape, 9, t)
        inp = m2_step_dev(st, shape.in_dtype)
        y_rep = R.replay_decode_step(state, *inp, A)
        R.replay_flush(state, A)
        y_base = R.ssm_state_update_baseline(S, *inp, A)
        S_ref, y_ref = om.recurrence_step(S_ref, st.v, st.k, st.q, st.dt, init.A)
        assert_close(y_base, y_ref, what=f"baseline step {t}")
        assert_close(y_rep, y_ref, what=f"replay step {t}")
    assert_close(S, S_ref, what="baseline state")


def test_baseline_tiny_and_bf16_out():
    shape = wl.TINY_MAMBA2
    R = rs()
    init = wl.mamba2_init(shape, 5, fill_max=0)
    S = dev(init.S0)
    S_ref = init.S0.astype(np.float64)
    for t in range(32):
        st = wl.mamba2_step(shape, 5, t)
        y = R.ssm_state_update_baseline(S, *m2_step_dev(st, shape.in_dtype), dev(init.A),
                                        y_dtype=torch.bfloat16 if t % 2 else torch.float32)
        S_ref, y_ref = om.recurrence_step(S_ref, st.v, st.k, st.q, st.dt, init.A)
        assert_close(y, y_ref, *tol_for(y.dtype), what=f"step {t}")


def test_flush_anywhere_gpu():
    """Forcing flushes at random steps (flag written from the host) leaves every
    output unchanged."""
    shape = wl.Mamba2Shape(B=8, H=8, G=2, d=32, n=64, L=8, in_dtype=wl.BF16)
    R = rs()
    init = wl.mamba2_init(shape, 31)
    s1, s2 = m2_state(init), m2_state(init)
    A = dev(init.A)
    rng = np.random.default_rng(31)
    for t in range(20):
        inp = m2_step_dev(wl.mamba2_step(shape, 31, t), shape.in_dtype)
        y1 = R.replay_decode_step(s1, *inp, A)
        R.replay_flush(s1, A)
        y2 = R.replay_decode_step(s2, *inp, A)
        force = torch.from_numpy((rng.random(shape.B) < 0.4).astype(np.int32)).cuda()
        s2.flag.copy_(torch.maximum(s2.flag, force))
        R.replay_flush(s2, A)
        assert_close(y2, host(y1), what=f"step {t}")


def run_spec(shape, T, rounds, seed, sample=None, workspace=True, y_dtype=torch.float32):
    R = rs()
    init = wl.mamba2_init(shape, seed, fill_max=shape.L - T)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    state = m2_state(init, workspace)
    orc = oracle_replay(init, idx)
    A = dev(init.A)
    for r in range(rounds):
        st = wl.mamba2_step(shape, seed, r, T=T)
        acc = wl.accepted_counts(shape.B, T, seed, r)
        y = R.replay_spec_verify(state, *m2_step_dev(st, shape.in_dtype), A, y_dtype=y_dtype)
        Y_ref = orc.spec_verify(take(st.v, idx), take(st.k, idx), take(st.q, idx), take(st.dt, idx))
        np.testing.assert_array_equal(host(state.flag)[idx], orc.flag, err_msg=f"round {r}: flag")
        assert_close(y[idx], Y_ref, *tol_for(y_dtype), what=f"round {r}: y")
        R.replay_spec_commit(dev(acc, torch.int32), state.count, T, shape.L, state.err)
        orc.commit(take(acc, idx), T)
        R.replay_flush(state, A)
        orc.flush()
        check_pointers(state, orc, idx, f"round {r}")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0


@pytest.mark.parametrize("workspace", WORKSPACE)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_spec_verify_parity(T, workspace):
    shape = wl.Mamba2Shape(B=12, H=8, G=2, d=64, n=128, L=16, in_dtype=wl.BF16)
    run_spec(shape, T, rounds=12, seed=40 + T, workspace=workspace)


def test_spec_verify_small_shapes():
    run_spec(wl.Mamba2Shape(B=5, H=4, G=1, d=16, n=16, L=6, in_dtype=wl.F32), 3, rounds=10, seed=3)
    run_spec(wl.Mamba2Shape(B=5, H=6, G=3, d=36, n=32, L=9, in_dtype=wl.BF16), 4, rounds=10, seed=4)
    # two-launch verify: fp32 inputs with n = 32, ragged heads, bf16 with n = 64 and a 12-slot ring
    run_spec(wl.Mamba2Shape(B=4, H=6, G=3, d=20, n=32, L=8, in_dtype=wl.F32), 3, rounds=10, seed=5)
    run_spec(wl.Mamba2Shape(B=4, H=8, G=2, d=48, n=64, L=12, in_dtype=wl.BF16), 6, rounds=10, seed=6)


@pytest.mark.parametrize("T", [3, 7])
def test_spec_verify_bf16_out_tensor_core(T):
    """bf16 outputs, eight heads per group; n = 128, d = 64 with T >= 5 takes
    the tensor-core stream (two heads of a group per block), T = 3 the CUDA
    cores."""
    shape = wl.Mamba2Shape(B=6, H=16, G=2, d=64, n=128, L=16, in_dtype=wl.BF16)
    run_spec(shape, T, rounds=8, seed=80 + T, y_dtype=torch.bfloat16)


def test_spec_window_equal_to_ring():
    """T = L: every round starts with an empty buffer (fill 0), flags the early
    flush, and folds exactly the accepted drafts."""
    run_spec(wl.Mamba2Shape(B=5, H=8, G=2, d=64, n=128, L=4, in_dtype=wl.BF16), 4, rounds=8, seed=95)
    run_spec(wl.Mamba2Shape(B=3, H=4, G=2, d=32, n=64, L=2, in_dtype=wl.F32), 2, rounds=8, seed=96)


def test_spec_full_batch_sampled():
    """Batch 512, T = 4, L = 16, accepted ~ U{0..4}: sampled sequences."""
    run_spec(wl.SPEC_MAMBA2, 4, rounds=24, seed=wl.SEED_SPEC, sample=[0, 100, 311, 511])


@pytest.mark.parametrize("T", [1, 4, 6])
def test_snapshot_baseline_parity(T):
    shape = wl.Mamba2Shape(B=6, H=8, G=2, d=64, n=128, L=16, in_dtype=wl.BF16)
    R = rs()
    init = wl.mamba2_init(shape, 60 + T, fill_max=0)
    slots = torch.zeros(shape.B, T + 1, shape.H, shape.d, shape.n, device="cuda")
    slots[:, 0] = dev(init.S0)
    cur = torch.zeros(shape.B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    base = om.Mamba2SnapshotBaseline(init.S0, init.A, T)
    A = dev(init.A)
    for r in range(8):
        st = wl.mamba2_step(shape, 60 + T, r, T=T)
        y = R.ssm_spec_verify_baseline(slots, cur, *m2_step_dev(st, shape.in_dtype), A, err=err)
        Y_ref = base.verify(st.v, st.k, st.q, st.dt)
        assert_close(y, Y_ref, what=f"round {r}")
        acc = wl.accepted_counts(shape.B, T, 60 + T, r)
        R.ssm_spec_commit_baseline(dev(acc, torch.int32), cur, T, err)
        base.commit(acc)
        np.testing.assert_array_equal(host(cur), base.cur)
    for b in range(shape.B):
        assert_close(slots[b, int(base.cur[b])], base.state(b), what=f"state {b}")
    assert int(host(err)[0]) == 0


def test_device_error_bits():
    """Out-of-range bookkeeping sets the sticky error word and skips only the
    offending sequence; nothing faults."""
    shape = wl.Mamba2Shape(B=4, H=4, G=2, d=32, n=64, L=8, in_dtype=wl.BF16)
    R = rs()
    init = wl.mamba2_init(shape, 70)
    init.count[:] = [8, 2, -1, 3]  # 8 == L and -1 are out of range
    state = m2_state(init)
    A = dev(init.A)
    st = wl.mamba2_step(shape, 70, 0)
    y = torch.full((shape.B, shape.H, shape.d), float("nan"), device="cuda")
    R.replay_decode_step(state, *m2_step_dev(st, shape.in_dtype), A, y=y)
    torch.cuda.synchronize()
    assert int(host(state.err)[0]) == R.EBIT_COUNT_RANGE
    assert R.read_error(state.err) == R.EBIT_COUNT_RANGE
    np.testing.assert_array_equal(host(state.count), [8, 3, -1, 4])
    yh = host(y)
    assert np.all(np.isnan(yh[[0, 2]])) and np.all(np.isfinite(yh[[1, 3]]))
    assert int(host(state.sync).sum()) == 0
    # verify window that does not fit, then an accepted count out of range
    state.err.zero_()
    state.count.copy_(dev(np.array([7, 1, 2, 0]), torch.int32))
    st4 = wl.mamba2_step(shape, 70, 1, T=2)
    R.replay_spec_verify(state, *m2_step_dev(st4, shape.in_dtype), A)
    torch.cuda.synchronize()
    assert int(host(state.err)[0]) == R.EBIT_WINDOW
    state.err.zero_()
    R.replay_spec_commit(dev(np.array([0, 3, 1, -1]), torch.int32), state.count, 2, shape.L, state.err)
    torch.cuda.synchronize()
    assert int(host(state.err)[0]) == R.EBIT_ACCEPTED
    np.testing.assert_array_equal(host(state.count), [7, 1, 3, 0])


def test_checkpoint_resume_bit_identical():
    """Copy the caller-owned state to the host mid-run, restore it into fresh
    buffers, continue: outputs are bit-identical to the uninterrupted run."""
    shape = wl.Mamba2Shape(B=8, H=8, G=2, d=64, n=128, L=8, in_dtype=wl.BF16)
    R = rs()
    init = wl.mamba2_init(shape, 80)
    state = m2_state(init)
    A = dev(init.A)
    steps = [m2_step_dev(wl.mamba2_step(shape, 80, t), shape.in_dtype) for t in range(14)]
    snap = None
    ys = []
    for t, inp in enumerate(steps):
        if t == 5:
            # the workspace is scratch: not part of the checkpoint
            snap = {f: getattr(state, f).cpu().clone() for f in state.__dataclass_fields__ if f != "work"}
        ys.append(R.replay_decode_step(state, *inp, A).clone())
        R.replay_flush(state, A)
    restored = R.Mamba2State(**{f: v.cuda() for f, v in snap.items()}).add_workspace()
    for t, inp in enumerate(steps[5:], start=5):
        y = R.replay_decode_step(restored, *inp, A)
        R.replay_flush(restored, A)
        assert torch.equal(y, ys[t])
    assert torch.equal(restored.S0, state.S0)


def test_tensor_core_verify_window_error_skips_the_sequence():
    """As above for the Mamba-2 tensor-core verify (T = 5)."""
    R = rs()
    shape = wl.Mamba2Shape(B=3, H=8, G=2, d=64, n=128, L=8, in_dtype=wl.BF16)
    T = 5
    init = wl.mamba2_init(shape, 97, fill_max=shape.L - T)
    init.count[:] = [1, 4, 3]  # 4 + 5 > 8
    state = m2_state(init)
    orc = oracle_replay(init, np.array([0, 2]))
    A = dev(init.A)
    st = wl.mamba2_step(shape, 97, 0, T=T)
    y = torch.full((shape.B, T, shape.H, shape.d), float("nan"), device="cuda")
    R.replay_spec_verify(state, *m2_step_dev(st, shape.in_dtype), A, y=y)
    assert R.read_error(state.err) == R.EBIT_WINDOW
    yh = host(y)
    assert np.all(np.isnan(yh[1]))
    Y_ref = orc.spec_verify(take(st.v, [0, 2]), take(st.k, [0, 2]), take(st.q, [0, 2]), take(st.dt, [0, 2]))
    assert_close(y[[0, 2]], Y_ref, what="valid sequences")


def run_fused_sampled(shape, seed, steps, idx, graph_steps=0):
    """replay_decode_step_fused with a workspace (the launch pair the benchmark
    times) over `steps` steps: sampled sequences' outputs and final S_0 against
    the oracle, every sequence's pointers against their closed form (the fused
    step folds a full buffer in place, so start never moves and count cycles
    through 0..L-1).  The last `graph_steps` steps are captured once in a CUDA
    graph per step and replayed, as the benchmark does."""
    R = rs()
    init = wl.mamba2_init(shape, seed)
    state = m2_state(init)
    orc = oracle_replay(init, idx)
    A = dev(init.A)
    start0, count0 = init.start.astype(np.int64), init.count.astype(np.int64)
    y = torch.empty(shape.B, shape.H, shape.d, device="cuda")
    for t in range(steps):
        st = wl.mamba2_step(shape, seed, t)
        inp = m2_step_dev(st, shape.in_dtype)
        if t >= steps - graph_steps:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            snap = {f: getattr(state, f).clone() for f in ("S0", "ring_v", "ring_k", "ring_dt", "start", "count")}
            with torch.cuda.graph(g, stream=s):
                R.replay_decode_step_fused(state, *inp, A, y=y)
            torch.cuda.current_stream().wait_stream(s)
            for f, v in snap.items():  # capture does not run the kernels, but be explicit
                assert torch.equal(getattr(state, f), v)
            g.replay()
        else:
            R.replay_decode_step_fused(state, *inp, A, y=y)
        y_ref = orc.decode_step(take(st.v, idx), take(st.k, idx), take(st.q, idx), take(st.dt, idx))
        orc.flush()
        assert_close(y[idx], y_ref, what=f"step {t}")
        tot = count0 + t + 1
        np.testing.assert_array_equal(host(state.count), tot % shape.L, err_msg=f"step {t}: count")
        np.testing.assert_array_equal(host(state.start), start0, err_msg=f"step {t}: start")
        np.testing.assert_array_equal(host(state.flag), np.zeros(shape.B), err_msg=f"step {t}: flag")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0
    assert int(host(state.sync).sum()) == 0


def test_nemotron_layer_fused_full_batch_sampled():
    """The benchmarked step at its own size: batch 256, H = 32, G = 8, d = 64,
    n = 128, L = 16, random fill, replay_decode_step_fused with the workspace
    (precompute + S_0 stream of 8192 blocks, several waves), 48 steps so every
    sequence folds three times; the last 8 steps replayed from CUDA graphs.
    Ten sampled sequences, the first and last blocks of the grid among them."""
    run_fused_sampled(wl.NEMOTRON_H_MAMBA2, wl.SEED_NEMOTRON, 48,
                      np.array([0, 1, 31, 37, 64, 128, 191, 200, 254, 255]), graph_steps=8)


@pytest.mark.parametrize("L", [4, 32])
def test_layer_sweep_fused_points(L):
    """The layer-sweep points at the sweep's dims (H = 32, G = 8, d = 64,
    n = 128) with the smallest and largest ring, batch 64, fused with a
    workspace: 2L + 8 steps, eight sampled sequences."""
    shape = wl.Mamba2Shape(B=64, H=32, G=8, d=64, n=128, L=L, in_dtype=wl.BF16)
    run_fused_sampled(shape, wl.SEED_SWEEP + L, 2 * L + 8, np.array([0, 5, 17, 32, 40, 51, 62, 63]))


def run_spec_fused(shape, T, rounds, seed, sample=None, workspace=True):
    """Rounds of replay_spec_verify_fused + replay_spec_commit (no separate
    flush) against the oracle doing flush, verify, commit: outputs within
    tolerance, pointers bit-exact every round, final S_0 after a last flush."""
    R = rs()
    init = wl.mamba2_init(shape, seed, fill_max=shape.L - T)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    state = m2_state(init, workspace)
    orc = oracle_replay(init, idx)
    A = dev(init.A)
    for r in range(rounds):
        st = wl.mamba2_step(shape, seed, r, T=T)
        acc = wl.accepted_counts(shape.B, T, seed, r)
        y = R.replay_spec_verify_fused(state, *m2_step_dev(st, shape.in_dtype), A)
        orc.flush()
        Y_ref = orc.spec_verify(take(st.v, idx), take(st.k, idx), take(st.q, idx), take(st.dt, idx))
        assert_close(y[idx], Y_ref, what=f"round {r}: y")
        check_pointers(state, orc, idx, f"round {r}")
        R.replay_spec_commit(dev(acc, torch.int32), state.count, T, shape.L, state.err)
        orc.commit(take(acc, idx), T)
        np.testing.assert_array_equal(host(state.count)[idx], orc.count, err_msg=f"round {r}: count after commit")
    R.replay_flush(state, A)
    orc.flush()
    check_pointers(state, orc, idx, "final flush")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0
    assert int(host(state.sync).sum()) == 0


@pytest.mark.parametrize("workspace", WORKSPACE)
@pytest.mark.parametrize("T", [1, 2, 3, 4, 6])
def test_spec_verify_fused_parity(T, workspace):
    """replay_spec_verify_fused == replay_flush + replay_spec_verify, over
    rounds whose early flushes empty windows whose slots the next drafts
    overwrite (c + T > L); two-launch (T <= 4 CUDA-core and T = 6 tensor-core
    streams) and one-launch verify."""
    shape = wl.Mamba2Shape(B=12, H=8, G=2, d=64, n=128, L=16, in_dtype=wl.BF16)
    run_spec_fused(shape, T, rounds=14, seed=140 + T, workspace=workspace)


def test_spec_verify_fused_small_shapes():
    # fp32 inputs with n = 32, ragged heads; T = L (every round flushes what it committed)
    run_spec_fused(wl.Mamba2Shape(B=4, H=6, G=3, d=20, n=32, L=8, in_dtype=wl.F32), 3, rounds=10, seed=141)
    run_spec_fused(wl.Mamba2Shape(B=5, H=8, G=2, d=64, n=128, L=4, in_dtype=wl.BF16), 4, rounds=8, seed=142)
    run_spec_fused(wl.Mamba2Shape(B=4, H=8, G=1, d=48, n=64, L=12, in_dtype=wl.BF16), 4, rounds=10, seed=143)


def test_spec_fused_full_batch_sampled():
    """The speculative workload at its own size: B = 512, T = 4, L = 16,
    accepted ~ U{0..4}, the pending flush, the verify and the commit, 24 rounds;
    ten sampled sequences against the oracle."""
    run_spec_fused(wl.SPEC_MAMBA2, 4, rounds=24, seed=wl.SEED_SPEC,
                   sample=[0, 1, 100, 255, 256, 311, 400, 480, 510, 511])


def test_fused_decode_output_feeds_next_step():
    """Each step's y (bf16) is the next step's v, passed as the same device
    buffer: the next step's precompute may start during the previous step's
    S_0 stream (programmatic dependent launch), so it must read its inputs
    only after that grid has finished.  Batch 128 (4096 streaming blocks, a
    tail the next precompute overlaps), 20 steps; the oracle gets the GPU's y
    as its next v."""
    R = rs()
    shape = wl.Mamba2Shape(B=128, H=32, G=8, d=64, n=128, L=8, in_dtype=wl.BF16)
    seed = 171
    init = wl.mamba2_init(shape, seed)
    idx = np.array([0, 1, 50, 64, 100, 127])
    state = m2_state(init)
    orc = oracle_replay(init, idx)
    A = dev(init.A)
    st0 = wl.mamba2_step(shape, seed, 0)
    bufs = [dev(st0.v, torch.bfloat16), torch.empty(shape.B, shape.H, shape.d, dtype=torch.bfloat16, device="cuda")]
    for t in range(20):
        st = wl.mamba2_step(shape, seed, t)
        _, k, q, dt = m2_step_dev(st, shape.in_dtype)
        v_in, y = bufs[t % 2], bufs[(t + 1) % 2]
        v_host = host(v_in.float())
        R.replay_decode_step_fused(state, v_in, k, q, dt, A, y=y)
        y_ref = orc.decode_step(take(v_host, idx), take(st.k, idx), take(st.q, idx), take(st.dt, idx))
        orc.flush()
        assert_close(y[idx], y_ref, 1e-2, 1e-3, what=f"step {t}: y")
    assert_close(state.S0[idx], orc.S0, what="final S0")
    assert int(host(state.err)[0]) == 0


def test_decode_runs_on_the_stream_passed():
    """stream= puts the call on that stream: while torch's current stream is
    still busy (a bounded sleep kernel), the output read back on the named
    stream is already the full result, equal to the same step on the current
    stream."""
    R = rs()
    shape = wl.Mamba2Shape(B=8, H=4, G=2, d=64, n=128, L=8, in_dtype=wl.BF16)
    seed = 23
    init = wl.mamba2_init(shape, seed)
    ref, out = m2_state(init), m2_state(init)
    A = dev(init.A)
    inp = m2_step_dev(wl.mamba2_step(shape, seed, 0), shape.in_dtype)
    y_ref = R.replay_decode_step_fused(ref, *inp, A)
    y = torch.full_like(y_ref, float("nan"))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    torch.cuda._sleep(400_000_000)  # keeps the current stream busy for about 0.2 s
    R.replay_decode_step_fused(out, *inp, A, y=y, stream=side)
    with torch.cuda.stream(side):
        y_side = y.cpu()  # a copy on `side`, which waits for `side` only
    busy = not torch.cuda.current_stream().query()
    torch.cuda.synchronize()
    assert busy, "the current stream finished before the read: the check says nothing"
    assert torch.equal(y_side, y_ref.cpu())
    for f in ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag"):
        assert torch.equal(getattr(out, f), getattr(ref, f)), f
