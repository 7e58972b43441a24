"""Per-sequence device bytes ("Results -- speculative decoding", maximum
concurrency at a fixed HBM budget, Fig. 11): the library's figures equal the
bytes of the tensors a state actually consists of, built here on the CPU from
their shapes (host-only calls; no kernel runs)."""
import pytest
import torch

from tests.test_abi import _lib_path


def _R():
    _lib_path()
    from ssm_decode_hybrid_gb300 import replayssm as R

    return R


def _nbytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts)


@pytest.mark.parametrize("T", [0, 1, 2, 4, 6, 8])
@pytest.mark.parametrize("shape", [(256, 32, 8, 64, 128, 16), (3, 4, 2, 16, 32, 4), (5, 8, 8, 128, 64, 32)])
def test_mamba2_seq_bytes_match_allocated_tensors(shape, T):
    R = _R()
    B, H, G, d, n, L = shape
    st = R.Mamba2State.empty(B, H, G, d, n, L, device="cpu", workspace=False).add_workspace(max_T=T)
    replay = _nbytes(st.S0, st.ring_v, st.ring_k, st.ring_dt, st.start, st.count, st.flag, st.sync, st.work)
    assert replay % B == 0
    assert R.seq_bytes(st.dims(), T, R.SEQ_REPLAY) == replay // B
    slots = torch.empty(B, T + 1, H, d, n) if T else torch.empty(B, H, d, n)
    cur = torch.empty(B, dtype=torch.int32)
    snap = _nbytes(slots, cur) if T else _nbytes(slots)
    assert R.seq_bytes(st.dims(), T, R.SEQ_SNAPSHOT) == snap // B


@pytest.mark.parametrize("T", [0, 1, 4, 6])
@pytest.mark.parametrize("u_dtype", [torch.float32, torch.bfloat16])
def test_gdn_seq_bytes_match_allocated_tensors(T, u_dtype):
    R = _R()
    B, Hv, Hk, dk, dv, L = 7, 32, 16, 128, 128, 16
    st = R.GdnState.empty(B, Hv, Hk, dk, dv, L, u_dtype=u_dtype, device="cpu", workspace_T=max(T, 1))
    replay = _nbytes(st.S0, st.ring_u, st.ring_k, st.ring_g, st.start, st.count, st.flag, st.sync, st.work)
    assert R.seq_bytes(st.dims(), T, R.SEQ_REPLAY) == replay // B
    snap = (T + 1) * 4 * Hv * dv * dk + 4 if T else 4 * Hv * dv * dk
    assert R.seq_bytes(st.dims(), T, R.SEQ_SNAPSHOT) == snap


def test_concurrency_ratio_grows_with_the_window():
    """The snapshot baseline holds T + 1 states per sequence, replay one
    checkpoint plus small input vectors, so the ratio of the batches that fit
    a budget grows with T and stays below T + 1."""
    R = _R()
    dims = R.M2Dims(256, 32, 8, 64, 128, 16, R.BF16, R.F32)
    budget = 184 * 2**30
    prev = 0.0
    for T in range(1, 7):
        rep = R.max_sequences(budget, dims, T, R.SEQ_REPLAY, layers=23)
        snap = R.max_sequences(budget, dims, T, R.SEQ_SNAPSHOT, layers=23)
        ratio = rep / snap
        assert prev < ratio < T + 1
        prev = ratio
    # one layer: the checkpoint is 1 MiB, the ring and workspace about 10% more
    rep_bytes = R.seq_bytes(dims, 4, R.SEQ_REPLAY)
    assert 2**20 < rep_bytes < 1.2 * 2**20


def test_invalid_arguments_give_zero():
    R = _R()
    dims = R.M2Dims(2, 4, 2, 64, 128, 16, R.BF16, R.F32)
    import ctypes

    assert R.LIB.replay_seq_bytes(ctypes.byref(dims), 9, 0) == 0
    assert R.LIB.replay_seq_bytes(ctypes.byref(dims), -1, 0) == 0
    assert R.LIB.replay_seq_bytes(ctypes.byref(dims), 4, 2) == 0
    bad = R.M2Dims(2, 3, 2, 64, 128, 16, R.BF16, R.F32)
    assert R.LIB.replay_seq_bytes(ctypes.byref(bad), 4, 0) == 0
    assert R.LIB.replay_seq_bytes(None, 4, 0) == 0


def test_layout_sizes_match_allocated_tensors():
    R = _R()
    st = R.Mamba2State.empty(5, 8, 2, 48, 64, 12, device="cpu", workspace=False)
    lay = R.layout_sizes(st.dims())
    assert (lay.S0, lay.ring_vec, lay.ring_k, lay.ring_decay, lay.per_seq) == (
        st.S0.numel(), st.ring_v.numel(), st.ring_k.numel(), st.ring_dt.numel(), st.start.numel())
    gst = R.GdnState.empty(3, 8, 4, 128, 64, 16, device="cpu", workspace_T=0)
    lay = R.layout_sizes(gst.dims())
    assert (lay.S0, lay.ring_vec, lay.ring_k, lay.ring_decay, lay.per_seq) == (
        gst.S0.numel(), gst.ring_u.numel(), gst.ring_k.numel(), gst.ring_g.numel(), gst.count.numel())
    import ctypes

    bad = R.M2Dims(2, 3, 2, 64, 128, 16, R.BF16, R.F32)
    assert R.LIB.rssm_m2_layout_sizes(ctypes.byref(bad), ctypes.byref(R.Layout())) == -1
    assert R.LIB.rssm_m2_layout_sizes(ctypes.byref(st.dims()), None) == -1
    assert R.LIB.rssm_read_error(None, None, None) == -1
