"""replay_decode_step_fused_noalloc: the fused decode step with the library's
own file-scope workspace gives the same outputs and state, bit for bit, as
replay_decode_step_fused with a caller workspace, over consecutive calls."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_util import dev, host, m2_state, m2_step_dev
from ssm_decode_hybrid_gb300 import workloads as wl

STATIC_WORK_FLOATS = 1 << 21


def _lib():
    from test_abi import _lib_path

    _lib_path()
    from ssm_decode_hybrid_gb300 import replayssm as R

    return R


@pytest.mark.skipif(torch.cuda.is_available(), reason="uses fake device pointers; CPU only")
def test_noalloc_rejects_shapes_beyond_its_workspace():
    R = _lib()
    fake = ctypes.c_void_p(0x10000)
    rep = R.M2Replay(*([fake] * 9))
    args = [fake] * 6 + [None]
    # 1024 x 32 heads x 84 floats > 2^21 floats: unsupported, refused before any CUDA call
    big = R.M2Dims(1024, 32, 8, 64, 128, 16, R.BF16, R.F32)
    assert big.B * big.H * 84 > STATIC_WORK_FLOATS
    assert R.LIB.replay_decode_step_fused_noalloc(ctypes.byref(big), ctypes.byref(rep), *args) == -2
    assert R.LIB.replay_decode_step_fused_noalloc(None, ctypes.byref(rep), *args) == -1


# records of 64 floats (d = 48, L = 12): 1024 x 32 heads fill the array exactly
LIMIT_SHAPE = wl.Mamba2Shape(B=1024, H=32, G=8, d=48, n=32, L=12, in_dtype=wl.BF16)
SHAPES = [
    wl.NEMOTRON_H_MAMBA2,  # batch 256: two-launch kernels
    LIMIT_SHAPE,  # B * H * record floats == the array's size
    wl.Mamba2Shape(B=4, H=6, G=3, d=20, n=32, L=3, in_dtype=wl.BF16),  # outside the two-launch kernels
]


def poison_static_workspace():
    """Fill the library's array with NaN-valued records: one call on the
    largest shape it holds, with NaN step sizes (every weight, abar and
    buffer term of every record becomes NaN), on a throwaway state.  A later
    call that read a slot it had not written would then produce NaN or a
    mismatch."""
    from ssm_decode_hybrid_gb300 import replayssm as R

    shape = LIMIT_SHAPE
    init = wl.mamba2_init(shape, 99)
    junk = m2_state(init, workspace=False)
    st = wl.mamba2_step(shape, 99, 0)
    v, k, q, dt = m2_step_dev(st, shape.in_dtype)
    dt.fill_(float("nan"))
    R.replay_decode_step_fused_noalloc(junk, v, k, q, dt, dev(init.A))
    torch.cuda.synchronize()
    del junk


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s.B}H{s.H}d{s.d}n{s.n}L{s.L}")
def test_noalloc_matches_fused_on_consecutive_calls(shape):
    from ssm_decode_hybrid_gb300 import replayssm as R

    assert shape.B * shape.H * ((4 + shape.L + shape.d + 3) & ~3) <= STATIC_WORK_FLOATS
    poison_static_workspace()
    seed = 4242
    init = wl.mamba2_init(shape, seed)
    ref = m2_state(init, workspace=True)
    out = m2_state(init, workspace=False)
    A = dev(init.A)
    for t in range(2):
        inp = m2_step_dev(wl.mamba2_step(shape, seed, t), shape.in_dtype)
        y_ref = R.replay_decode_step_fused(ref, *inp, A)
        y = R.replay_decode_step_fused_noalloc(out, *inp, A)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"call {t}: y differs"
        for f in ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag", "sync"):
            assert torch.equal(getattr(out, f), getattr(ref, f)), f"call {t}: {f} differs"
    assert out.work is None
    assert int(host(out.err)[0]) == 0 and int(host(ref.err)[0]) == 0
    assert np.all(host(out.count) < shape.L)


@pytest.mark.gpu
def test_noalloc_refuses_one_sequence_past_its_limit():
    """One sequence more than the array holds: RSSM_ERR_UNSUPPORTED, and
    nothing is launched (state and error word untouched)."""
    from ssm_decode_hybrid_gb300 import replayssm as R

    s = LIMIT_SHAPE
    assert s.B * s.H * ((4 + s.L + s.d + 3) & ~3) == STATIC_WORK_FLOATS
    over = wl.Mamba2Shape(B=s.B + 1, H=s.H, G=s.G, d=s.d, n=s.n, L=s.L, in_dtype=s.in_dtype)
    init = wl.mamba2_init(over, 7)
    out = m2_state(init, workspace=False)
    before = {f: getattr(out, f).clone() for f in ("S0", "ring_v", "start", "count", "flag")}
    y = torch.full((over.B, over.H, over.d), 7.0, device="cuda")
    with pytest.raises(R.ReplaySSMError, match=r"\(-2\)"):
        R.replay_decode_step_fused_noalloc(out, *m2_step_dev(wl.mamba2_step(over, 7, 0), over.in_dtype),
                                           dev(init.A), y=y)
    torch.cuda.synchronize()
    for f, v in before.items():
        assert torch.equal(getattr(out, f), v), f"{f} changed by a refused call"
    assert bool((y == 7.0).all())
    assert int(host(out.err)[0]) == 0
