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


SHAPES = [
    wl.NEMOTRON_H_MAMBA2,  # batch 256: two-launch kernels
    wl.Mamba2Shape(B=4, H=6, G=3, d=20, n=32, L=3, in_dtype=wl.BF16),  # outside the two-launch kernels
]


@pytest.mark.gpu
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"B{s.B}H{s.H}d{s.d}n{s.n}L{s.L}")
def test_noalloc_matches_fused_on_consecutive_calls(shape):
    from ssm_decode_hybrid_gb300 import replayssm as R

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
