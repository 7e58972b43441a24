"""GPU parity of the convolution-state decode step (conv_state_update) against
the fp64 oracle (oracle/conv.py), through the C ABI.

State updates are copies and compared bit for bit; outputs within
|gpu - ref| <= max(1e-3 |ref|, 1e-4) for fp32 and max(1e-2 |ref|, 1e-3) for
bf16 outputs (the oracle's exact value against the kernel's rounded one).
"""
import numpy as np
import pytest
import torch

from gpu_util import TORCH_DT, assert_close, dev, host, m2_state, tol_for
from oracle import conv as oc
from oracle import mamba2 as om
from ssm_decode_hybrid_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def rs():
    from ssm_decode_hybrid_gb300 import replayssm

    return replayssm


def run(shape, steps, seed, silu=True, bias=True, sample=None):
    R = rs()
    init = wl.conv_init(shape, seed)
    t = TORCH_DT[shape.io_dtype]
    state = dev(init.state, t)
    weight, b = dev(init.weight), (dev(init.bias) if bias else None)
    idx = np.arange(shape.B) if sample is None else np.asarray(sample)
    ref_state = init.state[idx].astype(np.float64)
    rtol, atol = tol_for(t)
    for step in range(steps):
        u = wl.conv_input(shape, seed, step)
        x, bo, co = R.conv_state_update(state, dev(u, t), weight, b, shape.dx, shape.dbc, silu=silu)
        ref_state, out = oc.conv_state_step(ref_state, u[idx], init.weight, init.bias if bias else None, silu)
        rx, rb, rc = oc.split_xbc(out, shape.dx, shape.dbc)
        assert_close(x[idx], rx, rtol, atol, what=f"step {step}: x")
        if shape.dbc:
            assert_close(bo[idx], rb, rtol, atol, what=f"step {step}: B")
            assert_close(co[idx], rc, rtol, atol, what=f"step {step}: C")
        np.testing.assert_array_equal(host(state)[idx], ref_state, err_msg=f"step {step}: state")


@pytest.mark.parametrize("shape", [
    wl.ConvShape(B=3, dx=40, dbc=12, W=4, io_dtype=wl.BF16),
    wl.ConvShape(B=2, dx=37, dbc=5, W=3, io_dtype=wl.F32),
    wl.ConvShape(B=4, dx=64, dbc=0, W=2, io_dtype=wl.BF16),
    wl.ConvShape(B=1, dx=9, dbc=3, W=8, io_dtype=wl.F32),
], ids=lambda s: f"B{s.B}x{s.dx}+2x{s.dbc}W{s.W}{s.io_dtype}")
def test_conv_step_parity(shape):
    run(shape, steps=6, seed=900 + shape.W)


def test_conv_step_without_activation_or_bias():
    run(wl.ConvShape(B=3, dx=24, dbc=8, W=4, io_dtype=wl.F32), steps=4, seed=910, silu=False, bias=False)


def test_conv_step_nemotron_layer_sampled():
    """The Nemotron-H layer's convolution (x 32 x 64, B and C 8 x 128, W = 4)
    at batch 256: sampled sequences."""
    run(wl.ConvShape(B=256, dx=2048, dbc=1024, W=4, io_dtype=wl.BF16), steps=3, seed=920, sample=[0, 77, 255])


def test_conv_feeds_the_decode_step():
    """The step's x, B, C are the decode step's v, k, q: convolution then
    replay_decode_step equals the two oracles composed."""
    R = rs()
    ms = wl.Mamba2Shape(B=4, H=8, G=2, d=16, n=32, L=8, in_dtype=wl.BF16)
    cs = wl.ConvShape(B=ms.B, dx=ms.H * ms.d, dbc=ms.G * ms.n, W=4, io_dtype=wl.BF16)
    cinit, minit = wl.conv_init(cs, 930), wl.mamba2_init(ms, 930)
    state, weight, bias = dev(cinit.state, torch.bfloat16), dev(cinit.weight), dev(cinit.bias)
    st = m2_state(minit)
    A = dev(minit.A)
    orc = om.Mamba2Replay(minit.S0, minit.A, minit.ring_v, minit.ring_k, minit.ring_dt, minit.start, minit.count)
    ref_state = cinit.state.astype(np.float64)
    rng = np.random.default_rng(931)
    for step in range(5):
        u = wl.conv_input(cs, 930, step)
        dt = np.log1p(np.exp(rng.standard_normal((ms.B, ms.H)))).astype(np.float32)
        x, bo, co = R.conv_state_update(state, dev(u, torch.bfloat16), weight, bias, cs.dx, cs.dbc)
        y = R.replay_decode_step_fused(st, x.view(ms.B, ms.H, ms.d), bo.view(ms.B, ms.G, ms.n),
                                       co.view(ms.B, ms.G, ms.n), dev(dt), A)
        ref_state, out = oc.conv_state_step(ref_state, u, cinit.weight, cinit.bias)
        rx, rb, rc = oc.split_xbc(out, cs.dx, cs.dbc)
        # the decode step consumes the kernel's bf16-rounded x, B, C, as a model would
        v_in, k_in, q_in = (host(t) for t in (x, bo, co))
        np.testing.assert_allclose(v_in, rx, rtol=1e-2, atol=1e-3)
        y_ref = orc.decode_step(v_in.reshape(ms.B, ms.H, ms.d), k_in.reshape(ms.B, ms.G, ms.n),
                                q_in.reshape(ms.B, ms.G, ms.n), dt)
        if orc.flag.any():
            orc.flush()
        assert_close(y, y_ref, what=f"step {step}: y")
