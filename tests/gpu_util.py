"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
build library state from them, and compare against the oracle.

Tolerance (fp32 state and accumulation): |gpu - ref| <= max(1e-3 |ref|, 1e-4)
element by element; bf16 outputs: max(1e-2 |ref|, 1e-2 * 1e-2 ...) see
``tol_for``.  Integer bookkeeping is compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

from ssm_decode_hybrid_gb300 import workloads as wl

TORCH_DT = {wl.F32: torch.float32, wl.BF16: torch.bfloat16}

RTOL_F32, ATOL_F32 = 1e-3, 1e-4
RTOL_BF16, ATOL_BF16 = 1e-2, 1e-3


def tol_for(y_dtype):
    return (RTOL_BF16, ATOL_BF16) if y_dtype == torch.bfloat16 else (RTOL_F32, ATOL_F32)


def dev(x, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64) if t.is_floating_point() else t.cpu().numpy()


def assert_close(gpu, ref, rtol=RTOL_F32, atol=ATOL_F32, what=""):
    g = host(gpu) if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, f"{what}: shape {g.shape} vs {r.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    bound = np.maximum(rtol * np.abs(r), atol)
    bad = np.abs(g - r) > bound
    if np.any(bad):
        idx = np.argwhere(bad)[0]
        diag = np.max(np.abs(g - r) / np.maximum(np.abs(r), atol))
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements off, first at {tuple(idx)}: "
                             f"gpu={g[tuple(idx)]!r} ref={r[tuple(idx)]!r}; max scaled err {diag:.3e}")


def m2_state(init: wl.Mamba2Init, workspace: bool = True):
    """Device state from a seeded init; workspace=True attaches the decode
    workspace (two-launch decode), False leaves it out (single-launch decode)."""
    from ssm_decode_hybrid_gb300 import replayssm as rs

    s = init.shape
    t = TORCH_DT[s.in_dtype]
    B = s.B
    st = rs.Mamba2State(
        S0=dev(init.S0), ring_v=dev(init.ring_v, t), ring_k=dev(init.ring_k, t), ring_dt=dev(init.ring_dt),
        start=dev(init.start, torch.int32), count=dev(init.count, torch.int32),
        flag=torch.zeros(B, dtype=torch.int32, device="cuda"), sync=torch.zeros(B, dtype=torch.int32, device="cuda"),
        err=torch.zeros(1, dtype=torch.int32, device="cuda"))
    if workspace:
        st.add_workspace(max_T=8)
        st.work.fill_(float("nan"))  # scratch: nothing may depend on its prior contents
    return st


def m2_step_dev(step: wl.Mamba2Step, in_dtype: str):
    t = TORCH_DT[in_dtype]
    return dev(step.v, t), dev(step.k, t), dev(step.q, t), dev(step.dt)


def gdn_state(init: wl.GdnInit, workspace_T: int = 8):
    """Device state from a seeded init; workspace_T > 0 attaches a workspace for
    calls of up to that many drafts (two-launch kernels), 0 leaves it out."""
    from ssm_decode_hybrid_gb300 import replayssm as rs

    s = init.shape
    B = s.B
    st = rs.GdnState(
        S0=dev(init.S0), ring_u=dev(init.ring_u, TORCH_DT[s.u_dtype]), ring_k=dev(init.ring_k, TORCH_DT[s.in_dtype]),
        ring_g=dev(init.ring_g), start=dev(init.start, torch.int32), count=dev(init.count, torch.int32),
        flag=torch.zeros(B, dtype=torch.int32, device="cuda"), sync=torch.zeros(B, dtype=torch.int32, device="cuda"),
        err=torch.zeros(1, dtype=torch.int32, device="cuda"))
    if workspace_T:
        st.add_workspace(workspace_T)
        st.work.fill_(float("nan"))  # scratch: nothing may depend on its prior contents
    return st


def gdn_step_dev(step: wl.GdnStep, in_dtype: str):
    t = TORCH_DT[in_dtype]
    return dev(step.q, t), dev(step.k, t), dev(step.v, t), dev(step.beta), dev(step.g)


def take(x, idx):
    """Rows `idx` of the leading (batch) axis."""
    return np.ascontiguousarray(np.asarray(x)[idx])
