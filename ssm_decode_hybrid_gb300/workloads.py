"""Seeded synthetic inputs for the ReplaySSM decode path.

This module draws random inputs only. It holds none of the method's
arithmetic (no decays, no outer products, no reads of a state): the same
arrays feed the CUDA path and the CPU checker, so neither side can bend them.

Distributions follow the workload descriptions of "ReplaySSM: Cache SSM
Inputs, Not State" (experimental setup: fp32 SSM state, bf16 buffer vectors,
batch 256, window 4):

* Mamba-2: S_0 ~ N(0, 0.1^2); v, k, q ~ N(0, 1); Delta = softplus(N(0, 1));
  A = -exp(U(0, 1)) per head.  Delta arrives after the softplus, so the
  kernels see a positive step size and nothing else is applied to it.
* Gated DeltaNet: k, q are N(0, 1) vectors divided by their L2 norm; v ~ N(0, 1);
  beta = sigmoid(N(0, 1)); g = -softplus(N(0, 1)); S_0 ~ N(0, 0.1^2).
  Buffered corrections u of pre-filled entries are drawn as N(0, 0.5^2), the
  size a correction beta (v - alpha S k) has under these inputs.

Values are drawn in float32 and, where the workload stores them in bf16,
rounded to bf16 once here; the arrays returned are float32 numpy arrays whose
values are exactly representable in the stated dtype.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round a float32 array to `dtype` (round to nearest even), returned as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F32:
        return x
    if dtype == BF16:
        return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    raise ValueError(dtype)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    nrm = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / nrm).astype(np.float32)


# --------------------------------------------------------------------------
# Mamba-2
# --------------------------------------------------------------------------


@dataclasses.dataclass
class Mamba2Shape:
    B: int
    H: int
    G: int
    d: int
    n: int
    L: int
    in_dtype: str = BF16


@dataclasses.dataclass
class Mamba2Init:
    """Checkpoint, per-head decay parameter and a pre-filled ring buffer."""

    shape: Mamba2Shape
    S0: np.ndarray  # [B,H,d,n] f32
    A: np.ndarray  # [H] f32, negative
    ring_v: np.ndarray  # [B,H,L,d] (values in in_dtype)
    ring_k: np.ndarray  # [B,G,L,n]
    ring_dt: np.ndarray  # [B,H,L] f32
    start: np.ndarray  # [B] int32, slot of the oldest committed entry
    count: np.ndarray  # [B] int32, committed entries


def mamba2_init(shape: Mamba2Shape, seed: int, fill_max: int | None = None,
                random_start: bool = True) -> Mamba2Init:
    """Draw S_0, A and a ring buffer holding U{0..fill_max} committed entries.

    fill_max defaults to L-1 (a buffer is never full between steps). Slots
    outside the committed window hold random values too, so that a kernel that
    reads past `count` produces a visible mismatch.
    """
    s = shape
    rng = np.random.default_rng([seed, 0])
    S0 = (0.1 * rng.standard_normal((s.B, s.H, s.d, s.n))).astype(np.float32)
    A = (-np.exp(rng.uniform(0.0, 1.0, size=s.H))).astype(np.float32)
    ring_v = round_to(rng.standard_normal((s.B, s.H, s.L, s.d)).astype(np.float32), s.in_dtype)
    ring_k = round_to(rng.standard_normal((s.B, s.G, s.L, s.n)).astype(np.float32), s.in_dtype)
    ring_dt = _softplus(rng.standard_normal((s.B, s.H, s.L)).astype(np.float32))
    fm = s.L - 1 if fill_max is None else fill_max
    count = rng.integers(0, fm + 1, size=s.B).astype(np.int32)
    if random_start:
        start = rng.integers(0, s.L, size=s.B).astype(np.int32)
    else:
        start = np.zeros(s.B, dtype=np.int32)
    return Mamba2Init(s, S0, A, ring_v, ring_k, ring_dt, start, count)


@dataclasses.dataclass
class Mamba2Step:
    """Inputs of one decode step (T=None) or one T-token verify round."""

    v: np.ndarray  # [B,H,d] or [B,T,H,d]
    k: np.ndarray  # [B,G,n] or [B,T,G,n]
    q: np.ndarray  # [B,G,n] or [B,T,G,n]
    dt: np.ndarray  # [B,H] or [B,T,H]


def mamba2_step(shape: Mamba2Shape, seed: int, step: int, T: int | None = None) -> Mamba2Step:
    s = shape
    rng = np.random.default_rng([seed, 1, step])
    lead = (s.B,) if T is None else (s.B, T)
    v = round_to(rng.standard_normal(lead + (s.H, s.d)).astype(np.float32), s.in_dtype)
    k = round_to(rng.standard_normal(lead + (s.G, s.n)).astype(np.float32), s.in_dtype)
    q = round_to(rng.standard_normal(lead + (s.G, s.n)).astype(np.float32), s.in_dtype)
    dt = _softplus(rng.standard_normal(lead + (s.H,)).astype(np.float32))
    return Mamba2Step(v, k, q, dt)


def accepted_counts(B: int, T: int, seed: int, rnd: int) -> np.ndarray:
    """Accepted draft count per sequence for one verify round, U{0..T}."""
    rng = np.random.default_rng([seed, 2, rnd])
    return rng.integers(0, T + 1, size=B).astype(np.int32)


# --------------------------------------------------------------------------
# Gated DeltaNet
# --------------------------------------------------------------------------


@dataclasses.dataclass
class GdnShape:
    B: int
    Hv: int  # value heads
    Hk: int  # key heads (k, q shared by Hv // Hk value heads)
    dk: int
    dv: int
    L: int
    in_dtype: str = BF16
    u_dtype: str = F32


@dataclasses.dataclass
class GdnInit:
    shape: GdnShape
    S0: np.ndarray  # [B,Hv,dv,dk] f32
    ring_u: np.ndarray  # [B,Hv,L,dv] (values in u_dtype)
    ring_k: np.ndarray  # [B,Hk,L,dk] (values in in_dtype, unit rows)
    ring_g: np.ndarray  # [B,Hv,L] f32, log decays (negative)
    start: np.ndarray  # [B] int32
    count: np.ndarray  # [B] int32


def gdn_init(shape: GdnShape, seed: int, fill_max: int | None = None,
             random_start: bool = True) -> GdnInit:
    s = shape
    rng = np.random.default_rng([seed, 10])
    S0 = (0.1 * rng.standard_normal((s.B, s.Hv, s.dv, s.dk))).astype(np.float32)
    ring_u = round_to((0.5 * rng.standard_normal((s.B, s.Hv, s.L, s.dv))).astype(np.float32), s.u_dtype)
    ring_k = round_to(_unit_rows(rng.standard_normal((s.B, s.Hk, s.L, s.dk)).astype(np.float32)), s.in_dtype)
    ring_g = (-_softplus(rng.standard_normal((s.B, s.Hv, s.L)).astype(np.float32))).astype(np.float32)
    fm = s.L - 1 if fill_max is None else fill_max
    count = rng.integers(0, fm + 1, size=s.B).astype(np.int32)
    if random_start:
        start = rng.integers(0, s.L, size=s.B).astype(np.int32)
    else:
        start = np.zeros(s.B, dtype=np.int32)
    return GdnInit(s, S0, ring_u, ring_k, ring_g, start, count)


@dataclasses.dataclass
class GdnStep:
    q: np.ndarray  # [B,Hk,dk] or [B,T,Hk,dk]
    k: np.ndarray  # [B,Hk,dk] or [B,T,Hk,dk]
    v: np.ndarray  # [B,Hv,dv] or [B,T,Hv,dv]
    beta: np.ndarray  # [B,Hv] or [B,T,Hv]
    g: np.ndarray  # [B,Hv] or [B,T,Hv]


def gdn_step(shape: GdnShape, seed: int, step: int, T: int | None = None) -> GdnStep:
    s = shape
    rng = np.random.default_rng([seed, 11, step])
    lead = (s.B,) if T is None else (s.B, T)
    q = round_to(_unit_rows(rng.standard_normal(lead + (s.Hk, s.dk)).astype(np.float32)), s.in_dtype)
    k = round_to(_unit_rows(rng.standard_normal(lead + (s.Hk, s.dk)).astype(np.float32)), s.in_dtype)
    v = round_to(rng.standard_normal(lead + (s.Hv, s.dv)).astype(np.float32), s.in_dtype)
    beta = _sigmoid(rng.standard_normal(lead + (s.Hv,)).astype(np.float32))
    g = (-_softplus(rng.standard_normal(lead + (s.Hv,)).astype(np.float32))).astype(np.float32)
    return GdnStep(q, k, v, beta, g)


# --------------------------------------------------------------------------
# Named workloads (sizes of the pages' experiments)
# --------------------------------------------------------------------------

TINY_MAMBA2 = Mamba2Shape(B=1, H=4, G=1, d=16, n=16, L=4, in_dtype=F32)
NEMOTRON_H_MAMBA2 = Mamba2Shape(B=256, H=32, G=8, d=64, n=128, L=16, in_dtype=BF16)
SPEC_MAMBA2 = Mamba2Shape(B=512, H=32, G=8, d=64, n=128, L=16, in_dtype=BF16)
GDN_LAYER = GdnShape(B=256, Hv=32, Hk=16, dk=128, dv=128, L=16, in_dtype=BF16, u_dtype=F32)

SEED_TINY = 1000
SEED_NEMOTRON = 1001
SEED_SWEEP = 1002
SEED_SPEC = 1003
SEED_GDN = 1004


# ---------------------------------------------------------------------------
# device-side generators for timing-only workloads (no oracle comparison)
# ---------------------------------------------------------------------------


def mamba2_state_tensors_device(shape: Mamba2Shape, seed: int, device, fill_max: int | None = None):
    """S_0, ring buffer and pointers of one Mamba-2 layer drawn directly on the
    device with a seeded torch generator, from the same distributions as
    mamba2_init (for sizes where host generation would dominate).  Returns a
    dict of tensors keyed like Mamba2Init's fields."""
    import torch

    s = shape
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if s.in_dtype == BF16 else torch.float32
    fm = s.L - 1 if fill_max is None else fill_max

    def normal(*size):
        return torch.randn(*size, generator=g, device=device, dtype=torch.float32)

    return {
        "S0": 0.1 * normal(s.B, s.H, s.d, s.n),
        "A": -torch.exp(torch.rand(s.H, generator=g, device=device)),
        "ring_v": normal(s.B, s.H, s.L, s.d).to(dt),
        "ring_k": normal(s.B, s.G, s.L, s.n).to(dt),
        "ring_dt": torch.nn.functional.softplus(normal(s.B, s.H, s.L)),
        "start": torch.randint(0, s.L, (s.B,), generator=g, device=device, dtype=torch.int32),
        "count": torch.randint(0, fm + 1, (s.B,), generator=g, device=device, dtype=torch.int32),
    }


def gdn_state_tensors_device(shape: GdnShape, seed: int, device, fill_max: int | None = None):
    """S_0, ring buffer and pointers of one GDN layer drawn on the device, from
    the same distributions as gdn_init.  Returns a dict keyed like GdnInit."""
    import torch

    s = shape
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if s.in_dtype == BF16 else torch.float32
    ut = torch.bfloat16 if s.u_dtype == BF16 else torch.float32
    fm = s.L - 1 if fill_max is None else fill_max

    def normal(*size):
        return torch.randn(*size, generator=g, device=device, dtype=torch.float32)

    k = normal(s.B, s.Hk, s.L, s.dk)
    return {
        "S0": 0.1 * normal(s.B, s.Hv, s.dv, s.dk),
        "ring_u": (0.5 * normal(s.B, s.Hv, s.L, s.dv)).to(ut),
        "ring_k": (k / k.norm(dim=-1, keepdim=True)).to(dt),
        "ring_g": -torch.nn.functional.softplus(normal(s.B, s.Hv, s.L)),
        "start": torch.randint(0, s.L, (s.B,), generator=g, device=device, dtype=torch.int32),
        "count": torch.randint(0, fm + 1, (s.B,), generator=g, device=device, dtype=torch.int32),
    }


def mamba2_round_device(shape: Mamba2Shape, seed: int, T: int, device):
    """Inputs (v, k, q, dt) of one T-draft verify round drawn on the device,
    distributed as mamba2_step's."""
    import torch

    s = shape
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if s.in_dtype == BF16 else torch.float32

    def normal(*size):
        return torch.randn(*size, generator=g, device=device, dtype=torch.float32)

    return (normal(s.B, T, s.H, s.d).to(dt), normal(s.B, T, s.G, s.n).to(dt), normal(s.B, T, s.G, s.n).to(dt),
            torch.nn.functional.softplus(normal(s.B, T, s.H)))


def gdn_round_device(shape: GdnShape, seed: int, T: int, device):
    """Inputs (q, k, v, beta, g) of one T-draft GDN verify round drawn on the
    device, distributed as gdn_step's."""
    import torch

    s = shape
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = torch.bfloat16 if s.in_dtype == BF16 else torch.float32

    def normal(*size):
        return torch.randn(*size, generator=gen, device=device, dtype=torch.float32)

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)

    return (unit(normal(s.B, T, s.Hk, s.dk)).to(dt), unit(normal(s.B, T, s.Hk, s.dk)).to(dt),
            normal(s.B, T, s.Hv, s.dv).to(dt), torch.sigmoid(normal(s.B, T, s.Hv)),
            -torch.nn.functional.softplus(normal(s.B, T, s.Hv)))


def accepted_counts_device(B: int, T: int, seed: int, device):
    """Accepted draft counts U{0..T} for one round, drawn on the device."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, T + 1, (B,), generator=g, device=device, dtype=torch.int32)


@dataclasses.dataclass
class ConvShape:
    """Convolution state of a Mamba-2 layer: conv_dim = dx + 2 dbc channels,
    width W (the state keeps W - 1 columns)."""

    B: int
    dx: int
    dbc: int
    W: int = 4
    io_dtype: str = BF16


@dataclasses.dataclass
class ConvInit:
    shape: ConvShape
    state: np.ndarray  # [B, C, W-1] (values in io_dtype)
    weight: np.ndarray  # [C, W] f32
    bias: np.ndarray  # [C] f32


def conv_init(shape: ConvShape, seed: int) -> ConvInit:
    """State ~ N(0, 1) in io_dtype, weight ~ N(0, 0.5^2), bias ~ N(0, 0.1^2)."""
    s = shape
    C = s.dx + 2 * s.dbc
    rng = np.random.default_rng([seed, 20])
    state = round_to(rng.standard_normal((s.B, C, s.W - 1)).astype(np.float32), s.io_dtype)
    weight = (0.5 * rng.standard_normal((C, s.W))).astype(np.float32)
    bias = (0.1 * rng.standard_normal(C)).astype(np.float32)
    return ConvInit(s, state, weight, bias)


def conv_input(shape: ConvShape, seed: int, step: int) -> np.ndarray:
    """The in-projection's x|B|C column of one decode step, N(0, 1) in io_dtype."""
    rng = np.random.default_rng([seed, 21, step])
    return round_to(rng.standard_normal((shape.B, shape.dx + 2 * shape.dbc)).astype(np.float32), shape.io_dtype)
