"""Python binding of libreplayssm (ctypes).  Argument marshalling only: every
step of the decode path runs in the library's CUDA kernels.

Tensors must be CUDA tensors on the current device, contiguous, in the
layouts documented in ``include/replayssm.h``.  Calls are asynchronous on
torch's current stream, or on the ``torch.cuda.Stream`` passed as ``stream=``.
A missing library raises at import time; a non-zero status raises
``ReplaySSMError``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# REPLAYSSM_LIB points the binding at another build of the same library.
LIB_PATH = os.environ.get("REPLAYSSM_LIB") or os.path.join(_HERE, "libreplayssm.so")

F32, BF16 = 0, 1
SEQ_REPLAY, SEQ_SNAPSHOT = 0, 1
EBIT_COUNT_RANGE, EBIT_WINDOW, EBIT_ACCEPTED, EBIT_CUR, EBIT_TIMEOUT = 1, 2, 4, 8, 16
_DT = {torch.float32: F32, torch.bfloat16: BF16}


class ReplaySSMError(RuntimeError):
    pass


class M2Dims(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in ("B", "H", "G", "d", "n", "L", "in_dtype", "y_dtype")]


class M2Replay(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in
                ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag", "sync", "err", "work")] + \
               [("work_bytes", ctypes.c_int64)]


class GdnDims(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in ("B", "Hv", "Hk", "dk", "dv", "L", "in_dtype", "u_dtype", "y_dtype")]


class Layout(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int64) for f in ("S0", "ring_vec", "ring_k", "ring_decay", "per_seq")]


class ConvDims(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in ("B", "dx", "dbc", "W", "io_dtype", "silu")]


class GdnReplay(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in
                ("S0", "ring_u", "ring_k", "ring_g", "start", "count", "flag", "sync", "err", "work")] + \
               [("work_bytes", ctypes.c_int64)]


EXPORTS = (
    "ssm_state_update_baseline", "replay_decode_step", "replay_decode_step_fused", "replay_flush",
    "replay_spec_verify",
    "replay_spec_verify_fused", "replay_spec_commit", "ssm_spec_verify_baseline", "ssm_spec_commit_baseline",
    "gdn_state_update_baseline", "gdn_replay_decode", "gdn_replay_flush", "gdn_replay_verify",
    "gdn_replay_verify_fused",
    "gdn_spec_verify_baseline", "rssm_version", "rssm_status_string", "rssm_last_cuda_error",
    "replay_decode_workspace_bytes", "replay_decode_step_fused_noalloc",
    "gdn_replay_decode_fused", "gdn_replay_workspace_bytes", "replay_verify_workspace_bytes",
    "replay_seq_bytes", "gdn_replay_seq_bytes", "conv_state_update",
    "rssm_m2_layout_sizes", "rssm_gdn_layout_sizes", "rssm_read_error",
)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m ssm_decode_hybrid_gb300.build` "
                          "(the ReplaySSM path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int32
    sig = {
        "ssm_state_update_baseline": [ctypes.POINTER(M2Dims), P, P, P, P, P, P, P, P],
        "replay_decode_step": [ctypes.POINTER(M2Dims), ctypes.POINTER(M2Replay), P, P, P, P, P, P, P],
        "replay_decode_step_fused": [ctypes.POINTER(M2Dims), ctypes.POINTER(M2Replay), P, P, P, P, P, P, P],
        "replay_decode_step_fused_noalloc": [ctypes.POINTER(M2Dims), ctypes.POINTER(M2Replay), P, P, P, P, P, P, P],
        "replay_flush": [ctypes.POINTER(M2Dims), ctypes.POINTER(M2Replay), P, P],
        "replay_spec_verify": [ctypes.POINTER(M2Dims), ctypes.POINTER(M2Replay), I, P, P, P, P, P, P, P],
        "replay_spec_verify_fused": [ctypes.POINTER(M2Dims), ctypes.POINTER(M2Replay), I, P, P, P, P, P, P, P],
        "replay_spec_commit": [I, I, I, P, P, P, P],
        "ssm_spec_verify_baseline": [ctypes.POINTER(M2Dims), I, P, P, P, P, P, P, P, P, P, P],
        "ssm_spec_commit_baseline": [I, I, P, P, P, P],
        "gdn_state_update_baseline": [ctypes.POINTER(GdnDims), P, P, P, P, P, P, P, P],
        "gdn_replay_decode": [ctypes.POINTER(GdnDims), ctypes.POINTER(GdnReplay), P, P, P, P, P, P, P],
        "gdn_replay_decode_fused": [ctypes.POINTER(GdnDims), ctypes.POINTER(GdnReplay), P, P, P, P, P, P, P],
        "gdn_replay_flush": [ctypes.POINTER(GdnDims), ctypes.POINTER(GdnReplay), P],
        "gdn_replay_verify": [ctypes.POINTER(GdnDims), ctypes.POINTER(GdnReplay), I, P, P, P, P, P, P, P],
        "gdn_replay_verify_fused": [ctypes.POINTER(GdnDims), ctypes.POINTER(GdnReplay), I, P, P, P, P, P, P, P],
        "gdn_spec_verify_baseline": [ctypes.POINTER(GdnDims), I, P, P, P, P, P, P, P, P, P, P],
        "conv_state_update": [ctypes.POINTER(ConvDims), P, P, P, P, P, P, P, P],
        "rssm_m2_layout_sizes": [ctypes.POINTER(M2Dims), ctypes.POINTER(Layout)],
        "rssm_gdn_layout_sizes": [ctypes.POINTER(GdnDims), ctypes.POINTER(Layout)],
        "rssm_read_error": [P, ctypes.POINTER(ctypes.c_int32), P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int32
    lib.rssm_version.restype = ctypes.c_int32
    lib.rssm_version.argtypes = []
    lib.rssm_status_string.restype = ctypes.c_char_p
    lib.rssm_status_string.argtypes = [ctypes.c_int32]
    lib.rssm_last_cuda_error.restype = ctypes.c_char_p
    lib.rssm_last_cuda_error.argtypes = []
    lib.replay_decode_workspace_bytes.restype = ctypes.c_int64
    lib.replay_decode_workspace_bytes.argtypes = [ctypes.POINTER(M2Dims)]
    lib.replay_verify_workspace_bytes.restype = ctypes.c_int64
    lib.replay_verify_workspace_bytes.argtypes = [ctypes.POINTER(M2Dims), ctypes.c_int32]
    lib.gdn_replay_workspace_bytes.restype = ctypes.c_int64
    lib.gdn_replay_workspace_bytes.argtypes = [ctypes.POINTER(GdnDims), ctypes.c_int32]
    lib.replay_seq_bytes.restype = ctypes.c_int64
    lib.replay_seq_bytes.argtypes = [ctypes.POINTER(M2Dims), ctypes.c_int32, ctypes.c_int32]
    lib.gdn_replay_seq_bytes.restype = ctypes.c_int64
    lib.gdn_replay_seq_bytes.argtypes = [ctypes.POINTER(GdnDims), ctypes.c_int32, ctypes.c_int32]
    return lib


LIB = _load()


def _check(status: int, what: str):
    if status != 0:
        msg = LIB.rssm_status_string(status).decode()
        if status == -3:
            msg += ": " + LIB.rssm_last_cuda_error().decode()
        raise ReplaySSMError(f"{what} failed ({status}): {msg}")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    return ctypes.c_void_p((torch.cuda.current_stream() if stream is None else stream).cuda_stream)


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise ValueError(f"{name} must be int32")


# ---------------------------------------------------------------------------
# state containers
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Mamba2State:
    """Checkpoint + ring buffer of one Mamba-2 layer (device tensors)."""

    S0: torch.Tensor  # [B,H,d,n] f32
    ring_v: torch.Tensor  # [B,H,L,d] in dtype
    ring_k: torch.Tensor  # [B,G,L,n] in dtype
    ring_dt: torch.Tensor  # [B,H,L] f32
    start: torch.Tensor  # [B] i32
    count: torch.Tensor  # [B] i32
    flag: torch.Tensor  # [B] i32
    sync: torch.Tensor  # [B] i32, zero
    err: torch.Tensor  # [1] i32
    work: torch.Tensor | None = None  # decode workspace (f32, decode_workspace_bytes) or None

    @classmethod
    def empty(cls, B, H, G, d, n, L, dtype=torch.bfloat16, device="cuda", workspace=True):
        z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=device)  # noqa: E731
        st = cls(z(B, H, d, n), z(B, H, L, d, dt=dtype), z(B, G, L, n, dt=dtype), z(B, H, L),
                 z(B, dt=torch.int32), z(B, dt=torch.int32), z(B, dt=torch.int32), z(B, dt=torch.int32),
                 z(1, dt=torch.int32))
        if workspace:
            st.add_workspace()
        return st

    def add_workspace(self, max_T: int = 0):
        """Attach a workspace, which lets the decode step (and verify rounds of
        up to max_T drafts) run as a precompute launch plus a launch that
        streams S_0."""
        nbytes = decode_workspace_bytes(self.dims())
        if max_T:
            nbytes = max(nbytes, verify_workspace_bytes(self.dims(), max_T))
        self.work = torch.empty(nbytes // 4, dtype=torch.float32, device=self.S0.device)
        return self

    @property
    def shape(self):
        B, H, d, n = self.S0.shape
        return B, H, self.ring_k.shape[1], d, n, self.ring_v.shape[2]

    def dims(self, y_dtype=torch.float32) -> M2Dims:
        B, H, G, d, n, L = self.shape
        return M2Dims(B, H, G, d, n, L, _dt(self.ring_v), _DT[y_dtype])

    def struct(self) -> M2Replay:
        _f32(self.S0, "S0")
        _f32(self.ring_dt, "ring_dt")
        for name in ("start", "count", "flag", "sync", "err"):
            _i32(getattr(self, name), name)
        if self.work is not None:
            _f32(self.work, "work")
        ptrs = [_ptr(getattr(self, f)) for f in
                ("S0", "ring_v", "ring_k", "ring_dt", "start", "count", "flag", "sync", "err", "work")]
        return M2Replay(*ptrs, 0 if self.work is None else self.work.numel() * 4)


@dataclasses.dataclass
class GdnState:
    """Checkpoint + ring buffer of cached corrections of one GDN layer."""

    S0: torch.Tensor  # [B,Hv,dv,dk] f32
    ring_u: torch.Tensor  # [B,Hv,L,dv] u dtype
    ring_k: torch.Tensor  # [B,Hk,L,dk] in dtype
    ring_g: torch.Tensor  # [B,Hv,L] f32
    start: torch.Tensor
    count: torch.Tensor
    flag: torch.Tensor
    sync: torch.Tensor
    err: torch.Tensor
    work: torch.Tensor | None = None  # workspace (f32, gdn_workspace_bytes) or None

    @classmethod
    def empty(cls, B, Hv, Hk, dk, dv, L, dtype=torch.bfloat16, u_dtype=torch.float32, device="cuda",
              workspace_T=4):
        z = lambda *s, dt=torch.float32: torch.zeros(*s, dtype=dt, device=device)  # noqa: E731
        st = cls(z(B, Hv, dv, dk), z(B, Hv, L, dv, dt=u_dtype), z(B, Hk, L, dk, dt=dtype), z(B, Hv, L),
                 z(B, dt=torch.int32), z(B, dt=torch.int32), z(B, dt=torch.int32), z(B, dt=torch.int32),
                 z(1, dt=torch.int32))
        if workspace_T:
            st.add_workspace(workspace_T)
        return st

    def add_workspace(self, max_T: int = 4):
        """Attach a workspace for decode steps and verify rounds of up to max_T
        drafts, which lets them run as a precompute launch plus a launch that
        streams S_0."""
        nbytes = gdn_workspace_bytes(self.dims(), max_T)
        self.work = torch.empty(nbytes // 4, dtype=torch.float32, device=self.S0.device)
        return self

    @property
    def shape(self):
        B, Hv, dv, dk = self.S0.shape
        return B, Hv, self.ring_k.shape[1], dk, dv, self.ring_u.shape[2]

    def dims(self, y_dtype=torch.float32) -> GdnDims:
        B, Hv, Hk, dk, dv, L = self.shape
        return GdnDims(B, Hv, Hk, dk, dv, L, _dt(self.ring_k), _dt(self.ring_u), _DT[y_dtype])

    def struct(self) -> GdnReplay:
        _f32(self.S0, "S0")
        _f32(self.ring_g, "ring_g")
        for name in ("start", "count", "flag", "sync", "err"):
            _i32(getattr(self, name), name)
        if self.work is not None:
            _f32(self.work, "work")
        ptrs = [_ptr(getattr(self, f)) for f in
                ("S0", "ring_u", "ring_k", "ring_g", "start", "count", "flag", "sync", "err", "work")]
        return GdnReplay(*ptrs, 0 if self.work is None else self.work.numel() * 4)


# ---------------------------------------------------------------------------
# Mamba-2 calls
# ---------------------------------------------------------------------------


def gdn_workspace_bytes(dims: GdnDims, max_T: int = 1) -> int:
    """Bytes of the optional GDN workspace for calls with up to max_T drafts."""
    n = int(LIB.gdn_replay_workspace_bytes(ctypes.byref(dims), int(max_T)))
    if n <= 0:
        raise ReplaySSMError("gdn_replay_workspace_bytes: invalid arguments")
    return n


def verify_workspace_bytes(dims: M2Dims, max_T: int) -> int:
    """Bytes of the optional Mamba-2 workspace for verify rounds of up to max_T drafts."""
    n = int(LIB.replay_verify_workspace_bytes(ctypes.byref(dims), int(max_T)))
    if n <= 0:
        raise ReplaySSMError("replay_verify_workspace_bytes: invalid arguments")
    return n


def decode_workspace_bytes(dims: M2Dims) -> int:
    """Bytes of the optional Mamba-2 decode workspace for these dims."""
    n = int(LIB.replay_decode_workspace_bytes(ctypes.byref(dims)))
    if n <= 0:
        raise ReplaySSMError("replay_decode_workspace_bytes: invalid dims")
    return n


def seq_bytes(dims, T: int, kind: int) -> int:
    """Device bytes one sequence holds per layer (replay_seq_bytes or
    gdn_replay_seq_bytes, chosen by the type of dims); kind SEQ_REPLAY or
    SEQ_SNAPSHOT, T the speculative window (0: standard decode)."""
    fn = LIB.gdn_replay_seq_bytes if isinstance(dims, GdnDims) else LIB.replay_seq_bytes
    n = int(fn(ctypes.byref(dims), int(T), int(kind)))
    if n <= 0:
        raise ReplaySSMError("seq_bytes: invalid arguments")
    return n


def max_sequences(budget_bytes: int, dims, T: int, kind: int, layers: int = 1) -> int:
    """Largest batch whose per-sequence state for `layers` layers fits in budget_bytes."""
    return int(budget_bytes) // (int(layers) * seq_bytes(dims, T, kind))


def _out(y, shape, dtype, device):
    if y is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return y


def ssm_state_update_baseline(S, v, k, q, dt, A, y=None, y_dtype=torch.float32, stream=None):
    """Baseline decode step: S <- a S + dt v k^T in place, returns y = S q."""
    _f32(S, "S")
    B, H, d, n = S.shape
    G = k.shape[1]
    y = _out(y, (B, H, d), y_dtype, S.device)
    dims = M2Dims(B, H, G, d, n, 1, _dt(v), _dt(y))
    _check(LIB.ssm_state_update_baseline(ctypes.byref(dims), _ptr(S), _ptr(v), _ptr(k), _ptr(q), _ptr(dt), _ptr(A),
                                         _ptr(y), _stream(stream)), "ssm_state_update_baseline")
    return y


def replay_decode_step(state: Mamba2State, v, k, q, dt, A, y=None, y_dtype=torch.float32, stream=None):
    B, H, G, d, n, L = state.shape
    y = _out(y, (B, H, d), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.replay_decode_step(ctypes.byref(dims), ctypes.byref(st), _ptr(v), _ptr(k), _ptr(q), _ptr(dt), _ptr(A),
                                  _ptr(y), _stream(stream)), "replay_decode_step")
    return y


def replay_decode_step_fused(state: Mamba2State, v, k, q, dt, A, y=None, y_dtype=torch.float32, stream=None):
    """Decode step with the full-buffer flush in the same launch."""
    B, H, G, d, n, L = state.shape
    y = _out(y, (B, H, d), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.replay_decode_step_fused(ctypes.byref(dims), ctypes.byref(st), _ptr(v), _ptr(k), _ptr(q), _ptr(dt),
                                        _ptr(A), _ptr(y), _stream(stream)), "replay_decode_step_fused")
    return y


def replay_decode_step_fused_noalloc(state: Mamba2State, v, k, q, dt, A, y=None, y_dtype=torch.float32,
                                     stream=None):
    """replay_decode_step_fused with the library's own workspace (state.work is
    not used); allocates nothing when y is given."""
    B, H, G, d, n, L = state.shape
    y = _out(y, (B, H, d), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.replay_decode_step_fused_noalloc(ctypes.byref(dims), ctypes.byref(st), _ptr(v), _ptr(k), _ptr(q),
                                                _ptr(dt), _ptr(A), _ptr(y), _stream(stream)),
           "replay_decode_step_fused_noalloc")
    return y


def replay_flush(state: Mamba2State, A, stream=None):
    dims = state.dims()
    st = state.struct()
    _check(LIB.replay_flush(ctypes.byref(dims), ctypes.byref(st), _ptr(A), _stream(stream)), "replay_flush")


def replay_spec_verify(state: Mamba2State, v, k, q, dt, A, y=None, y_dtype=torch.float32, stream=None):
    """v [B,T,H,d]; k, q [B,T,G,n]; dt [B,T,H]; returns y [B,T,H,d]."""
    B, H, G, d, n, L = state.shape
    T = v.shape[1]
    y = _out(y, (B, T, H, d), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.replay_spec_verify(ctypes.byref(dims), ctypes.byref(st), T, _ptr(v), _ptr(k), _ptr(q), _ptr(dt),
                                  _ptr(A), _ptr(y), _stream(stream)), "replay_spec_verify")
    return y


def replay_spec_verify_fused(state: Mamba2State, v, k, q, dt, A, y=None, y_dtype=torch.float32, stream=None):
    """replay_flush, then replay_spec_verify, in one call.  Arguments as
    replay_spec_verify."""
    B, H, G, d, n, L = state.shape
    T = v.shape[1]
    y = _out(y, (B, T, H, d), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.replay_spec_verify_fused(ctypes.byref(dims), ctypes.byref(st), T, _ptr(v), _ptr(k), _ptr(q),
                                        _ptr(dt), _ptr(A), _ptr(y), _stream(stream)), "replay_spec_verify_fused")
    return y


def replay_spec_commit(accepted, count, T: int, L: int, err=None, stream=None):
    _i32(accepted, "accepted")
    _i32(count, "count")
    _check(LIB.replay_spec_commit(count.shape[0], T, L, _ptr(accepted), _ptr(count), _ptr(err), _stream(stream)),
           "replay_spec_commit")


def ssm_spec_verify_baseline(slots, cur, v, k, q, dt, A, y=None, err=None, y_dtype=torch.float32, stream=None):
    """slots [B,T+1,H,d,n] f32; cur [B] i32; inputs as replay_spec_verify."""
    _f32(slots, "slots")
    B, T1, H, d, n = slots.shape
    T = T1 - 1
    G = k.shape[2]
    y = _out(y, (B, T, H, d), y_dtype, slots.device)
    dims = M2Dims(B, H, G, d, n, 1, _dt(v), _dt(y))
    _check(LIB.ssm_spec_verify_baseline(ctypes.byref(dims), T, _ptr(slots), _ptr(cur), _ptr(v), _ptr(k), _ptr(q),
                                        _ptr(dt), _ptr(A), _ptr(y), _ptr(err), _stream(stream)), "ssm_spec_verify_baseline")
    return y


def ssm_spec_commit_baseline(accepted, cur, T: int, err=None, stream=None):
    _check(LIB.ssm_spec_commit_baseline(cur.shape[0], T, _ptr(accepted), _ptr(cur), _ptr(err), _stream(stream)),
           "ssm_spec_commit_baseline")


# ---------------------------------------------------------------------------
# GDN calls
# ---------------------------------------------------------------------------


def gdn_state_update_baseline(S, q, k, v, beta, g, y=None, y_dtype=torch.float32, stream=None):
    _f32(S, "S")
    B, Hv, dv, dk = S.shape
    Hk = k.shape[1]
    y = _out(y, (B, Hv, dv), y_dtype, S.device)
    dims = GdnDims(B, Hv, Hk, dk, dv, 1, _dt(k), F32, _dt(y))
    _check(LIB.gdn_state_update_baseline(ctypes.byref(dims), _ptr(S), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                         _ptr(y), _stream(stream)), "gdn_state_update_baseline")
    return y


def gdn_replay_decode(state: GdnState, q, k, v, beta, g, y=None, y_dtype=torch.float32, stream=None):
    B, Hv, Hk, dk, dv, L = state.shape
    y = _out(y, (B, Hv, dv), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.gdn_replay_decode(ctypes.byref(dims), ctypes.byref(st), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                 _ptr(y), _stream(stream)), "gdn_replay_decode")
    return y


def gdn_replay_decode_fused(state: GdnState, q, k, v, beta, g, y=None, y_dtype=torch.float32, stream=None):
    """GDN decode step with the full-buffer flush in the same launches."""
    B, Hv, Hk, dk, dv, L = state.shape
    y = _out(y, (B, Hv, dv), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.gdn_replay_decode_fused(ctypes.byref(dims), ctypes.byref(st), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                       _ptr(g), _ptr(y), _stream(stream)), "gdn_replay_decode_fused")
    return y


def gdn_replay_flush(state: GdnState, stream=None):
    dims = state.dims()
    st = state.struct()
    _check(LIB.gdn_replay_flush(ctypes.byref(dims), ctypes.byref(st), _stream(stream)), "gdn_replay_flush")


def gdn_replay_verify(state: GdnState, q, k, v, beta, g, y=None, y_dtype=torch.float32, stream=None):
    """q, k [B,T,Hk,dk]; v [B,T,Hv,dv]; beta, g [B,T,Hv]; returns y [B,T,Hv,dv]."""
    B, Hv, Hk, dk, dv, L = state.shape
    T = v.shape[1]
    y = _out(y, (B, T, Hv, dv), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.gdn_replay_verify(ctypes.byref(dims), ctypes.byref(st), T, _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                 _ptr(g), _ptr(y), _stream(stream)), "gdn_replay_verify")
    return y


def gdn_replay_verify_fused(state: GdnState, q, k, v, beta, g, y=None, y_dtype=torch.float32, stream=None):
    """gdn_replay_flush, then gdn_replay_verify, in one call.  Arguments as
    gdn_replay_verify."""
    B, Hv, Hk, dk, dv, L = state.shape
    T = v.shape[1]
    y = _out(y, (B, T, Hv, dv), y_dtype, state.S0.device)
    dims = state.dims(y.dtype)
    st = state.struct()
    _check(LIB.gdn_replay_verify_fused(ctypes.byref(dims), ctypes.byref(st), T, _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(beta), _ptr(g), _ptr(y), _stream(stream)), "gdn_replay_verify_fused")
    return y


def gdn_spec_verify_baseline(slots, cur, q, k, v, beta, g, y=None, err=None, y_dtype=torch.float32, stream=None):
    _f32(slots, "slots")
    B, T1, Hv, dv, dk = slots.shape
    T = T1 - 1
    Hk = k.shape[2]
    y = _out(y, (B, T, Hv, dv), y_dtype, slots.device)
    dims = GdnDims(B, Hv, Hk, dk, dv, 1, _dt(k), F32, _dt(y))
    _check(LIB.gdn_spec_verify_baseline(ctypes.byref(dims), T, _ptr(slots), _ptr(cur), _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(beta), _ptr(g), _ptr(y), _ptr(err), _stream(stream)),
           "gdn_spec_verify_baseline")
    return y


def conv_state_update(state, u, weight, bias, dx: int, dbc: int, silu: bool = True, out=None, stream=None):
    """Convolution-state decode step: state [B][dx+2dbc][W-1] (updated in
    place), u [B][dx+2dbc] (same dtype, bf16 or f32), weight f32 [dx+2dbc][W],
    bias f32 [dx+2dbc] or None.  Returns (x [B][dx], b [B][dbc], c [B][dbc])
    in the state's dtype, or writes into `out` = (x, b, c)."""
    B, C, Wm1 = state.shape
    if C != dx + 2 * dbc or tuple(u.shape) != (B, C) or u.dtype != state.dtype:
        raise ValueError("state/u shapes or dtypes do not match dx + 2 dbc channels")
    _f32(weight, "weight")
    if bias is not None:
        _f32(bias, "bias")
    if out is None:
        out = tuple(torch.empty(B, n, dtype=state.dtype, device=state.device) for n in (dx, dbc, dbc))
    dims = ConvDims(B, dx, dbc, Wm1 + 1, _dt(state), 1 if silu else 0)
    _check(LIB.conv_state_update(ctypes.byref(dims), _ptr(state), _ptr(u), _ptr(weight), _ptr(bias),
                                 *(_ptr(t) if t.numel() else None for t in out), _stream(stream)), "conv_state_update")
    return out


def layout_sizes(dims) -> Layout:
    """Element counts of one layer's arrays (rssm_m2_layout_sizes or
    rssm_gdn_layout_sizes, chosen by the type of dims)."""
    out = Layout()
    fn = LIB.rssm_gdn_layout_sizes if isinstance(dims, GdnDims) else LIB.rssm_m2_layout_sizes
    _check(fn(ctypes.byref(dims), ctypes.byref(out)), "layout_sizes")
    return out


def read_error(err: torch.Tensor, stream=None) -> int:
    """The sticky device error word, read on torch's current stream or on
    `stream` (this waits for that stream)."""
    _i32(err, "err")
    v = ctypes.c_int32(0)
    _check(LIB.rssm_read_error(_ptr(err), ctypes.byref(v), _stream(stream)), "rssm_read_error")
    return int(v.value)


def version() -> int:
    return int(LIB.rssm_version())
