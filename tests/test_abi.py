"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments on the host before any launch (CPU only: no kernel runs)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "replayssm.h")


def _lib_path():
    from ssm_decode_hybrid_gb300 import build

    if not os.path.exists(build.LIB):
        build.build()
    return build.LIB


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"^RSSM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = set(declared_symbols())
    for required in ("ssm_state_update_baseline", "replay_decode_step", "replay_flush", "replay_spec_verify",
                     "replay_spec_commit", "gdn_replay_decode", "gdn_replay_flush", "gdn_replay_verify"):
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(_lib_path())
    for name in declared_symbols():
        assert hasattr(lib, name), f"missing export {name}"


def test_binding_covers_exports():
    _lib_path()
    from ssm_decode_hybrid_gb300 import replayssm as R

    assert set(declared_symbols()) == set(R.EXPORTS)
    assert R.version() == 200
    assert R.LIB.rssm_status_string(-1) == b"invalid argument"
    assert R.LIB.rssm_status_string(-2) == b"unsupported shape or dtype"


def test_every_launching_call_takes_a_stream():
    """Every binding call that passes a stream to the library accepts
    stream= (default None: torch's current stream), and the calls the
    library exposes with a stream argument are all covered."""
    import inspect

    _lib_path()
    from ssm_decode_hybrid_gb300 import replayssm as R

    src = inspect.getsource(R)
    callers = set(re.findall(r"^def (\w+)\(", src, flags=re.M)) - {"_stream"}
    with_stream = {n for n in callers if "_stream(stream)" in inspect.getsource(getattr(R, n))}
    assert "replay_decode_step_fused" in with_stream and "gdn_replay_verify" in with_stream
    for name in with_stream:
        p = inspect.signature(getattr(R, name)).parameters
        assert "stream" in p and p["stream"].default is None, name
    assert not re.search(r"(?<![\w.])_stream\(\)", src), "a call still takes torch's current stream only"
    header = open(HEADER).read()
    takes_stream = set(re.findall(r"^RSSM_API\s+[\w\s\*]+?\b(\w+)\s*\([^;]*?rssm_stream_t", header, flags=re.M | re.S))
    wrapped = {"rssm_read_error": "read_error"}
    for sym in takes_stream:
        assert wrapped.get(sym, sym) in with_stream, f"{sym} takes a stream but its binding has no stream="


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-validation test uses fake device pointers; CPU only")
def test_host_validation_rejects_bad_arguments():
    _lib_path()
    from ssm_decode_hybrid_gb300 import replayssm as R

    L = R.LIB
    P = ctypes.c_void_p
    fake = P(0x10000)  # aligned, never dereferenced: every call below fails validation first
    mis = P(0x10004)  # 4-byte but not 16-byte aligned

    def dims(**kw):
        base = dict(B=2, H=4, G=2, d=64, n=128, L=16, in_dtype=R.BF16, y_dtype=R.F32)
        base.update(kw)
        return R.M2Dims(*base.values())

    rep = R.M2Replay(*([fake] * 9))
    args = [fake, fake, fake, fake, fake, fake, None]
    assert L.replay_decode_step(None, ctypes.byref(rep), *args) == -1
    assert L.replay_decode_step(ctypes.byref(dims(H=3)), ctypes.byref(rep), *args) == -1  # H % G
    assert L.replay_decode_step(ctypes.byref(dims(n=96)), ctypes.byref(rep), *args) == -2
    assert L.replay_decode_step(ctypes.byref(dims(d=66)), ctypes.byref(rep), *args) == -2
    assert L.replay_decode_step(ctypes.byref(dims(L=33)), ctypes.byref(rep), *args) == -2
    assert L.replay_decode_step(ctypes.byref(dims(in_dtype=7)), ctypes.byref(rep), *args) == -1
    assert L.replay_decode_step(ctypes.byref(dims(B=0)), ctypes.byref(rep), *args) == -1
    assert L.replay_decode_step(ctypes.byref(dims()), None, *args) == -1
    bad = R.M2Replay(mis, *([fake] * 8))  # misaligned S0
    assert L.replay_decode_step(ctypes.byref(dims()), ctypes.byref(bad), *args) == -1
    badwork = R.M2Replay(*([fake] * 9), mis)  # misaligned decode workspace
    assert L.replay_decode_step(ctypes.byref(dims()), ctypes.byref(badwork), *args) == -1
    assert L.replay_decode_step_fused(ctypes.byref(dims()), ctypes.byref(badwork), *args) == -1
    cd = R.ConvDims(2, 8, 4, 4, R.BF16, 1)
    cargs = [fake, fake, fake, None, fake, fake, fake, None]
    for bad in (R.ConvDims(2, 8, 4, 1, R.BF16, 1), R.ConvDims(2, 8, 4, 9, R.BF16, 1), R.ConvDims(0, 8, 4, 4, R.BF16, 1),
                R.ConvDims(2, 0, 4, 4, R.BF16, 1), R.ConvDims(2, 8, -1, 4, R.BF16, 1), R.ConvDims(2, 8, 4, 4, 5, 1),
                R.ConvDims(2, 8, 4, 4, R.BF16, 2)):
        assert L.conv_state_update(ctypes.byref(bad), *cargs) == -1
    assert L.conv_state_update(None, *cargs) == -1
    assert L.conv_state_update(ctypes.byref(cd), fake, fake, P(0x10002), None, fake, fake, fake,
                               None) == -1  # misaligned weight
    assert L.conv_state_update(ctypes.byref(cd), fake, fake, fake, None, fake, None, fake, None) == -1  # no B output
    nosync = R.M2Replay(*([fake] * 7), None, fake)
    assert L.replay_decode_step(ctypes.byref(dims()), ctypes.byref(nosync), *args) == -1
    assert L.replay_flush(ctypes.byref(dims()), ctypes.byref(nosync), fake, None) == -1
    # verify: T out of range
    vargs = [fake, fake, fake, fake, fake, fake, None]
    assert L.replay_spec_verify(ctypes.byref(dims()), ctypes.byref(rep), 0, *vargs) == -1
    assert L.replay_spec_verify(ctypes.byref(dims(L=4)), ctypes.byref(rep), 5, *vargs) == -1
    assert L.replay_spec_verify(ctypes.byref(dims()), ctypes.byref(rep), 9, *vargs) == -2
    assert L.replay_spec_commit(2, 5, 4, fake, fake, None, None) == -1  # T > L
    assert L.replay_spec_commit(0, 1, 4, fake, fake, None, None) == -1
    assert L.ssm_spec_commit_baseline(2, 0, fake, fake, None, None) == -1
    # baseline: misaligned k
    assert L.ssm_state_update_baseline(ctypes.byref(dims()), fake, fake, mis, fake, fake, fake, fake, None) == -1

    gd = R.GdnDims(2, 4, 2, 128, 128, 16, R.BF16, R.F32, R.F32)
    grep = R.GdnReplay(*([fake] * 9))
    gargs = [fake, fake, fake, fake, fake, fake, None]
    bad_g = R.GdnDims(2, 4, 3, 128, 128, 16, R.BF16, R.F32, R.F32)  # Hv % Hk
    assert L.gdn_replay_decode(ctypes.byref(bad_g), ctypes.byref(grep), *gargs) == -1
    bad_g = R.GdnDims(2, 4, 2, 256, 128, 16, R.BF16, R.F32, R.F32)  # dk unsupported
    assert L.gdn_replay_decode(ctypes.byref(bad_g), ctypes.byref(grep), *gargs) == -2
    assert L.gdn_replay_verify(ctypes.byref(gd), ctypes.byref(grep), 17, *gargs) == -1
    assert L.gdn_replay_flush(ctypes.byref(gd), None, None) == -1


def test_decode_workspace_size_query():
    """Host-only size query: B * H records of 4 + L + d floats rounded up to 16 bytes."""
    _lib_path()
    from ssm_decode_hybrid_gb300 import replayssm as R

    def nbytes(B, H, G, d, n, L):
        return R.LIB.replay_decode_workspace_bytes(ctypes.byref(R.M2Dims(B, H, G, d, n, L, R.BF16, R.F32)))

    assert nbytes(256, 32, 8, 64, 128, 16) == 256 * 32 * 84 * 4
    assert nbytes(3, 4, 2, 20, 32, 3) == 3 * 4 * 28 * 4
    assert nbytes(1, 1, 1, 4, 16, 1) == 12 * 4
    assert nbytes(2, 3, 2, 64, 128, 16) == 0  # H % G != 0
    assert R.LIB.replay_decode_workspace_bytes(None) == 0
