"""Parity tests against the bounds-checked build of the library.

The bounds-checked variant (compiled with -DRSSM_CHECKED) checks every ring
slot a kernel writes and every pointer value it decodes from a workspace
record against its extent; a failed check sets RSSM_EBIT_BOUNDS in the
error word and the access is redirected or the item skipped, never out of
the caller's arrays.  It stands in for a memory sanitizer on the GPU.  This
test compiles that variant, then runs a representative set of the parity
tests in a fresh process bound to it (REPLAYSSM_LIB): every kernel family
(one- and two-launch decode, fused decode, verify on the CUDA and tensor
cores, the fused verify, the flush, GDN decode and chunked verify).  Each of
those tests also checks that the error word stays zero, so a check that
fires fails them.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SELECTED = [
    "tests/test_gpu_mamba2.py::test_tiny_config_parity",
    "tests/test_gpu_mamba2.py::test_decode_parity",
    "tests/test_gpu_mamba2.py::test_decode_fused_parity",
    "tests/test_gpu_mamba2.py::test_spec_verify_parity",
    "tests/test_gpu_mamba2.py::test_spec_verify_fused_parity",
    "tests/test_gpu_gdn.py::test_decode_parity",
    "tests/test_gpu_gdn.py::test_decode_fused_parity",
    "tests/test_gpu_gdn.py::test_chunked_verify_parity",
]


def test_parity_under_the_bounds_checked_build():
    from ssm_decode_hybrid_gb300 import build

    lib = build.build(checked=True)
    env = dict(os.environ, REPLAYSSM_LIB=lib)
    probe = subprocess.run(
        [sys.executable, "-c", "from ssm_decode_hybrid_gb300 import replayssm as R; print(R.LIB_PATH)"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip() == lib
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider", *SELECTED],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-2000:])
    assert " passed" in r.stdout
