"""The checked build (libcoda_checked.so, compiled with -DCODA_CHECKED).

Every staged load and store of the epilogues (and every gamma load) is checked
against its tensor's extent, every TMA box start against its tensor map's
extent and the 16-byte alignment of its innermost coordinate, and every
workspace index against its size; a failed check records
CODA_ERR_DEVICE_BOUNDS and skips the access, it never traps.  The GPU test runs the small, ragged, split-tail, column-plan and
no-allocation parity cases against that library in a child process (the
binding picks the library when the process starts) and requires every case to
match the oracle with a clean status word.  The CPU test checks that the
checked library builds and exports the same symbols as the normal one.
"""

import ctypes
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_checked_library_builds_and_exports_the_same_symbols():
    sys.path.insert(0, ROOT)
    from gemm_epilogue_fusion_gemm0_gb300 import build as b
    from gemm_epilogue_fusion_gemm0_gb300.binding import EXPORTS

    path = b.build(checked=True)
    assert path == b.LIB_PATH_CHECKED and os.path.exists(path)
    lib = ctypes.CDLL(path)
    for name in EXPORTS:
        assert hasattr(lib, name), name


@pytest.mark.gpu
def test_checked_build_parity_cases_with_a_clean_status():
    env = dict(os.environ, CODA_CHECKED_BUILD="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert "checked cases ok" in r.stdout, out[-4000:]
