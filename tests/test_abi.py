"""C-ABI checks that need no GPU: the library builds, loads and exports every
symbol include/coda.h declares; workspace sizes; argument validation that
returns before anything touches a device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coda.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g

    g.build()
    from gemm_epilogue_fusion_gemm0_gb300 import binding as B

    return B


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"CODA_API\s+[\w\s\*]+?\b(coda_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = declared_symbols()
    for must in ("coda_fwd", "coda_bwd_dgrad", "coda_fwd_workspace_bytes",
                 "coda_bwd_dgrad_workspace_bytes", "coda_get_device_status", "coda_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    raw = lib.raw()
    for name in declared_symbols():
        assert hasattr(raw, name), name
    assert set(declared_symbols()) == set(lib.EXPORTS)


def test_status_strings(lib):
    for code, name in lib.STATUS_NAMES.items():
        assert lib.status_string(code) == name


def _split_tail_bytes_for_tiles(tiles):
    # min(T, 160) slots of 256 x 256 fp32 partials, a u64 flag per 128-row half of each
    # (rounded up to 256 B); the launch counter is the workspace's first 256 bytes
    slots = min(tiles, 160)
    return slots * 256 * 256 * 4 + -(-(slots * 16) // 256) * 256


def _split_tail_bytes(M, d, N1):
    # the forward's region: T = 256 x 256 tiles of the larger GEMM
    return _split_tail_bytes_for_tiles(-(-M // 256) * max(-(-d // 256), -(-N1 // 256)))


def test_workspace_sizes(lib):
    # Every workspace starts with the 256-byte slot of the launch counter.  The forward:
    # the slot, hg [M,d] bf16 + partial sums [2 * ceil(d/256), M] fp32, each rounded up to
    # 256 B, then the split-tail region
    M, d, N1 = 8192, 4096, 28672
    assert _split_tail_bytes(M, d, N1) == 160 * 262144 + 2560
    assert lib.coda_fwd_workspace_bytes(M, d, N1) == (
        256 + M * d * 2 + 32 * M * 4 + _split_tail_bytes(M, d, N1))
    assert lib.coda_fwd_unfused_workspace_bytes(M, d, N1) == 256 + M * d * 2
    # the slot, qpart [2 * 32, M] fp32 + flags [2 * ceil(M/256) * 32] u64 (one per 128-row
    # slab and column tile, for up to 2 * ceil(d/256) = 32 column tiles per row block), then
    # min(3 T, 192) partial slots of 2 x 128 x 256 fp32 and their 2 flags each for the
    # pieces of the last row blocks (T = 32 x 16 tiles of 256 x 256)
    assert lib.coda_bwd_dgrad_workspace_bytes(M, d, N1) == (
        256 + 64 * M * 4 + 64 * 32 * 8 + 192 * 262144 + 192 * 16)
    # 256; 2 * 2 x 300 fp32 = 4800 -> 4864; 4 slabs x 2 tiles x 8 = 64 -> 256; 3 x 2 x 1
    # tiles = 6 slots of 256 KiB; 6 x 16 = 96 -> 256
    assert lib.coda_bwd_dgrad_workspace_bytes(300, 256, 512) == 256 + 4864 + 256 + 6 * 262144 + 256
    assert lib.coda_fwd_workspace_bytes(0, d, N1) == 0
    assert _split_tail_bytes(300, 328, 776) == 8 * 262144 + 256  # 2 x 4 tiles
    assert lib.coda_fwd_workspace_bytes(300, 328, 776) == (  # ragged: rounded up
        256 + 196864 + 4864 + _split_tail_bytes(300, 328, 776))
    assert lib.coda_fwd_workspace_bytes(10, 12, 16) == 0  # d % 8 != 0: unsupported
    # the slot, the SwiGLU statistic's partials [2 * ceil(N1/2 / 256), M] fp32, then the piece
    # slots of its tile-local data gradient as for coda_bwd_dgrad (3 x 2 x 1 tiles = 6)
    assert lib.coda_bwd_swiglu_dgrad_workspace_bytes(300, 256, 1024, 512) == (
        256 + 4864 + 6 * 262144 + 256)
    # the slot, then hq [M, d] E4M3 codes and the partial sums
    assert lib.coda_fwd_fp8_workspace_bytes(300, 256, 512) == 256 + 76800 + 2560
    # the full backward: the data gradient's workspace, h2 [M, d] bf16, the dgamma partials
    # [4 * 128-row slabs, d] fp32 and the split-tail region sized for its largest GEMM
    tiles = max(-(-d // 256) * -(-max(d, N1) // 256), -(-M // 256) * -(-d // 256))
    assert lib.coda_bwd_workspace_bytes(M, d, N1) == (
        lib.coda_bwd_dgrad_workspace_bytes(M, d, N1) + M * d * 2 + 4 * 64 * d * 4
        + _split_tail_bytes_for_tiles(tiles))


FAKE = 0x10000  # a 16-byte-aligned address that is never dereferenced


def _fwd(lib, M=128, d=256, N1=512, eps=1e-5, ptrs=None, ws=FAKE, wsb=1 << 30):
    p = [FAKE] * 8 if ptrs is None else ptrs
    return lib.raw().coda_fwd(p[0], p[1], p[2], p[3], p[4], eps, M, d, N1, p[5], p[6], p[7],
                              ws, wsb, None)


def _bwd(lib, M=128, d=256, N1=512, ptrs=None, ws=FAKE, wsb=1 << 30):
    p = [FAKE] * 6 if ptrs is None else ptrs
    return lib.raw().coda_bwd_dgrad(p[0], p[1], p[2], p[3], p[4], M, d, N1, p[5], ws, wsb, None)


def test_argument_validation_before_any_launch(lib):
    E = {v: k for k, v in lib.STATUS_NAMES.items()}
    assert _fwd(lib, M=-1) == E["CODA_ERR_INVALID_ARG"]
    assert _fwd(lib, d=0) == E["CODA_ERR_INVALID_ARG"]
    assert _fwd(lib, M=0) == E["CODA_OK"]  # empty batch: no-op
    assert _fwd(lib, d=260) == E["CODA_ERR_UNSUPPORTED_SHAPE"]
    assert _fwd(lib, N1=100) == E["CODA_ERR_UNSUPPORTED_SHAPE"]
    assert _fwd(lib, ptrs=[FAKE] * 7 + [0]) == E["CODA_ERR_INVALID_ARG"]
    assert _fwd(lib, ptrs=[FAKE + 8] + [FAKE] * 7) == E["CODA_ERR_MISALIGNED"]
    assert _fwd(lib, eps=float("nan")) == E["CODA_ERR_INVALID_ARG"]
    assert _fwd(lib, eps=-1.0) == E["CODA_ERR_INVALID_ARG"]
    assert _fwd(lib, wsb=100) == E["CODA_ERR_WORKSPACE_TOO_SMALL"]
    assert _fwd(lib, ws=0) == E["CODA_ERR_WORKSPACE_TOO_SMALL"]
    assert _bwd(lib, M=-5) == E["CODA_ERR_INVALID_ARG"]
    assert _bwd(lib, M=0) == E["CODA_OK"]
    assert _bwd(lib, d=12) == E["CODA_ERR_UNSUPPORTED_SHAPE"]
    assert _bwd(lib, ptrs=[FAKE] * 5 + [FAKE + 4]) == E["CODA_ERR_MISALIGNED"]
    assert _bwd(lib, wsb=8) == E["CODA_ERR_WORKSPACE_TOO_SMALL"]


def test_swiglu_argument_validation(lib):
    E = {v: k for k, v in lib.STATUS_NAMES.items()}
    raw = lib.raw()

    def call(N1=512, y=0, a=FAKE):
        return raw.coda_fwd_swiglu(FAKE, FAKE, FAKE, FAKE, FAKE, 1e-5, 128, 256, N1, FAKE, FAKE,
                                   y, a, FAKE, 1 << 30, None)

    assert call(N1=520) == E["CODA_ERR_UNSUPPORTED_SHAPE"]  # N1/2 rows must be 16-byte multiples
    assert call(a=0) == E["CODA_ERR_INVALID_ARG"]
    assert call(y=FAKE + 2) == E["CODA_ERR_MISALIGNED"]


def test_full_backward_workspace_and_validation(lib):
    E = {v: k for k, v in lib.STATUS_NAMES.items()}
    M, d, N1 = 8192, 4096, 28672
    # dgrad workspace + h2 [M, d] bf16 + dgamma partials [4 * 64 slabs, d] fp32
    # + a split-tail region sized for the largest of dW1 (d x N1), dx (M x d), dW0 (d x d)
    tiles = max(-(-d // 256) * -(-max(d, N1) // 256), -(-M // 256) * -(-d // 256))
    assert lib.coda_bwd_workspace_bytes(M, d, N1) == (
        lib.coda_bwd_dgrad_workspace_bytes(M, d, N1) + M * d * 2 + 4 * 64 * d * 4
        + _split_tail_bytes_for_tiles(tiles))
    raw = lib.raw()

    def call(res=0, M=128, wsb=1 << 30, dgamma=FAKE):
        return raw.coda_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, res, M, 256, 512, FAKE, FAKE,
                            dgamma, FAKE, FAKE, FAKE, wsb, None)

    assert call(M=-1) == E["CODA_ERR_INVALID_ARG"]
    assert call(M=0) == E["CODA_OK"]
    assert call(dgamma=0) == E["CODA_ERR_INVALID_ARG"]
    assert call(res=FAKE + 4) == E["CODA_ERR_MISALIGNED"]
    assert call(wsb=64) == E["CODA_ERR_WORKSPACE_TOO_SMALL"]


def test_fp8_argument_validation(lib):
    E = {v: k for k, v in lib.STATUS_NAMES.items()}
    raw = lib.raw()

    def call(d=256, sx=0.1, shg=0.1):
        return raw.coda_fwd_fp8(FAKE, sx, FAKE, 0.1, FAKE, FAKE, FAKE, 0.1, shg, 1e-5, 128, d, 512,
                                FAKE, FAKE, FAKE, FAKE, 1 << 30, None)

    assert call(d=264) == E["CODA_ERR_UNSUPPORTED_SHAPE"]  # FP8 rows need d % 16 == 0
    assert call(sx=0.0) == E["CODA_ERR_INVALID_ARG"]
    assert call(shg=float("nan")) == E["CODA_ERR_INVALID_ARG"]
    assert lib.coda_fwd_fp8_workspace_bytes(8192, 4096, 28672) == 256 + 8192 * 4096 + 32 * 8192 * 4


def test_no_device_is_reported_without_gpu(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is visible")
    E = {v: k for k, v in lib.STATUS_NAMES.items()}
    assert _fwd(lib) == E["CODA_ERR_NO_DEVICE"]
    assert _bwd(lib) == E["CODA_ERR_NO_DEVICE"]


def test_binding_refuses_to_load_without_the_library(tmp_path):
    """The product path has no CPU fallback: importing the binding from a copy of
    the package without libcoda.so raises ImportError."""
    import shutil
    import subprocess
    import sys

    pkg = "gemm_epilogue_fusion_gemm0_gb300"
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), pkg)
    dst = tmp_path / pkg
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.so", "*.so.tmp", "csrc", "__pycache__"))
    code = ("import importlib, sys\n"
            "try:\n"
            f"    importlib.import_module('{pkg}.binding')\n"
            "except ImportError as e:\n"
            "    print('ImportError:', e); sys.exit(0)\n"
            "sys.exit(1)\n")
    res = subprocess.run([sys.executable, "-c", code], cwd=tmp_path, capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "libcoda.so not found" in res.stdout


def test_binding_checks_tensors_before_calling_the_library(lib):
    """The binding refuses, before any C call, tensors that are not CUDA tensors
    and a workspace that is not one either; a raw stream handle passes through."""
    import torch

    M, d, N1 = 4, 8, 8
    bf = torch.bfloat16
    dy, W1 = torch.zeros(M, N1, dtype=bf), torch.zeros(d, N1, dtype=bf)
    h, r, g = torch.zeros(M, d, dtype=bf), torch.ones(M), torch.ones(d, dtype=bf)
    with pytest.raises(TypeError, match="dy must be a CUDA tensor"):
        lib.coda_bwd_dgrad(dy, W1, h, r, g, ws=torch.zeros(16, dtype=torch.uint8))
    call = lib._Call("probe", torch.device("cuda", 0))
    with pytest.raises(TypeError, match="workspace"):
        call.ws(torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(TypeError, match="x must be a CUDA tensor"):
        call.t(h, bf, (M, d), "x")
    assert lib._stream_ptr(1234) == 1234
