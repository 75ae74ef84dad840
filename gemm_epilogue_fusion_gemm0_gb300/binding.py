"""ctypes binding of libcoda.so (include/coda.h), same names as the C ABI.

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity and passed as raw device pointers together with the current CUDA
stream.  Every step of the computation runs in the library's kernels; if the
library is missing this module raises at import time.  A process started with
CODA_CHECKED_BUILD=1 loads the checked build (libcoda_checked.so) instead.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH, LIB_PATH_CHECKED

LIB = LIB_PATH_CHECKED if os.environ.get("CODA_CHECKED_BUILD") == "1" else LIB_PATH

if not os.path.exists(LIB):
    raise ImportError(
        f"{os.path.basename(LIB)} not found at {LIB}: build it first "
        "(python -c 'import __graft_entry__ as g; g.build()')"
    )

_lib = ctypes.CDLL(LIB)

CODA_OK = 0
CODA_ERR_INVALID_ARG = 1
CODA_ERR_UNSUPPORTED_SHAPE = 2
CODA_ERR_MISALIGNED = 3
CODA_ERR_WORKSPACE_TOO_SMALL = 4
CODA_ERR_LAUNCH = 5
CODA_ERR_DEVICE_TIMEOUT = 6
CODA_ERR_NO_DEVICE = 7
CODA_ERR_UNSUPPORTED_DEVICE = 8
CODA_ERR_DEVICE_BOUNDS = 9
STATUS_NAMES = {
    0: "CODA_OK",
    1: "CODA_ERR_INVALID_ARG",
    2: "CODA_ERR_UNSUPPORTED_SHAPE",
    3: "CODA_ERR_MISALIGNED",
    4: "CODA_ERR_WORKSPACE_TOO_SMALL",
    5: "CODA_ERR_LAUNCH",
    6: "CODA_ERR_DEVICE_TIMEOUT",
    7: "CODA_ERR_NO_DEVICE",
    8: "CODA_ERR_UNSUPPORTED_DEVICE",
    9: "CODA_ERR_DEVICE_BOUNDS",
}

_vp, _i64, _sz, _f32, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float, ctypes.c_uint64
_st = ctypes.c_int

EXPORTS = {
    # name: (restype, argtypes)
    "coda_fwd_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "coda_bwd_dgrad_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "coda_fwd_unfused_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "coda_fwd": (_st, [_vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "coda_fwd_unfused": (_st, [_vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "coda_bwd_dgrad": (_st, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "coda_get_device_status": (_st, [_vp, ctypes.POINTER(ctypes.c_uint32)]),
    "coda_set_wait_timeout_ns": (None, [_u64]),
    "coda_status_string": (ctypes.c_char_p, [_st]),
    "coda_watchdog_selftest": (_st, [_u64, _vp]),
    "coda_set_launch_events": (None, [_vp, ctypes.c_int]),
    "coda_bwd_dgrad_noalloc": (_st, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]),
    "coda_set_mma_mode": (_st, [ctypes.c_int]),
    "coda_bwd_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "coda_bwd": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                       _vp, _sz, _vp]),
    "coda_bwd_swiglu_dgrad_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "coda_bwd_swiglu_dgrad": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp,
                                    _vp, _vp, _vp, _sz, _vp]),
    "coda_fwd_swiglu": (_st, [_vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                              _sz, _vp]),
    "coda_get_mma_mode": (ctypes.c_int, []),
    "coda_set_fold_rowreduce": (_st, [ctypes.c_int]),
    "coda_set_split_tail": (_st, [ctypes.c_int]),
    "coda_set_col_plan": (_st, [ctypes.c_int]),
    "coda_set_serpentine_k": (_st, [ctypes.c_int]),
    "coda_get_serpentine_k": (ctypes.c_int, []),
    "coda_set_dgrad_pieces": (_st, [ctypes.c_int]),
    "coda_get_dgrad_pieces": (ctypes.c_int, []),
    "coda_dgrad_piece_plan": (ctypes.c_int, [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int32)]),
    "coda_fwd_fp8_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "coda_fwd_fp8": (_st, [_vp, _f32, _vp, _f32, _vp, _vp, _vp, _f32, _f32, _f32, _i64, _i64, _i64, _vp,
                           _vp, _vp, _vp, _sz, _vp]),
}

for _name, (_res, _args) in EXPORTS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class CodaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def status_string(status: int) -> str:
    return _lib.coda_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != CODA_OK:
        raise CodaError(status, where)


def _stream_ptr(stream, device=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if not hasattr(stream, "cuda_stream"):
        return int(stream)  # a raw cudaStream_t handle
    if device is not None and stream.device != device:
        raise ValueError(f"the stream is on {stream.device}, the call's tensors on {device}")
    return int(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype: torch.dtype, shape: tuple, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class _Call:
    """Marshalling for one call: every tensor must be a contiguous CUDA tensor
    of the stated dtype and shape on the device of the call's first tensor,
    and the C function runs with that device current (the C ABI works on the
    current device, so a tensor on another one would hand the kernels a
    pointer they cannot use)."""

    def __init__(self, where: str, device: torch.device):
        self.where, self.device = where, torch.device(device)

    def t(self, t, dtype, shape, name) -> int:
        p = _dev(t, dtype, shape, name)
        if t.device != self.device:
            raise ValueError(f"{self.where}: {name} is on {t.device}, the call's first tensor on "
                             f"{self.device}")
        return p

    def opt(self, t, dtype, shape, name):
        return None if t is None else self.t(t, dtype, shape, name)

    def ws(self, ws) -> tuple:
        if not isinstance(ws, torch.Tensor) or not ws.is_cuda or not ws.is_contiguous():
            raise TypeError(f"{self.where}: the workspace must be a contiguous CUDA tensor")
        if ws.device != self.device:
            raise ValueError(f"{self.where}: the workspace is on {ws.device}, the call's first "
                             f"tensor on {self.device}")
        return ws.data_ptr(), ws.numel() * ws.element_size()

    def run(self, fn, *args, stream=None) -> None:
        if self.device.index == torch.cuda.current_device():
            _check(fn(*args, _stream_ptr(stream, self.device)), self.where)
            return
        with torch.cuda.device(self.device):
            _check(fn(*args, _stream_ptr(stream, self.device)), self.where)


# --------------------------------------------------------------------------- sizes
def coda_fwd_workspace_bytes(M: int, d: int, N1: int) -> int:
    return int(_lib.coda_fwd_workspace_bytes(M, d, N1))


def coda_fwd_unfused_workspace_bytes(M: int, d: int, N1: int) -> int:
    return int(_lib.coda_fwd_unfused_workspace_bytes(M, d, N1))


def coda_bwd_dgrad_workspace_bytes(M: int, d: int, N1: int) -> int:
    return int(_lib.coda_bwd_dgrad_workspace_bytes(M, d, N1))


def workspace(nbytes: int, device) -> torch.Tensor:
    """A device byte buffer of at least `nbytes` (torch allocates it)."""
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


# --------------------------------------------------------------------------- calls
def _fwd_common(fn, wsfn, x, W0, z, gamma, W1, eps, h, r, y, ws, stream):
    M, d = x.shape
    N1 = W1.shape[1]
    dev = x.device
    if h is None:
        h = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
    if r is None:
        r = torch.empty((M,), dtype=torch.float32, device=dev)
    if y is None:
        y = torch.empty((M, N1), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = workspace(wsfn(M, d, N1), dev)
    bf = torch.bfloat16
    c = _Call(fn.__name__, dev)
    c.run(fn, c.t(x, bf, (M, d), "x"), c.t(W0, bf, (d, d), "W0"), c.t(z, bf, (M, d), "z"),
          c.t(gamma, bf, (d,), "gamma"), c.t(W1, bf, (d, N1), "W1"), float(eps), M, d, N1,
          c.t(h, bf, (M, d), "h"), c.t(r, torch.float32, (M,), "r"), c.t(y, bf, (M, N1), "y"),
          *c.ws(ws), stream=stream)
    return h, r, y


def coda_fwd(x, W0, z, gamma, W1, eps, h=None, r=None, y=None, ws=None, stream=None):
    """Fused forward; returns (h, r, y).  Outputs are allocated if not given."""
    return _fwd_common(_lib.coda_fwd, coda_fwd_workspace_bytes, x, W0, z, gamma, W1, eps,
                       h, r, y, ws, stream)


def coda_fwd_unfused(x, W0, z, gamma, W1, eps, h=None, r=None, y=None, ws=None, stream=None):
    """Unfused reference sequence (measurement only); returns (h, r, y)."""
    return _fwd_common(_lib.coda_fwd_unfused, coda_fwd_unfused_workspace_bytes, x, W0, z, gamma,
                       W1, eps, h, r, y, ws, stream)


def coda_fwd_swiglu(x, W0, z, gamma, W1, eps, h=None, r=None, a=None, y=None, want_y=False,
                    ws=None, stream=None):
    """Fused forward with the SwiGLU gated activation; W1 = [W_gate | W_up].
    Returns (h, r, a) or (h, r, a, y) with want_y=True (pre-activation)."""
    M, d = x.shape
    N1 = W1.shape[1]
    dev = x.device
    bf = torch.bfloat16
    h = torch.empty((M, d), dtype=bf, device=dev) if h is None else h
    r = torch.empty((M,), dtype=torch.float32, device=dev) if r is None else r
    a = torch.empty((M, N1 // 2), dtype=bf, device=dev) if a is None else a
    if want_y and y is None:
        y = torch.empty((M, N1), dtype=bf, device=dev)
    if ws is None:
        ws = workspace(coda_fwd_workspace_bytes(M, d, N1), dev)
    c = _Call("coda_fwd_swiglu", dev)
    c.run(_lib.coda_fwd_swiglu,
          c.t(x, bf, (M, d), "x"), c.t(W0, bf, (d, d), "W0"), c.t(z, bf, (M, d), "z"),
          c.t(gamma, bf, (d,), "gamma"), c.t(W1, bf, (d, N1), "W1"), float(eps), M, d, N1,
          c.t(h, bf, (M, d), "h"), c.t(r, torch.float32, (M,), "r"), c.opt(y, bf, (M, N1), "y"),
          c.t(a, bf, (M, N1 // 2), "a"), *c.ws(ws), stream=stream)
    return (h, r, a, y) if y is not None else (h, r, a)


def coda_fwd_fp8_workspace_bytes(M: int, d: int, N1: int) -> int:
    return int(_lib.coda_fwd_fp8_workspace_bytes(M, d, N1))


def coda_fwd_fp8(x_q, sx, W0_q, sW0, z, gamma, W1_q, sW1, s_hg, eps, h=None, r=None, y=None,
                 ws=None, stream=None):
    """FP8 forward: x_q, W0_q, W1_q are float8_e4m3fn (or uint8) code tensors with
    per-tensor scales; returns (h, r, y)."""
    M, d = x_q.shape
    N1 = W1_q.shape[1]
    dev = x_q.device
    bf = torch.bfloat16
    h = torch.empty((M, d), dtype=bf, device=dev) if h is None else h
    r = torch.empty((M,), dtype=torch.float32, device=dev) if r is None else r
    y = torch.empty((M, N1), dtype=bf, device=dev) if y is None else y
    if ws is None:
        ws = workspace(coda_fwd_fp8_workspace_bytes(M, d, N1), dev)
    c = _Call("coda_fwd_fp8", dev)

    def code(t, shape, name):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must hold E4M3 codes (float8_e4m3fn or uint8)")
        return c.t(t, t.dtype, shape, name)

    c.run(_lib.coda_fwd_fp8,
          code(x_q, (M, d), "x_q"), float(sx), code(W0_q, (d, d), "W0_q"), float(sW0),
          c.t(z, bf, (M, d), "z"), c.t(gamma, bf, (d,), "gamma"), code(W1_q, (d, N1), "W1_q"),
          float(sW1), float(s_hg), float(eps), M, d, N1, c.t(h, bf, (M, d), "h"),
          c.t(r, torch.float32, (M,), "r"), c.t(y, bf, (M, N1), "y"), *c.ws(ws), stream=stream)
    return h, r, y


def coda_bwd_dgrad(dy, W1, h, r, gamma, dh=None, ws=None, stream=None):
    """Fused RMSNorm-branch data gradient; returns dh."""
    M, N1 = dy.shape
    d = W1.shape[0]
    if dh is None:
        dh = torch.empty((M, d), dtype=torch.bfloat16, device=dy.device)
    if ws is None:
        ws = workspace(coda_bwd_dgrad_workspace_bytes(M, d, N1), dy.device)
    bf = torch.bfloat16
    c = _Call("coda_bwd_dgrad", dy.device)
    c.run(_lib.coda_bwd_dgrad,
          c.t(dy, bf, (M, N1), "dy"), c.t(W1, bf, (d, N1), "W1"), c.t(h, bf, (M, d), "h"),
          c.t(r, torch.float32, (M,), "r"), c.t(gamma, bf, (d,), "gamma"), M, d, N1,
          c.t(dh, bf, (M, d), "dh"), *c.ws(ws), stream=stream)
    return dh


def coda_bwd_swiglu_dgrad_workspace_bytes(M: int, d: int, N1: int, Dout: int) -> int:
    return int(_lib.coda_bwd_swiglu_dgrad_workspace_bytes(M, d, N1, Dout))


def coda_bwd_swiglu_dgrad(dout, W2, y, W1, h, r, gamma, dy=None, s=None, dh=None, ws=None,
                          stream=None):
    """SwiGLU backward (statistic formed upstream) + tile-local RMSNorm-branch
    data gradient; returns (dy, s, dh)."""
    M, Dout = dout.shape
    half = W2.shape[0]
    N1 = 2 * half
    d = W1.shape[0]
    dev = dout.device
    bf = torch.bfloat16
    dy = torch.empty((M, N1), dtype=bf, device=dev) if dy is None else dy
    s = torch.empty((M,), dtype=torch.float32, device=dev) if s is None else s
    dh = torch.empty((M, d), dtype=bf, device=dev) if dh is None else dh
    if ws is None:
        ws = workspace(coda_bwd_swiglu_dgrad_workspace_bytes(M, d, N1, Dout), dev)
    c = _Call("coda_bwd_swiglu_dgrad", dev)
    c.run(_lib.coda_bwd_swiglu_dgrad,
          c.t(dout, bf, (M, Dout), "dout"), c.t(W2, bf, (half, Dout), "W2"),
          c.t(y, bf, (M, N1), "y"), c.t(W1, bf, (d, N1), "W1"), c.t(h, bf, (M, d), "h"),
          c.t(r, torch.float32, (M,), "r"), c.t(gamma, bf, (d,), "gamma"), M, d, N1, Dout,
          c.t(dy, bf, (M, N1), "dy"), c.t(s, torch.float32, (M,), "s"), c.t(dh, bf, (M, d), "dh"),
          *c.ws(ws), stream=stream)
    return dy, s, dh


def coda_bwd_workspace_bytes(M: int, d: int, N1: int) -> int:
    return int(_lib.coda_bwd_workspace_bytes(M, d, N1))


def coda_bwd(dy, x, W0, W1, h, r, gamma, dh_res=None, out=None, ws=None, stream=None):
    """All gradients of the chain; returns dict dh (= dz), dx, dgamma, dW0, dW1."""
    M, N1 = dy.shape
    d = W1.shape[0]
    dev = dy.device
    bf, f32 = torch.bfloat16, torch.float32
    o = dict(out or {})
    o.setdefault("dh", torch.empty((M, d), dtype=bf, device=dev))
    o.setdefault("dx", torch.empty((M, d), dtype=bf, device=dev))
    o.setdefault("dgamma", torch.empty((d,), dtype=f32, device=dev))
    o.setdefault("dW0", torch.empty((d, d), dtype=f32, device=dev))
    o.setdefault("dW1", torch.empty((d, N1), dtype=f32, device=dev))
    if ws is None:
        ws = workspace(coda_bwd_workspace_bytes(M, d, N1), dev)
    c = _Call("coda_bwd", dev)
    c.run(_lib.coda_bwd,
          c.t(dy, bf, (M, N1), "dy"), c.t(x, bf, (M, d), "x"), c.t(W0, bf, (d, d), "W0"),
          c.t(W1, bf, (d, N1), "W1"), c.t(h, bf, (M, d), "h"), c.t(r, f32, (M,), "r"),
          c.t(gamma, bf, (d,), "gamma"), c.opt(dh_res, bf, (M, d), "dh_res"),
          M, d, N1, c.t(o["dh"], bf, (M, d), "dh"), c.t(o["dx"], bf, (M, d), "dx"),
          c.t(o["dgamma"], f32, (d,), "dgamma"), c.t(o["dW0"], f32, (d, d), "dW0"),
          c.t(o["dW1"], f32, (d, N1), "dW1"), *c.ws(ws), stream=stream)
    return o


def coda_get_device_status(stream=None) -> tuple[int, int]:
    """(status, detail) after synchronising the stream; clears the status."""
    detail = ctypes.c_uint32(0)
    st = _lib.coda_get_device_status(_stream_ptr(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def coda_set_mma_mode(mode: int) -> None:
    """0: single-CTA 128x256 tiles; 1: CTA-pair 256x256 tiles (tcgen05 cta_group::2)."""
    _check(_lib.coda_set_mma_mode(int(mode)), "coda_set_mma_mode")


def coda_set_fold_rowreduce(enable: int) -> None:
    """1: r is formed in GEMM1's epilogue (2 launches); 0: separate reduction (default)."""
    _check(_lib.coda_set_fold_rowreduce(int(enable)), "coda_set_fold_rowreduce")


def coda_set_split_tail(enable: int) -> None:
    """1: the forward's CTA-pair GEMMs split their last tiles along K (default); 0: whole tiles."""
    _check(_lib.coda_set_split_tail(int(enable)), "coda_set_split_tail")


def coda_set_col_plan(enable: int) -> None:
    """1 (2): the CTA-pair data gradients may use narrower column tiles, widths in steps of
    16 (64), that spread evenly over the pairs; 0: 256-column tiles (default)."""
    _check(_lib.coda_set_col_plan(int(enable)), "coda_set_col_plan")


def coda_set_serpentine_k(enable: int) -> None:
    """1: the CTA-pair data gradients load every other wave's K blocks backwards; 0: forwards
    (default)."""
    _check(_lib.coda_set_serpentine_k(int(enable)), "coda_set_serpentine_k")


def coda_get_serpentine_k() -> int:
    return int(_lib.coda_get_serpentine_k())


def coda_set_dgrad_pieces(enable: int) -> None:
    """1 (default): the CTA-pair data gradients may cut their last row blocks' tiles into K
    pieces when whole tiles would leave the last wave partly idle; 0: whole tiles."""
    _check(_lib.coda_set_dgrad_pieces(int(enable)), "coda_set_dgrad_pieces")


def coda_get_dgrad_pieces() -> int:
    return int(_lib.coda_get_dgrad_pieces())


def coda_dgrad_piece_plan(M: int, d: int, N1: int, npairs: int, tile_local: bool = False):
    """The data gradient's piece plan on `npairs` CTA pairs as (tiles whole, pieces,
    first levelled pair, levelling pieces per such pair), or None for whole tiles."""
    out = (ctypes.c_int32 * 4)()
    rc = int(_lib.coda_dgrad_piece_plan(M, d, N1, int(npairs), int(bool(tile_local)), out))
    if rc < 0:
        raise ValueError("coda_dgrad_piece_plan: invalid arguments")
    return tuple(int(v) for v in out) if rc == 1 else None


def coda_get_mma_mode() -> int:
    return int(_lib.coda_get_mma_mode())


def coda_set_wait_timeout_ns(ns: int) -> None:
    _lib.coda_set_wait_timeout_ns(int(ns))


def coda_watchdog_selftest(timeout_ns: int, stream=None) -> int:
    return int(_lib.coda_watchdog_selftest(int(timeout_ns), _stream_ptr(stream)))


_events_keepalive = None


def coda_set_launch_events(events) -> None:
    """Measurement hook: record events[k] after the k-th kernel launch of each
    following coda_* call (events: list of torch.cuda.Event, or None)."""
    global _events_keepalive
    if not events:
        _lib.coda_set_launch_events(None, 0)
        _events_keepalive = None
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event lazily, on first record
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[int(e.cuda_event) for e in events])
    _events_keepalive = (arr, events)
    _lib.coda_set_launch_events(ctypes.cast(arr, ctypes.c_void_p), len(events))


def raw() -> ctypes.CDLL:
    """The loaded library (for direct C-ABI calls, e.g. with bad arguments)."""
    return _lib
