"""coda_bwd_dgrad_noalloc: the data gradient for callers that cannot allocate.

Some callers must not allocate device memory when they run the backward (code
inside an allocator or memory-pool callback, runtimes that forbid allocation
mid-step, embedders with all device memory reserved up front).  This entry
point keeps its scratch in a fixed array inside the library instead of a
caller-provided workspace.  The test calls it through the C ABI twice in a
row, on different inputs, and checks each result against coda_bwd_dgrad on
the same inputs and against the fp64 oracle, with the parity tests'
data-gradient tolerance (the two entry points may tile the columns
differently, so they agree up to fp32 summation order).  It checks that a call made after
the library is loaded on the device leaves the device's free memory unchanged,
and that a shape beyond the static maximum is refused without a launch.

The file name makes pytest collect it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
from gemm_epilogue_fusion_gemm0_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_DH = 2e-2


@pytest.fixture(scope="module")
def B():
    import __graft_entry__ as g

    g.build()
    from gemm_epilogue_fusion_gemm0_gb300 import binding

    torch.cuda.set_device(0)
    return binding


def _saved_forward(B, M, d, N1, seed):
    dev = torch.device("cuda:0")
    t = synth.make_forward_inputs(M, d, N1, seed=seed)
    g = {k: v.to(dev) for k, v in t.items() if k != "_rng"}
    h, r, _ = B.coda_fwd(g["x"], g["W0"], g["z"], g["gamma"], g["W1"], 1e-5)
    dy = synth.make_grad_output(t["_rng"], M, N1).to(dev)
    return dy, g["W1"], h, r, g["gamma"]


def _noalloc(B, dy, W1, h, r, gamma, dh):
    M, N1 = dy.shape
    d = W1.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return B.raw().coda_bwd_dgrad_noalloc(
        ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(W1.data_ptr()),
        ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(r.data_ptr()),
        ctypes.c_void_p(gamma.data_ptr()), M, d, N1, ctypes.c_void_p(dh.data_ptr()),
        ctypes.c_void_p(stream))


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def test_noalloc_dgrad_matches_workspace_dgrad_twice(B):
    cases = [(300, 328, 776, 11), (1024, 2048, 4096, 12)]  # ragged, then several tiles
    for (M, d, N1, seed) in cases:
        dy, W1, h, r, gamma = _saved_forward(B, M, d, N1, seed)
        ref = B.coda_bwd_dgrad(dy, W1, h, r, gamma)
        got = torch.full_like(ref, float("nan"))
        assert _noalloc(B, dy, W1, h, r, gamma, got) == B.CODA_OK
        st, detail = B.coda_get_device_status()
        assert st == B.CODA_OK, (B.status_string(st), hex(detail))
        a, b = f64(got), f64(ref)
        assert np.all(np.isfinite(a))
        assert oracle.normwise_rel_err(a, b) <= TOL_DH
        # on its own: the oracle's data gradient from the same saved h, r
        o = oracle.backward_dgrad(f64(dy), f64(W1), f64(h), f64(r), f64(gamma)).dh
        assert oracle.normwise_rel_err(a, o) <= TOL_DH


def test_noalloc_dgrad_leaves_free_device_memory_unchanged(B):
    """Once the library is loaded on the device (any earlier call), a call
    allocates nothing: the device's free memory is the same before and after."""
    M, d, N1 = 640, 512, 1280
    dy, W1, h, r, gamma = _saved_forward(B, M, d, N1, 13)
    dh = torch.empty_like(h)
    assert _noalloc(B, dy, W1, h, r, gamma, dh) == B.CODA_OK  # warm: library loaded
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(2):
        assert _noalloc(B, dy, W1, h, r, gamma, dh) == B.CODA_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert B.coda_get_device_status() == (B.CODA_OK, 0)


def test_noalloc_dgrad_rejects_shapes_beyond_static_scratch(B):
    dev = torch.device("cuda:0")
    bf = torch.bfloat16
    # ceil(8192/256) * 16512 = 528384 partials > 524288: refused before any launch
    M, d, N1 = 16512, 8192, 64
    dy = torch.zeros((M, N1), dtype=bf, device=dev)
    W1 = torch.zeros((d, N1), dtype=bf, device=dev)
    h = torch.zeros((M, d), dtype=bf, device=dev)
    r = torch.ones((M,), dtype=torch.float32, device=dev)
    gamma = torch.ones((d,), dtype=bf, device=dev)
    dh = torch.zeros((M, d), dtype=bf, device=dev)
    assert _noalloc(B, dy, W1, h, r, gamma, dh) == B.CODA_ERR_UNSUPPORTED_SHAPE
    assert B.coda_get_device_status() == (B.CODA_OK, 0)
