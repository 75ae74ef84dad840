"""Parity cases run against the checked build (libcoda_checked.so).

Run by tests/test_checked_build.py in a child process with
CODA_CHECKED_BUILD=1, so that the binding loads the library compiled with
-DCODA_CHECKED: every staged epilogue load and store, gamma load, TMA box
start and workspace index is checked on the device, and a failed check records
CODA_ERR_DEVICE_BOUNDS in the status word instead of touching memory.  Every
case below compares with the fp64 oracle (the parity tests' own helpers and
tolerances) and then requires a clean status word.  Prints one line per case
and "checked cases ok" at the end; exits non-zero on the first failure.
"""

import ctypes
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)
sys.path.insert(0, HERE)

import torch  # noqa: E402

import test_parity_gpu as T  # noqa: E402  (the parity tests' helpers and shapes)
from gemm_epilogue_fusion_gemm0_gb300 import binding as B  # noqa: E402
from gemm_epilogue_fusion_gemm0_gb300 import synth  # noqa: E402
from gemm_epilogue_fusion_gemm0_gb300.build import LIB_PATH_CHECKED  # noqa: E402


def clean(name):
    st, detail = B.coda_get_device_status()
    assert st == B.CODA_OK, (name, B.status_string(st), hex(detail))
    print("ok", name, flush=True)


def noalloc(M, d, N1, seed):
    dev = torch.device("cuda:0")
    t = synth.make_forward_inputs(M, d, N1, seed=seed)
    g = {k: v.to(dev) for k, v in t.items() if k != "_rng"}
    h, r, _ = B.coda_fwd(g["x"], g["W0"], g["z"], g["gamma"], g["W1"], 1e-5)
    dy_cpu = synth.make_grad_output(t["_rng"], M, N1)
    dy = dy_cpu.to(dev)
    dh = torch.empty_like(h)
    st = B.raw().coda_bwd_dgrad_noalloc(
        ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(g["W1"].data_ptr()),
        ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(r.data_ptr()),
        ctypes.c_void_p(g["gamma"].data_ptr()), M, d, N1, ctypes.c_void_p(dh.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == B.CODA_OK, st
    bref = T.oracle.backward_dgrad(T.f64(dy_cpu), T.f64(t["W1"]), T.f64(h), T.f64(r), T.f64(t["gamma"]))
    T.check("dh (no allocation)", T.f64(dh), bref.dh, T.TOL_DH)


def main():
    assert os.environ.get("CODA_CHECKED_BUILD") == "1" and B.LIB == LIB_PATH_CHECKED, B.LIB
    torch.cuda.set_device(0)
    small = [(128, 256, 512), (300, 328, 776), (640, 512, 1280), (1, 8, 8), (129, 64, 264)]
    for mode in (0, 1):
        B.coda_set_mma_mode(mode)
        for (M, d, N1) in small:
            T.run_case(B, M, d, N1, 1e-5)
            clean(f"fwd + dgrad {M}x{d}x{N1} mode {mode}")
        T.run_swiglu(B, 300, 328, 784, 1e-5)
        clean(f"swiglu fwd mode {mode}")
        T.run_swiglu_bwd(B, 300, 328, 784, 264, 1e-5)
        clean(f"swiglu bwd mode {mode}")
        T.run_full_bwd(B, 300, 328, 776, 1e-5)
        clean(f"full bwd mode {mode}")
        T.test_workspace_shared_across_shapes_and_entry_points(B, mode)
        clean(f"one workspace for several shapes mode {mode}")
    B.coda_set_mma_mode(1)
    T.run_fp8(B, 300, 336, 784, 1e-5)
    clean("fp8 fwd")
    for (M, d, N1) in T.SPLIT_SHAPES:
        T.test_split_tail_forward_matches_oracle(B, M, d, N1)
        clean(f"split tail {M}x{d}x{N1}")
    T.test_one_workspace_for_split_forward_and_dgrad(B)
    clean("one workspace for a split forward and the dgrad")
    for shape, slots in T.PIECE_SHAPES:
        T.test_dgrad_pieces_match_oracle(B, shape, slots)
        clean(f"dgrad in K pieces {shape}")
    for shape in T.SWIGLU_PIECE_SHAPES:
        T.test_swiglu_backward_in_pieces_matches_oracle(B, *shape)
        clean(f"swiglu backward in K pieces {shape}")
    for (M, d, N1) in T.SWEEP_SHAPES[:4]:
        T.test_split_tail_shape_sweep(B, M, d, N1)
        clean(f"split sweep {M}x{d}x{N1}")
    for (M, d, N1) in T.PLAN_SHAPES:
        T.test_dgrad_column_plans_match_oracle(B, M, d, N1)
        clean(f"column plan {M}x{d}x{N1}")
    for (M, d, N1, seed) in [(300, 328, 776, 11), (1024, 2048, 4096, 12)]:
        noalloc(M, d, N1, seed)
        clean(f"no-allocation dgrad {M}x{d}x{N1}")
    print("checked cases ok", flush=True)


if __name__ == "__main__":
    main()
