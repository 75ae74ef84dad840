"""Oracle for the CODA GEMM -> residual -> RMSNorm -> GEMM chain.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import anything from this
package.  The CUDA library never calls it, and nothing here calls the CUDA
library: the two share no code.
"""

from .coda_oracle import (  # noqa: F401
    ForwardResult,
    BackwardResult,
    FullBackwardResult,
    backward_full,
    round_e4m3,
    forward_fp8,
    E4M3_MAX,
    residual_gemm,
    mean_square,
    inverse_rms,
    rmsnorm,
    forward,
    backward_dgrad,
    normwise_rel_err,
    silu,
    swiglu,
    forward_swiglu,
    backward_swiglu,
    backward_rmsnorm_given_s,
)
