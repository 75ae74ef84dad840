"""Seeded synthetic inputs for the GEMM -> residual -> RMSNorm -> GEMM chain.

This module only draws random numbers and rounds them to bfloat16; it holds
none of the chain's arithmetic.  Both the CUDA path (tests, bench) and the
oracle comparison consume exactly the tensors made here.

Distributions (the Llama-shaped workloads the method is evaluated on):
  x, z   ~ N(0, 1)
  W0, W1 ~ N(0, 1/d)         (second argument of N is the variance)
  gamma  = 1 + N(0, 0.1)
  dy     ~ N(0, 1e-2)
Values are drawn as float32 from one ``numpy.random.default_rng(seed)`` in the
fixed order x, z, W0, W1, gamma (then dy), then rounded to bfloat16 with
round-to-nearest-even.  Weights are stored [in, out] (W0 [d, d], W1 [d, N1]).
Workloads too large to draw on the host in seconds (billions of elements) are
drawn on the device instead by ``make_inputs_on_device``: the same
distributions and order from a seeded torch generator (a different stream).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int       # tokens (rows)
    d: int       # hidden size
    N1: int      # output width of the second GEMM
    eps: float

    @property
    def fwd_flops(self) -> int:
        """Algorithmic FLOPs of the forward: the two GEMMs only."""
        return 2 * self.M * self.d * self.d + 2 * self.M * self.d * self.N1

    @property
    def bwd_flops(self) -> int:
        """Algorithmic FLOPs of the data-gradient GEMM dy @ W1^T."""
        return 2 * self.M * self.N1 * self.d


# The five evaluation shapes: tiny, and the hidden sizes of Llama-3-style
# 1B / 7B / 70B models (W1 is the gate|up projection, N1 = 2 * ffn).
WORKLOADS = {
    "tiny": Workload("tiny", 128, 256, 512, 1e-5),
    "llama1b": Workload("llama1b", 8192, 2048, 16384, 1e-5),
    "llama7b": Workload("llama7b", 8192, 4096, 28672, 1e-5),
    "llama70b": Workload("llama70b", 4096, 8192, 57344, 1e-6),
}


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> bfloat16 CPU tensor, round-to-nearest-even."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng, shape, var: float) -> np.ndarray:
    a = rng.standard_normal(shape, dtype=np.float32)
    if var != 1.0:
        a *= np.float32(np.sqrt(var))
    return a


def make_forward_inputs(M: int, d: int, N1: int, seed: int = 0) -> dict:
    """bf16 CPU tensors x [M,d], z [M,d], W0 [d,d], W1 [d,N1], gamma [d]."""
    rng = np.random.default_rng(seed)
    x = to_bf16(_normal(rng, (M, d), 1.0))
    z = to_bf16(_normal(rng, (M, d), 1.0))
    W0 = to_bf16(_normal(rng, (d, d), 1.0 / d))
    W1 = to_bf16(_normal(rng, (d, N1), 1.0 / d))
    gamma = to_bf16(1.0 + _normal(rng, (d,), 0.1))
    return {"x": x, "z": z, "W0": W0, "W1": W1, "gamma": gamma, "_rng": rng}


def make_grad_output(rng_or_seed, M: int, N1: int) -> torch.Tensor:
    """bf16 CPU tensor dy [M, N1] ~ N(0, 1e-2).  Pass the ``_rng`` returned by
    ``make_forward_inputs`` to continue its stream (the documented order)."""
    rng = rng_or_seed
    if not isinstance(rng, np.random.Generator):
        rng = np.random.default_rng(rng_or_seed)
    return to_bf16(_normal(rng, (M, N1), 1e-2))


def make_dgrad_inputs(M: int, d: int, N1: int, seed: int = 0) -> dict:
    """bf16 CPU tensors for a data gradient on its own, without running a
    forward: h [M, d] ~ N(0, 2) (the spread of x @ W0 + z with the forward's
    distributions), W1 [d, N1] ~ N(0, 1/d), gamma [d] = 1 + N(0, 0.1) and
    dy [M, N1] ~ N(0, 1e-2), drawn in that order from default_rng(seed)."""
    rng = np.random.default_rng(seed)
    h = to_bf16(_normal(rng, (M, d), 2.0))
    W1 = to_bf16(_normal(rng, (d, N1), 1.0 / d))
    gamma = to_bf16(1.0 + _normal(rng, (d,), 0.1))
    dy = to_bf16(_normal(rng, (M, N1), 1e-2))
    return {"h": h, "W1": W1, "gamma": gamma, "dy": dy}


def make_residual_grad(rng, M: int, d: int) -> torch.Tensor:
    """bf16 CPU tensor dh_res [M, d] ~ N(0, 1e-2): the gradient reaching h
    through the residual stream; drawn after dy from the same generator."""
    return to_bf16(_normal(rng, (M, d), 1e-2))


def make_down_proj_backward(rng, M: int, N1: int, Dout: int) -> dict:
    """bf16 CPU tensors for the backward through the gated activation and the
    down projection: W2 [N1/2, Dout] ~ N(0, 2/N1) and dout [M, Dout] ~ N(0, 1e-2),
    drawn in that order from `rng` (continue the forward generator)."""
    half = N1 // 2
    W2 = to_bf16(_normal(rng, (half, Dout), 1.0 / half))
    dout = to_bf16(_normal(rng, (M, Dout), 1e-2))
    return {"W2": W2, "dout": dout}


E4M3_MAX = 448.0


def to_e4m3(a: np.ndarray):
    """Per-tensor amax scaling to FP8 E4M3: returns (codes as a float8_e4m3fn
    CPU tensor, scale) with value = code * scale and max |code| = 448."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    scale = float(np.max(np.abs(a))) / E4M3_MAX
    if scale == 0.0:
        scale = 1.0
    codes = torch.from_numpy(a / np.float32(scale)).to(torch.float8_e4m3fn)
    return codes, scale


def make_fp8_forward_inputs(M: int, d: int, N1: int, seed: int = 0) -> dict:
    """The FP8 forward's inputs: the same draws as make_forward_inputs, with x,
    W0 and W1 carried as E4M3 codes plus per-tensor scales; z and gamma bf16.
    The scale of GEMM1's FP8 operand h * gamma is fixed from the input
    distributions: h = x @ W0 + z has variance 2, so 6 standard deviations of h
    times max |gamma| maps to the largest E4M3 code."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (M, d), 1.0)
    z = to_bf16(_normal(rng, (M, d), 1.0))
    W0 = _normal(rng, (d, d), 1.0 / d)
    W1 = _normal(rng, (d, N1), 1.0 / d)
    gamma = to_bf16(1.0 + _normal(rng, (d,), 0.1))
    xq, sx = to_e4m3(x)
    W0q, sW0 = to_e4m3(W0)
    W1q, sW1 = to_e4m3(W1)
    g_amax = float(gamma.abs().max().to(torch.float32))
    s_hg = 6.0 * float(np.sqrt(2.0)) * g_amax / E4M3_MAX
    return {"x_q": xq, "sx": sx, "W0_q": W0q, "sW0": sW0, "W1_q": W1q, "sW1": sW1, "z": z,
            "gamma": gamma, "s_hg": s_hg}


def sample_rows(M: int, n: int, seed: int = 1) -> np.ndarray:
    """Sorted seeded sample of n distinct row indices in [0, M), always
    containing the first row, both sides of the first 128-row tile boundary
    and the last row."""
    must = [r for r in (0, 127, 128, M - 1) if 0 <= r < M]
    if n >= M:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    pool = np.setdiff1d(np.arange(M), np.array(must))
    extra = rng.choice(pool, size=max(0, n - len(set(must))), replace=False)
    return np.unique(np.concatenate([np.array(must, dtype=np.int64), extra]))


def make_inputs_on_device(M: int, d: int, N1: int, seed: int, device) -> dict:
    """bf16 tensors x, z [M,d], W0 [d,d], W1 [d,N1], gamma [d] and dy [M,N1] on
    `device`, with the distributions above, drawn as float32 in that order from
    one ``torch.Generator(device).manual_seed(seed)`` and rounded to bf16."""
    gen = torch.Generator(device=device).manual_seed(seed)

    def normal(shape, var):
        a = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if var != 1.0:
            a.mul_(float(np.float32(np.sqrt(var))))
        return a.to(torch.bfloat16)

    x = normal((M, d), 1.0)
    z = normal((M, d), 1.0)
    W0 = normal((d, d), 1.0 / d)
    W1 = normal((d, N1), 1.0 / d)
    gamma = (1.0 + torch.randn((d,), generator=gen, device=device, dtype=torch.float32)
             * float(np.float32(np.sqrt(0.1)))).to(torch.bfloat16)
    dy = normal((M, N1), 1e-2)
    return {"x": x, "z": z, "W0": W0, "W1": W1, "gamma": gamma, "dy": dy}
