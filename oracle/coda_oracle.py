"""Plain fp64 CPU oracle of the CODA GEMM -> residual -> RMSNorm -> GEMM chain.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``, never by the library.

What it computes is the *unfused* definition of the chain, step by step, in
float64 with numpy (``@`` is the only library primitive used).  No blocking,
fusion or reordering is done here; the GPU path's reparameterised form
``y = r * ((h * gamma) @ W1)`` is deliberately NOT used, so that the oracle can
check it.

Sources (web pages on the method; cited by title and section):

* [CODA-blog] "CODA：将 Transformer 块重写为 GEMM-Epilogue 程序以消除显存瓶颈"
  (blog.hotdry.top), section "GEMM-Residual-RMSNorm-GEMM 重参数化": the chain
  y = RMSNorm(x @ W0 + z, gamma) @ W1 with a per-row inverse-RMS factor r.
* [CODA-blog], section "反向传播的 GEMM-Epilogue 结构": the row statistic
  s = sum over columns of (grad_h2 * h2) = sum over columns of (grad_y * y).
* The RMSNorm backward itself is textbook calculus: with
  r = (mean_j h_j^2 + eps)^(-1/2) one has dr/dh_j = -r^3 h_j / d.

Readings where the pages are silent (each also listed in the design notes):

* the mean of h^2 is taken over the d features, and eps sits inside the
  square root (standard RMSNorm);
* r multiplies the row *after* the residual add and *before* gamma; gamma is
  an elementwise weight over the d features;
* the backward returns the RMSNorm-branch gradient only (no upstream residual
  gradient is added) and uses the r it is given, as saved by the forward.

Inputs are float64 arrays (the GPU's bf16 tensors widened exactly).  Rows are
independent, so callers may pass any subset of rows of x, z, h, r and grad_y.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class ForwardResult:
    h: np.ndarray   # [M, d]  new residual stream x @ W0 + z
    r: np.ndarray   # [M]     inverse RMS factor per row
    y: np.ndarray   # [M, N1] RMSNorm(h, gamma) @ W1


@dataclass
class FullBackwardResult:
    dh: np.ndarray      # [M, d]  total gradient at h (RMSNorm branch + upstream residual); = dz
    dx: np.ndarray      # [M, d]
    dgamma: np.ndarray  # [d]
    dW0: np.ndarray     # [d, d]
    dW1: np.ndarray     # [d, N1]
    h2: np.ndarray      # [M, d]  normalised activation RMSNorm(h, gamma)


@dataclass
class BackwardResult:
    dh: np.ndarray   # [M, d]  gradient w.r.t. h through the RMSNorm branch
    s: np.ndarray    # [M]     row statistic sum_j grad_h2 * h2
    dh2: np.ndarray  # [M, d]  gradient w.r.t. the normalised activation h2


def _f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return a


def residual_gemm(x, W0, z) -> np.ndarray:
    """h = x @ W0 + z  ([CODA-blog] reparameterisation section, inner term
    of RMSNorm(x @ W0 + z, gamma)).  W0 is stored [in, out]."""
    return _f64(x) @ _f64(W0) + _f64(z)


def mean_square(h) -> np.ndarray:
    """ms[m] = (1/d) * sum_j h[m, j]^2 -- mean over the d features."""
    h = _f64(h)
    return np.sum(h * h, axis=1) / h.shape[1]


def inverse_rms(ms, eps: float) -> np.ndarray:
    """r[m] = 1 / sqrt(ms[m] + eps), the per-row inverse RMS factor
    ([CODA-blog] reparameterisation section)."""
    return 1.0 / np.sqrt(_f64(ms) + float(eps))


def rmsnorm(h, gamma, r) -> np.ndarray:
    """h2 = RMSNorm(h, gamma) = (r[m] * h[m, j]) * gamma[j]."""
    return (_f64(r)[:, None] * _f64(h)) * _f64(gamma)[None, :]


def forward(x, W0, z, gamma, W1, eps: float) -> ForwardResult:
    """Unfused forward y = RMSNorm(x @ W0 + z, gamma) @ W1.

    Steps, in the order the definition gives them:
      1. h  = x @ W0 + z
      2. ms = mean_j h^2
      3. r  = 1 / sqrt(ms + eps)
      4. h2 = r * h * gamma
      5. y  = h2 @ W1            (W1 stored [in, out])
    """
    h = residual_gemm(x, W0, z)
    r = inverse_rms(mean_square(h), eps)
    h2 = rmsnorm(h, gamma, r)
    y = h2 @ _f64(W1)
    return ForwardResult(h=h, r=r, y=y)


def backward_dgrad(dy, W1, h, r, gamma) -> BackwardResult:
    """RMSNorm-branch data gradient of the chain, given the saved h and r.

    Steps:
      1. dh2 = dy @ W1^T                       (the dgrad GEMM)
      2. g   = gamma * dh2                     (through the elementwise weight)
      3. dh  = r * g - (r^3 / d) * h * sum_j g_j h_j
             (chain rule through r = (mean h^2 + eps)^(-1/2))
    Also returns s = sum_j dh2_j * h2_j, the row statistic that [CODA-blog]
    ("反向传播的 GEMM-Epilogue 结构") moves to the GEMM boundary; s equals
    r * sum_j g_j h_j, so dh = r * g - (r^2 * s / d) * h.
    """
    dy = _f64(dy)
    h = _f64(h)
    r = _f64(r)
    gamma = _f64(gamma)
    d = h.shape[1]
    dh2 = dy @ _f64(W1).T
    g = gamma[None, :] * dh2
    gh = np.sum(g * h, axis=1)
    dh = r[:, None] * g - ((r ** 3) / d * gh)[:, None] * h
    s = np.sum(dh2 * rmsnorm(h, gamma, r), axis=1)
    return BackwardResult(dh=dh, s=s, dh2=dh2)


def backward_full(dy, x, W0, W1, h, r, gamma, dh_res=None) -> FullBackwardResult:
    """All gradients of the chain h = x @ W0 + z, y = RMSNorm(h, gamma) @ W1,
    given dy, the saved h and r, and optionally the gradient dh_res that
    reaches h through the residual stream.

    Steps:
      1. dh2, dh (RMSNorm branch) from backward_dgrad
      2. dh_tot = dh + dh_res                       (= dz, since h = ... + z)
      3. h2 = RMSNorm(h, gamma);  dgamma = sum_m dh2 * (r * h)  (dh2/dgamma_j = r h_j)
      4. dW1 = h2^T dy
      5. dx = dh_tot @ W0^T,  dW0 = x^T dh_tot
    """
    b = backward_dgrad(dy, W1, h, r, gamma)
    dh_tot = b.dh if dh_res is None else b.dh + _f64(dh_res)
    h = _f64(h)
    r = _f64(r)
    h2 = rmsnorm(h, gamma, r)
    dgamma = np.sum(b.dh2 * (r[:, None] * h), axis=0)
    dW1 = h2.T @ _f64(dy)
    dx = dh_tot @ _f64(W0).T
    dW0 = _f64(x).T @ dh_tot
    return FullBackwardResult(dh=dh_tot, dx=dx, dgamma=dgamma, dW0=dW0, dW1=dW1, h2=h2)


def silu(t) -> np.ndarray:
    """silu(t) = t * sigmoid(t) = t / (1 + exp(-t))."""
    t = _f64(t)
    with np.errstate(over="ignore"):
        return t / (1.0 + np.exp(-t))


def swiglu(y) -> np.ndarray:
    """Gated activation on a [gate | up] pre-activation (CODA blog, section
    "五类 Epilogue 原语", SwiGLU gating; the pairing is the one of section
    "成对激活的寄存器级融合"): with y = [g | u] split into two equal column
    halves, a[:, j] = silu(g[:, j]) * u[:, j]."""
    y = _f64(y)
    half = y.shape[1] // 2
    return silu(y[:, :half]) * y[:, half:]


def forward_swiglu(x, W0, z, gamma, W1, eps: float):
    """The chain followed by the gated activation: returns (ForwardResult, a)
    with a = swiglu(RMSNorm(x @ W0 + z, gamma) @ W1), W1 = [W_gate | W_up]."""
    f = forward(x, W0, z, gamma, W1, eps)
    return f, swiglu(f.y)


def backward_swiglu(dout, W2, y):
    """Backward of out = swiglu(y) @ W2 to the pre-activation y = [g | u].

    Steps:
      1. da = dout @ W2^T                        (W2 stored [in = N1/2, out])
      2. dg = da * u * silu'(g),  du = da * silu(g)
         with silu'(t) = sig(t) * (1 + t * (1 - sig(t))), sig the logistic
      3. dy = [dg | du]
    Also returns s = sum_n dy[:, n] * y[:, n], the row statistic of the RMSNorm
    backward, formed where dy and y meet (CODA blog, section
    "反向传播的 GEMM-Epilogue 结构": s = sum_cols(grad_y * y))."""
    dout = _f64(dout)
    y = _f64(y)
    half = y.shape[1] // 2
    g, u = y[:, :half], y[:, half:]
    da = dout @ _f64(W2).T
    with np.errstate(over="ignore"):
        sig = 1.0 / (1.0 + np.exp(-g))
    dg = da * u * sig * (1.0 + g * (1.0 - sig))
    du = da * g * sig
    dy = np.concatenate([dg, du], axis=1)
    s = np.sum(dy * y, axis=1)
    return dy, s


def backward_rmsnorm_given_s(dh2, h, r, gamma, s):
    """RMSNorm-branch backward with the row statistic supplied from outside:
    dh = r * gamma * dh2 - (r^2 * s / d) * h.  Equal to backward_dgrad's dh when
    s = sum_j dh2_j * h2_j (the identity r * sum(g * h) = s)."""
    dh2 = _f64(dh2)
    h = _f64(h)
    r = _f64(r)
    d = h.shape[1]
    return r[:, None] * _f64(gamma)[None, :] * dh2 - ((r ** 2) * _f64(s) / d)[:, None] * h


E4M3_MAX = 448.0


def round_e4m3(v) -> np.ndarray:
    """Round to the nearest FP8 E4M3 value (ties to even), saturating at +-448.

    E4M3 (the 'fn' variant: no infinities): 1 sign bit, 4 exponent bits with
    bias 7, 3 mantissa bits.  Normal values have |v| >= 2^-6 and spacing
    2^(e - 3) in the binade [2^e, 2^(e+1)); below 2^-6 the spacing is the
    subnormal step 2^-9."""
    v = _f64(v)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)              # subnormal range shares the 2^-9 step
    step = np.exp2(e - 3.0)
    q = np.round(a / step) * step        # numpy rounds half to even
    q = np.minimum(q, E4M3_MAX)
    return np.sign(v) * q


def forward_fp8(x_q, sx, W0_q, sW0, z, gamma, W1_q, sW1, s_hg, eps: float):
    """The chain with FP8 (E4M3) operands and per-tensor scales; the values of
    the FP8 tensors are code * scale.

    Steps:
      1. h  = (x_q sx) @ (W0_q sW0) + z
      2. r  = 1 / sqrt(mean_j h^2 + eps)
      3. hq = round_e4m3(h * gamma / s_hg)    (GEMM1's operand, quantised once)
      4. y  = r * ((hq s_hg) @ (W1_q sW1))
    Returns (ForwardResult, hq)."""
    h = (_f64(x_q) * sx) @ (_f64(W0_q) * sW0) + _f64(z)
    r = inverse_rms(mean_square(h), eps)
    hq = round_e4m3(h * _f64(gamma)[None, :] / s_hg)
    y = r[:, None] * ((hq * s_hg) @ (_f64(W1_q) * sW1))
    return ForwardResult(h=h, r=r, y=y), hq


def normwise_rel_err(got, ref) -> float:
    """||got - ref||_F / ||ref||_F in float64 (the parity metric)."""
    got = _f64(got)
    ref = _f64(ref)
    num = np.linalg.norm((got - ref).ravel())
    den = np.linalg.norm(ref.ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)
