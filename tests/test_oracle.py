"""Pins for the fp64 oracle (CPU only).

The oracle is checked against things other than itself:
  * a hand-worked example with exact closed-form answers (tests/golden),
  * brute-force scalar loops on tiny shapes,
  * library routines: torch.nn.functional.rms_norm and torch autograd (fp64),
  * central finite differences of the loss sum(dy * y),
  * invariants: unit RMS before gamma when eps = 0, scale invariance of the
    RMSNorm backward, the reparameterisation identity
    r * ((h * gamma) @ W1) == RMSNorm(h, gamma) @ W1 and the row-statistic
    identity sum(dy * y) == sum(dh2 * h2) (CODA blog, blog.hotdry.top,
    sections "GEMM-Residual-RMSNorm-GEMM 重参数化" and
    "反向传播的 GEMM-Epilogue 结构").
The last test plants plausible mistakes in the oracle and checks that each
one is caught by at least one of these pins.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import coda_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")

TINY_SHAPES = [(1, 1, 1), (2, 3, 4), (3, 8, 5), (5, 17, 7), (4, 33, 3), (7, 6, 33)]


def _exact(expr: str) -> float:
    """Evaluate 'p/q' or 'sqrt(a/b)*p/q' exactly (Fraction + one sqrt)."""
    expr = expr.replace(" ", "")
    if expr.startswith("sqrt("):
        inner, rest = expr[5:].split(")", 1)
        root = math.sqrt(Fraction(inner))
        mult = Fraction(rest[1:]) if rest.startswith("*") else Fraction(1)
        return root * float(mult)
    return float(Fraction(expr))


def _rand_case(rng, M, d, N1, eps=None):
    x = rng.standard_normal((M, d))
    z = rng.standard_normal((M, d))
    W0 = rng.standard_normal((d, d)) / math.sqrt(d)
    W1 = rng.standard_normal((d, N1)) / math.sqrt(d)
    gamma = 1.0 + 0.3 * rng.standard_normal(d)
    dy = 0.1 * rng.standard_normal((M, N1))
    if eps is None:
        eps = float(rng.choice([0.0, 1e-6, 1e-5, 0.5]))
    return x, W0, z, gamma, W1, dy, eps


# ----------------------------------------------------------------------------
# pin checks (each raises AssertionError on a mismatch); reused by the
# planted-mistake test below
# ----------------------------------------------------------------------------

def pin_golden():
    g = json.load(open(GOLDEN))
    f = O.forward(g["x"], g["W0"], g["z"], g["gamma"], g["W1"], g["eps"])
    ex = g["expected"]
    ev = np.vectorize(_exact, otypes=[float])
    np.testing.assert_allclose(f.h, ev(np.array(ex["h"])), rtol=1e-14, atol=0)
    np.testing.assert_allclose(f.r, ev(np.array(ex["r"])), rtol=1e-14, atol=0)
    np.testing.assert_allclose(f.y, ev(np.array(ex["y"])), rtol=1e-13, atol=1e-15)
    b = O.backward_dgrad(g["dy"], g["W1"], f.h, f.r, g["gamma"])
    np.testing.assert_allclose(b.dh, ev(np.array(ex["dh"])), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(b.s, ev(np.array(ex["s"])), rtol=1e-13, atol=0)


def _brute_forward(x, W0, z, gamma, W1, eps):
    M, d = len(x), len(W0)
    N1 = len(W1[0])
    h = [[0.0] * d for _ in range(M)]
    for m in range(M):
        for j in range(d):
            acc = 0.0
            for k in range(d):
                acc += x[m][k] * W0[k][j]
            h[m][j] = acc + z[m][j]
    r = []
    for m in range(M):
        ss = 0.0
        for j in range(d):
            ss += h[m][j] * h[m][j]
        r.append(1.0 / math.sqrt(ss / d + eps))
    y = [[0.0] * N1 for _ in range(M)]
    for m in range(M):
        for n in range(N1):
            acc = 0.0
            for j in range(d):
                acc += (h[m][j] * r[m] * gamma[j]) * W1[j][n]
            y[m][n] = acc
    return np.array(h), np.array(r), np.array(y)


def _brute_backward(dy, W1, h, r, gamma):
    M, d = len(h), len(h[0])
    N1 = len(W1[0])
    dh = np.zeros((M, d))
    for m in range(M):
        dh2 = [0.0] * d
        for j in range(d):
            acc = 0.0
            for n in range(N1):
                acc += dy[m][n] * W1[j][n]
            dh2[j] = acc
        # d/dh_i of sum_j dh2_j * gamma_j * h_j * r(h), r = (sum h^2/d + eps)^-1/2
        dot = 0.0
        for j in range(d):
            dot += dh2[j] * gamma[j] * h[m][j]
        for i in range(d):
            drdhi = -(r[m] ** 3) * h[m][i] / d
            dh[m][i] = dh2[i] * gamma[i] * r[m] + dot * drdhi
    return dh


def pin_bruteforce(seed=0):
    rng = np.random.default_rng(seed)
    for (M, d, N1) in TINY_SHAPES:
        x, W0, z, gamma, W1, dy, eps = _rand_case(rng, M, d, N1)
        f = O.forward(x, W0, z, gamma, W1, eps)
        h, r, y = _brute_forward(x.tolist(), W0.tolist(), z.tolist(), gamma.tolist(), W1.tolist(), eps)
        np.testing.assert_allclose(f.h, h, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(f.r, r, rtol=1e-12, atol=0)
        np.testing.assert_allclose(f.y, y, rtol=1e-11, atol=1e-12)
        b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)
        dh = _brute_backward(dy.tolist(), W1.tolist(), f.h.tolist(), f.r.tolist(), gamma.tolist())
        np.testing.assert_allclose(b.dh, dh, rtol=1e-10, atol=1e-12)


def pin_torch_library(seed=1):
    """torch.nn.functional.rms_norm and autograd in fp64 on the CPU."""
    rng = np.random.default_rng(seed)
    for (M, d, N1) in [(6, 16, 9), (3, 40, 24), (8, 5, 5)]:
        x, W0, z, gamma, W1, dy, eps = _rand_case(rng, M, d, N1, eps=1e-5)
        f = O.forward(x, W0, z, gamma, W1, eps)
        th = torch.tensor(x) @ torch.tensor(W0) + torch.tensor(z)
        th.requires_grad_(True)
        ty = torch.nn.functional.rms_norm(th, (d,), weight=torch.tensor(gamma), eps=eps) @ torch.tensor(W1)
        np.testing.assert_allclose(f.h, th.detach().numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(f.y, ty.detach().numpy(), rtol=1e-10, atol=1e-12)
        ty.backward(torch.tensor(dy))
        b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)
        np.testing.assert_allclose(b.dh, th.grad.numpy(), rtol=1e-9, atol=1e-12)


def pin_finite_differences(seed=2):
    """Central differences of L(h) = sum(dy * y(h)), r recomputed from h."""
    rng = np.random.default_rng(seed)
    M, d, N1 = 3, 6, 5
    x, W0, z, gamma, W1, dy, eps = _rand_case(rng, M, d, N1, eps=1e-3)
    f = O.forward(x, W0, z, gamma, W1, eps)
    b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)

    def loss(h):
        r = 1.0 / np.sqrt(np.mean(h * h, axis=1) + eps)
        return float(np.sum(dy * ((r[:, None] * h * gamma) @ W1)))

    step = 1e-6
    fd = np.zeros_like(f.h)
    for m in range(M):
        for j in range(d):
            hp = f.h.copy()
            hm = f.h.copy()
            hp[m, j] += step
            hm[m, j] -= step
            fd[m, j] = (loss(hp) - loss(hm)) / (2 * step)
    np.testing.assert_allclose(b.dh, fd, rtol=1e-5, atol=1e-8)


def pin_invariants(seed=3):
    rng = np.random.default_rng(seed)
    for (M, d, N1) in [(5, 12, 7), (4, 64, 16)]:
        # eps = 0: RMSNorm before gamma has unit RMS, and the backward is
        # orthogonal to h (RMSNorm is scale invariant).
        x, W0, z, gamma, W1, dy, _ = _rand_case(rng, M, d, N1)
        f = O.forward(x, W0, z, gamma, W1, 0.0)
        u = f.r[:, None] * f.h
        np.testing.assert_allclose(np.sqrt(np.mean(u * u, axis=1)), 1.0, rtol=1e-13)
        b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)
        scale = np.linalg.norm(f.h, axis=1) * np.linalg.norm(b.dh, axis=1)
        assert np.all(np.abs(np.sum(f.h * b.dh, axis=1)) <= 1e-12 * scale + 1e-300)
        # eps > 0: sum_j h_j dh_j = r * sum(g*h) * eps / (ms + eps)
        eps = 0.25
        f = O.forward(x, W0, z, gamma, W1, eps)
        b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)
        ms = np.mean(f.h * f.h, axis=1)
        gh = np.sum(gamma * b.dh2 * f.h, axis=1)
        np.testing.assert_allclose(np.sum(f.h * b.dh, axis=1), f.r * gh * eps / (ms + eps),
                                   rtol=1e-10, atol=1e-13)
        # rms(r*h) = sqrt(ms / (ms + eps))
        u = f.r[:, None] * f.h
        np.testing.assert_allclose(np.sqrt(np.mean(u * u, axis=1)), np.sqrt(ms / (ms + eps)), rtol=1e-13)


def pin_reparameterisation(seed=4):
    """r * ((h * gamma) @ W1) == RMSNorm(h, gamma) @ W1, and
    sum(dy * y) == sum(dh2 * h2) == s (the two identities of the method)."""
    rng = np.random.default_rng(seed)
    for (M, d, N1) in [(6, 10, 12), (3, 32, 64)]:
        x, W0, z, gamma, W1, dy, eps = _rand_case(rng, M, d, N1, eps=1e-5)
        f = O.forward(x, W0, z, gamma, W1, eps)
        fused = f.r[:, None] * ((f.h * gamma[None, :]) @ W1)
        np.testing.assert_allclose(fused, f.y, rtol=1e-11, atol=1e-13)
        b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)
        np.testing.assert_allclose(np.sum(dy * f.y, axis=1), b.s, rtol=1e-10, atol=1e-13)


def pin_special_case_plain_rmsnorm(seed=5):
    """W0 = I, z = 0, gamma = 1, W1 = I reduces the chain to a plain RMSNorm
    of x (checked against torch's rms_norm)."""
    rng = np.random.default_rng(seed)
    M, d = 4, 24
    x = rng.standard_normal((M, d))
    eye = np.eye(d)
    for eps in (0.0, 1e-5):
        f = O.forward(x, eye, np.zeros((M, d)), np.ones(d), eye, eps)
        ref = torch.nn.functional.rms_norm(torch.tensor(x), (d,), eps=eps).numpy()
        np.testing.assert_allclose(f.y, ref, rtol=1e-12, atol=1e-14)


ALL_PINS = [pin_golden, pin_bruteforce, pin_torch_library, pin_finite_differences,
            pin_invariants, pin_reparameterisation, pin_special_case_plain_rmsnorm]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin()


def test_normwise_rel_err():
    a = np.array([[3.0, 4.0]])
    assert O.normwise_rel_err(a, a) == 0.0
    assert abs(O.normwise_rel_err(a + np.array([[0.0, 0.5]]), a) - 0.1) < 1e-15


def test_oracle_rows_are_independent():
    """Row subsets give exactly the rows of the full result (parity at full
    size relies on this)."""
    rng = np.random.default_rng(7)
    x, W0, z, gamma, W1, dy, eps = _rand_case(rng, 9, 16, 8, eps=1e-5)
    full = O.forward(x, W0, z, gamma, W1, eps)
    rows = np.array([0, 4, 8])
    sub = O.forward(x[rows], W0, z[rows], gamma, W1, eps)
    np.testing.assert_array_equal(sub.y, full.y[rows])
    np.testing.assert_array_equal(sub.r, full.r[rows])


# ----------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# ----------------------------------------------------------------------------

def _bwd_mutant(kind):
    def bwd(dy, W1, h, r, gamma):
        dy, h, r, gamma = (np.asarray(a, dtype=np.float64) for a in (dy, h, r, gamma))
        d = h.shape[1]
        dh2 = dy @ np.asarray(W1, dtype=np.float64).T
        g = dh2 if kind == "no_gamma" else gamma[None, :] * dh2
        gh = np.sum(g * h, axis=1)
        p = 2 if kind == "r_squared" else 3
        coef = ((r ** p) / d * gh)[:, None] * h
        dh = r[:, None] * g + coef if kind == "sign" else r[:, None] * g - coef
        if kind == "dropped_term":
            dh = r[:, None] * g
        s = np.sum(dh2 * O.rmsnorm(h, gamma, r), axis=1)
        return O.BackwardResult(dh=dh, s=s, dh2=dh2)
    return bwd


MUTANTS = {
    "dropped_residual": ("residual_gemm", lambda x, W0, z: np.asarray(x, float) @ np.asarray(W0, float)),
    "transposed_W0": ("residual_gemm",
                      lambda x, W0, z: np.asarray(x, float) @ np.asarray(W0, float).T + np.asarray(z, float)),
    "mean_over_d_minus_1": ("mean_square",
                            lambda h: np.sum(np.asarray(h, float) ** 2, axis=1) / max(np.shape(h)[1] - 1, 1)),
    "eps_outside_sqrt": ("inverse_rms", lambda ms, eps: 1.0 / np.sqrt(np.asarray(ms, float)) + eps),
    "dropped_gamma": ("rmsnorm", lambda h, gamma, r: np.asarray(r, float)[:, None] * np.asarray(h, float)),
    "bwd_sign": ("backward_dgrad", _bwd_mutant("sign")),
    "bwd_r_squared": ("backward_dgrad", _bwd_mutant("r_squared")),
    "bwd_no_gamma": ("backward_dgrad", _bwd_mutant("no_gamma")),
    "bwd_dropped_term": ("backward_dgrad", _bwd_mutant("dropped_term")),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(O, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} was not caught by any pin"


# ----------------------------------------------------------------------------
# SwiGLU extension (gated activation on the [gate | up] output of the chain)
# ----------------------------------------------------------------------------

def pin_swiglu_bruteforce(seed=8):
    rng = np.random.default_rng(seed)
    for (M, d, N1) in [(3, 5, 4), (4, 9, 10), (2, 16, 32)]:
        x, W0, z, gamma, W1, _, eps = _rand_case(rng, M, d, N1, eps=1e-5)
        f, a = O.forward_swiglu(x, W0, z, gamma, W1, eps)
        _, _, y = _brute_forward(x.tolist(), W0.tolist(), z.tolist(), gamma.tolist(), W1.tolist(), eps)
        half = N1 // 2
        ref = np.zeros((M, half))
        for m in range(M):
            for j in range(half):
                g, u = y[m][j], y[m][half + j]
                ref[m, j] = g / (1.0 + math.exp(-g)) * u
        np.testing.assert_allclose(a, ref, rtol=1e-11, atol=1e-13)


def pin_swiglu_library(seed=9):
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((7, 12)) * 3.0
    ref = (torch.nn.functional.silu(torch.tensor(y[:, :6])) * torch.tensor(y[:, 6:])).numpy()
    np.testing.assert_allclose(O.swiglu(y), ref, rtol=1e-13, atol=1e-15)


def pin_swiglu_closed_forms():
    # silu(0) = 0; silu(t) -> t for t >> 0, -> 0 for t << 0; up = 1 gives silu(gate)
    y = np.array([[0.0, 50.0, -50.0, 1.0, 2.0, 3.0, 4.0, 1.0]])
    a = O.swiglu(y)
    assert a[0, 0] == 0.0
    np.testing.assert_allclose(a[0, 1], 50.0 * 3.0, rtol=1e-15)  # gate 50, up 3
    assert abs(a[0, 2]) < 1e-18
    np.testing.assert_allclose(a[0, 3], 1.0 / (1.0 + math.exp(-1.0)), rtol=1e-15)
    # the gate is the first half and the up projection the second half
    assert O.swiglu(np.array([[1.0, 0.0]]))[0, 0] == 0.0


SWIGLU_PINS = [pin_swiglu_bruteforce, pin_swiglu_library, pin_swiglu_closed_forms]


@pytest.mark.parametrize("pin", SWIGLU_PINS, ids=lambda p: p.__name__)
def test_swiglu_pin(pin):
    pin()


@pytest.mark.parametrize("name,fn", [
    ("gate_up_swapped", lambda y: O.silu(np.asarray(y, float)[:, np.asarray(y).shape[1] // 2:])
     * np.asarray(y, float)[:, :np.asarray(y).shape[1] // 2]),
    ("interleaved_pairs", lambda y: O.silu(np.asarray(y, float)[:, 0::2]) * np.asarray(y, float)[:, 1::2]),
    ("sigmoid_not_silu", lambda y: 1.0 / (1.0 + np.exp(-np.asarray(y, float)[:, :np.asarray(y).shape[1] // 2]))
     * np.asarray(y, float)[:, np.asarray(y).shape[1] // 2:]),
])
def test_swiglu_planted_mistake_is_caught(name, fn, monkeypatch):
    monkeypatch.setattr(O, "swiglu", fn)
    failed = []
    for pin in SWIGLU_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} was not caught"


# ----------------------------------------------------------------------------
# SwiGLU backward and the statistic formed upstream
# ----------------------------------------------------------------------------

def _swiglu_case(rng, M=4, half=5, dout_w=6):
    y = rng.standard_normal((M, 2 * half)) * 2.0
    W2 = rng.standard_normal((half, dout_w)) / math.sqrt(half)
    dout = rng.standard_normal((M, dout_w)) * 0.3
    return y, W2, dout


def pin_swiglu_bwd_autograd(seed=10):
    """torch autograd of out = (silu(g) * u) @ W2 in fp64."""
    rng = np.random.default_rng(seed)
    for shape in [(4, 5, 6), (3, 16, 8)]:
        y, W2, dout = _swiglu_case(rng, *shape)
        ty = torch.tensor(y, requires_grad=True)
        half = y.shape[1] // 2
        out = (torch.nn.functional.silu(ty[:, :half]) * ty[:, half:]) @ torch.tensor(W2)
        out.backward(torch.tensor(dout))
        dy, s = O.backward_swiglu(dout, W2, y)
        np.testing.assert_allclose(dy, ty.grad.numpy(), rtol=1e-11, atol=1e-13)


def pin_swiglu_bwd_finite_differences(seed=11):
    rng = np.random.default_rng(seed)
    y, W2, dout = _swiglu_case(rng, 3, 4, 5)
    dy, _ = O.backward_swiglu(dout, W2, y)
    half = y.shape[1] // 2

    def loss(yy):
        return float(np.sum(dout * ((yy[:, :half] / (1 + np.exp(-yy[:, :half]))) * yy[:, half:] @ W2)))

    fd = np.zeros_like(y)
    for i in range(y.shape[0]):
        for j in range(y.shape[1]):
            yp, ym = y.copy(), y.copy()
            yp[i, j] += 1e-6
            ym[i, j] -= 1e-6
            fd[i, j] = (loss(yp) - loss(ym)) / 2e-6
    np.testing.assert_allclose(dy, fd, rtol=1e-6, atol=1e-9)


def pin_statistic_upstream_equals_definition(seed=12):
    """s formed upstream (sum dy * y) equals sum_j dh2_j h2_j of the definition,
    and the given-s RMSNorm backward equals backward_dgrad."""
    rng = np.random.default_rng(seed)
    M, d, N1, dw = 5, 12, 10, 7
    x, W0, z, gamma, W1, _, eps = _rand_case(rng, M, d, N1, eps=1e-5)
    f = O.forward(x, W0, z, gamma, W1, eps)
    W2 = rng.standard_normal((N1 // 2, dw)) / math.sqrt(N1 // 2)
    dout = rng.standard_normal((M, dw)) * 0.2
    dy, s = O.backward_swiglu(dout, W2, f.y)
    b = O.backward_dgrad(dy, W1, f.h, f.r, gamma)
    np.testing.assert_allclose(s, b.s, rtol=1e-10, atol=1e-13)
    dh = O.backward_rmsnorm_given_s(b.dh2, f.h, f.r, gamma, s)
    np.testing.assert_allclose(dh, b.dh, rtol=1e-9, atol=1e-13)


SWIGLU_BWD_PINS = [pin_swiglu_bwd_autograd, pin_swiglu_bwd_finite_differences,
                   pin_statistic_upstream_equals_definition]


@pytest.mark.parametrize("pin", SWIGLU_BWD_PINS, ids=lambda p: p.__name__)
def test_swiglu_bwd_pin(pin):
    pin()


def _swiglu_bwd_mutant(kind):
    def bwd(dout, W2, y):
        y = np.asarray(y, float)
        half = y.shape[1] // 2
        g, u = y[:, :half], y[:, half:]
        da = np.asarray(dout, float) @ np.asarray(W2, float).T
        sig = 1.0 / (1.0 + np.exp(-g))
        dsilu = sig if kind == "dsilu_is_sigmoid" else sig * (1.0 + g * (1.0 - sig))
        dg = da * u * dsilu
        du = da * g * sig
        dy = np.concatenate([du, dg] if kind == "halves_swapped" else [dg, du], axis=1)
        return dy, np.sum(dy * y, axis=1)
    return bwd


@pytest.mark.parametrize("kind", ["dsilu_is_sigmoid", "halves_swapped"])
def test_swiglu_bwd_planted_mistake_is_caught(kind, monkeypatch):
    monkeypatch.setattr(O, "backward_swiglu", _swiglu_bwd_mutant(kind))
    failed = []
    for pin in SWIGLU_BWD_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed


def test_given_s_planted_mistake_is_caught(monkeypatch):
    # r^3 instead of r^2 in the given-s form
    monkeypatch.setattr(O, "backward_rmsnorm_given_s",
                        lambda dh2, h, r, gamma, s: np.asarray(r)[:, None] * np.asarray(gamma)[None, :]
                        * np.asarray(dh2) - ((np.asarray(r) ** 3) * np.asarray(s) / np.shape(h)[1])[:, None]
                        * np.asarray(h))
    with pytest.raises(AssertionError):
        pin_statistic_upstream_equals_definition()


# ----------------------------------------------------------------------------
# Full backward of the chain (all parameter and input gradients)
# ----------------------------------------------------------------------------

def pin_full_backward_autograd(seed=13):
    """torch autograd (fp64) of L = sum(dy * y) + sum(dh_res * h) through
    h = x @ W0 + z, y = rms_norm(h, gamma) @ W1."""
    rng = np.random.default_rng(seed)
    for (M, d, N1) in [(5, 8, 6), (3, 16, 12)]:
        x, W0, z, gamma, W1, dy, eps = _rand_case(rng, M, d, N1, eps=1e-5)
        dh_res = 0.2 * rng.standard_normal((M, d))
        T = {k: torch.tensor(v, requires_grad=True) for k, v in
             dict(x=x, W0=W0, z=z, gamma=gamma, W1=W1).items()}
        th = T["x"] @ T["W0"] + T["z"]
        ty = torch.nn.functional.rms_norm(th, (d,), weight=T["gamma"], eps=eps) @ T["W1"]
        loss = torch.sum(torch.tensor(dy) * ty) + torch.sum(torch.tensor(dh_res) * th)
        loss.backward()
        f = O.forward(x, W0, z, gamma, W1, eps)
        b = O.backward_full(dy, x, W0, W1, f.h, f.r, gamma, dh_res)
        np.testing.assert_allclose(b.dh, T["z"].grad.numpy(), rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(b.dx, T["x"].grad.numpy(), rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(b.dW0, T["W0"].grad.numpy(), rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(b.dW1, T["W1"].grad.numpy(), rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(b.dgamma, T["gamma"].grad.numpy(), rtol=1e-9, atol=1e-12)


def pin_full_backward_finite_differences(seed=14):
    """Central differences of L = sum(dy * y) in gamma and W0 (no upstream term)."""
    rng = np.random.default_rng(seed)
    M, d, N1 = 3, 5, 4
    x, W0, z, gamma, W1, dy, eps = _rand_case(rng, M, d, N1, eps=1e-3)

    def loss(W0_, gamma_):
        f = O.forward(x, W0_, z, gamma_, W1, eps)
        return float(np.sum(dy * f.y))

    f = O.forward(x, W0, z, gamma, W1, eps)
    b = O.backward_full(dy, x, W0, W1, f.h, f.r, gamma)
    step = 1e-6
    for j in range(d):
        gp, gm = gamma.copy(), gamma.copy()
        gp[j] += step
        gm[j] -= step
        fd = (loss(W0, gp) - loss(W0, gm)) / (2 * step)
        np.testing.assert_allclose(b.dgamma[j], fd, rtol=1e-5, atol=1e-8)
    for (i, j) in [(0, 0), (2, 3), (4, 1)]:
        wp, wm = W0.copy(), W0.copy()
        wp[i, j] += step
        wm[i, j] -= step
        fd = (loss(wp, gamma) - loss(wm, gamma)) / (2 * step)
        np.testing.assert_allclose(b.dW0[i, j], fd, rtol=1e-5, atol=1e-8)


FULL_BWD_PINS = [pin_full_backward_autograd, pin_full_backward_finite_differences]


@pytest.mark.parametrize("pin", FULL_BWD_PINS, ids=lambda p: p.__name__)
def test_full_backward_pin(pin):
    pin()


def _full_bwd_mutant(kind):
    orig = O.backward_full

    def bwd(dy, x, W0, W1, h, r, gamma, dh_res=None):
        res = orig(dy, x, W0, W1, h, r, gamma, dh_res)
        if kind == "dgamma_without_r":
            bd = O.backward_dgrad(dy, W1, h, r, gamma)
            res.dgamma = np.sum(bd.dh2 * np.asarray(h, float), axis=0)
        elif kind == "dW1_from_h_not_h2":
            res.dW1 = np.asarray(h, float).T @ np.asarray(dy, float)
        elif kind == "dx_without_residual_grad" and dh_res is not None:
            res.dx = (res.dh - np.asarray(dh_res, float)) @ np.asarray(W0, float).T
        elif kind == "dW0_transposed":
            res.dW0 = res.dW0.T
        return res
    return bwd


@pytest.mark.parametrize("kind", ["dgamma_without_r", "dW1_from_h_not_h2", "dx_without_residual_grad",
                                  "dW0_transposed"])
def test_full_backward_planted_mistake_is_caught(kind, monkeypatch):
    monkeypatch.setattr(O, "backward_full", _full_bwd_mutant(kind))
    failed = []
    for pin in FULL_BWD_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, kind


# ----------------------------------------------------------------------------
# FP8 (E4M3) variant
# ----------------------------------------------------------------------------

def pin_e4m3_rounding_library(seed=15):
    """round_e4m3 against torch's float8_e4m3fn conversion on in-range values."""
    rng = np.random.default_rng(seed)
    v = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 1e-2,
                        rng.uniform(-448, 448, 2000), [0.0, 448.0, -448.0, 2.0 ** -9, 2.0 ** -6]])
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    # float32 first, as torch converts from float32: compare on values exact in float32
    got = O.round_e4m3(v.astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def pin_e4m3_closed_forms():
    # exact grid points stay; halfway points go to the even mantissa; saturation
    assert O.round_e4m3(np.array([1.0, 1.125, 448.0, 2.0 ** -9]))[[0, 1, 2, 3]].tolist() == \
        [1.0, 1.125, 448.0, 2.0 ** -9]
    assert O.round_e4m3(np.array([1.0625]))[0] == 1.0      # between 1 and 1.125: tie to even 1.0
    assert O.round_e4m3(np.array([1.1875]))[0] == 1.25     # tie between 1.125 and 1.25 -> 1.25
    assert O.round_e4m3(np.array([1000.0, -1e6]))[[0, 1]].tolist() == [448.0, -448.0]
    assert O.round_e4m3(np.array([2.0 ** -10]))[0] == 0.0  # tie between 0 and 2^-9 -> 0
    assert O.round_e4m3(np.array([3 * 2.0 ** -10]))[0] == 2.0 ** -8  # tie 2^-9/2^-8 -> even


def pin_fp8_forward_reduces_to_bf16_definition(seed=16):
    """With operands exactly representable and s_hg making h * gamma land on the
    E4M3 grid, forward_fp8 equals the plain forward of the dequantised inputs."""
    rng = np.random.default_rng(seed)
    M, d, N1 = 4, 8, 6
    grid = np.array([-2.0, -1.0, -0.5, 0.0, 0.5, 1.0, 2.0])
    x_q = rng.choice(grid, (M, d))
    W0_q = np.zeros((d, d))  # h = z: keeps h * gamma on the grid
    z = rng.choice(grid, (M, d))
    gamma = np.ones(d)
    W1_q = rng.choice(grid, (d, N1))
    f, hq = O.forward_fp8(x_q, 0.5, W0_q, 0.25, z, gamma, W1_q, 0.125, 1.0, 1e-5)
    ref = O.forward(x_q * 0.5, W0_q * 0.25, z, gamma, W1_q * 0.125, 1e-5)
    np.testing.assert_allclose(f.y, ref.y, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(hq, z)


def pin_fp8_forward_bruteforce(seed=17):
    """Scalar loops over the four steps, with rounding by torch's E4M3 conversion."""
    rng = np.random.default_rng(seed)
    M, d, N1 = 3, 5, 4
    x_q = O.round_e4m3(rng.standard_normal((M, d)) * 20)
    W0_q = O.round_e4m3(rng.standard_normal((d, d)) * 20)
    W1_q = O.round_e4m3(rng.standard_normal((d, N1)) * 20)
    z = rng.standard_normal((M, d))
    gamma = 1 + 0.3 * rng.standard_normal(d)
    sx, sW0, sW1, s_hg, eps = 0.05, 0.01, 0.02, 0.03, 1e-5
    f, _ = O.forward_fp8(x_q, sx, W0_q, sW0, z, gamma, W1_q, sW1, s_hg, eps)
    for m in range(M):
        h = [sum(x_q[m][k] * sx * W0_q[k][j] * sW0 for k in range(d)) + z[m][j] for j in range(d)]
        r = 1.0 / math.sqrt(sum(v * v for v in h) / d + eps)
        hq = [float(torch.tensor(min(max(h[j] * gamma[j] / s_hg, -448.0), 448.0),
                                 dtype=torch.float64).to(torch.float8_e4m3fn).to(torch.float64))
              for j in range(d)]
        for n in range(N1):
            y = r * sum(hq[j] * s_hg * W1_q[j][n] * sW1 for j in range(d))
            assert abs(f.y[m, n] - y) <= 1e-12 * (1 + abs(y))


FP8_PINS = [pin_e4m3_rounding_library, pin_e4m3_closed_forms,
            pin_fp8_forward_reduces_to_bf16_definition, pin_fp8_forward_bruteforce]


@pytest.mark.parametrize("pin", FP8_PINS, ids=lambda p: p.__name__)
def test_fp8_pin(pin):
    pin()


@pytest.mark.parametrize("kind", ["ties_away_from_zero", "three_bits_too_many", "no_saturation"])
def test_e4m3_planted_mistake_is_caught(kind, monkeypatch):
    orig = O.round_e4m3

    def mutant(v):
        v = np.asarray(v, float)
        a = np.abs(v)
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6.0)
        if kind == "ties_away_from_zero":
            step = np.exp2(e - 3.0)
            q = np.floor(a / step + 0.5) * step
            return np.sign(v) * np.minimum(q, 448.0)
        if kind == "three_bits_too_many":
            step = np.exp2(e - 6.0)
            return np.sign(v) * np.minimum(np.round(a / step) * step, 448.0)
        q = orig(np.clip(v, -1e9, 1e9))
        return np.where(np.abs(v) > 448.0, v, q)

    monkeypatch.setattr(O, "round_e4m3", mutant)
    failed = []
    for pin in FP8_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, kind
