"""Host-side checks of the seeded input generator (CPU only)."""

import numpy as np
import torch

from gemm_epilogue_fusion_gemm0_gb300 import synth


def test_shapes_dtypes_and_determinism():
    a = synth.make_forward_inputs(64, 32, 48, seed=0)
    b = synth.make_forward_inputs(64, 32, 48, seed=0)
    for k, shape in (("x", (64, 32)), ("z", (64, 32)), ("W0", (32, 32)), ("W1", (32, 48)), ("gamma", (32,))):
        assert a[k].dtype == torch.bfloat16 and tuple(a[k].shape) == shape
        assert torch.equal(a[k], b[k])
    dy1 = synth.make_grad_output(a["_rng"], 64, 48)
    dy2 = synth.make_grad_output(b["_rng"], 64, 48)
    assert torch.equal(dy1, dy2) and dy1.dtype == torch.bfloat16
    c = synth.make_forward_inputs(64, 32, 48, seed=1)
    assert not torch.equal(a["x"], c["x"])


def test_distributions():
    M, d, N1 = 512, 256, 512
    t = synth.make_forward_inputs(M, d, N1, seed=3)
    f = lambda k: t[k].to(torch.float64).numpy()
    assert abs(f("x").std() - 1.0) < 0.02 and abs(f("x").mean()) < 0.02
    assert abs(f("W0").std() - (1 / d) ** 0.5) < 0.003
    assert abs(f("W1").std() - (1 / d) ** 0.5) < 0.003
    assert abs(f("gamma").mean() - 1.0) < 0.08 and abs(f("gamma").std() - 0.1 ** 0.5) < 0.05
    dy = synth.make_grad_output(t["_rng"], M, N1).to(torch.float64).numpy()
    assert abs(dy.std() - 0.1) < 0.003


def test_bf16_rounding_is_nearest_even():
    # 1 + 2^-8 is halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even -> 1
    v = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8], dtype=np.float32)
    out = synth.to_bf16(v).to(torch.float64).numpy()
    assert out[0] == 1.0 and out[1] == 1.0 + 2 * 2.0 ** -7


def test_sample_rows():
    rows = synth.sample_rows(8192, 512, seed=1)
    assert len(rows) == 512 and len(np.unique(rows)) == 512
    for r in (0, 127, 128, 8191):
        assert r in rows
    assert np.all(np.diff(rows) > 0)
    assert np.array_equal(synth.sample_rows(100, 512), np.arange(100))


def test_device_generator_shapes_determinism_and_distributions():
    """make_inputs_on_device (used for workloads too large to draw on the
    host) run on the CPU device: shapes, dtypes, seeding, distributions."""
    a = synth.make_inputs_on_device(512, 256, 384, seed=5, device="cpu")
    b = synth.make_inputs_on_device(512, 256, 384, seed=5, device="cpu")
    c = synth.make_inputs_on_device(512, 256, 384, seed=6, device="cpu")
    shapes = {"x": (512, 256), "z": (512, 256), "W0": (256, 256), "W1": (256, 384),
              "gamma": (256,), "dy": (512, 384)}
    for k, shp in shapes.items():
        assert tuple(a[k].shape) == shp and a[k].dtype == torch.bfloat16, k
        assert torch.equal(a[k], b[k]), k
        assert not torch.equal(a[k], c[k]), k
    std = {k: float(a[k].float().std()) for k in shapes}
    assert abs(std["x"] - 1.0) < 0.02 and abs(std["z"] - 1.0) < 0.02
    assert abs(std["W0"] - 256 ** -0.5) < 0.003 and abs(std["W1"] - 256 ** -0.5) < 0.003
    assert abs(std["dy"] - 0.1) < 0.003
    assert abs(float(a["gamma"].float().mean()) - 1.0) < 0.06 and abs(std["gamma"] - 0.1 ** 0.5) < 0.06


def test_dgrad_input_generator():
    """make_dgrad_inputs: shapes, dtypes, seeding and the stated distributions."""
    a = synth.make_dgrad_inputs(512, 256, 384, seed=9)
    b = synth.make_dgrad_inputs(512, 256, 384, seed=9)
    shapes = {"h": (512, 256), "W1": (256, 384), "gamma": (256,), "dy": (512, 384)}
    for k, shp in shapes.items():
        assert tuple(a[k].shape) == shp and a[k].dtype == torch.bfloat16, k
        assert torch.equal(a[k], b[k]), k
    f = lambda k: a[k].to(torch.float64).numpy()
    assert abs(f("h").std() - 2.0 ** 0.5) < 0.03 and abs(f("h").mean()) < 0.03
    assert abs(f("W1").std() - (1 / 256) ** 0.5) < 0.003
    assert abs(f("gamma").mean() - 1.0) < 0.08
    assert abs(f("dy").std() - 0.1) < 0.003
