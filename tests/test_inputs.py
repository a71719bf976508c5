"""Seeded input generator: determinism, bf16 rounding, distributions (CPU)."""
import numpy as np
import pytest
import torch

from memory_fusion_gb300 import inputs


def test_round_to_bf16_matches_torch_rne():
    rng = np.random.Generator(np.random.PCG64(0))
    a = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, -1e-40], np.float32)])
    mine = inputs.round_to_bf16(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
    np.testing.assert_array_equal(mine.view(np.uint32), ref.view(np.uint32))


def test_bf16_bits_roundtrip():
    a = inputs.round_to_bf16(np.linspace(-3, 3, 1001, dtype=np.float32))
    bits = inputs.bf16_bits(a)
    back = (bits.astype(np.uint32) << 16).view(np.float32)
    np.testing.assert_array_equal(back, a)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(t, a)


def test_gemm_inputs_deterministic_and_shaped():
    a = inputs.gemm_inputs(64, 96, 32, 5, x_std=0.5, w_std=0.25)
    b = inputs.gemm_inputs(64, 96, 32, 5, x_std=0.5, w_std=0.25)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    assert a["X"].shape == (64, 32) and a["W"].shape == (32, 96)
    assert a["bias"].shape == (96,) and a["gamma"].dtype == np.float32
    assert np.array_equal(inputs.round_to_bf16(a["X"]), a["X"])
    c = inputs.gemm_inputs(64, 96, 32, 6, x_std=0.5, w_std=0.25)
    assert not np.array_equal(a["X"], c["X"])


def test_stitch_inputs_distribution():
    d = inputs.stitch_inputs(2000, 64, 3)
    A, b = d["A"], d["row_bias"]
    assert A.dtype == np.float32 and b.dtype == np.float32
    assert abs(A.std() - 2.0) < 0.02
    assert b.min() >= -1.0 and b.max() < 1.0


@pytest.mark.parametrize("name", ["ln_tiny_128x512x256", "softmax_4096x2048x128"])
def test_workload_moments(name):
    w = inputs.WORKLOADS[name]
    d = inputs.workload_inputs(name)
    assert abs(d["X"].std() / w.x_std - 1) < 0.05
    assert abs(d["W"].std() / w.w_std - 1) < 0.05


def test_workload_bytes_and_flops():
    w = inputs.WORKLOADS["gelu_ln_16384x4096x4096"]
    assert w.flops == 2 * 16384 * 4096 * 4096
    assert w.unavoidable_bytes == 302039040
    assert inputs.WORKLOADS["softmax_4096x2048x128"].unavoidable_bytes == 18350080
    assert inputs.WORKLOADS["wide_ln_8192x16384x2048"].unavoidable_bytes == 369295360
    assert inputs.WORKLOADS["ln_tiny_128x512x256"].unavoidable_bytes == 464896
    assert inputs.WORKLOADS["stitch_750000x32"].unavoidable_bytes == 195000000
    assert inputs.WORKLOADS["stitch_64x30000"].unavoidable_bytes == 15360256
