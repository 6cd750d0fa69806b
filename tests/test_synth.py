"""The seeded generator: determinism, piecewise generation, distributions, storage rounding."""
import numpy as np
import torch

import synth


def test_deterministic_and_piecewise():
    a = np.empty(200_000, np.float32)
    synth.fill(a, "normal", 0.0, 1.0, seed=3, tensor_id=synth.X_ID)
    b = np.empty(200_000, np.float32)
    synth.fill(b[:70_001], "normal", 0.0, 1.0, seed=3, tensor_id=synth.X_ID, offset=0)
    synth.fill(b[70_001:], "normal", 0.0, 1.0, seed=3, tensor_id=synth.X_ID, offset=70_001)
    assert np.array_equal(a, b)
    c = np.empty(200_000, np.float32)
    synth.fill(c, "normal", 0.0, 1.0, seed=3, tensor_id=synth.X_ID, nthreads=1)
    assert np.array_equal(a, c)


def test_streams_differ_by_seed_and_id():
    a = np.empty(1000, np.float32)
    b = np.empty(1000, np.float32)
    synth.fill(a, "uniform", -1, 1, seed=0, tensor_id=0)
    synth.fill(b, "uniform", -1, 1, seed=0, tensor_id=2)
    assert not np.array_equal(a, b)
    synth.fill(b, "uniform", -1, 1, seed=1, tensor_id=0)
    assert not np.array_equal(a, b)


def test_distributions():
    n = 1 << 20
    u = np.empty(n, np.float32)
    synth.fill(u, "uniform", -1, 1, seed=0, tensor_id=0)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 5e-3 and abs(u.var() - 1 / 3) < 5e-3
    z = np.empty(n, np.float32)
    synth.fill(z, "normal", 0, 0.02, seed=2, tensor_id=1)
    assert abs(z.mean()) < 1e-4 and abs(z.std() - 0.02) < 2e-4
    i = np.empty(n, np.float32)
    synth.fill(i, "integer", -3, 3, seed=5, tensor_id=0)
    assert set(np.unique(i).tolist()) == {-3, -2, -1, 0, 1, 2, 3}


def test_16bit_storage_rounds_like_torch():
    f = np.empty(1 << 18, np.float32)
    synth.fill(f, "normal", 0, 1, seed=9, tensor_id=0)
    # spread magnitudes over fp16's normal and subnormal ranges and bf16's range
    scale = np.float32(2.0) ** np.linspace(-30, 15, f.size).astype(np.float32)
    f = (f * scale).astype(np.float32)
    tb = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    th = torch.from_numpy(f).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    ours_b = np.array([synth.f32_to_bf16_bits(float(v)) for v in f[::7]], np.uint16)
    ours_h = np.array([synth.f32_to_f16_bits(float(v)) for v in f[::7]], np.uint16)
    assert np.array_equal(ours_b, tb[::7])
    assert np.array_equal(ours_h, th[::7])


def test_fill_torch_tensor_16bit():
    t = synth.tensor((4, 8, 8, 16), torch.bfloat16, "normal", 0, 1, seed=3, tensor_id=0)
    f = np.empty(t.numel(), np.float32)
    synth.fill(f, "normal", 0, 1, seed=3, tensor_id=0)
    assert torch.equal(t.flatten(), torch.from_numpy(f).to(torch.bfloat16))
    h = synth.tensor((1000,), torch.float16, "normal", 0, 1, seed=4, tensor_id=2)
    f = np.empty(1000, np.float32)
    synth.fill(f, "normal", 0, 1, seed=4, tensor_id=2)
    assert torch.equal(h, torch.from_numpy(f).to(torch.float16))
