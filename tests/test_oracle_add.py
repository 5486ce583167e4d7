"""Pins for oracle.add: IEEE binary32 special cases and the library float32 add."""
import numpy as np
import torch

from oracle.add import add_f32


def test_add_special_cases():
    x = np.array([1.0, 1.0, 2.0 ** -149, -2.0 ** -149, np.inf, 3e38, 1.0], np.float32)
    y = np.array([2.0 ** -24, 3 * 2.0 ** -24, 2.0 ** -149, 2.0 ** -149, -np.inf, 3e38, -1.0], np.float32)
    out = add_f32(x, y)
    assert out[0] == 1.0                      # tie -> even
    assert out[1] == np.float32(1 + 2.0 ** -22)  # tie -> even (up)
    assert out[2] == np.float32(2.0 ** -148)  # subnormals are kept (no flush to zero)
    assert out[3] == 0.0
    assert np.isnan(out[4])
    assert np.isinf(out[5])
    assert out[6] == 0.0 and not np.signbit(out[6])


def test_add_matches_torch_cpu():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((300, 257)) * np.exp(rng.uniform(-90, 80, (300, 257)))).astype(np.float32)
    y = (rng.standard_normal((300, 257)) * np.exp(rng.uniform(-90, 80, (300, 257)))).astype(np.float32)
    ref = (torch.from_numpy(x) + torch.from_numpy(y)).numpy()
    assert np.array_equal(add_f32(x, y).view(np.uint32), ref.view(np.uint32))


def test_add_exact_when_sum_is_representable():
    rng = np.random.default_rng(8)
    x = rng.integers(-2 ** 20, 2 ** 20, 1000).astype(np.float32)
    y = rng.integers(-2 ** 20, 2 ** 20, 1000).astype(np.float32)
    assert np.array_equal(add_f32(x, y), (x.astype(np.int64) + y.astype(np.int64)).astype(np.float32))


def test_scale_exact_and_rounded():
    from oracle.add import scale_f32
    x = np.array([1.0, 2.0 ** -149, 3e38, 1.0 + 2.0 ** -23, -0.0], np.float32)
    two = scale_f32(x, 2.0)
    assert two[0] == 2.0 and two[1] == np.float32(2.0 ** -148) and np.isinf(two[2]) and np.signbit(two[4])
    three = scale_f32(np.array([1.0 + 2.0 ** -23], np.float32), 3.0)
    # 3 * (1 + 2^-23) = 3 + 1.5 ulp (ulp 2^-22 in [2, 4)): a tie between 3 + 2^-22 (odd) and 3 + 2^-21 (even)
    assert three[0] == np.float32(3.0 + 2.0 ** -21)
    rng = np.random.default_rng(1)
    y = rng.standard_normal(1000).astype(np.float32)
    assert np.array_equal(scale_f32(y, 3.0), (torch.from_numpy(y) * 3.0).numpy())
