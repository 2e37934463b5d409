"""The fp64 oracle against its pins (CPU only)."""
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(oracle_mod, pin):
    pin()


def test_storage_rounding_matches_library_conversions(oracle_mod):
    """round_to_storage against numpy's float32 cast and torch's bf16 cast, on fp32 inputs
    (torch converts through fp32, so only fp32-representable inputs give a single rounding)."""
    import numpy as np
    import torch
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    a = np.concatenate([a, [0.0, -0.0, 1.0, 1.00390625, 1.01171875, -3.0e38]]).astype(np.float64)
    assert np.array_equal(oracle_mod.round_to_storage(a, "bf16"),
                          torch.from_numpy(a).float().to(torch.bfloat16).double().numpy())
    b = rng.standard_normal(100000) * 1e3
    assert np.array_equal(oracle_mod.round_to_storage(b, "f32"), b.astype(np.float32))
