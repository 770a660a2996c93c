"""The parity gate's storage allowance (CPU): half an ulp of bf16/fp16 at the
reference value, checked against torch's own rounding."""
import numpy as np
import pytest
import torch

from tests.parity import check, half_ulp


@pytest.mark.parametrize("storage,dtype", [("bf16", torch.bfloat16), ("fp16", torch.float16)])
def test_half_ulp_bounds_the_storage_rounding(storage, dtype):
    rng = np.random.default_rng(3)
    v = rng.standard_normal(20000) * 6
    # torch rounds float64 to fp16 through float32: allow that first rounding
    rounded = torch.from_numpy(v).to(dtype).double().numpy()
    assert (np.abs(rounded - v) <= half_ulp(v, storage) + np.abs(v) * 2.0 ** -24).all()
    # and it is attained: some element rounds by more than 90% of it
    assert (np.abs(rounded - v) > 0.9 * half_ulp(v, storage)).any()


def test_storage_allowance_is_on_top_of_the_tolerance():
    ref = np.array([[9.0, 1.0, -12.0, 0.5]])
    ok = ref + np.array([[0.031 + 0.019, 0.0039 + 0.019, -0.031 - 0.019, 0.0]])
    check(ok, ref, "within", unit_scale=True, storage="bf16", cos_min=0.99)
    bad = ref + np.array([[0.0, 0.03, 0.0, 0.0]])
    with pytest.raises(AssertionError):
        check(bad, ref, "beyond", unit_scale=True, storage="bf16", cos_min=0.99)
