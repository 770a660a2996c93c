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
    ref = np.array([[0.5, 1.0, -1.5, 0.2]])                      # rms < 1: scale 1
    hu = half_ulp(ref, "bf16")
    ok = ref + np.sign(ref) * (hu + 0.019)
    check(ok, ref, "within", unit_scale=True, storage="bf16", cos_min=0.99)
    bad = ref + np.array([[0.0, 0.03, 0.0, 0.0]])                # 0.026 past half an ulp
    with pytest.raises(AssertionError):
        check(bad, ref, "beyond", unit_scale=True, storage="bf16", cos_min=0.99)


def test_outputs_larger_than_unit_scale_scale_the_tolerance():
    ref = np.array([[3.0, -3.0, 3.0, -3.0]])                     # rms 3
    check(ref + 0.055, ref, "within", unit_scale=True, cos_min=0.99)
    with pytest.raises(AssertionError):
        check(ref + 0.065, ref, "beyond", unit_scale=True, cos_min=0.99)
