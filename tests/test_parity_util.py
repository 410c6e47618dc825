"""CPU checks of the parity helpers the GPU tests rely on."""
import numpy as np
import torch

from parity_util import assert_close_bf16_stored, bf16_ulp


def test_bf16_ulp_is_the_spacing_of_bf16_numbers():
    rng = np.random.default_rng(0)
    v = torch.from_numpy(rng.standard_normal(4096) * 10.0 ** rng.integers(-30, 30, 4096))
    b = v.to(torch.bfloat16)
    # the next bf16 value away from zero: the bit pattern plus one (sign and
    # magnitude format)
    nb = (b.view(torch.int16) + 1).view(torch.bfloat16)
    gap = (nb.double() - b.double()).abs().numpy()
    assert np.array_equal(bf16_ulp(b.double().numpy()), gap)


def test_bf16_stored_accepts_one_ulp_and_rejects_two():
    ref = np.array([5.0, 0.25, 100.0])
    one = ref + bf16_ulp(ref)
    assert_close_bf16_stored(one, ref, 1.0, 1e-3)
    two = ref.copy()
    two[2] += 2 * bf16_ulp(ref[2])
    try:
        assert_close_bf16_stored(two, ref, 1.0, 1e-3)
    except AssertionError:
        return
    raise AssertionError("two ulps accepted")
