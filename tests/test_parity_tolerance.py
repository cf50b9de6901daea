"""The parity tolerance helper itself (CPU): it accepts the exact result
rounded to the output dtype and rejects a result that is off by a real error."""
import numpy as np
import pytest
import torch

from parity_util import compare


def _round(x, dtype):
    return torch.tensor(x).to(dtype).double().numpy()


def test_bf16_rounding_of_exact_result_passes():
    rng = np.random.default_rng(0)
    o_ref = rng.uniform(-3.5, 3.5, size=(64, 128))
    a_ref = np.abs(o_ref) + 0.1
    compare(_round(o_ref, torch.bfloat16), None, o_ref, None, 3.6, "bf16 exact",
            torch.bfloat16, a_ref)


def test_fp16_rounding_of_exact_result_passes():
    rng = np.random.default_rng(1)
    o_ref = rng.uniform(-3.5, 3.5, size=(64, 128))
    compare(_round(o_ref, torch.float16), None, o_ref, None, 3.6, "fp16 exact")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_real_error_fails(dtype):
    o_ref = np.zeros((4, 8))
    o = o_ref.copy()
    o[2, 3] = 0.05  # 0.05 > 2e-3 * 3.6 and > the rounding terms at |O_ref| = 0
    with pytest.raises(AssertionError):
        compare(o, None, o_ref, None, 3.6, "planted", dtype, np.full_like(o_ref, 0.5))


def test_lse_bound():
    o = np.zeros((2, 2))
    with pytest.raises(AssertionError):
        compare(o, np.array([1.0, 2.0 + 2e-3]), o, np.array([1.0, 2.0]), 1.0, "lse")
    compare(o, np.array([1.0, 2.0 + 5e-4]), o, np.array([1.0, 2.0]), 1.0, "lse ok")
