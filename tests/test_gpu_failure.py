"""The failure path on the GPU without a fault: a bounded wait on a barrier
that nothing arrives on gives up, the status word reports FA_ERR_TIMEOUT, and
the context stays usable for the next attention call."""
import pytest
import torch

from attention_forward_02_gb300 import inputs

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_forward_02_gb300 as fa
    import oracle
    from parity_util import check_full, run_gpu
    stream = torch.cuda.current_stream().cuda_stream
    assert fa.fa_last_device_status(stream) == 0          # clean start
    assert fa.fa_selftest_wait_timeout(2000, stream) == 0  # ~2 ms wait that must expire
    assert fa.fa_last_device_status(stream) == 5           # FA_ERR_TIMEOUT, and cleared
    assert fa.fa_last_device_status(stream) == 0
    q, k, v = inputs.make_qkv(1, 2, 300, 64, "fp16", (3, 4, 5))
    o, lse = run_gpu(q, k, v, 0.125, True)
    check_full(oracle.get(), q, k, v, 0.125, True, o, lse, "after timeout self-test")
