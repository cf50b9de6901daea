"""fa1_fwd_noalloc: the allocation-free entry point for callers that cannot call
cudaMalloc themselves (for example code inside a host framework that only hands
it fixed input and output buffers).  It keeps its scratch in a fixed array in
the library, so this test calls it straight through the C ABI and compares it
with fa1_fwd, which takes a caller workspace, and with the fp64 oracle, on two
calls in a row with different inputs (the second call must not be affected by
what the first one left in the shared array).  Collected last on purpose."""
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
from parity_util import LSE_TOL, O_TOL_REL_VMAX, check_full

pytestmark = pytest.mark.gpu


def _noalloc_call(q, k, v, o, lse, causal):
    from attention_forward_02_gb300 import _lib
    B, H, N, d = q.shape
    code = 0 if q.dtype == torch.float16 else 1
    return _lib.load().fa1_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), B, H, N, d, d ** -0.5, int(causal), code,
                                       torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    orc = oracle.get()
    cases = [((1, 2, 700, 64, "fp16", (91, 92, 93)), True),
             ((2, 3, 389, 128, "bf16", (94, 95, 96)), False)]
    for (B, H, N, d, dtype, seeds), causal in cases:
        q, k, v = (t.to(dev) for t in inputs.make_qkv(B, H, N, d, dtype, seeds))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        assert _noalloc_call(q, k, v, o, lse, causal) == 0
        o_ref, lse_ref = fa.fa1_fwd(q, k, v, scale=d ** -0.5, causal=causal)
        assert fa.fa_last_device_status(torch.cuda.current_stream().cuda_stream) == 0
        vmax = float(v.abs().max())
        assert float((o.double() - o_ref.double()).abs().max()) <= O_TOL_REL_VMAX * vmax
        assert float((lse.double() - lse_ref.double()).abs().max()) <= LSE_TOL
        # and against the oracle itself, element by element
        check_full(orc, q.cpu(), k.cpu(), v.cpu(), d ** -0.5, causal, o.cpu(), lse.cpu(),
                   "fa1_fwd_noalloc B%dH%dN%d d=%d %s causal=%s" % (B, H, N, d, dtype, causal))


def test_noalloc_rejects_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    B, H, N, d = 4, 32, 2048, 64  # needs 69 MB of scratch, above the 16 MiB array
    assert fa.fa1_fwd_workspace_size(B, H, N, d) > 16 << 20
    q = torch.zeros((B, H, N, d), dtype=torch.float16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    assert _noalloc_call(q, q, q, o, lse, False) == 2  # FA_ERR_UNSUPPORTED, nothing launched
