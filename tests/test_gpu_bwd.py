"""Backward pass (fa_bwd) against the fp64 oracle's gradients through the C
ABI: every tensor element within the bound derived in tests/bwd_util.py, for
both dtypes, both head dims, causal and not, ragged lengths, several heads."""
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
from bwd_util import check_bwd, run_gpu_fwd_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return oracle.get()


def _case(orc, B, H, N, d, dtype, causal, seed, q_scale=1.0):
    q, k, v = inputs.make_qkv(B, H, N, d, dtype, (seed, seed + 1, seed + 2), q_scale=q_scale)
    do = inputs.make_dout(B, H, N, d, dtype, seed + 3)
    scale = d ** -0.5
    gpu = run_gpu_fwd_bwd(q, k, v, do, scale, causal)
    return check_bwd(orc, q, k, v, do, scale, causal, gpu,
                     "bwd B%d H%d N%d d%d %s causal=%s" % (B, H, N, d, dtype, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_tiny(orc, causal):
    q, k, v, meta = inputs.make_workload("tiny")
    do = inputs.make_dout(meta["B"], meta["H"], meta["N"], meta["d"], meta["dtype"], 3)
    gpu = run_gpu_fwd_bwd(q, k, v, do, 0.125, causal)
    check_bwd(orc, q, k, v, do, 0.125, causal, gpu, "bwd tiny causal=%s" % causal)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 100, 128, 129, 384, 520])
def test_ragged(orc, dtype, d, causal, N):
    _case(orc, 1, 2, N, d, dtype, causal, 7000 + N)


@pytest.mark.parametrize("causal", [False, True])
def test_many_heads(orc, causal):
    _case(orc, 3, 3, 700, 64, "fp16", causal, 7100)


@pytest.mark.parametrize("causal", [False, True])
def test_stress_scores(orc, causal):
    # Q x 8: scaled scores with standard deviation about 8 (peaked softmax rows)
    _case(orc, 1, 2, 640, 128, "bf16", causal, 7200, q_scale=8.0)
