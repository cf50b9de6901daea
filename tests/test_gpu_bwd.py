"""Backward pass (fa_bwd) against the fp64 oracle's gradients through the C
ABI: every tensor element within the bound derived in tests/bwd_util.py, for
both dtypes, both head dims, causal and not, ragged lengths, several heads."""
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
import numpy as np

from bwd_util import check_bwd, check_bwd_heads, check_dq_rows, check_dv_identity, run_gpu_fwd_bwd

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


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 96])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 384])
def test_head_dims_32_96(orc, dtype, d, causal, N):
    _case(orc, 1, 2, N, d, dtype, causal, 7300 + N + d)


@pytest.mark.parametrize("causal", [False, True])
def test_many_heads(orc, causal):
    _case(orc, 3, 3, 700, 64, "fp16", causal, 7100)


@pytest.mark.parametrize("d,dtype", [(32, "bf16"), (64, "fp16"), (96, "fp16"), (128, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
def test_several_items_per_cta(orc, d, dtype, causal):
    # 2 x 40 heads x 5 key blocks = 400 (head, key block) items, more than the
    # 152 SMs: each persistent CTA walks two or three items, so ring slots and
    # barrier phases carry over item boundaries (causal: items of 1..5 blocks)
    _case(orc, 2, 40, 520, d, dtype, causal, 7400 + d)


@pytest.mark.parametrize("causal", [False, True])
def test_stress_scores(orc, causal):
    # Q x 8: scaled scores with standard deviation about 8 (peaked softmax rows)
    _case(orc, 1, 2, 640, 128, "bf16", causal, 7200, q_scale=8.0)


@pytest.mark.parametrize("causal", [False, True])
def test_base_sampled_heads(orc, causal):
    """Full base workload (B=4 H=32 N=2048 d=64 fp16) on the GPU; three heads
    compared element by element with the oracle."""
    q, k, v, meta = inputs.make_workload("base")
    do = inputs.make_dout(meta["B"], meta["H"], meta["N"], meta["d"], meta["dtype"],
                          inputs.DOUT_SEEDS["base"])
    gpu = run_gpu_fwd_bwd(q, k, v, do, 0.125, causal)
    check_bwd_heads(orc, q, k, v, do, 0.125, causal, gpu, [0, 77, 127],
                    "bwd base heads causal=%s" % causal)


@pytest.mark.parametrize("causal", [False, True])
def test_d128_one_head(orc, causal):
    """Full d128 workload (B=2 H=16 N=8192 d=128 bf16) on the GPU; one whole
    head (8192 x 8192 scores) compared element by element with the oracle."""
    q, k, v, meta = inputs.make_workload("d128")
    do = inputs.make_dout(meta["B"], meta["H"], meta["N"], meta["d"], meta["dtype"],
                          inputs.DOUT_SEEDS["d128"])
    scale = meta["d"] ** -0.5
    gpu = run_gpu_fwd_bwd(q, k, v, do, scale, causal)
    check_bwd_heads(orc, q, k, v, do, scale, causal, gpu, [21], "bwd d128 head 21 causal=%s" % causal)


@pytest.mark.parametrize("name", ["base", "d128", "long"])
@pytest.mark.parametrize("causal", [False, True])
def test_full_size_dq_rows(orc, name, causal):
    """The bench workloads at full size: sampled dQ rows (seeded, plus tile
    edges and the first and last rows) against the oracle's dQ rows."""
    q, k, v, meta = inputs.make_workload(name)
    B, H, N, d = meta["B"], meta["H"], meta["N"], meta["d"]
    do = inputs.make_dout(B, H, N, d, meta["dtype"], inputs.DOUT_SEEDS[name])
    scale = d ** -0.5
    o, lse, dq, dk, dv = run_gpu_fwd_bwd(q, k, v, do, scale, causal)
    rng = np.random.default_rng(808)
    heads = rng.choice(B * H, size=min(4, B * H), replace=False)
    rows = [(h, i) for h in heads for i in (0, 127, 128, N // 2, N - 1)]
    rows += [(int(rng.integers(B * H)), int(rng.integers(N))) for _ in range(24)]
    check_dq_rows(orc, q, k, v, do, o, lse, dq, np.array(rows), scale, causal,
                  "bwd %s dq rows causal=%s" % (name, causal))


@pytest.mark.parametrize("name", ["base", "d128", "long"])
@pytest.mark.parametrize("causal", [False, True])
def test_full_size_dv_identity(name, causal):
    """The bench workloads at full size, in the launch configuration bench.py
    times: every gradient finite, and sum_j dV_j = sum_i dO_i per head."""
    import attention_forward_02_gb300 as fa
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    q, k, v, meta = inputs.make_workload(name)
    do = inputs.make_dout(meta["B"], meta["H"], meta["N"], meta["d"], meta["dtype"],
                          inputs.DOUT_SEEDS[name])
    dev = torch.device("cuda:0")
    q, k, v, do = (t.to(dev) for t in (q, k, v, do))
    scale = meta["d"] ** -0.5
    o, lse = fa.fa_fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, scale=scale, causal=causal)
    st = fa.fa_last_device_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, fa.fa_status_str(st)
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    check_dv_identity(do, dv, "bwd %s causal=%s" % (name, causal))
