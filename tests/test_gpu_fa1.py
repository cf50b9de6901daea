"""The FA1-structured baseline (fa1_fwd) against the fp64 oracle through the C ABI,
same tolerance as fa_fwd; plus whole-tensor checks on the base and B=1 comparison
workloads and a row sample of the d=128 workload."""
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
from parity_util import check_full, check_rows, edge_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return oracle.get()


def run_fa1(q, k, v, scale, causal):
    import attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    o, lse = fa.fa1_fwd(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    st = fa.fa_last_device_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, "device status %s" % fa.fa_status_str(st)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_full(orc, causal):
    q, k, v, meta = inputs.make_workload("tiny")
    o, lse = run_fa1(q, k, v, 0.125, causal)
    check_full(orc, q, k, v, 0.125, causal, o, lse, "fa1 tiny causal=%s" % causal)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 127, 128, 129, 300, 640])
def test_ragged_full(orc, dtype, d, causal, N):
    q, k, v = inputs.make_qkv(1, 2, N, d, dtype, (4000 + N, 5000 + N, 6000 + N))
    o, lse = run_fa1(q, k, v, d ** -0.5, causal)
    check_full(orc, q, k, v, d ** -0.5, causal, o, lse, "fa1 N=%d d=%d %s causal=%s" % (N, d, dtype, causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 96])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 640])
def test_head_dims_32_96_full(orc, dtype, d, causal, N):
    q, k, v = inputs.make_qkv(1, 2, N, d, dtype, (4100 + N + d, 5100 + N, 6100 + d))
    o, lse = run_fa1(q, k, v, d ** -0.5, causal)
    check_full(orc, q, k, v, d ** -0.5, causal, o, lse, "fa1 N=%d d=%d %s causal=%s" % (N, d, dtype, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_stress_full(orc, causal):
    q, k, v = inputs.make_qkv(1, 4, 1024, 64, "fp16", (71, 72, 73), q_scale=8.0)
    o, lse = run_fa1(q, k, v, 0.125, causal)
    check_full(orc, q, k, v, 0.125, causal, o, lse, "fa1 stress causal=%s" % causal)


def test_matches_fa2_closely(orc):
    """Same inputs through both loop nests: both within the oracle bound, and
    close to each other (they differ only in rounding order)."""
    import attention_forward_02_gb300 as fa
    q, k, v = inputs.make_qkv(2, 3, 777, 128, "bf16", (81, 82, 83))
    dev = torch.device("cuda:0")
    o1, l1 = run_fa1(q, k, v, 128 ** -0.5, True)
    o2, l2 = fa.fa_fwd(q.to(dev), k.to(dev), v.to(dev), scale=128 ** -0.5, causal=True)
    assert float((o1.float() - o2.float()).abs().max()) <= 2e-2
    assert float((l1 - l2).abs().max()) <= 1e-3


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name", ["base", "sweep_b1"])
def test_full_size_whole_tensor(orc, name, causal):
    q, k, v, meta = inputs.make_workload(name)
    d = meta["d"]
    o, lse = run_fa1(q, k, v, d ** -0.5, causal)
    check_full(orc, q, k, v, d ** -0.5, causal, o, lse, "fa1 %s causal=%s (whole tensor)" % (name, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_d128_sampled(orc, causal):
    q, k, v, meta = inputs.make_workload("d128")
    B, H, N, d = meta["B"], meta["H"], meta["N"], meta["d"]
    o, lse = run_fa1(q, k, v, d ** -0.5, causal)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    rows = edge_rows(B, H, N, inputs.sample_rows(B, H, N, 64, 8000 + B))
    check_rows(orc, q, k, v, d ** -0.5, causal, o, lse, rows, "fa1 d128 causal=%s" % causal)
