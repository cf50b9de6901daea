"""Decoding attention (fa_decode, split-KV) against the fp64 oracle through
the C ABI, with the forward pass's tolerance (the CUDA-core path keeps P in
fp32; the tensor-core path (3-16 queries, 2 at d = 128) rounds P to the input
type before the P V product, as the forward does); full checks at the bench
sizes."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
from parity_util import compare, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return oracle.get()


def run_decode(q, k, v, scale, causal):
    import attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    o, lse = fa.fa_decode(q.to(dev), k.to(dev), v.to(dev), scale=scale, causal=causal)
    st = fa.fa_last_device_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, "device status %s" % fa.fa_status_str(st)
    return o.cpu(), lse.cpu()


def check(orc, q, k, v, scale, causal, what):
    o, lse = run_decode(q, k, v, scale, causal)
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    o_ref, lse_ref = orc.attention_decode(qf, kf, vf, scale, causal=causal)
    a_ref = None
    if v.dtype == torch.bfloat16:
        a_ref, _ = orc.attention_decode(qf, kf, np.abs(vf), scale, causal=causal)
    return compare(to_f64(o), to_f64(lse), o_ref, lse_ref, float(v.abs().max()), what, v.dtype, a_ref)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 100), (1, 128), (1, 129), (3, 3), (3, 1000),
                                   (16, 16), (16, 4100), (5, 2048)])
def test_small(orc, dtype, d, causal, Nq, Nk):
    q, k, v = inputs.make_decode(2, 3, Nq, Nk, d, dtype, (9000 + Nk, 9100 + Nq, 9200 + d))
    check(orc, q, k, v, d ** -0.5, causal, "decode Nq%d Nk%d d%d %s causal=%s" % (Nq, Nk, d, dtype, causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 96])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(1, 129), (3, 1000), (16, 4100)])
def test_head_dims_32_96(orc, dtype, d, causal, Nq, Nk):
    q, k, v = inputs.make_decode(2, 3, Nq, Nk, d, dtype, (9400 + Nk, 9500 + Nq, 9600 + d))
    check(orc, q, k, v, d ** -0.5, causal, "decode Nq%d Nk%d d%d %s causal=%s" % (Nq, Nk, d, dtype, causal))


def test_peaked_scores(orc):
    # q x 8: scaled scores with a standard deviation about 8 (the running max moves)
    q, k, v = inputs.make_decode(1, 4, 2, 5000, 128, "fp16", (9301, 9302, 9303))
    check(orc, q * 8, k, v, 128 ** -0.5, True, "decode peaked")


@pytest.mark.parametrize("name", sorted(inputs.DECODE_WORKLOADS))
def test_workload_full(orc, name):
    """The bench's decoding workloads, every output row checked."""
    q, k, v, meta = inputs.make_decode_workload(name)
    check(orc, q, k, v, meta["d"] ** -0.5, meta["causal"], "decode workload %s" % name)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(2, 2), (2, 300), (3, 3), (3, 300), (4, 4097), (8, 1500), (15, 2000),
                                   (16, 129)])
def test_tensor_core_path(orc, dtype, causal, Nq, Nk):
    """d = 128 with 2-16 queries: both products on the tensor cores (queries
    padded to 16, ragged key tails, one or several chunks per head)."""
    q, k, v = inputs.make_decode(3, 5, Nq, Nk, 128, dtype, (9700 + Nk, 9800 + Nq, 9900))
    check(orc, q, k, v, 128 ** -0.5, causal, "decode tc Nq%d Nk%d %s causal=%s" % (Nq, Nk, dtype, causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 96])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(3, 300), (5, 700), (8, 1500), (16, 129)])
def test_tensor_core_path_head_dims(orc, dtype, d, causal, Nq, Nk):
    """Head dims below 128 on the tensor cores: K = d in the score product; the
    O^T product keeps M = 128 with the V tile's columns past d zero (TMA
    zero-fills them for d = 96; a zeroed second block for d <= 64)."""
    q, k, v = inputs.make_decode(2, 5, Nq, Nk, d, dtype, (9600 + Nk, 9650 + Nq, 9690 + d))
    check(orc, q, k, v, d ** -0.5, causal, "decode tc Nq%d Nk%d d%d %s causal=%s" % (Nq, Nk, d, dtype, causal))


def test_tensor_core_many_items(orc):
    """More (head, chunk) items than SMs: every CTA runs several items, so the
    Q buffers, the O accumulator hand-over and the ring wrap many times."""
    q, k, v = inputs.make_decode(4, 40, 3, 3000, 128, "bf16", (9911, 9912, 9913))
    check(orc, q, k, v, 128 ** -0.5, True, "decode tc many items")


@pytest.mark.parametrize("Nq", [1, 4])
def test_rising_scores(orc, Nq):
    """Scores that grow along the keys (about 2 log2 units per 128-key tile):
    the running reference moves again and again inside a chunk, so the
    accumulated O and row sums are rescaled many times."""
    q, k, v = inputs.make_decode(1, 3, Nq, 5000, 128, "fp16", (9921, 9922, 9923))
    q = (q.float().abs() + 1.0).to(q.dtype)
    ramp = torch.linspace(0.0, 3.0, 5000).view(1, 1, 5000, 1)
    k = (k.float() + ramp).to(k.dtype)
    check(orc, q, k, v, 128 ** -0.5, False, "decode rising Nq%d" % Nq)
