"""CPU check of the backward tolerance in tests/bwd_util.py: a float32
emulation of the kernel's roundings (O and LSE from an fp32 forward, O rounded
to the input dtype, P and dS rounded to the input dtype before their
products, fp32 accumulation, outputs rounded once) stays inside the bound,
and a planted error of a few units in the last place of the output does not."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
from bwd_util import check_bwd


def emulate(q, k, v, do, scale, causal):
    dt = q.dtype
    qf, kf, vf, dof = (t.float() for t in (q, k, v, do))
    s = scale * qf @ kf.transpose(-1, -2)
    n = s.shape[-1]
    if causal:
        s = s.masked_fill(~torch.ones(n, n, dtype=torch.bool).tril(), float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    p = torch.exp(s - lse[..., None])
    o = (p.to(dt).float() @ vf).to(dt)
    pr = p.to(dt).float()
    dp = dof @ vf.transpose(-1, -2)
    dd = (dof * o.float()).sum(-1)
    ds = (pr * (dp - dd[..., None]) * scale).to(dt).float()
    dq = (ds @ kf).to(dt)
    dk = (ds.transpose(-1, -2) @ qf).to(dt)
    dv = (pr.transpose(-1, -2) @ dof).to(dt)
    return o, lse, dq, dk, dv


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_emulated_kernel_is_inside_the_bound(orc, dtype, causal):
    q, k, v = inputs.make_qkv(1, 2, 200, 64, dtype, (1, 2, 3))
    do = inputs.make_dout(1, 2, 200, 64, dtype, 4)
    res = check_bwd(orc, q, k, v, do, 0.125, causal, emulate(q, k, v, do, 0.125, causal),
                    "emulated %s causal=%s" % (dtype, causal))
    # the bound is a worst case: the emulation sits well inside it
    assert max(res["dq_max_ratio"], res["dk_max_ratio"], res["dv_max_ratio"]) < 0.5


@pytest.mark.parametrize("name", ["dq", "dk", "dv"])
def test_planted_error_fails(orc, name):
    q, k, v = inputs.make_qkv(1, 1, 96, 64, "fp16", (5, 6, 7))
    do = inputs.make_dout(1, 1, 96, 64, "fp16", 8)
    out = list(emulate(q, k, v, do, 0.125, False))
    idx = {"dq": 2, "dk": 3, "dv": 4}[name]
    t = out[idx].float()
    t[0, 0, 17, 5] += 0.02 * float(t.abs().max())
    out[idx] = t.to(q.dtype)
    with pytest.raises(AssertionError):
        check_bwd(orc, q, k, v, do, 0.125, False, out, "planted %s" % name)


@pytest.mark.parametrize("causal", [False, True])
def test_dv_identity_holds_for_the_emulation(causal):
    """The full-size dV identity passes on the emulated kernel and fails when
    one dV element is off by 0.5."""
    from bwd_util import check_dv_identity
    q, k, v = inputs.make_qkv(1, 2, 300, 64, "fp16", (21, 22, 23))
    do = inputs.make_dout(1, 2, 300, 64, "fp16", 24)
    o, lse, dq, dk, dv = emulate(q, k, v, do, 0.125, causal)
    assert check_dv_identity(do, dv, "emulated") < 0.5
    bad = dv.float().clone()
    bad[0, 1, 7, 3] += 0.5
    with pytest.raises(AssertionError):
        check_dv_identity(do, bad.to(dv.dtype), "planted dv")


@pytest.mark.parametrize("causal", [False, True])
def test_dq_rows_check_on_the_emulation(orc, causal):
    """The sampled-row dQ check passes on the emulated kernel, and fails on a
    planted error of a quarter of the row's largest entry (the bf16 bound is a
    worst case over the row's cancelling terms, near 15 % of |dQ| here)."""
    from bwd_util import check_dq_rows
    q, k, v = inputs.make_qkv(1, 2, 260, 64, "bf16", (31, 32, 33))
    do = inputs.make_dout(1, 2, 260, 64, "bf16", 34)
    o, lse, dq, dk, dv = emulate(q, k, v, do, 0.125, causal)
    rows = np.array([[0, 0], [0, 129], [1, 259], [1, 64]])
    assert check_dq_rows(orc, q, k, v, do, o, lse, dq, rows, 0.125, causal, "emulated") < 0.5
    bad = dq.float().clone()
    bad[0, 1, 259, 7] += 0.25 * float(bad[0, 1, 259].abs().max())
    with pytest.raises(AssertionError):
        check_dq_rows(orc, q, k, v, do, o, lse, bad.to(dq.dtype), rows, 0.125, causal, "planted")
