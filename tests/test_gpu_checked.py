"""The checked build (libfa_gb300_checked.so: the same sources compiled with
FA_BOUNDS_CHECK, whose kernels check every shared-memory and tensor-memory
address and every ring-slot, buffer and barrier index before using it; see
include/fa.h).  It stands in for a memory checker: these tests run the four
entry points of the checked library on small cases of every head dim, both
dtypes and both variants, and require a clean status word (no failed check,
no expired wait) and results within the oracle tolerances.  A self-test first
shows that the checks do fire on addresses outside the shared window and the
tensor-memory columns (evaluated only, nothing is accessed)."""
import numpy as np
import pytest
import torch

import oracle
from attention_forward_02_gb300 import inputs
from bwd_util import check_bwd
from parity_util import check_full, compare, to_f64

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_BOUNDS = 0, 6


@pytest.fixture(scope="module")
def chk():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_forward_02_gb300 import _lib
    lib = _lib.load_checked()
    assert lib.fa_checked_build() == 1
    assert _lib.load().fa_checked_build() == 0  # the product library has no checks
    return lib


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _code(t):
    return 0 if t.dtype == torch.float16 else 1


def _status(lib):
    st = lib.fa_last_device_status(_stream())
    assert st == FA_OK, "checked build: %s" % lib.fa_status_str(st).decode()


def test_checks_fire_on_out_of_range_addresses(chk):
    assert chk.fa_last_device_status(_stream()) == FA_OK
    assert chk.fa_selftest_bounds_check(_stream()) == FA_OK
    assert chk.fa_last_device_status(_stream()) == FA_ERR_BOUNDS  # and cleared
    assert chk.fa_last_device_status(_stream()) == FA_OK


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 640])
def test_forward_checked(chk, orc, dtype, d, causal, N):
    q, k, v = inputs.make_qkv(2, 3, N, d, dtype, (5000 + N, 5100 + d, 5200))
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((2, 3, N), dtype=torch.float32, device=dev)
    assert chk.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      2, 3, N, d, d ** -0.5, int(causal), _code(qd), _stream()) == FA_OK
    _status(chk)
    check_full(orc, q, k, v, d ** -0.5, causal, o, lse, "checked fwd N%d d%d %s causal=%s"
               % (N, d, dtype, causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_checked(chk, orc, dtype, d, causal):
    B, H, N = 1, 2, 300
    q, k, v = inputs.make_qkv(B, H, N, d, dtype, (5300 + d, 5400, 5500))
    do = inputs.make_dout(B, H, N, d, dtype, 5600 + d)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd)
    ws_bytes = chk.fa_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    scale = d ** -0.5
    assert chk.fa_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      B, H, N, d, scale, int(causal), _code(qd), _stream()) == FA_OK
    assert chk.fa_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                      dod.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                      ws_bytes, B, H, N, d, scale, int(causal), _code(qd), _stream()) == FA_OK
    _status(chk)
    check_bwd(orc, q, k, v, do, scale, causal, (o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()),
              "checked bwd N%d d%d %s causal=%s" % (N, d, dtype, causal))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("d", [32, 64, 96, 128])
@pytest.mark.parametrize("Nq,Nk,causal", [(1, 1000, False), (4, 2100, True), (16, 300, True)])
def test_decode_checked(chk, orc, dtype, d, Nq, Nk, causal):
    B, H = 2, 3
    q, k, v = inputs.make_decode(B, H, Nq, Nk, d, dtype, (5700 + Nk, 5800 + Nq, 5900 + d))
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws_bytes = chk.fa_decode_workspace_size(B, H, Nq, Nk, d)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    scale = d ** -0.5
    assert chk.fa_decode(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         ws.data_ptr(), ws_bytes, B, H, Nq, Nk, d, scale, int(causal), _code(qd),
                         _stream()) == FA_OK
    _status(chk)
    qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
    o_ref, lse_ref = orc.attention_decode(qf, kf, vf, scale, causal=causal)
    a_ref = None
    if v.dtype == torch.bfloat16:
        a_ref, _ = orc.attention_decode(qf, kf, np.abs(vf), scale, causal=causal)
    compare(to_f64(o), to_f64(lse), o_ref, lse_ref, float(v.abs().max()),
            "checked decode Nq%d Nk%d d%d %s" % (Nq, Nk, d, dtype), v.dtype, a_ref)


@pytest.mark.parametrize("d,dtype", [(64, "fp16"), (128, "bf16")])
@pytest.mark.parametrize("causal", [False, True])
def test_fa1_checked(chk, orc, d, dtype, causal):
    B, H, N = 1, 2, 520
    q, k, v = inputs.make_qkv(B, H, N, d, dtype, (6000 + d, 6100, 6200))
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws_bytes = chk.fa1_fwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    assert chk.fa1_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       ws.data_ptr(), ws_bytes, B, H, N, d, d ** -0.5, int(causal), _code(qd),
                       _stream()) == FA_OK
    _status(chk)
    check_full(orc, q, k, v, d ** -0.5, causal, o, lse, "checked fa1 d%d %s causal=%s" % (d, dtype, causal))
