"""Helpers for the GPU-vs-oracle parity tests.

Tolerance (fp16/bf16 inputs, fp32 accumulation), O_ref and LSE_ref from the
fp64 oracle on the same rounded inputs:

  fp16:  max |O_gpu - O_ref| <= 2e-3 * max|V|
  bf16:  |O_gpu - O_ref| <= 2e-3 * max|V| + u * (|O_ref| + A_ref)   element-wise
  both:  max |LSE_gpu - LSE_ref| <= 1e-3

For bf16 the fixed bound alone is below what the format can hold on short
rows: the method rounds P to V's dtype before the second product (P.to(V's
dtype) in "Triton으로 FlashAttention 1·2 forward 구현하기", section "출력 누적
방식") and the output is stored in bf16.  Each rounding has unit roundoff
u = 2^-8 for bf16, so the two add at most u * sum_j w_j |v_j| (= u * A_ref,
A_ref being the oracle's output with |V| as values) and u * |O_ref| on top of
the fp32 accumulation error that the fixed bound covers.  For fp16
(u = 2^-11) the same terms stay inside the fixed bound, so fp16 keeps it alone.
"""
import json
import os

import numpy as np
import torch

O_TOL_REL_VMAX = 2e-3
LSE_TOL = 1e-3
UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}


def to_f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_gpu(q, k, v, scale, causal, with_lse=True):
    import attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = fa.fa_fwd(qd, kd, vd, scale=scale, causal=causal, return_lse=with_lse)
    st = fa.fa_last_device_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, "device status %s" % fa.fa_status_str(st)
    return o, lse


def check_full(orc, q, k, v, scale, causal, o, lse, what=""):
    o_ref, lse_ref = orc.attention_fwd(to_f64(q), to_f64(k), to_f64(v), scale, causal=causal)
    a_ref = None
    if v.dtype == torch.bfloat16:
        a_ref, _ = orc.attention_fwd(to_f64(q), to_f64(k), np.abs(to_f64(v)), scale, causal=causal)
    return compare(to_f64(o), None if lse is None else to_f64(lse), o_ref, lse_ref,
                   float(v.abs().max()), what, v.dtype, a_ref)


def check_rows(orc, q, k, v, scale, causal, o, lse, rows, what=""):
    """Compare sampled rows (bh, i) of the GPU output with the oracle."""
    B, H, N, d = q.shape
    o_ref, lse_ref = orc.attention_rows(to_f64(q), to_f64(k), to_f64(v), rows, scale,
                                        causal=causal)
    a_ref = None
    if v.dtype == torch.bfloat16:
        a_ref, _ = orc.attention_rows(to_f64(q), to_f64(k), np.abs(to_f64(v)), rows, scale,
                                      causal=causal)
    og = o.reshape(B * H, N, d)[torch.as_tensor(rows[:, 0]), torch.as_tensor(rows[:, 1])]
    lg = None if lse is None else lse.reshape(B * H, N)[torch.as_tensor(rows[:, 0]),
                                                         torch.as_tensor(rows[:, 1])]
    return compare(to_f64(og), None if lg is None else to_f64(lg), o_ref, lse_ref,
                   float(v.abs().max()), what, v.dtype, a_ref)


def compare(o, lse, o_ref, lse_ref, vmax, what="", dtype=torch.float16, a_ref=None):
    assert np.all(np.isfinite(o)), "%s: non-finite O" % what
    err = np.abs(o - o_ref)
    e_max = float(err.max()) if err.size else 0.0
    e_999 = float(np.quantile(err, 0.999)) if err.size else 0.0
    fixed = O_TOL_REL_VMAX * vmax
    if dtype == torch.bfloat16:
        assert a_ref is not None, "bf16 needs the |V| oracle output"
        bound = fixed + UNIT_ROUNDOFF[dtype] * (np.abs(o_ref) + a_ref)
    else:
        bound = np.full(err.shape, fixed)
    excess = err - bound
    worst = int(np.argmax(excess)) if err.size else 0
    assert err.size == 0 or excess.flat[worst] <= 0.0, (
        "%s: |dO| = %.4g > bound %.4g at flat index %d (max|dO| %.4g, fixed bound %.4g, "
        "p99.9 %.3g)" % (what, err.flat[worst], bound.flat[worst], worst, e_max, fixed, e_999))
    res = dict(o_max_err=e_max, o_p999_err=e_999, o_fixed_bound=fixed,
               frac_within_fixed=float(np.mean(err <= fixed)) if err.size else 1.0)
    if lse is not None:
        assert np.all(np.isfinite(lse)), "%s: non-finite LSE" % what
        le = float(np.abs(lse - lse_ref).max()) if lse.size else 0.0
        res["lse_max_err"] = le
        assert le <= LSE_TOL, "%s: max|dLSE| = %.4g > %g" % (what, le, LSE_TOL)
    log = os.environ.get("FA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(dict(what=what, dtype=str(dtype), **res)) + "\n")
    return res


def edge_rows(B, H, N, extra):
    """Seeded row sample plus the rows at tile edges and the ragged tail."""
    from attention_forward_02_gb300 import inputs
    rows = [tuple(r) for r in extra]
    edges = sorted({0, 1, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1})
    for bh in range(B * H):
        for i in edges:
            if 0 <= i < N:
                rows.append((bh, i))
    return np.unique(np.array(rows, dtype=np.int64).reshape(-1, 2), axis=0)
