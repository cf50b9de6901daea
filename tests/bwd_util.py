"""Helpers for the backward-pass parity tests (GPU fa_bwd against the fp64
oracle's gradients on the same rounded inputs).

Tolerance, element by element, derived from the roundings the kernel makes
(u = unit roundoff of the dtype: 2^-11 fp16, 2^-8 bf16).  With exact
P, dP = dO V^T, D_i = sum_c dO_ic O_ic and A_i = sum_c |dO_ic| |O_ic|:
  * P is recomputed from the forward's LSE (error dL_i, measured against the
    oracle's LSE) and rounded to the input dtype: relative error
    r_i = 2u + |dL_i| (one u of margin for exp2 and fp32 scores);
  * D comes from the stored (rounded) O: error <= 2u A_i;
  * dS = P (dP - D) scale is rounded to the input dtype (one more u);
  * dQ, dK, dV are accumulated in fp32 and rounded once (u |ref|).
So
  T_ij    = scale P_ij ((r_i + u) |dP_ij - D_i| + 2u A_i)
  |ddQ|  <= T |K|   + u |dQ_ref| + f
  |ddK|  <= T^T |Q| + u |dK_ref| + f
  |ddV|  <= (r P)^T |dO| + u |dV_ref| + f
with f = 1e-5 max|ref| for the fp32 accumulation.  P, dP, D, A here only size
the bound; the expected values are the oracle's.
"""
import json
import os

import numpy as np
import torch

UNIT_ROUNDOFF = {torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}
FLOOR_REL = 1e-5


def to_f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def run_gpu_fwd_bwd(q, k, v, do, scale, causal):
    """Forward then backward on cuda:0; returns CPU (o, lse, dq, dk, dv)."""
    import attention_forward_02_gb300 as fa
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    o, lse = fa.fa_fwd(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = fa.fa_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal)
    st = fa.fa_last_device_status(torch.cuda.current_stream(dev).cuda_stream)
    assert st == 0, "device status %s" % fa.fa_status_str(st)
    return o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


def _magnitudes(q, k, v, do, o, scale, causal):
    """Per head: exact P, |dP - D|, A (fp64, full matrices; small sizes only)."""
    s = scale * np.einsum("hid,hjd->hij", q, k)
    n = s.shape[-1]
    if causal:
        s = np.where(np.tril(np.ones((n, n), dtype=bool)), s, -np.inf)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    dp = np.einsum("hid,hjd->hij", do, v)
    dd = np.einsum("hid,hid->hi", do, o)
    a = np.einsum("hid,hid->hi", np.abs(do), np.abs(o))
    return p, np.abs(dp - dd[..., None]), a


def check_bwd(orc, q, k, v, do, scale, causal, gpu, what=""):
    """gpu = (o, lse, dq, dk, dv) from run_gpu_fwd_bwd; q, k, v, do CPU tensors."""
    o_g, lse_g, dq_g, dk_g, dv_g = gpu
    B, H, N, d = q.shape
    u = UNIT_ROUNDOFF[q.dtype]
    qf, kf, vf, dof = (to_f64(t) for t in (q, k, v, do))
    dq_r, dk_r, dv_r = orc.attention_bwd(qf, kf, vf, dof, scale, causal=causal)
    _, lse_r = orc.attention_fwd(qf, kf, vf, scale, causal=causal)
    hq, hk, hv, hdo = (x.reshape(B * H, N, d) for x in (qf, kf, vf, dof))
    ho = to_f64(o_g).reshape(B * H, N, d)
    p, adp, a = _magnitudes(hq, hk, hv, hdo, ho, scale, causal)
    dl = np.abs(to_f64(lse_g) - lse_r).reshape(B * H, N)
    r = 2 * u + dl
    t = scale * p * ((r + u)[..., None] * adp + 2 * u * a[..., None])
    bounds = {
        "dq": np.einsum("hij,hjd->hid", t, np.abs(hk)),
        "dk": np.einsum("hij,hid->hjd", t, np.abs(hq)),
        "dv": np.einsum("hij,hid->hjd", r[..., None] * p, np.abs(hdo)),
    }
    res = {}
    for name, g, ref in (("dq", dq_g, dq_r), ("dk", dk_g, dk_r), ("dv", dv_g, dv_r)):
        gf = to_f64(g).reshape(B * H, N, d)
        rf = ref.reshape(B * H, N, d)
        assert np.all(np.isfinite(gf)), "%s: non-finite %s" % (what, name)
        bound = bounds[name] + u * np.abs(rf) + FLOOR_REL * max(float(np.abs(rf).max()), 1e-30)
        err = np.abs(gf - rf)
        ratio = err / bound
        worst = int(np.argmax(ratio))
        res[name + "_max_err"] = float(err.max())
        res[name + "_max_ratio"] = float(ratio.flat[worst])
        res[name + "_ref_max"] = float(np.abs(rf).max())
        assert ratio.flat[worst] <= 1.0, (
            "%s: |d%s| = %.4g > bound %.4g at flat index %d (ref %.4g, max|ref| %.4g)" %
            (what, name, err.flat[worst], bound.flat[worst], worst, rf.flat[worst],
             float(np.abs(rf).max())))
    log = os.environ.get("FA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(dict(what=what, dtype=str(q.dtype), **res)) + "\n")
    return res
