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


def _bounds(q, k, v, do, o, dl, scale, causal, u, block=256):
    """Per-head bound tensors for dQ, dK, dV (see the module docstring), built
    over query-row blocks so that only [block, N] slices of P exist at once.
    q, k, v, do, o: [BH, N, d] fp64; dl: [BH, N] measured LSE error."""
    BH, N, d = q.shape
    bq, bk, bv = np.zeros_like(q), np.zeros_like(q), np.zeros_like(q)
    ak, aq, ado = np.abs(k), np.abs(q), np.abs(do)
    for i0 in range(0, N, block):
        i1 = min(N, i0 + block)
        s = scale * np.einsum("hid,hjd->hij", q[:, i0:i1], k)
        if causal:
            allowed = np.arange(N)[None, :] <= np.arange(i0, i1)[:, None]
            s = np.where(allowed[None], s, -np.inf)
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=-1, keepdims=True)
        dp = np.einsum("hid,hjd->hij", do[:, i0:i1], v)
        dd = np.einsum("hid,hid->hi", do[:, i0:i1], o[:, i0:i1])
        a = np.einsum("hid,hid->hi", ado[:, i0:i1], np.abs(o[:, i0:i1]))
        r = 2 * u + dl[:, i0:i1]
        t = scale * p * ((r + u)[..., None] * np.abs(dp - dd[..., None]) + 2 * u * a[..., None])
        bq[:, i0:i1] = np.einsum("hij,hjd->hid", t, ak)
        bk += np.einsum("hij,hid->hjd", t, aq[:, i0:i1])
        bv += np.einsum("hij,hid->hjd", r[..., None] * p, ado[:, i0:i1])
    return {"dq": bq, "dk": bk, "dv": bv}


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
    dl = np.abs(to_f64(lse_g) - lse_r).reshape(B * H, N)
    bounds = _bounds(hq, hk, hv, hdo, ho, dl, scale, causal, u)
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


def check_bwd_heads(orc, q, k, v, do, scale, causal, gpu, heads, what=""):
    """check_bwd restricted to the listed (flattened batch*head) heads."""
    B, H, N, d = q.shape
    sel = torch.as_tensor(heads)

    def pick(t, shape):
        return t.reshape(B * H, *shape)[sel].reshape(1, len(heads), *shape)

    sub = tuple(pick(t, (N, d)) for t in (q, k, v, do))
    o_g, lse_g, dq_g, dk_g, dv_g = gpu
    gsub = (pick(o_g, (N, d)), pick(lse_g, (N,)), pick(dq_g, (N, d)), pick(dk_g, (N, d)),
            pick(dv_g, (N, d)))
    return check_bwd(orc, *sub, scale, causal, gsub, what)


def check_dv_identity(do, dv, what=""):
    """Rows of P sum to 1, so per head and column c, sum_j dV_jc = sum_i dO_ic
    at any size.  Bound from the per-element dV bound above summed over j
    (sum_j P_ij = 1), with r = 3u: |err| <= r sum_i |dO_ic| + u sum_j |dV_jc|."""
    u = UNIT_ROUNDOFF[do.dtype]
    dtype = str(do.dtype)
    do, dv = do.detach().to(torch.float64), dv.detach().to(torch.float64)
    err = (dv.sum(2) - do.sum(2)).abs()
    bound = 3 * u * do.abs().sum(2) + u * dv.abs().sum(2)
    ratio = float((err / bound).max())
    assert ratio <= 1.0, "%s: sum_j dV_j vs sum_i dO_i ratio %.3g > 1" % (what, ratio)
    log = os.environ.get("FA_PARITY_LOG")
    if log:
        with open(log, "a") as fh:
            fh.write(json.dumps(dict(what=what, dtype=dtype, dv_identity_ratio=ratio)) + "\n")
    return ratio


def check_dq_rows(orc, q, k, v, do, o, lse, dq, rows, scale, causal, what=""):
    """Sampled rows (flattened head, query) of the GPU dQ at any size against
    the oracle's dQ rows (each O(N d)), with the dQ bound of the module
    docstring evaluated for those rows.  Tensors: CPU [B, H, N, d]; lse and
    the GPU o, dq as returned by the kernels."""
    B, H, N, d = q.shape
    u = UNIT_ROUNDOFF[q.dtype]
    qf, kf, vf, dof = (to_f64(t) for t in (q, k, v, do))
    ref = orc.attention_bwd_rows(qf, kf, vf, dof, rows, scale, causal=causal)
    _, lse_r = orc.attention_rows(qf, kf, vf, rows, scale, causal=causal)
    hq, hk, hv, hdo = (x.reshape(B * H, N, d) for x in (qf, kf, vf, dof))
    ho = to_f64(o).reshape(B * H, N, d)
    lg = to_f64(lse).reshape(B * H, N)
    gq = to_f64(dq).reshape(B * H, N, d)
    worst = 0.0
    for r, (bh, i) in enumerate(rows):
        nk = i + 1 if causal else N
        s = scale * hk[bh, :nk] @ hq[bh, i]
        p = np.exp(s - s.max())
        p /= p.sum()
        dp = hv[bh, :nk] @ hdo[bh, i]
        dd = float(hdo[bh, i] @ ho[bh, i])
        a = float(np.abs(hdo[bh, i]) @ np.abs(ho[bh, i]))
        rr = 2 * u + abs(lg[bh, i] - lse_r[r])
        t = scale * p * ((rr + u) * np.abs(dp - dd) + 2 * u * a)
        bound = t @ np.abs(hk[bh, :nk]) + u * np.abs(ref[r]) + FLOOR_REL * max(float(np.abs(ref).max()), 1e-30)
        err = np.abs(gq[bh, i] - ref[r])
        assert np.all(np.isfinite(gq[bh, i])), "%s: non-finite dq row %s" % (what, (bh, i))
        ratio = float((err / bound).max())
        worst = max(worst, ratio)
        assert ratio <= 1.0, "%s: dq row (%d, %d): err %.4g > bound %.4g" % (
            what, bh, i, float(err.max()), float(bound[np.argmax(err / bound)]))
    log = os.environ.get("FA_PARITY_LOG")
    if log:
        with open(log, "a") as fh:
            fh.write(json.dumps(dict(what=what, dtype=str(q.dtype), dq_rows_max_ratio=worst,
                                     rows=len(rows))) + "\n")
    return worst
