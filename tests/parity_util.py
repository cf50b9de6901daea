"""Helpers for the GPU-vs-oracle parity tests.

Tolerance (stated for fp16/bf16 inputs with fp32 accumulation):
  max |O_gpu - O_ref| <= 2e-3 * max|V|   and   max |LSE_gpu - LSE_ref| <= 1e-3
where O_ref, LSE_ref come from the fp64 oracle on the same (rounded) inputs.
"""
import numpy as np
import torch

O_TOL_REL_VMAX = 2e-3
LSE_TOL = 1e-3


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
    return compare(to_f64(o), None if lse is None else to_f64(lse), o_ref, lse_ref,
                   float(v.abs().max()), what)


def check_rows(orc, q, k, v, scale, causal, o, lse, rows, what=""):
    """Compare sampled rows (bh, i) of the GPU output with the oracle."""
    B, H, N, d = q.shape
    o_ref, lse_ref = orc.attention_rows(to_f64(q), to_f64(k), to_f64(v), rows, scale,
                                        causal=causal)
    og = o.reshape(B * H, N, d)[torch.as_tensor(rows[:, 0]), torch.as_tensor(rows[:, 1])]
    lg = None if lse is None else lse.reshape(B * H, N)[torch.as_tensor(rows[:, 0]),
                                                         torch.as_tensor(rows[:, 1])]
    return compare(to_f64(og), None if lg is None else to_f64(lg), o_ref, lse_ref,
                   float(v.abs().max()), what)


def compare(o, lse, o_ref, lse_ref, vmax, what=""):
    assert np.all(np.isfinite(o)), "%s: non-finite O" % what
    err = np.abs(o - o_ref)
    e_max = float(err.max()) if err.size else 0.0
    e_999 = float(np.quantile(err, 0.999)) if err.size else 0.0
    bound = O_TOL_REL_VMAX * vmax
    assert e_max <= bound, "%s: max|dO| = %.4g > %.4g (p99.9 %.3g)" % (what, e_max, bound, e_999)
    res = dict(o_max_err=e_max, o_p999_err=e_999, o_bound=bound)
    if lse is not None:
        assert np.all(np.isfinite(lse)), "%s: non-finite LSE" % what
        le = float(np.abs(lse - lse_ref).max()) if lse.size else 0.0
        assert le <= LSE_TOL, "%s: max|dLSE| = %.4g > %g" % (what, le, LSE_TOL)
        res["lse_max_err"] = le
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
