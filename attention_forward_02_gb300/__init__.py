"""GB300-native (sm_103a) FlashAttention-2 style attention.

``fa_fwd(q, k, v, ...)`` computes O = softmax(Q K^T * scale) V and the row
log-sum-exp for contiguous [B, H, N, d] fp16/bf16 CUDA tensors by calling the
C ABI (include/fa.h) of the in-tree CUDA library on the current torch stream;
``fa_bwd`` computes the gradients of q, k, v from the forward's o and lse;
``fa_decode`` runs a few query rows per head against a long KV sequence
(split-KV).
PyTorch only supplies device memory and the stream; every step of the
computation runs in the library's kernel.  There is no CPU or eager fallback:
without the built library, or off a CUDA device, calls raise ``FAError``.
"""
from ._lib import (FA_BF16, FA_FP16, FAError, fa1_fwd_raw, fa1_fwd_workspace_size,
                   fa_abi_version, fa_bwd_raw, fa_bwd_workspace_size, fa_decode_raw,
                   fa_decode_workspace_size, fa_fwd_raw, fa_last_device_status,
                   fa_selftest_bounds_check, fa_selftest_wait_timeout, fa_status_str, lib_path,
                   load, load_checked)

__all__ = ["fa_fwd", "fa_fwd_raw", "fa1_fwd", "fa1_fwd_raw", "fa1_fwd_workspace_size",
           "fa_bwd", "fa_bwd_raw", "fa_bwd_workspace_size",
           "fa_decode", "fa_decode_raw", "fa_decode_workspace_size",
           "fa_last_device_status", "fa_selftest_wait_timeout", "fa_selftest_bounds_check",
           "fa_status_str", "fa_abi_version", "FAError", "load", "load_checked", "lib_path"]


def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise FAError(2, "dtype must be float16 or bfloat16, got %s" % t.dtype)


def _check_qkv(q, k, v):
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise FAError(1, "%s must be a CUDA tensor" % name)
        if t.dim() != 4 or not t.is_contiguous():
            raise FAError(1, "%s must be a contiguous [B, H, N, d] tensor" % name)
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise FAError(1, "q, k, v must share shape and dtype")


def _outputs(q, o, lse, return_lse):
    import torch
    B, H, N, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or not o.is_cuda:
        raise FAError(1, "o must be a contiguous CUDA tensor shaped and typed like q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    if lse is not None and (lse.shape != (B, H, N) or lse.dtype != torch.float32
                            or not lse.is_contiguous() or not lse.is_cuda):
        raise FAError(1, "lse must be a contiguous CUDA float32 tensor of shape [B, H, N]")
    return o, lse


def fa1_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, return_lse=True, workspace=None,
            stream=None):
    """The FA1-structured baseline (same arguments and results as fa_fwd).

    workspace: optional CUDA uint8 tensor of at least fa1_fwd_workspace_size
    bytes; allocated with torch when None."""
    import torch
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    code = _dtype_code(q)
    if scale is None:
        scale = float(d) ** -0.5
    o, lse = _outputs(q, o, lse, return_lse)
    need = fa1_fwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa1_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                         lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), B, H, N, d, float(scale),
                         int(bool(causal)), code, stream.cuda_stream)
    if st != 0:
        raise FAError(st, "fa1_fwd")
    return o, lse


def fa_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, return_lse=True, stream=None):
    """Attention forward on CUDA tensors q, k, v of shape [B, H, N, d].

    o / lse: optional preallocated outputs ([B,H,N,d] in q's dtype and
    [B,H,N] fp32); allocated with torch when None (lse only if return_lse).
    scale defaults to 1/sqrt(d).  Returns (o, lse) (lse None if not requested).
    The call is asynchronous on ``stream`` (default: torch's current stream).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise FAError(1, "%s must be a CUDA tensor" % name)
        if t.dim() != 4 or not t.is_contiguous():
            raise FAError(1, "%s must be a contiguous [B, H, N, d] tensor" % name)
    if k.shape != q.shape or v.shape != q.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise FAError(1, "q, k, v must share shape and dtype")
    B, H, N, d = q.shape
    code = _dtype_code(q)
    if scale is None:
        scale = float(d) ** -0.5
    if o is None:
        o = torch.empty_like(q)
    elif o.shape != q.shape or o.dtype != q.dtype or not o.is_contiguous() or not o.is_cuda:
        raise FAError(1, "o must be a contiguous CUDA tensor shaped and typed like q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    if lse is not None and (lse.shape != (B, H, N) or lse.dtype != torch.float32
                            or not lse.is_contiguous() or not lse.is_cuda):
        raise FAError(1, "lse must be a contiguous CUDA float32 tensor of shape [B, H, N]")
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                        lse.data_ptr() if lse is not None else None, B, H, N, d, float(scale),
                        int(bool(causal)), code, stream.cuda_stream)
    if st != 0:
        raise FAError(st, "fa_fwd")
    return o, lse


def fa_bwd(q, k, v, o, lse, dout, scale=None, causal=False, dq=None, dk=None, dv=None,
           workspace=None, stream=None):
    """Attention backward: gradients (dq, dk, dv) of a loss given dout = dL/do.

    q, k, v, o, dout: contiguous [B, H, N, d] CUDA tensors of one dtype (o the
    forward output for q, k, v); lse: the forward's [B, H, N] fp32 log-sum-exp.
    scale and causal must be the forward's.  dq/dk/dv: optional preallocated
    outputs; workspace: optional CUDA uint8 tensor of at least
    fa_bwd_workspace_size bytes (allocated with torch when None)."""
    import torch
    _check_qkv(q, k, v)
    for name, t in (("o", o), ("dout", dout)):
        if (not isinstance(t, torch.Tensor) or not t.is_cuda or t.shape != q.shape
                or t.dtype != q.dtype or not t.is_contiguous()):
            raise FAError(1, "%s must be a contiguous CUDA tensor shaped and typed like q" % name)
    B, H, N, d = q.shape
    if (not isinstance(lse, torch.Tensor) or not lse.is_cuda or lse.shape != (B, H, N)
            or lse.dtype != torch.float32 or not lse.is_contiguous()):
        raise FAError(1, "lse must be a contiguous CUDA float32 tensor of shape [B, H, N]")
    code = _dtype_code(q)
    if scale is None:
        scale = float(d) ** -0.5
    outs = []
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t is None:
            t = torch.empty_like(q)
        elif t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or not t.is_cuda:
            raise FAError(1, "%s must be a contiguous CUDA tensor shaped and typed like q" % name)
        outs.append(t)
    dq, dk, dv = outs
    need = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(), B, H, N,
                        d, float(scale), int(bool(causal)), code, stream.cuda_stream)
    if st != 0:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv


def fa_decode(q, k, v, o=None, lse=None, scale=None, causal=False, return_lse=True, workspace=None,
              stream=None):
    """Decoding attention: q [B, H, Nq, d] (1 <= Nq <= 16) against k, v
    [B, H, Nk, d] (Nk >= Nq), CUDA tensors of one 16-bit dtype.  causal puts
    the queries at the end of the sequence.  Returns (o, lse)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise FAError(1, "%s must be a CUDA tensor" % name)
        if t.dim() != 4 or not t.is_contiguous():
            raise FAError(1, "%s must be a contiguous [B, H, N, d] tensor" % name)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if (k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != d
            or k.dtype != q.dtype or v.dtype != q.dtype):
        raise FAError(1, "k, v must be [B, H, Nk, d] like q")
    code = _dtype_code(q)
    if scale is None:
        scale = float(d) ** -0.5
    o, lse = _outputs(q, o, lse, return_lse)
    need = fa_decode_workspace_size(B, H, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        st = fa_decode_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr() if lse is not None else None, workspace.data_ptr(),
                           workspace.numel() * workspace.element_size(), B, H, Nq, Nk, d,
                           float(scale), int(bool(causal)), code, stream.cuda_stream)
    if st != 0:
        raise FAError(st, "fa_decode")
    return o, lse
