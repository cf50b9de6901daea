"""ctypes binding of the C ABI in include/fa.h (argument marshalling only).

The shared library is built in-tree by ``attention_forward_02_gb300.build``.
There is no fallback: if the library is missing or fails to load, every call
raises ``FAError``.
"""
import ctypes
import os

from .build import LIB, LIB_CHECKED

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_CUDA = 4
FA_ERR_TIMEOUT = 5
FA_ERR_BOUNDS = 6
FA_FP16 = 0
FA_BF16 = 1

# every symbol include/fa.h declares
EXPORTS = ("fa_fwd", "fa1_fwd_workspace_size", "fa1_fwd", "fa1_fwd_noalloc", "fa_bwd_workspace_size",
           "fa_bwd", "fa_decode_workspace_size", "fa_decode", "fa_last_device_status",
           "fa_selftest_wait_timeout", "fa_selftest_bounds_check", "fa_checked_build",
           "fa_status_str", "fa_abi_version")

_lib = None
_lib_checked = None


class FAError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        name = status_name(status)
        super().__init__("%s%s" % (name, (": " + what) if what else ""))


def status_name(status):
    names = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
             4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_BOUNDS"}
    return names.get(int(status), "FA_ERR_UNKNOWN(%d)" % int(status))


def load(path=None):
    """Load (once) and return the CUDA library; raise if it is not built."""
    global _lib
    if _lib is None:
        _lib = _open(path or LIB)
    return _lib


def load_checked():
    """Load (once) and return the checked build of the library (the same
    entry points with device-side address checks; see include/fa.h)."""
    global _lib_checked
    if _lib_checked is None:
        _lib_checked = _open(LIB_CHECKED)
    return _lib_checked


def _open(path):
    if not os.path.exists(path):
        raise FAError(FA_ERR_CUDA, "CUDA library %s is not built; run "
                      "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.restype = i
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.fa1_fwd_workspace_size.restype = ctypes.c_size_t
    lib.fa1_fwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa1_fwd.restype = i
    lib.fa1_fwd.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, f, i, i, vp]
    lib.fa1_fwd_noalloc.restype = i
    lib.fa1_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, f, i,
                           i, vp]
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_decode.restype = i
    lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_size_t, i, i, i, i, i, f, i, i, vp]
    lib.fa_last_device_status.restype = i
    lib.fa_last_device_status.argtypes = [vp]
    lib.fa_selftest_wait_timeout.restype = i
    lib.fa_selftest_wait_timeout.argtypes = [i, vp]
    lib.fa_selftest_bounds_check.restype = i
    lib.fa_selftest_bounds_check.argtypes = [vp]
    lib.fa_checked_build.restype = i
    lib.fa_checked_build.argtypes = []
    lib.fa_status_str.restype = ctypes.c_char_p
    lib.fa_status_str.argtypes = [i]
    lib.fa_abi_version.restype = i
    lib.fa_abi_version.argtypes = []
    return lib


def lib_path():
    return LIB


def fa_fwd_raw(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream):
    """Direct call of the C entry point with integer pointers; returns the status."""
    return load().fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, stream)


def fa1_fwd_workspace_size(B, H, N, d):
    return load().fa1_fwd_workspace_size(B, H, N, d)


def fa1_fwd_raw(q, k, v, o, lse, ws, ws_bytes, B, H, N, d, scale, causal, dtype, stream):
    """Direct call of the FA1-structured entry point; returns the status."""
    return load().fa1_fwd(q, k, v, o, lse, ws, ws_bytes, B, H, N, d, scale, causal, dtype, stream)


def fa_bwd_workspace_size(B, H, N, d):
    return load().fa_bwd_workspace_size(B, H, N, d)


def fa_bwd_raw(q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes, B, H, N, d, scale, causal, dtype,
               stream):
    """Direct call of the backward entry point; returns the status."""
    return load().fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes, B, H, N, d, scale, causal,
                         dtype, stream)


def fa_decode_workspace_size(B, H, Nq, Nk, d):
    return load().fa_decode_workspace_size(B, H, Nq, Nk, d)


def fa_decode_raw(q, k, v, o, lse, ws, ws_bytes, B, H, Nq, Nk, d, scale, causal, dtype, stream):
    """Direct call of the decoding entry point; returns the status."""
    return load().fa_decode(q, k, v, o, lse, ws, ws_bytes, B, H, Nq, Nk, d, scale, causal, dtype,
                            stream)


def fa_last_device_status(stream=None):
    return load().fa_last_device_status(stream)


def fa_selftest_wait_timeout(limit_us, stream=None):
    return load().fa_selftest_wait_timeout(int(limit_us), stream)


def fa_selftest_bounds_check(stream=None):
    return load().fa_selftest_bounds_check(stream)


def fa_status_str(status):
    return load().fa_status_str(int(status)).decode()


def fa_abi_version():
    return load().fa_abi_version()
