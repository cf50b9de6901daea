"""fp64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE.

Only tests/, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, loads or calls it, and the two share no code.

The arithmetic lives in ``attention_oracle.c`` (plain C, fp64); this module
only marshals numpy arrays through ctypes.  What it computes, per head and
query row i (allowed keys: all, or j <= i when causal):

    s_j = scale * <q_i, k_j>,  m = max s_j,  l = sum exp(s_j - m),
    o_i = sum exp(s_j - m) v_j / l,  lse_i = m + ln l

following "3.6 어텐션 I — 메모리 문제·FlashAttention 원리" sections 3.6.4
(stable softmax, online recurrence), 3.6.6 (causal skip of j > i) and 3.6.7
(L = m + log l), and the formula in the section "커널 구조는 단순한데, 디테일이
지옥임" of "FlashAttention-2를 CuTe로 밑바닥부터 구현하며 겪은 GPU 커널 지옥기".

Every function is pinned by tests/test_oracle_pins.py and
tests/test_oracle_mutations.py (no function here is "parity unpinned").
"""
import ctypes
import os

import numpy as np

from .build import LIB, build_oracle

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


class OracleError(RuntimeError):
    pass


class Oracle:
    """ctypes front-end for one build of the oracle library."""

    def __init__(self, lib_path=None):
        path = lib_path or build_oracle()
        self.path = path
        self._lib = ctypes.CDLL(path)
        L = self._lib
        L.oracle_attention_rows.restype = ctypes.c_int
        L.oracle_attention_rows.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                            ctypes.c_long, ctypes.c_double, ctypes.c_int,
                                            _lp, ctypes.c_long, _dp, _dp, ctypes.c_int]
        L.oracle_attention_fwd.restype = ctypes.c_int
        L.oracle_attention_fwd.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                           ctypes.c_long, ctypes.c_double, ctypes.c_int,
                                           _dp, _dp, ctypes.c_int]
        L.oracle_scores_row.restype = ctypes.c_int
        L.oracle_scores_row.argtypes = [_dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                        ctypes.c_double, ctypes.c_int, _dp,
                                        ctypes.POINTER(ctypes.c_long)]
        L.oracle_online_row.restype = ctypes.c_int
        L.oracle_online_row.argtypes = [_dp, _dp, ctypes.c_long, ctypes.c_long, _lp, _lp,
                                        ctypes.c_long, _dp, _dp, _dp, _dp]
        L.oracle_attention_bwd.restype = ctypes.c_int
        L.oracle_attention_bwd.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                           ctypes.c_long, ctypes.c_double, ctypes.c_int,
                                           _dp, _dp, _dp, ctypes.c_int]
        L.oracle_attention_bwd_rows.restype = ctypes.c_int
        L.oracle_attention_bwd_rows.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                                ctypes.c_long, ctypes.c_double, ctypes.c_int,
                                                ctypes.POINTER(ctypes.c_long), ctypes.c_long, _dp,
                                                ctypes.c_int]
        L.oracle_attention_decode.restype = ctypes.c_int
        L.oracle_attention_decode.argtypes = [_dp, _dp, _dp, ctypes.c_long, ctypes.c_long,
                                              ctypes.c_long, ctypes.c_long, ctypes.c_double,
                                              ctypes.c_int, _dp, _dp, ctypes.c_int]
        L.oracle_abi_version.restype = ctypes.c_int

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _f64(a):
        return np.ascontiguousarray(np.asarray(a, dtype=np.float64))

    @staticmethod
    def _ptr(a, t=_dp):
        return a.ctypes.data_as(t)

    @staticmethod
    def default_threads():
        return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                   else (os.cpu_count() or 1))

    # -- plain definition --------------------------------------------------
    def attention_fwd(self, q, k, v, scale, causal=False, threads=None):
        """q, k, v: [B, H, N, d] (any float dtype, converted exactly to fp64).

        Returns (o [B,H,N,d] fp64, lse [B,H,N] fp64)."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
            raise OracleError("q, k, v must share a [B,H,N,d] shape")
        B, H, N, d = q.shape
        o = np.empty_like(q)
        lse = np.empty((B, H, N), dtype=np.float64)
        st = self._lib.oracle_attention_fwd(self._ptr(q), self._ptr(k), self._ptr(v),
                                            B * H, N, d, float(scale), int(bool(causal)),
                                            self._ptr(o), self._ptr(lse),
                                            threads or self.default_threads())
        if st != 0:
            raise OracleError("oracle_attention_fwd returned %d" % st)
        return o, lse

    def attention_rows(self, q, k, v, rows, scale, causal=False, threads=None):
        """Plain definition on selected rows.

        q, k, v: [B, H, N, d]; rows: int array [R, 2] of (bh, i) with
        bh = b * H + h.  Returns (o [R, d], lse [R]) in fp64."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        B, H, N, d = q.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
        R = rows.shape[0]
        o = np.empty((R, d), dtype=np.float64)
        lse = np.empty((R,), dtype=np.float64)
        st = self._lib.oracle_attention_rows(self._ptr(q), self._ptr(k), self._ptr(v),
                                             B * H, N, d, float(scale), int(bool(causal)),
                                             self._ptr(rows, _lp), R, self._ptr(o),
                                             self._ptr(lse), threads or self.default_threads())
        if st != 0:
            raise OracleError("oracle_attention_rows returned %d" % st)
        return o, lse

    def scores_row(self, q, k, i, scale, causal=False):
        """Scaled scores of query row i of one head (q, k: [N, d])."""
        q, k = self._f64(q), self._f64(k)
        N, d = q.shape
        s = np.empty((N,), dtype=np.float64)
        n = ctypes.c_long(0)
        st = self._lib.oracle_scores_row(self._ptr(q), self._ptr(k), N, d, int(i),
                                         float(scale), int(bool(causal)), self._ptr(s),
                                         ctypes.byref(n))
        if st != 0:
            raise OracleError("oracle_scores_row returned %d" % st)
        return s[: n.value].copy()

    def attention_decode(self, q, k, v, scale, causal=False, threads=None):
        """Nq queries q [B,H,Nq,d] against Nk >= Nq keys k, v [B,H,Nk,d];
        causal aligns the queries with the end of the keys.  Returns
        (o [B,H,Nq,d], lse [B,H,Nq]) fp64."""
        q, k, v = self._f64(q), self._f64(k), self._f64(v)
        if q.ndim != 4 or k.ndim != 4 or k.shape != v.shape or q.shape[:2] != k.shape[:2] \
                or q.shape[3] != k.shape[3]:
            raise OracleError("q [B,H,Nq,d], k and v [B,H,Nk,d] expected")
        B, H, Nq, d = q.shape
        Nk = k.shape[2]
        o = np.empty_like(q)
        lse = np.empty((B, H, Nq))
        st = self._lib.oracle_attention_decode(self._ptr(q), self._ptr(k), self._ptr(v), B * H, Nq,
                                               Nk, d, float(scale), int(bool(causal)), self._ptr(o),
                                               self._ptr(lse), threads or self.default_threads())
        if st != 0:
            raise OracleError("oracle_attention_decode returned %d" % st)
        return o, lse

    def attention_bwd(self, q, k, v, g, scale, causal=False, threads=None):
        """Gradients (dq, dk, dv) of sum(o * g) for the plain definition.

        q, k, v, g: [B, H, N, d]; returns three fp64 arrays of that shape."""
        q, k, v, g = self._f64(q), self._f64(k), self._f64(v), self._f64(g)
        if q.ndim != 4 or any(t.shape != q.shape for t in (k, v, g)):
            raise OracleError("q, k, v, g must share a [B,H,N,d] shape")
        B, H, N, d = q.shape
        dq, dk, dv = np.empty_like(q), np.empty_like(q), np.empty_like(q)
        st = self._lib.oracle_attention_bwd(self._ptr(q), self._ptr(k), self._ptr(v),
                                            self._ptr(g), B * H, N, d, float(scale),
                                            int(bool(causal)), self._ptr(dq), self._ptr(dk),
                                            self._ptr(dv), threads or self.default_threads())
        if st != 0:
            raise OracleError("oracle_attention_bwd returned %d" % st)
        return dq, dk, dv

    def attention_bwd_rows(self, q, k, v, g, rows, scale, causal=False, threads=None):
        """dq of the listed query rows; rows: int array [n, 2] of (flattened
        head, query index).  Returns [n, d] fp64."""
        q, k, v, g = self._f64(q), self._f64(k), self._f64(v), self._f64(g)
        if q.ndim != 4 or any(t.shape != q.shape for t in (k, v, g)):
            raise OracleError("q, k, v, g must share a [B,H,N,d] shape")
        B, H, N, d = q.shape
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
        out = np.empty((len(rows), d))
        st = self._lib.oracle_attention_bwd_rows(
            self._ptr(q), self._ptr(k), self._ptr(v), self._ptr(g), B * H, N, d, float(scale),
            int(bool(causal)), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_long)), len(rows),
            self._ptr(out), threads or self.default_threads())
        if st != 0:
            raise OracleError("oracle_attention_bwd_rows returned %d" % st)
        return out

    # -- online recurrence -------------------------------------------------
    def online_row(self, s, v, blocks):
        """Online softmax over one row.

        s: [n] scores; v: [n] or [n, d] values; blocks: list of (start, length)
        in processing order.  Returns dict with o (normalised [d]), l, m and
        trace: a list of per-block dicts (m_tilde, m_new, alpha, l, O)."""
        s = self._f64(s).reshape(-1)
        v = self._f64(v)
        if v.ndim == 1:
            v = v.reshape(-1, 1)
        n, d = v.shape
        starts = np.ascontiguousarray(np.array([b[0] for b in blocks], dtype=np.int64))
        lens = np.ascontiguousarray(np.array([b[1] for b in blocks], dtype=np.int64))
        nb = len(blocks)
        o = np.empty((d,), dtype=np.float64)
        l = ctypes.c_double(0.0)
        m = ctypes.c_double(0.0)
        trace = np.empty((nb, 4 + d), dtype=np.float64)
        st = self._lib.oracle_online_row(self._ptr(s), self._ptr(v), n, d,
                                         self._ptr(starts, _lp), self._ptr(lens, _lp), nb,
                                         self._ptr(o), ctypes.byref(l), ctypes.byref(m),
                                         self._ptr(trace))
        if st != 0:
            raise OracleError("oracle_online_row returned %d" % st)
        tr = [dict(m_tilde=t[0], m_new=t[1], alpha=t[2], l=t[3], O=t[4:].copy()) for t in trace]
        return dict(o=o, l=l.value, m=m.value, trace=tr)


_DEFAULT = None


def get():
    """The oracle built from this package's source (built on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
