"""The C-ABI library builds, loads and exports every symbol include/fa.h
declares; argument errors are rejected before any CUDA call.  CPU only: no
call here reaches a kernel launch."""
import ctypes
import os
import re

import pytest

import attention_forward_02_gb300 as fa
from attention_forward_02_gb300 import _lib
from attention_forward_02_gb300.build import INCLUDE, build_library

HEADER = os.path.join(INCLUDE, "fa.h")


@pytest.fixture(scope="module")
def lib():
    build_library()
    return fa.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_checked_build_exports_the_same_symbols(lib):
    """The checked build (device-side address checks) is the same ABI."""
    chk = _lib.load_checked()
    for name in declared_functions():
        assert hasattr(chk, name), name
    assert chk.fa_checked_build() == 1 and lib.fa_checked_build() == 0
    assert chk.fa_abi_version() == lib.fa_abi_version()


def test_abi_version_matches_header(lib):
    m = re.search(r"#define FA_ABI_VERSION (\d+)", open(HEADER).read())
    assert fa.fa_abi_version() == int(m.group(1))


def test_status_strings(lib):
    names = ["FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_MISALIGNED",
             "FA_ERR_CUDA", "FA_ERR_TIMEOUT", "FA_ERR_BOUNDS"]
    for code, name in enumerate(names):
        assert fa.fa_status_str(code) == name
        assert _lib.status_name(code) == name
    assert fa.fa_status_str(99) == "FA_ERR_UNKNOWN"


# Fake, well-separated, 16-byte-aligned "device" addresses: every call below
# must be rejected (or be an empty problem) before the library touches CUDA.
Q, K, V, O, L = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def call(q=Q, k=K, v=V, o=O, lse=L, B=1, H=2, N=256, d=64, scale=0.125, causal=0, dtype=0):
    return fa.fa_fwd_raw(q, k, v, o, lse, B, H, N, d, scale, causal, dtype, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(d=48), 2), (dict(d=16), 2), (dict(d=256), 2),
    (dict(dtype=7), 2), (dict(scale=-1.0), 2),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(causal=2), 1), (dict(B=-1), 1), (dict(N=-5), 1),
    (dict(q=0), 1), (dict(o=0), 1),
    (dict(q=Q + 2), 3), (dict(k=K + 8), 3), (dict(o=O + 4), 3), (dict(lse=L + 2), 3),
    (dict(o=Q + 4096), 1),          # output overlaps q
    (dict(lse=O + 64), 1),          # lse overlaps o
    (dict(B=65536, H=65536), 2),    # more CTAs than a 1-D grid allows
    (dict(N=0), 0), (dict(B=0), 0), (dict(H=0, q=0, o=0), 0),  # empty problems
], ids=lambda x: str(x))
def test_argument_checks(lib, kwargs, status):
    assert call(**kwargs) == status


def test_fa1_workspace_size(lib):
    assert fa.fa1_fwd_workspace_size(4, 32, 2048, 64) == 4 * 32 * 2048 * 66 * 4
    assert fa.fa1_fwd_workspace_size(1, 1, 1, 128) == 130 * 4
    assert fa.fa1_fwd_workspace_size(1, 1, 1, 96) == 98 * 4
    assert fa.fa1_fwd_workspace_size(1, 1, 1, 48) == 0
    assert fa.fa1_fwd_workspace_size(-1, 1, 1, 64) == 0


W = 0x60000000


def call_fa1(ws=W, ws_bytes=1 << 30, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=2, N=256, d=64, scale=0.125, causal=0, dtype=0)
    a.update(kw)
    return fa.fa1_fwd_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], ws, ws_bytes, a["B"], a["H"],
                          a["N"], a["d"], a["scale"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(ws=0), 1), (dict(ws_bytes=100), 1), (dict(ws=W + 8), 3), (dict(ws=Q), 1),
    (dict(d=48), 2), (dict(causal=3), 1), (dict(N=0), 0),
], ids=lambda x: str(x))
def test_fa1_argument_checks(lib, kwargs, status):
    assert call_fa1(**kwargs) == status


def test_bwd_workspace_size(lib):
    # fp32 dQ accumulator [BH, Npad, d] + two fp32 row vectors, Npad = N rounded up to 128
    assert fa.fa_bwd_workspace_size(4, 32, 2048, 64) == 4 * 32 * 2048 * 66 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 1, 128) == 128 * 130 * 4
    assert fa.fa_bwd_workspace_size(2, 3, 200, 64) == 6 * 256 * 66 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 1, 96) == 128 * 98 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 1, 48) == 0
    assert fa.fa_bwd_workspace_size(1, -1, 1, 64) == 0


DO, DQ, DK, DV = 0x70000000, 0x80000000, 0x90000000, 0xA0000000


def call_bwd(ws=W, ws_bytes=1 << 30, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, do=DO, dq=DQ, dk=DK, dv=DV, B=1, H=2, N=256, d=64,
             scale=0.125, causal=0, dtype=0)
    a.update(kw)
    return fa.fa_bwd_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["do"], a["dq"], a["dk"],
                         a["dv"], ws, ws_bytes, a["B"], a["H"], a["N"], a["d"], a["scale"],
                         a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(lse=0), 1), (dict(do=0), 1), (dict(dq=0), 1), (dict(dk=0), 1), (dict(dv=0), 1),
    (dict(ws=0), 1), (dict(ws_bytes=100), 1),
    (dict(do=DO + 8), 3), (dict(dq=DQ + 2), 3), (dict(dv=DV + 4), 3), (dict(ws=W + 8), 3),
    (dict(dk=DQ + 64), 1),          # two outputs overlap
    (dict(dq=DO), 1),               # an output overlaps dout
    (dict(ws=L), 1),                # the workspace overlaps lse
    (dict(d=48), 2), (dict(dtype=5), 2), (dict(causal=2), 1),
    (dict(scale=float("nan")), 1),
    (dict(N=0), 0), (dict(B=0), 0),
], ids=lambda x: str(x))
def test_bwd_argument_checks(lib, kwargs, status):
    assert call_bwd(**kwargs) == status


def test_decode_workspace_size(lib):
    # one chunk per 128 keys at most, (m, l, O[d]) fp32 per query
    assert fa.fa_decode_workspace_size(8, 32, 1, 16384, 128) == 256 * 128 * 1 * 130 * 4
    assert fa.fa_decode_workspace_size(1, 1, 4, 129, 64) == 2 * 4 * 66 * 4
    assert fa.fa_decode_workspace_size(1, 1, 17, 1000, 64) == 0   # Nq > 16
    assert fa.fa_decode_workspace_size(1, 1, 4, 3, 64) == 0       # Nk < Nq
    assert fa.fa_decode_workspace_size(1, 1, 1, 10, 96) == 1 * 98 * 4
    assert fa.fa_decode_workspace_size(1, 1, 1, 10, 48) == 0


def call_decode(ws=W, ws_bytes=1 << 30, **kw):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=2, Nq=1, Nk=256, d=64, scale=0.125, causal=0, dtype=0)
    a.update(kw)
    return fa.fa_decode_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], ws, ws_bytes, a["B"], a["H"],
                            a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(Nq=17), 2), (dict(Nq=0), 2), (dict(Nk=0), 1), (dict(Nq=4, Nk=3), 1),
    (dict(d=48), 2), (dict(dtype=3), 2), (dict(causal=5), 1), (dict(scale=float("nan")), 1),
    (dict(q=0), 1), (dict(ws=0), 1), (dict(ws_bytes=10), 1),
    (dict(k=K + 8), 3), (dict(lse=L + 1), 3), (dict(ws=W + 4), 3),
    (dict(o=K), 1), (dict(ws=V), 1),
    (dict(B=0), 0), (dict(H=0), 0),
], ids=lambda x: str(x))
def test_decode_argument_checks(lib, kwargs, status):
    assert call_decode(**kwargs) == status


def test_selftest_rejects_bad_limit_before_cuda(lib):
    assert fa.fa_selftest_wait_timeout(0) == 1
    assert fa.fa_selftest_wait_timeout(2_000_000) == 1


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(fa.FAError):
        _lib.load(str(tmp_path / "missing.so"))


def test_cpu_tensors_are_rejected():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 1, 128, 64, dtype=torch.float16)
    with pytest.raises(fa.FAError):
        fa.fa_fwd(x, x, x)
