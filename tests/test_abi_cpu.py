"""The C-ABI library loads and exports every entry point of include/attn.h, and
its host-side argument checks return their status codes before any launch.

No call here reaches a kernel: every argument set is rejected (or is a no-op)
on the host, so these run without a GPU.
"""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available to build the library")


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_11_gb300 import _build, _lib
    _build.build()
    return _lib.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(", text, re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = declared_functions()
    for n in ("attn_fwd", "attn_decode_paged", "merge_partials", "attn_decode_workspace_size", "attn_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    expect = ["ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED", "ATTN_ERR_WORKSPACE", "ATTN_ERR_CUDA",
              "ATTN_ERR_DEVICE_CHECK"]
    for code, s in enumerate(expect):
        assert lib.attn_status_string(code).decode() == s
    assert lib.attn_status_string(99).decode() == "ATTN_STATUS_UNKNOWN"


# fake device addresses: never dereferenced because every call below is rejected on the host
A = ctypes.c_void_p(0x10000)
MIS = ctypes.c_void_p(0x10008)  # 8-byte aligned only
NULL = None
INVALID, UNSUPPORTED, WORKSPACE, OK = 1, 2, 3, 0


def fwd(lib, q=A, k=A, v=A, o=A, lse=A, B=1, H=4, Hkv=2, N=128, d=128, causal=0, scale=0.1, dtype=1):
    return lib.attn_fwd(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, dtype, None)


def test_attn_fwd_argument_checks(lib):
    assert fwd(lib, q=NULL) == INVALID
    assert fwd(lib, o=NULL) == INVALID
    assert fwd(lib, k=MIS) == INVALID
    assert fwd(lib, lse=ctypes.c_void_p(0x10002)) == INVALID   # the LSE needs 4-byte alignment
    assert fwd(lib, H=6, Hkv=4) == INVALID
    assert fwd(lib, Hkv=0) == INVALID
    assert fwd(lib, N=-1) == INVALID
    assert fwd(lib, scale=0.0) == INVALID
    assert fwd(lib, scale=-1.0) == INVALID
    assert fwd(lib, scale=float("nan")) == INVALID
    assert fwd(lib, scale=float("inf")) == INVALID
    assert fwd(lib, dtype=7) == INVALID
    assert fwd(lib, d=96) == UNSUPPORTED
    assert fwd(lib, d=256, dtype=0) == UNSUPPORTED
    # empty problems are no-ops that launch nothing
    assert fwd(lib, N=0) == OK
    assert fwd(lib, B=0) == OK
    assert fwd(lib, H=0, q=NULL) == OK


def dec(lib, q=A, kp=A, vp=A, pt=A, kl=A, o=A, lse=A, B=2, H=32, Hkv=8, d=128, ps=16, maxp=4, P=8, scale=0.1,
        splits=2, ws=A, ws_bytes=1 << 20):
    return lib.attn_decode_paged(q, kp, vp, pt, kl, o, lse, B, H, Hkv, d, ps, maxp, P, scale, splits, ws, ws_bytes,
                                 None)


def test_attn_decode_paged_argument_checks(lib):
    assert dec(lib, q=NULL) == INVALID
    assert dec(lib, kl=NULL) == INVALID
    assert dec(lib, ws=NULL) == INVALID
    assert dec(lib, kp=NULL) == INVALID
    assert dec(lib, pt=NULL) == INVALID
    assert dec(lib, vp=MIS) == INVALID
    assert dec(lib, H=30, Hkv=8) == INVALID
    assert dec(lib, scale=0.0) == INVALID
    assert dec(lib, d=96) == UNSUPPORTED
    assert dec(lib, ps=32) == UNSUPPORTED
    assert dec(lib, H=64, Hkv=2) == UNSUPPORTED     # group of 32 query heads per KV head
    need = lib.attn_decode_workspace_size(2, 32, 128, 2)
    assert dec(lib, ws_bytes=need - 1) == WORKSPACE
    assert dec(lib, B=0) == OK


def test_workspace_size_arithmetic(lib):
    B, H, d, S = 64, 32, 128, 32
    n = B * H * S
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.attn_decode_workspace_size(B, H, d, S) == 2 * a256(4 * n) + a256(4 * n * d)
    assert lib.attn_decode_workspace_size(0, H, d, S) == 0
    assert lib.attn_decode_workspace_size(B, H, d, 0) == 0


def test_merge_partials_argument_checks(lib):
    f = lambda **kw: lib.merge_partials(kw.get("m", A), kw.get("l", A), kw.get("ot", A), kw.get("np", NULL),  # noqa: E731
                                        kw.get("B", 2), kw.get("H", 4), kw.get("S", 3), kw.get("d", 128),
                                        kw.get("o", A), kw.get("dt", 1), kw.get("lse", A), None)
    assert f(S=0) == INVALID
    assert f(m=NULL) == INVALID
    assert f(ot=MIS) == INVALID
    assert f(dt=5) == INVALID
    assert f(d=32) == UNSUPPORTED
    assert f(B=0) == OK


def test_device_error_rejects_null(lib):
    assert lib.attn_device_error(None, 0) == INVALID


def test_fwd_host_rejects_bad_streams_before_any_work(lib):
    """attn_fwd_host checks its streams and pointers on the host (no GPU needed)."""
    vp = ctypes.c_void_p
    buf = ctypes.create_string_buffer(64)
    p = ctypes.cast(buf, vp)
    s1, s2 = vp(0x1000), vp(0x2000)
    args = lambda cin, cout: (p, p, p, p, None, p, p, p, p, None, 1, 1, 1, 1, 64, 0, ctypes.c_float(0.125), 1, None,
                              cin, cout)
    assert lib.attn_fwd_host(*args(None, s2)) == INVALID      # no copy-in stream
    assert lib.attn_fwd_host(*args(s1, s1)) == INVALID        # copy streams coincide
    assert lib.attn_fwd_host(*args(s1, None)) == INVALID
    bad = list(args(s1, s2))
    bad[0] = None                                              # no host q
    assert lib.attn_fwd_host(*bad) == INVALID
    zero = list(args(s1, s2))
    zero[13] = 0                                               # N == 0: no-op
    assert lib.attn_fwd_host(*zero) == 0
