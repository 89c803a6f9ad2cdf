"""ctypes binding over libattn.so: the C ABI of include/attn.h, same names.

Only argument marshalling happens here: shapes and dtypes are read from
torch tensors, outputs the caller did not supply are allocated with torch,
and the raw device pointers plus the current CUDA stream are handed to the
library.  Every step of the computation runs in the library's kernels.  If
the library has not been built, every call raises instead of falling back to
anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple

import torch

from ._build import LIB_PATH

ATTN_F32 = 0
ATTN_BF16 = 1
_STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_WORKSPACE",
           4: "ATTN_ERR_CUDA", 5: "ATTN_ERR_DEVICE_CHECK"}

_lock = threading.Lock()
_handle = None


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}")
        self.status = status


def library_path() -> str:
    return LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libattn.so (built by ``exact_tiled_attention_11_gb300._build.build``)."""
    global _handle
    with _lock:
        if _handle is not None:
            return _handle
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.restype = i32
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, vp]
        lib.attn_fwd_host.restype = i32
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32,
                                      vp, vp, vp]
        lib.attn_fwd_cross.restype = i32
        lib.attn_fwd_cross.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp]
        lib.attn_fwd_varlen.restype = i32
        lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, f32, vp]
        lib.attn_fwd_paged.restype = i32
        lib.attn_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                       i32, f32, vp]
        lib.attn_cascade_workspace_size.restype = sz
        lib.attn_cascade_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.attn_cascade_decode.restype = i32
        lib.attn_cascade_decode.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32,
                                            f32, i32, vp, sz, vp]
        lib.attn_decode_workspace_size.restype = sz
        lib.attn_decode_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.attn_decode_max_splits.restype = i32
        lib.attn_decode_max_splits.argtypes = [i32, i32, i32, i32]
        lib.attn_decode_paged.restype = i32
        lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                          vp, sz, vp]
        lib.attn_decode_paged_noalloc.restype = i32
        lib.attn_decode_paged_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                                  i32, vp]
        lib.merge_partials.restype = i32
        lib.merge_partials.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, vp, i32, vp, vp]
        lib.attn_fp8_padded_keys.restype = i32
        lib.attn_fp8_padded_keys.argtypes = [i32]
        lib.attn_fp8_quantize.restype = i32
        lib.attn_fp8_quantize.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
        lib.attn_fwd_fp8.restype = i32
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, vp]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [i32]
        lib.attn_device_error.restype = i32
        lib.attn_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
        lib.attn_selftest_wait_timeout.restype = i32
        lib.attn_selftest_wait_timeout.argtypes = [vp, vp]
        lib.attn_clock_probe.restype = i32
        lib.attn_clock_probe.argtypes = [vp, vp, vp]
        _handle = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, status: int):
    if status != 0:
        raise AttnError(fn, status)


def _need(t, name, dtype=None, ndim=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(status).decode()


def attn_fwd(q, k, v, o=None, lse=None, *, causal=False, scale=None, stream=None):
    """Exact attention forward pass.  q [B, H, N, d]; k, v [B, Hkv, N, d]; bf16 or fp32.

    Returns (o [B, H, N, d] in q's dtype, lse [B, H, N] fp32)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, 4)
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("attn_fwd takes bf16 or fp32 tensors")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, device=q.device)
    _need(o, "o", q.dtype, 4)
    _need(lse, "lse", torch.float32, 3)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    dt = ATTN_BF16 if q.dtype == torch.bfloat16 else ATTN_F32
    _check("attn_fwd", lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                    1 if causal else 0, scale, dt, _stream(stream, q.device)))
    return o, lse


_COPY_STREAMS = {}


def _copy_streams(device):
    """Two side streams per device for attn_fwd_host's copies (created once)."""
    key = torch.device(device).index
    if key not in _COPY_STREAMS:
        _COPY_STREAMS[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    return _COPY_STREAMS[key]


def attn_fwd_host(q, k, v, o=None, lse=None, *, device=None, buffers=None, causal=False, scale=None, stream=None,
                  copy_streams=None):
    """attn_fwd on host tensors (q [B, H, N, d], k, v [B, Hkv, N, d], bf16 or fp32, CPU,
    contiguous; pinned for overlap).  The copies in and out are pipelined with the
    attention inside the call.  ``buffers`` = (q_dev, k_dev, v_dev, o_dev, lse_dev) on the
    device (allocated when not given).  Returns (o, lse) on the host; the results are
    complete once ``stream`` (default: the current stream) has reached this point."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        if t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype or t.dim() != 4:
            raise ValueError(f"{n} must be a contiguous 4-D host tensor of q's dtype")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("attn_fwd_host takes bf16 or fp32 tensors")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None:
        lse = torch.empty(B, H, N, dtype=torch.float32, pin_memory=True)
    if buffers is None:
        buffers = (torch.empty(q.shape, dtype=q.dtype, device=dev), torch.empty(k.shape, dtype=q.dtype, device=dev),
                   torch.empty(k.shape, dtype=q.dtype, device=dev), torch.empty(q.shape, dtype=q.dtype, device=dev),
                   torch.empty(B, H, N, dtype=torch.float32, device=dev))
    qd, kd, vd, od, ld = buffers
    for t, n in ((qd, "q_dev"), (kd, "k_dev"), (vd, "v_dev"), (od, "o_dev")):
        _need(t, n, q.dtype, 4)
    _need(ld, "lse_dev", torch.float32, 3)
    cin, cout = _copy_streams(dev) if copy_streams is None else copy_streams
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    dt = ATTN_BF16 if q.dtype == torch.bfloat16 else ATTN_F32
    _check("attn_fwd_host", lib.attn_fwd_host(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(od), _ptr(ld),
        B, H, Hkv, N, d, 1 if causal else 0, scale, dt, _stream(stream, dev),
        ctypes.c_void_p(cin.cuda_stream), ctypes.c_void_p(cout.cuda_stream)))
    return o, lse


def attn_fwd_cross(q, k, v, o=None, lse=None, *, causal=False, scale=None, stream=None):
    """Attention of Nq query rows against Nk keys.  q [B, H, Nq, d]; k, v [B, Hkv, Nk, d];
    causal masking is aligned to the last key (row i attends keys j <= i + Nk - Nq).

    Returns (o [B, H, Nq, d] in q's dtype, lse [B, H, Nq] fp32)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, 4)
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("attn_fwd_cross takes bf16 or fp32 tensors")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Nk, d] matching q")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=q.device)
    _need(o, "o", q.dtype, 4)
    _need(lse, "lse", torch.float32, 3)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    dt = ATTN_BF16 if q.dtype == torch.bfloat16 else ATTN_F32
    _check("attn_fwd_cross", lib.attn_fwd_cross(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq, Nk,
                                                d, 1 if causal else 0, scale, dt, _stream(stream, q.device)))
    return o, lse


def attn_fwd_varlen(q, k, v, qo_indptr, kv_indptr, max_q_len, o=None, lse=None, *, causal=False, scale=None,
                    stream=None):
    """Ragged batch: q [total_q, H, d], k, v [total_k, Hkv, d] bf16; qo_indptr, kv_indptr
    [B + 1] int32 (device); max_q_len the longest sequence's query count.
    Returns (o [total_q, H, d] bf16, lse [total_q, H] fp32)."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 3)
    _need(qo_indptr, "qo_indptr", torch.int32, 1)
    _need(kv_indptr, "kv_indptr", torch.int32, 1)
    total_q, H, d = q.shape
    total_k, Hkv, _ = k.shape
    B = qo_indptr.shape[0] - 1
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(total_q, H, dtype=torch.float32, device=q.device)
    _check("attn_fwd_varlen", lib.attn_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(qo_indptr), _ptr(kv_indptr), B, H, Hkv, int(max_q_len),
        total_q, total_k, d, 1 if causal else 0, (1.0 / d ** 0.5) if scale is None else float(scale),
        _stream(stream, q.device)))
    return o, lse


def attn_fwd_paged(q, k_pages, v_pages, page_table, kv_lens, qo_indptr, max_q_len, o=None, lse=None, *,
                   causal=True, scale=None, stream=None):
    """Ragged query chunks q [total_q, H, d] (qo_indptr [B + 1]) against each sequence's
    paged cache (k_pages, v_pages [P, Hkv, 16, d], page_table [B, max_pages], kv_lens [B]).
    Returns (o [total_q, H, d] bf16, lse [total_q, H] fp32)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    _need(qo_indptr, "qo_indptr", torch.int32, 1)
    total_q, H, d = q.shape
    P, Hkv, ps, _ = k_pages.shape
    B = kv_lens.shape[0]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(total_q, H, dtype=torch.float32, device=q.device)
    _check("attn_fwd_paged", lib.attn_fwd_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens), _ptr(qo_indptr), _ptr(o), _ptr(lse),
        B, H, Hkv, int(max_q_len), total_q, d, ps, page_table.shape[1], P, 1 if causal else 0,
        (1.0 / d ** 0.5) if scale is None else float(scale), _stream(stream, q.device)))
    return o, lse


class Fp8Inputs(NamedTuple):
    """FP8 blocks of one attention call (see attn_fp8_quantize in include/attn.h)."""
    q8: torch.Tensor        # [B, H, Nq, 128] uint8 e4m3 codes of q M
    k8: torch.Tensor        # [B, Hkv, Nk, 128] uint8 e4m3 codes of k M
    v8t: torch.Tensor       # [B, Hkv, 128, Nk_pad] uint8 e4m3 codes of v, transposed
    q_scale: torch.Tensor   # [B, H, ceil(Nq / 128)] fp32
    k_scale: torch.Tensor   # [B, Hkv, ceil(Nk / 128)] fp32
    v_scale: torch.Tensor   # [B, Hkv, ceil(Nk / 128)] fp32


def attn_fp8_padded_keys(Nk: int) -> int:
    return int(load_library().attn_fp8_padded_keys(Nk))


def attn_fp8_quantize(q, k, v, signs=None, out: Fp8Inputs = None, *, stream=None) -> Fp8Inputs:
    """Block-quantise bf16 q [B, H, Nq, 128], k, v [B, Hkv, Nk, 128] to e4m3, after the
    orthogonal transform diag(signs) H / sqrt(128) of q and k (signs [128] fp32 +-1 on the
    device, or None for no transform).  Allocates the outputs unless ``out`` is given."""
    lib = load_library()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, Hkv, Nk, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Nk, d] matching q")
    if signs is not None:
        _need(signs, "signs", torch.float32, 1)
        if signs.numel() != d:
            raise ValueError(f"signs must hold {d} values")
    if out is None:
        dev = q.device
        nq, nk = -(-Nq // 128), -(-Nk // 128)
        out = Fp8Inputs(torch.empty(B, H, Nq, d, dtype=torch.uint8, device=dev),
                        torch.empty(B, Hkv, Nk, d, dtype=torch.uint8, device=dev),
                        torch.empty(B, Hkv, d, attn_fp8_padded_keys(Nk), dtype=torch.uint8, device=dev),
                        torch.empty(B, H, nq, dtype=torch.float32, device=dev),
                        torch.empty(B, Hkv, nk, dtype=torch.float32, device=dev),
                        torch.empty(B, Hkv, nk, dtype=torch.float32, device=dev))
    _check("attn_fp8_quantize", lib.attn_fp8_quantize(
        _ptr(q), _ptr(k), _ptr(v), None if signs is None else _ptr(signs), _ptr(out.q8), _ptr(out.k8),
        _ptr(out.v8t), _ptr(out.q_scale), _ptr(out.k_scale), _ptr(out.v_scale), B, H, Hkv, Nq, Nk, d,
        _stream(stream, q.device)))
    return out


def attn_fwd_fp8(x: Fp8Inputs, o=None, lse=None, *, causal=False, scale=None, stream=None):
    """Attention over FP8 blocks from attn_fp8_quantize.  Returns (o [B, H, Nq, 128] bf16,
    lse [B, H, Nq] fp32)."""
    lib = load_library()
    _need(x.q8, "q8", torch.uint8, 4)
    _need(x.k8, "k8", torch.uint8, 4)
    _need(x.v8t, "v8t", torch.uint8, 4)
    for t, n in ((x.q_scale, "q_scale"), (x.k_scale, "k_scale"), (x.v_scale, "v_scale")):
        _need(t, n, torch.float32, 3)
    B, H, Nq, d = x.q8.shape
    Hkv, Nk = x.k8.shape[1], x.k8.shape[2]
    if x.v8t.shape != (B, Hkv, d, attn_fp8_padded_keys(Nk)):
        raise ValueError("v8t must be [B, Hkv, d, Nk_pad]")
    if o is None:
        o = torch.empty(B, H, Nq, d, dtype=torch.bfloat16, device=x.q8.device)
    if lse is None:
        lse = torch.empty(B, H, Nq, dtype=torch.float32, device=x.q8.device)
    _need(o, "o", torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    scale = (1.0 / d ** 0.5) if scale is None else float(scale)
    _check("attn_fwd_fp8", lib.attn_fwd_fp8(
        _ptr(x.q8), _ptr(x.k8), _ptr(x.v8t), _ptr(x.q_scale), _ptr(x.k_scale), _ptr(x.v_scale), _ptr(o), _ptr(lse),
        B, H, Hkv, Nq, Nk, d, 1 if causal else 0, scale, _stream(stream, x.q8.device)))
    return o, lse


def attn_decode_workspace_size(B: int, H: int, d: int, max_splits: int) -> int:
    return int(load_library().attn_decode_workspace_size(B, H, d, max_splits))


def attn_decode_max_splits(B: int, H: int, Hkv: int, max_pages_per_seq: int) -> int:
    return int(load_library().attn_decode_max_splits(B, H, Hkv, max_pages_per_seq))


def attn_decode_paged(q, k_pages, v_pages, page_table, kv_lens, o=None, lse=None, *, scale=None, num_splits=0,
                      workspace=None, stream=None):
    """Split-KV decode over a paged cache.  q [B, H, d] bf16; k_pages, v_pages
    [P, Hkv, page_size, d] bf16; page_table [B, max_pages] int32; kv_lens [B] int32.

    Returns (o [B, H, d] bf16, lse [B, H] fp32).  ``workspace`` (uint8, device)
    is allocated here when not given."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    B, H, d = q.shape
    P, Hkv, ps, _ = k_pages.shape
    maxp = page_table.shape[1]
    if o is None:
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    S = num_splits if num_splits > 0 else lib.attn_decode_max_splits(B, H, Hkv, max(maxp, 1))
    need = lib.attn_decode_workspace_size(B, H, d, max(S, 1))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check("attn_decode_paged", lib.attn_decode_paged(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens), _ptr(o), _ptr(lse),
        B, H, Hkv, d, ps, maxp, P, (1.0 / d ** 0.5) if scale is None else float(scale), int(num_splits),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, q.device)))
    return o, lse


def attn_cascade_workspace_size(B: int, H: int, d: int, max_splits: int) -> int:
    return int(load_library().attn_cascade_workspace_size(B, H, d, max_splits))


def attn_cascade_decode(q, prefix_k, prefix_v, k_pages, v_pages, page_table, kv_lens, o=None, lse=None, *,
                        scale=None, num_splits=0, workspace=None, stream=None):
    """Decode for requests sharing one prefix: q [B, H, d] bf16; prefix_k, prefix_v
    [Hkv, prefix_len, d] bf16; each request's own suffix as in attn_decode_paged
    (kv_lens counts suffix tokens).  Returns (o [B, H, d] bf16, lse [B, H] fp32)."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(prefix_k, "prefix_k", torch.bfloat16, 3)
    _need(prefix_v, "prefix_v", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    B, H, d = q.shape
    P, Hkv, ps, _ = k_pages.shape
    Lp = prefix_k.shape[1]
    if prefix_k.shape != (Hkv, Lp, d) or prefix_v.shape != prefix_k.shape:
        raise ValueError("prefix_k and prefix_v must be [Hkv, prefix_len, d]")
    maxp = page_table.shape[1]
    if o is None:
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=q.device)
    S = num_splits if num_splits > 0 else lib.attn_decode_max_splits(B, H, Hkv, max(maxp, 1))
    if workspace is None:
        workspace = torch.empty(max(lib.attn_cascade_workspace_size(B, H, d, max(S, 1)), 256), dtype=torch.uint8,
                                device=q.device)
    _check("attn_cascade_decode", lib.attn_cascade_decode(
        _ptr(q), _ptr(prefix_k), _ptr(prefix_v), Lp, _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens),
        _ptr(o), _ptr(lse), B, H, Hkv, d, ps, maxp, P, (1.0 / d ** 0.5) if scale is None else float(scale),
        int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, q.device)))
    return o, lse


def attn_decode_paged_noalloc(q, k_pages, v_pages, page_table, kv_lens, o, lse, *, scale=None, num_splits=0,
                              stream=None):
    """attn_decode_paged with the library's fixed device scratch array instead of a
    workspace, for callers that cannot allocate device memory.  ``o`` [B, H, d] bf16
    and ``lse`` [B, H] fp32 must be given; nothing is allocated."""
    lib = load_library()
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(kv_lens, "kv_lens", torch.int32, 1)
    _need(o, "o", torch.bfloat16, 3)
    _need(lse, "lse", torch.float32, 2)
    B, H, d = q.shape
    P, Hkv, ps, _ = k_pages.shape
    _check("attn_decode_paged_noalloc", lib.attn_decode_paged_noalloc(
        _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens), _ptr(o), _ptr(lse),
        B, H, Hkv, d, ps, page_table.shape[1], P, (1.0 / d ** 0.5) if scale is None else float(scale),
        int(num_splits), _stream(stream, q.device)))
    return o, lse


def merge_partials(m, l, o_tilde, num_parts=None, *, out_dtype=torch.bfloat16, o=None, lse=None, stream=None):
    """Exact merge of partials: m, l [B, H, S] fp32, o_tilde [B, H, S, d] fp32,
    num_parts [B] int32 or None.  Returns (o [B, H, d] out_dtype, lse [B, H] fp32)."""
    lib = load_library()
    _need(m, "m", torch.float32, 3)
    _need(l, "l", torch.float32, 3)
    _need(o_tilde, "o_tilde", torch.float32, 4)
    B, H, S, d = o_tilde.shape
    if num_parts is not None:
        _need(num_parts, "num_parts", torch.int32, 1)
    if o is None:
        o = torch.empty(B, H, d, dtype=out_dtype, device=m.device)
    if lse is None:
        lse = torch.empty(B, H, dtype=torch.float32, device=m.device)
    dt = ATTN_BF16 if o.dtype == torch.bfloat16 else ATTN_F32
    _check("merge_partials", lib.merge_partials(_ptr(m), _ptr(l), _ptr(o_tilde), _ptr(num_parts), B, H, S, d,
                                                _ptr(o), dt, _ptr(lse), _stream(stream, m.device)))
    return o, lse


def attn_device_error(clear: bool = False) -> int:
    """The OR of the kernels' device error words (synchronises the device)."""
    code = ctypes.c_uint32(0)
    _check("attn_device_error", load_library().attn_device_error(ctypes.byref(code), 1 if clear else 0))
    return int(code.value)


def attn_selftest_wait_timeout(device=None, stream=None) -> list:
    """Run the bounded-wait self-test kernel (about one wait limit of GPU time) and
    return [gave_up_warp0, gave_up_warp1]; afterwards attn_device_error() carries
    ATTN_DEVERR_WAIT_TIMEOUT."""
    device = torch.device("cuda") if device is None else torch.device(device)
    gave_up = torch.full((2,), -1, dtype=torch.int32, device=device)
    _check("attn_selftest_wait_timeout",
           load_library().attn_selftest_wait_timeout(_ptr(gave_up), _stream(stream, gave_up.device)))
    return [int(x) for x in gave_up.cpu()]


def attn_clock_probe(out, match=None, stream=None) -> None:
    """Queue a clock probe on ``stream``: ``out`` (4 int64 on the device) receives the
    global timer (ns), one SM's clock64, that SM's id and a claim flag (1 once written).
    With ``match`` (an earlier probe's ``out``) it records on the same SM.  Two probes
    around work give its average SM clock: 1000 * d(clock64) / d(timer) MHz."""
    if not (out.is_cuda and out.dtype == torch.int64 and out.numel() >= 4 and out.is_contiguous()):
        raise ValueError("attn_clock_probe: out must be a contiguous CUDA int64 tensor of 4 elements")
    if match is not None and not (match.is_cuda and match.dtype == torch.int64 and match.numel() >= 4):
        raise ValueError("attn_clock_probe: match must be an earlier probe's output")
    _check("attn_clock_probe", load_library().attn_clock_probe(_ptr(out), None if match is None else _ptr(match),
                                                               _stream(stream, out.device)))
