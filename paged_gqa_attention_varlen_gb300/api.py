"""Python binding of libpgqa (include/pgqa.h): argument marshalling only.

Every step of the attention path runs in the CUDA library; this module checks tensor
dtypes/shapes/devices, allocates outputs with torch, and passes raw pointers and the
current CUDA stream through ctypes.  There is no fallback: if the library is missing
or cannot be loaded, importing this module raises.
"""
from __future__ import annotations

import ctypes
import math
from pathlib import Path

import torch

from . import build as _build

_LIB_PATH = _build.LIB

PGQA_OK = 0
STATUS_NAMES = {
    0: "ok", -1: "invalid argument", -2: "unsupported shape", -3: "workspace",
    -4: "CUDA error", -5: "device timeout", -6: "device bounds", -7: "no device",
    -8: "device capacity (work list larger than the workspace)",
}

ABI_FUNCTIONS = (
    "pgqa_ragged_prefill_bf16", "pgqa_paged_prefill_bf16", "pgqa_paged_decode_bf16",
    "pgqa_paged_prefill_bf16_strided", "pgqa_paged_decode_bf16_strided",
    "pgqa_paged_decode_e4m3", "pgqa_paged_prefill_e4m3",
    "ragged_prefill_bf16", "paged_prefill_bf16", "paged_decode_bf16", "pgqa_set_workspace", "pgqa_workspace_bytes_prefill",
    "pgqa_workspace_bytes_decode", "pgqa_get_device_status", "pgqa_status_string",
    "pgqa_version", "pgqa_paged_decode_bf16_noalloc", "pgqa_selftest_expired_wait",
)


class PgqaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: status {code} ({STATUS_NAMES.get(code, 'unknown')})")
        self.code = code


def _load(path: Path):
    if not path.exists():
        raise ImportError(
            f"libpgqa not built ({path} missing): run `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` first; there is no CPU fallback")
    lib = ctypes.CDLL(str(path))
    p, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    sz, i64 = ctypes.c_size_t, ctypes.c_int64
    prefill_args = [p, p, p, p, p, p, p, i, i, i, i, i, f, p]
    decode_args = [p, p, p, p, p, i, i, i, p, p, i, i, i, i, f, p]
    for name in ("pgqa_ragged_prefill_bf16", "ragged_prefill_bf16"):
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = prefill_args, i
    for name in ("pgqa_paged_decode_bf16", "paged_decode_bf16"):
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = decode_args, i
    paged_prefill_args = [p, p, p, p, p, p, p, i, p, i, i, i, i, i, i, i, f, p]
    for name in ("pgqa_paged_prefill_bf16", "paged_prefill_bf16"):
        fn = getattr(lib, name)
        fn.argtypes, fn.restype = paged_prefill_args, i
    lib.pgqa_paged_prefill_bf16_strided.argtypes = [p, p, p, p, p, p, p, i, p, i, i, i64, i64, i64,
                                                    i, i, i, i, i, f, p]
    lib.pgqa_paged_prefill_bf16_strided.restype = i
    lib.pgqa_paged_decode_bf16_strided.argtypes = [p, p, p, p, p, i, i, i, i64, i64, i64, p, p, i,
                                                   i, i, i, f, p]
    lib.pgqa_paged_decode_bf16_strided.restype = i
    lib.pgqa_paged_decode_e4m3.argtypes = [p, p, p, p, p, i, i, i, i64, i64, i64, f, f, p, p, i, i,
                                           i, i, f, p]
    lib.pgqa_paged_decode_e4m3.restype = i
    lib.pgqa_paged_prefill_e4m3.argtypes = [p, p, p, p, p, p, p, i, p, i, i, i64, i64, i64, f, f,
                                            i, i, i, i, i, i, f, p]
    lib.pgqa_paged_prefill_e4m3.restype = i
    lib.pgqa_set_workspace.argtypes, lib.pgqa_set_workspace.restype = [p, sz], i
    lib.pgqa_workspace_bytes_prefill.argtypes = [i, i64, i, i]
    lib.pgqa_workspace_bytes_prefill.restype = sz
    lib.pgqa_workspace_bytes_decode.argtypes = [i, i, i, i, i]
    lib.pgqa_workspace_bytes_decode.restype = sz
    lib.pgqa_get_device_status.argtypes, lib.pgqa_get_device_status.restype = [p], i
    lib.pgqa_status_string.argtypes, lib.pgqa_status_string.restype = [i], ctypes.c_char_p
    lib.pgqa_version.argtypes, lib.pgqa_version.restype = [], i
    lib.pgqa_selftest_expired_wait.argtypes = [p]
    lib.pgqa_selftest_expired_wait.restype = i
    return lib


lib = _load(_LIB_PATH)


def library_path() -> str:
    return str(_LIB_PATH)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _with_rows(t):
    """t itself, or a one-row stand-in when t has no rows (a tensor without elements has no
    device address to pass; the calls never read rows their indptr does not cover)."""
    return t if t.shape[0] > 0 else torch.zeros((1,) + tuple(t.shape[1:]), dtype=t.dtype,
                                                device=t.device)


def _pool_with_page(t, page_size, hk, d, strides):
    """t itself, or a zeroed stand-in spanning one page under `strides` when the pool has no
    pages.  The call still gets num_pages = 0, so any page id a request names is reported
    out of bounds; the stand-in only gives the pool a device address."""
    if t.shape[0] > 0:
        return t
    _, slot_s, head_s = strides
    span = (page_size - 1) * slot_s + (hk - 1) * head_s + d
    return torch.zeros(span, dtype=t.dtype, device=t.device)


def _stream(stream, dev=None):
    """The stream handle for a call on device `dev` (default: its current stream)."""
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    elif dev is not None and stream.device != dev:
        raise ValueError(f"stream is on {stream.device}, the tensors on {dev}")
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, dim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, got {t.dim()}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


_E4M3_DTYPES = (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8))


def _page_pools(k_pages, v_pages, kv_layout, dev, allow_e4m3=False):
    """Shape and element strides of the K/V page pools.

    kv_layout "NHD": tensors [num_pages, page_size, Hk, d]; "HND": [num_pages, Hk,
    page_size, d].  Any strides are accepted as long as d is contiguous and K and V share
    them (for instance a per-layer slice of a larger cache).  bf16 pools, or with
    allow_e4m3 one-byte E4M3 pools (uint8 or float8_e4m3fn).  Returns (num_pages,
    page_size, Hk, d, (page_stride, slot_stride, head_stride), contiguous_nhd).
    """
    ok_types = (torch.bfloat16,) + (_E4M3_DTYPES if allow_e4m3 else ())
    for t, name in ((k_pages, "k_pages"), (v_pages, "v_pages")):
        if not isinstance(t, torch.Tensor) or t.dtype not in ok_types:
            raise TypeError(f"{name} must be a torch.Tensor of dtype {ok_types}")
        if not t.is_cuda or t.device != dev:
            raise ValueError(f"{name} must be a CUDA tensor on {dev}")
        if t.dim() != 4 or t.stride(-1) != 1:
            raise ValueError(f"{name} must be 4-D with a contiguous last (head_dim) axis")
    if (k_pages.shape != v_pages.shape or k_pages.stride() != v_pages.stride() or
            k_pages.element_size() != v_pages.element_size()):
        raise ValueError("k_pages and v_pages must have the same dtype size, shape and strides")
    if kv_layout == "NHD":
        num_pages, page_size, hk, d = k_pages.shape
        page_s, slot_s, head_s, _ = k_pages.stride()
    elif kv_layout == "HND":
        num_pages, hk, page_size, d = k_pages.shape
        page_s, head_s, slot_s, _ = k_pages.stride()
    else:
        raise ValueError(f"kv_layout must be 'NHD' or 'HND', got {kv_layout!r}")
    contiguous_nhd = kv_layout == "NHD" and k_pages.is_contiguous() and v_pages.is_contiguous()
    return num_pages, page_size, hk, d, (page_s, slot_s, head_s), contiguous_nhd


def ragged_prefill(q, k, v, q_indptr, kv_indptr, causal=True, sm_scale=None, out=None,
                   lse=None, return_lse=True, stream=None):
    """Ragged batched prefill (pgqa_ragged_prefill_bf16).

    q [total_q, Hq, d], k/v [total_kv, Hk, d] bf16 on one CUDA device; q_indptr /
    kv_indptr [batch + 1] int32 on the same device.  Returns (o, lse) with
    o [total_q, Hq, d] bf16 and lse [total_q, Hq] fp32 (None if return_lse is False).
    """
    dev = q.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(k, "k", torch.bfloat16, 3, dev)
    _check(v, "v", torch.bfloat16, 3, dev)
    _check(q_indptr, "q_indptr", torch.int32, 1, dev)
    _check(kv_indptr, "kv_indptr", torch.int32, 1, dev)
    total_q, hq, d = q.shape
    hk = k.shape[1]
    if k.shape != v.shape or k.shape[2] != d:
        raise ValueError("k and v must be [total_kv, Hk, d] with q's d")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if lse is None and return_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2, dev)
    batch = q_indptr.numel() - 1
    if total_q == 0:  # no query rows in any request: nothing to compute or write
        return out, lse
    k, v = _with_rows(k), _with_rows(v)  # no keys at all: every row gets zeros, lse -inf
    with torch.cuda.device(dev):  # the library works on the current device
        rc = lib.pgqa_ragged_prefill_bf16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                          _ptr(q_indptr), _ptr(kv_indptr), batch, hq, hk, d,
                                          int(bool(causal)), float(sm_scale),
                                          _stream(stream, dev))
    if rc != PGQA_OK:
        raise PgqaError(rc, "pgqa_ragged_prefill_bf16")
    return out, lse


def paged_prefill(q, k_pages, v_pages, q_indptr, page_table, kv_lens, causal=True, sm_scale=None,
                  out=None, lse=None, return_lse=True, stream=None, kv_layout="NHD",
                  k_scale=1.0, v_scale=1.0, max_qo_len=None):
    """Paged prefill / append (pgqa_paged_prefill_bf16, or the _strided call for HND or
    non-contiguous page pools; pgqa_paged_prefill_e4m3 for FP8 E4M3 pools).

    q [total_q, Hq, d] bf16 with q_indptr [batch + 1] int32; k_pages / v_pages
    [num_pages, page_size, Hk, d] (kv_layout "NHD") or [num_pages, Hk, page_size, d]
    ("HND"), any strides with d contiguous, bf16 or E4M3 bytes (uint8 / float8_e4m3fn,
    element = e4m3 x k_scale / v_scale); page_table [batch, stride] int32; kv_lens [batch]
    int32 (keys per request, the cached prefix plus the new tokens); all on one CUDA device.
    For E4M3 pools max_qo_len is the most query rows any request has (q_indptr stays on
    the device; default: total_q, always an upper bound): with max_qo_len * G <= 16 the
    call takes the tensor-core multi-token path.  Returns (o [total_q, Hq, d] bf16,
    lse [total_q, Hq] fp32 or None).
    """
    dev = q.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(q_indptr, "q_indptr", torch.int32, 1, dev)
    _check(page_table, "page_table", torch.int32, 2, dev)
    _check(kv_lens, "kv_lens", torch.int32, 1, dev)
    total_q, hq, d = q.shape
    num_pages, page_size, hk, dk, strides, packed = _page_pools(k_pages, v_pages, kv_layout, dev,
                                                                allow_e4m3=True)
    e4m3 = k_pages.element_size() == 1
    batch = q_indptr.numel() - 1
    if e4m3 and max_qo_len is None:
        max_qo_len = max(total_q, 1)
    if dk != d:
        raise ValueError("k_pages / v_pages must have q's head_dim")
    if page_table.shape[0] != batch or kv_lens.numel() != batch:
        raise ValueError("page_table / kv_lens must have one row per request")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if lse is None and return_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2, dev)
    if total_q == 0:  # no query rows in any request: nothing to compute or write
        return out, lse
    name = ("pgqa_paged_prefill_e4m3" if e4m3 else
            "pgqa_paged_prefill_bf16" if packed else "pgqa_paged_prefill_bf16_strided")
    k_pages = _pool_with_page(k_pages, page_size, hk, d, strides)
    v_pages = _pool_with_page(v_pages, page_size, hk, d, strides)
    with torch.cuda.device(dev):  # the library works on the current device
        st = _stream(stream, dev)
        if e4m3:
            rc = lib.pgqa_paged_prefill_e4m3(
                _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(out), _ptr(lse), _ptr(q_indptr),
                _ptr(page_table), page_table.shape[1], _ptr(kv_lens), page_size, num_pages,
                *strides, float(k_scale), float(v_scale), batch, int(max_qo_len), hq, hk, d,
                int(bool(causal)), float(sm_scale), st)
        elif packed:
            rc = lib.pgqa_paged_prefill_bf16(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(out),
                                             _ptr(lse), _ptr(q_indptr), _ptr(page_table),
                                             page_table.shape[1], _ptr(kv_lens), page_size,
                                             num_pages, batch, hq, hk, d, int(bool(causal)),
                                             float(sm_scale), st)
        else:
            rc = lib.pgqa_paged_prefill_bf16_strided(
                _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(out), _ptr(lse), _ptr(q_indptr),
                _ptr(page_table), page_table.shape[1], _ptr(kv_lens), page_size, num_pages,
                *strides, batch, hq, hk, d, int(bool(causal)), float(sm_scale), st)
    if rc != PGQA_OK:
        raise PgqaError(rc, name)
    return out, lse


def paged_decode(q, k_pages, v_pages, page_table, kv_lens, sm_scale=None, out=None, lse=None,
                 return_lse=True, stream=None, kv_layout="NHD", k_scale=1.0, v_scale=1.0):
    """Paged decode (pgqa_paged_decode_bf16; the _strided call for HND or non-contiguous
    bf16 pools; pgqa_paged_decode_e4m3 for FP8 E4M3 pools).

    q [batch, Hq, d] bf16; k_pages / v_pages [num_pages, page_size, Hk, d] ("NHD") or
    [num_pages, Hk, page_size, d] ("HND"), any strides with d contiguous, either bf16 or
    E4M3 bytes (uint8 / float8_e4m3fn, element = e4m3 x k_scale / v_scale); page_table
    [batch, stride] int32; kv_lens [batch] int32; all on one CUDA device.
    Returns (o [batch, Hq, d] bf16, lse [batch, Hq] fp32 or None).
    """
    dev = q.device
    _check(q, "q", torch.bfloat16, 3, dev)
    _check(page_table, "page_table", torch.int32, 2, dev)
    _check(kv_lens, "kv_lens", torch.int32, 1, dev)
    batch, hq, d = q.shape
    num_pages, page_size, hk, dk, strides, packed = _page_pools(k_pages, v_pages, kv_layout, dev,
                                                                allow_e4m3=True)
    e4m3 = k_pages.element_size() == 1
    if dk != d:
        raise ValueError("k_pages / v_pages must have q's head_dim")
    if page_table.shape[0] != batch or kv_lens.numel() != batch:
        raise ValueError("page_table / kv_lens must have one row per request")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16, 3, dev)
    if lse is None and return_lse:
        lse = torch.empty((batch, hq), dtype=torch.float32, device=dev)
    if lse is not None:
        _check(lse, "lse", torch.float32, 2, dev)
    name = ("pgqa_paged_decode_e4m3" if e4m3 else
            "pgqa_paged_decode_bf16" if packed else "pgqa_paged_decode_bf16_strided")
    k_pages = _pool_with_page(k_pages, page_size, hk, d, strides)
    v_pages = _pool_with_page(v_pages, page_size, hk, d, strides)
    with torch.cuda.device(dev):  # the library works on the current device
        st = _stream(stream, dev)
        if e4m3:
            rc = lib.pgqa_paged_decode_e4m3(
                _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens),
                page_size, page_table.shape[1], num_pages, *strides, float(k_scale),
                float(v_scale), _ptr(out), _ptr(lse), batch, hq, hk, d, float(sm_scale), st)
        elif packed:
            rc = lib.pgqa_paged_decode_bf16(_ptr(q), _ptr(k_pages), _ptr(v_pages),
                                            _ptr(page_table), _ptr(kv_lens), page_size,
                                            page_table.shape[1], num_pages, _ptr(out), _ptr(lse),
                                            batch, hq, hk, d, float(sm_scale), st)
        else:
            rc = lib.pgqa_paged_decode_bf16_strided(
                _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(kv_lens),
                page_size, page_table.shape[1], num_pages, *strides, _ptr(out), _ptr(lse), batch,
                hq, hk, d, float(sm_scale), st)
    if rc != PGQA_OK:
        raise PgqaError(rc, name)
    return out, lse


def device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device status code of `device`
    (default: the current device, or the stream's)."""
    if device is None:
        device = stream.device if stream is not None else torch.device(
            "cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        return lib.pgqa_get_device_status(_stream(stream, device))


def selftest_expired_wait(stream=None, device=None):
    """Enqueue the library's failure-path self-test (pgqa_selftest_expired_wait): a wait
    that runs out after 2 s and leaves PGQA_ERR_DEVICE_TIMEOUT for device_status()."""
    if device is None:
        device = stream.device if stream is not None else torch.device(
            "cuda", torch.cuda.current_device())
    with torch.cuda.device(device):
        rc = lib.pgqa_selftest_expired_wait(_stream(stream, device))
    if rc != PGQA_OK:
        raise PgqaError(rc, "pgqa_selftest_expired_wait")


def set_workspace(buf: torch.Tensor | None, device=None):
    """Use a caller-owned uint8 CUDA tensor as the workspace of its device (None: back to
    lazy allocation on `device`, default the current device)."""
    if buf is None:
        with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
            rc = lib.pgqa_set_workspace(None, 0)
    else:
        if buf.dtype != torch.uint8 or not buf.is_cuda or not buf.is_contiguous():
            raise ValueError("workspace must be a contiguous uint8 CUDA tensor")
        with torch.cuda.device(buf.device):
            rc = lib.pgqa_set_workspace(_ptr(buf), buf.numel())
    if rc != PGQA_OK:
        raise PgqaError(rc, "pgqa_set_workspace")


def workspace_bytes_decode(batch, page_table_stride, page_size, num_qo_heads, head_dim):
    return lib.pgqa_workspace_bytes_decode(batch, page_table_stride, page_size, num_qo_heads,
                                           head_dim)


def workspace_bytes_prefill(batch, max_total_q, num_qo_heads, num_kv_heads):
    return lib.pgqa_workspace_bytes_prefill(batch, max_total_q, num_qo_heads, num_kv_heads)
