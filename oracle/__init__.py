"""Float64 CPU oracle for ragged and paged GQA attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product library never
imports, links or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``pgqa_oracle.c`` (plain loops, float64, OpenMP over output
rows); this module only compiles it with gcc and marshals arrays through ctypes.
Every function takes the *stored* bf16 tensors (their raw bit patterns) so that what
the oracle sees is exactly what the GPU sees.

Functions
  ragged_attention  -- ragged/varlen prefill (Atlas "Module flashinfer",
                       ragged_prefill_bf16_hd128 / _hd256).
  paged_attention   -- attention through an NHD page table; decode is the case
                       q_indptr = 0..batch (vllm-rlt PR "feat: add FlashInfer attention
                       backend for SM120 decode", Design notes).
  merge_states      -- merge of partial (V, LSE) states (FlashInfer documentation,
                       flashinfer.cascade, "Merge Attention States").
  paged_attention_e4m3 -- paged attention over a KV cache stored as FP8 E4M3 with one
                       scale per tensor (FlashInfer documentation, flashinfer_benchmark.py
                       "Attention Flags", --kv_dtype fp8_e4m3).
  e4m3_decode       -- the E4M3 byte decoder the previous function uses.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "pgqa_oracle.c"
_BUILD = _HERE / "_build"
_LIB = None


def _lib_path() -> Path:
    return _BUILD / f"libpgqa_oracle_{platform.machine()}.so"


def build(force: bool = False) -> Path:
    """Compile the C oracle with gcc (float64, no FP contraction, OpenMP)."""
    out = _lib_path()
    if force or not out.exists() or out.stat().st_mtime < _SRC.stat().st_mtime:
        _BUILD.mkdir(exist_ok=True)
        tmp = out.with_suffix(f".{os.getpid()}.tmp")
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
             "-o", str(tmp), str(_SRC), "-lm"],
            check=True)
        os.replace(tmp, out)
    return out


def _load():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(str(build()))
        p = ctypes.c_void_p
        i = ctypes.c_int
        lng = ctypes.c_long
        d = ctypes.c_double
        lib.pgqa_oracle_ragged.argtypes = [p, p, p, p, p, i, i, i, i, i, d, p, lng, p, p, i]
        lib.pgqa_oracle_ragged.restype = i
        lib.pgqa_oracle_paged.argtypes = [p, p, p, p, p, i, p, i, lng, i, i, i, i, i, d, p,
                                          lng, p, p, i]
        lib.pgqa_oracle_paged.restype = i
        lib.pgqa_oracle_merge_states.argtypes = [p, p, i, lng, i, p, p]
        lib.pgqa_oracle_merge_states.restype = None
        lib.pgqa_oracle_paged_e4m3.argtypes = [p, p, p, p, d, d, p, i, p, i, lng, i, i, i, i, i,
                                               d, p, lng, p, p, i]
        lib.pgqa_oracle_paged_e4m3.restype = i
        lib.pgqa_oracle_e4m3_decode.argtypes = [p, lng, p]
        lib.pgqa_oracle_e4m3_decode.restype = None
        lib.pgqa_oracle_threads.argtypes = []
        lib.pgqa_oracle_threads.restype = i
        _LIB = lib
    return _LIB


def threads() -> int:
    """Number of OpenMP threads the oracle uses by default."""
    return _load().pgqa_oracle_threads()


def _bf16_bits(x) -> np.ndarray:
    """Raw bf16 bit patterns of a torch bf16 tensor (any device) or a uint16 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must be uint16 bf16 bit patterns")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError(f"expected a bfloat16 tensor, got {x.dtype}")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


def _i32(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def all_rows(total_q: int, num_qo_heads: int) -> np.ndarray:
    return np.arange(total_q * num_qo_heads, dtype=np.int64)


def ragged_attention(q, k, v, q_indptr, kv_indptr, num_qo_heads, num_kv_heads, causal,
                     sm_scale, rows=None, nthreads: int = 0):
    """Float64 attention for the requested rows (t * Hq + h); returns (o [n, d], lse [n])."""
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    qi, ki = _i32(q_indptr), _i32(kv_indptr)
    batch = len(qi) - 1
    d = qb.shape[-1]
    if rows is None:
        rows = all_rows(qb.shape[0], num_qo_heads)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    rc = _load().pgqa_oracle_ragged(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(qi), _ptr(ki), batch,
                                    num_qo_heads, num_kv_heads, d, int(bool(causal)),
                                    float(sm_scale), _ptr(rows), len(rows), _ptr(o), _ptr(lse),
                                    int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, lse


def paged_attention(q, q_indptr, k_pages, v_pages, page_table, kv_lens, num_qo_heads,
                    num_kv_heads, causal, sm_scale, rows=None, nthreads: int = 0):
    """Float64 attention through a page table; returns (o [n, d], lse [n])."""
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k_pages), _bf16_bits(v_pages)
    qi, pt, kl = _i32(q_indptr), _i32(page_table), _i32(kv_lens)
    batch = len(kl)
    num_pages, page_size = kb.shape[0], kb.shape[1]
    d = kb.shape[-1]
    stride = pt.shape[1] if pt.ndim == 2 else 0
    if rows is None:
        rows = all_rows(qb.shape[0], num_qo_heads)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    rc = _load().pgqa_oracle_paged(_ptr(qb), _ptr(qi), _ptr(kb), _ptr(vb), _ptr(pt), stride,
                                   _ptr(kl), page_size, num_pages, batch, num_qo_heads,
                                   num_kv_heads, d, int(bool(causal)), float(sm_scale),
                                   _ptr(rows), len(rows), _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, lse


def _u8(x) -> np.ndarray:
    """Raw bytes of a uint8 / float8 torch tensor (any device) or a uint8 array."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint8:
            raise TypeError("numpy inputs must be uint8 bytes")
        return np.ascontiguousarray(x)
    import torch
    if x.element_size() != 1:
        raise TypeError(f"expected a one-byte dtype, got {x.dtype}")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.uint8).numpy())


def e4m3_decode(x) -> np.ndarray:
    """Values (float64) of E4M3 bytes."""
    b = _u8(x)
    out = np.empty(b.shape, dtype=np.float64)
    _load().pgqa_oracle_e4m3_decode(_ptr(b), b.size, _ptr(out))
    return out


def paged_attention_e4m3(q, q_indptr, k_pages, v_pages, k_scale, v_scale, page_table, kv_lens,
                         num_qo_heads, num_kv_heads, causal, sm_scale, rows=None,
                         nthreads: int = 0):
    """Float64 attention through a page table over E4M3 K/V bytes (element = e4m3 value x
    k_scale / v_scale); returns (o [n, d], lse [n])."""
    qb, kb, vb = _bf16_bits(q), _u8(k_pages), _u8(v_pages)
    qi, pt, kl = _i32(q_indptr), _i32(page_table), _i32(kv_lens)
    batch = len(kl)
    num_pages, page_size = kb.shape[0], kb.shape[1]
    d = kb.shape[-1]
    stride = pt.shape[1] if pt.ndim == 2 else 0
    if rows is None:
        rows = all_rows(qb.shape[0], num_qo_heads)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.empty((len(rows), d), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    rc = _load().pgqa_oracle_paged_e4m3(_ptr(qb), _ptr(qi), _ptr(kb), _ptr(vb), float(k_scale),
                                        float(v_scale), _ptr(pt), stride, _ptr(kl), page_size,
                                        num_pages, batch, num_qo_heads, num_kv_heads, d,
                                        int(bool(causal)), float(sm_scale), _ptr(rows), len(rows),
                                        _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, lse


def merge_states(v: np.ndarray, s: np.ndarray):
    """Merge partial states v [n_states, n_rows, d], s [n_states, n_rows] (float64)."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    s = np.ascontiguousarray(s, dtype=np.float64)
    n_states, n_rows, d = v.shape
    vo = np.empty((n_rows, d), dtype=np.float64)
    so = np.empty(n_rows, dtype=np.float64)
    _load().pgqa_oracle_merge_states(_ptr(v), _ptr(s), n_states, n_rows, d, _ptr(vo), _ptr(so))
    return vo, so
