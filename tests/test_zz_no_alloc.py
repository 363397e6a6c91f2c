"""pgqa_paged_decode_bf16_noalloc: the decode entry point that allocates nothing.

Callers that cannot allocate device memory -- work enqueued during CUDA-graph capture,
engines whose pool allocator owns all device memory, deployments that forbid allocation
after start-up -- use this variant; its split-KV scratch is a fixed 16 MiB static device
array inside the library.  These tests call it through the C ABI and check that its
results match pgqa_paged_decode_bf16 (which uses the lazily allocated workspace) within
the tolerance the parity tests use, on two calls in a row (the second call reuses the
array the first one left behind), and that sizes beyond the array are refused.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes when run on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu

O_ATOL, O_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


def _fn(lib):
    f = lib.pgqa_paged_decode_bf16_noalloc
    p, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [p, p, p, p, p, i, i, i, p, p, i, i, i, i, fl, p]
    f.restype = i
    return f


def _call(fn, pc, o, lse):
    P = ctypes.c_void_p
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(P(pc.q.data_ptr()), P(pc.k_pages.data_ptr()), P(pc.v_pages.data_ptr()),
              P(pc.page_table.data_ptr()), P(pc.kv_lens_t.data_ptr()), pc.page_size,
              pc.page_table.shape[1], pc.num_pages, P(o.data_ptr()), P(lse.data_ptr()),
              pc.batch, pc.num_qo_heads, pc.num_kv_heads, pc.head_dim, pc.sm_scale, stream)


def _close(o, lse, ro, rl):
    o, ro = o.double().cpu().numpy(), ro.double().cpu().numpy()
    lse, rl = lse.double().cpu().numpy(), rl.double().cpu().numpy()
    assert np.all(np.abs(o - ro) <= O_ATOL + O_RTOL * np.abs(ro))
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    fin = np.isfinite(rl)
    assert np.all(np.abs(lse[fin] - rl[fin]) <= LSE_ATOL)


def test_noalloc_decode_matches_workspace_decode_twice(cuda_lib):
    fn = _fn(cuda_lib.lib)
    pc = W.paged_case([1, 700, 1024, 2500, 4097, 33, 0], 32, 8, 128, page_size=16, seed=3,
                      device="cuda")
    ref_o, ref_l = cuda_lib.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table,
                                         pc.kv_lens_t, sm_scale=pc.sm_scale)
    torch.cuda.synchronize()
    for _ in range(2):
        o = torch.full_like(pc.q, 3.0)
        lse = torch.full(pc.q.shape[:2], 5.0, dtype=torch.float32, device="cuda")
        assert _call(fn, pc, o, lse) == 0
        torch.cuda.synchronize()
        _close(o, lse, ref_o, ref_l)


def test_noalloc_decode_refuses_sizes_beyond_its_array(cuda_lib):
    fn = _fn(cuda_lib.lib)
    # 256 requests with 32k-key tables need about 135 MB of partials: more than 16 MiB
    pc = W.paged_case([16] * 256, 32, 8, 128, page_size=16, stride=2048, seed=4, device="cuda")
    o = torch.zeros_like(pc.q)
    lse = torch.zeros(pc.q.shape[:2], dtype=torch.float32, device="cuda")
    assert _call(fn, pc, o, lse) == -3          # PGQA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((o == 0).all())
