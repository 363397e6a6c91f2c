"""pgqa_paged_decode_bf16_noalloc: the decode entry point that allocates nothing.

Some callers cannot let a library allocate device memory: serving engines that give all
free device memory to their own pool at start-up, and deployments that forbid allocation
once initialisation is over.  This entry point keeps its split-KV scratch in a fixed
16 MiB static device array inside the library instead of the lazily cudaMalloc'ed
workspace of pgqa_paged_decode_bf16.

The tests call it through the C ABI.  It runs the same plan, decode and merge kernels
with the same chunk rule as pgqa_paged_decode_bf16, so its results must equal that
call's bit for bit; they are also compared with the float64 oracle at the parity
tolerance.  Both checks are made on two calls in a row (the second call reuses the array
the first one left behind).  Sizes beyond the array must be refused.

This file is collected last so that a run stopping at the first failure has already run
every other test; it also passes when run on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows

pytestmark = pytest.mark.gpu


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


def test_noalloc_decode_matches_workspace_decode_twice(cuda_lib):
    fn = _fn(cuda_lib.lib)
    pc = W.paged_case([1, 700, 1024, 2500, 4097, 33, 0], 32, 8, 128, page_size=16, seed=3,
                      device="cuda")
    ref_o, ref_l = cuda_lib.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table,
                                         pc.kv_lens_t, sm_scale=pc.sm_scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    orc_o, orc_l = oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages,
                                          pc.page_table, pc.kv_lens_t, pc.num_qo_heads,
                                          pc.num_kv_heads, True, pc.sm_scale)
    for call in range(2):
        o = torch.full_like(pc.q, 3.0)
        lse = torch.full(pc.q.shape[:2], 5.0, dtype=torch.float32, device="cuda")
        assert _call(fn, pc, o, lse) == 0
        torch.cuda.synchronize()
        # the same kernels and chunk rule as the workspace decode: the same bits
        assert torch.equal(o, ref_o), f"call {call}: output differs from the workspace decode"
        assert torch.equal(lse, ref_l), f"call {call}: lse differs from the workspace decode"
        check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), orc_o, orc_l,
                   f"noalloc call {call}")


def test_noalloc_decode_refuses_sizes_beyond_its_array(cuda_lib):
    fn = _fn(cuda_lib.lib)
    # 256 requests with 32k-key tables need about 135 MB of partials: more than 16 MiB
    pc = W.paged_case([16] * 256, 32, 8, 128, page_size=16, stride=2048, seed=4, device="cuda")
    o = torch.zeros_like(pc.q)
    lse = torch.zeros(pc.q.shape[:2], dtype=torch.float32, device="cuda")
    assert _call(fn, pc, o, lse) == -3          # PGQA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert bool((o == 0).all())
