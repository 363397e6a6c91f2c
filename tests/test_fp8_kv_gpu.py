"""GPU parity of the paged decode over an FP8 E4M3 KV cache (pgqa_paged_decode_e4m3)
against the float64 oracle's E4M3 path.  E4M3 K/V with one scale per tensor is the
kv_dtype fp8_e4m3 of FlashInfer documentation, flashinfer_benchmark.py "Attention Flags"."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_paged_decode_all_rows, check_rows

pytestmark = pytest.mark.gpu

LENS = [0, 1, 15, 16, 17, 100, 1023, 1024, 1025, 3000, 4097]


def run(api, pc, **kw):
    o, lse = api.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens_t,
                              sm_scale=pc.sm_scale, k_scale=pc.meta["k_scale"],
                              v_scale=pc.meta["v_scale"], **kw)
    torch.cuda.synchronize()
    return o, lse


def oracle_e4m3(pc, rows=None):
    return oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages,
                                       pc.meta["k_scale"], pc.meta["v_scale"], pc.page_table,
                                       pc.kv_lens_t, pc.num_qo_heads, pc.num_kv_heads, True,
                                       pc.sm_scale, rows=rows)


@pytest.mark.parametrize("G,ps,ks,vs", [(1, 16, 0.5, 2.0), (2, 64, 1.0, 1.0), (4, 16, 0.25, 3.0),
                                        (8, 32, 2.0, 0.5)])
def test_e4m3_decode_against_oracle(cuda_lib, G, ps, ks, vs):
    hk = 8 // G if G < 8 else 2
    pc = W.paged_case_e4m3(LENS, G * hk, hk, 128, page_size=ps, seed=91 + G, device="cuda",
                           k_scale=ks, v_scale=vs)
    o, lse = run(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl, f"e4m3 G={G}")


def test_e4m3_nan_bytes_in_unused_tail_slots_are_invisible(cuda_lib):
    pc = W.paged_case_e4m3([20, 1030, 3], 32, 8, 128, page_size=16, seed=93, device="cuda")
    o1, l1 = run(cuda_lib, pc)
    for b, n in enumerate(pc.kv_lens):
        last = int(pc.page_table[b, (n - 1) // 16])
        pc.k_pages[last, n % 16:] = 0x7F   # E4M3 NaN
        pc.v_pages[last, n % 16:] = 0xFF
    o2, l2 = run(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    assert torch.isfinite(o2).all()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_e4m3_hnd_and_float8_dtype_match_packed_bitwise(cuda_lib):
    pc = W.paged_case_e4m3([700, 5, 2100], 16, 4, 128, page_size=32, seed=95, device="cuda")
    o, lse = run(cuda_lib, pc)
    k8 = pc.k_pages.view(torch.float8_e4m3fn)
    v8 = pc.v_pages.view(torch.float8_e4m3fn)
    o2, l2 = cuda_lib.paged_decode(pc.q, k8, v8, pc.page_table, pc.kv_lens_t,
                                   sm_scale=pc.sm_scale, k_scale=0.5, v_scale=2.0)
    kh = pc.k_pages.permute(0, 2, 1, 3).contiguous()
    vh = pc.v_pages.permute(0, 2, 1, 3).contiguous()
    o3, l3 = cuda_lib.paged_decode(pc.q, kh, vh, pc.page_table, pc.kv_lens_t, kv_layout="HND",
                                   sm_scale=pc.sm_scale, k_scale=0.5, v_scale=2.0)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    for a, b in ((o2, l2), (o3, l3)):
        assert torch.equal(a, o) and torch.equal(b, lse)


def test_e4m3_decode_workload_all_requests(cuda_lib):
    """The 256-request decode workload with its cache stored as FP8 E4M3 (the bf16 draws
    rounded by torch's float8_e4m3fn cast, scales 1), as the benchmark times it: all
    256 x 32 output rows compared with the oracle's E4M3 path."""
    pc = W.config("decode", device="cuda")
    pc.k_pages = pc.k_pages.to(torch.float8_e4m3fn).view(torch.uint8)
    pc.v_pages = pc.v_pages.to(torch.float8_e4m3fn).view(torch.uint8)
    pc.meta.update(k_scale=1.0, v_scale=1.0)
    o, lse = run(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    check_paged_decode_all_rows(pc, o, lse, oracle_e4m3, "e4m3 decode workload")
