"""GPU parity of the paged split-KV decode (pgqa_paged_decode_bf16) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_paged_decode_all_rows, check_rows

pytestmark = pytest.mark.gpu


def run_gpu(api, pc, **kw):
    o, lse = api.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens_t,
                              sm_scale=pc.sm_scale, **kw)
    torch.cuda.synchronize()
    return o, lse


def oracle_decode(pc):
    return oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                  pc.kv_lens_t, pc.num_qo_heads, pc.num_kv_heads, True,
                                  pc.sm_scale)


LENS = [0, 1, 15, 16, 17, 100, 1023, 1024, 1025, 2048, 3000, 4097]


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_lengths_and_groups(cuda_lib, G):
    hk = 8 // G if G < 8 else 2
    pc = W.paged_case(LENS, G * hk, hk, 128, page_size=16, seed=G, device="cuda")
    o, lse = run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_decode(pc)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl, f"G={G}")


@pytest.mark.parametrize("ps", [32, 64, 128])
def test_decode_page_sizes(cuda_lib, ps):
    """Larger pages: each is streamed as 16-token slices of the same page."""
    pc = W.paged_case(LENS + [5000], 32, 8, 128, page_size=ps, seed=31 + ps, device="cuda")
    o, lse = run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_decode(pc)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl, f"page {ps}")


@pytest.mark.parametrize("ps", [16, 64])
def test_decode_and_one_row_paged_prefill_agree(cuda_lib, ps):
    """Decode (split-KV + merge on the CUDA cores) and the one-row paged prefill (tensor
    cores, one pass) compute the same attention: they agree within the tolerance."""
    pc = W.paged_case([1, 700, 3000], 16, 4, 128, page_size=ps, seed=37 + ps, device="cuda")
    o_d, l_d = run_gpu(cuda_lib, pc)
    o_p, l_p = cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                                      pc.kv_lens_t, causal=True, sm_scale=pc.sm_scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_decode(pc)
    check_rows(o_d.reshape(-1, 128).float().cpu(), l_d.reshape(-1).cpu(), ro, rl, "decode")
    check_rows(o_p.reshape(-1, 128).float().cpu(), l_p.reshape(-1).cpu(), ro, rl, "prefill q=1")


def test_decode_single_request_long(cuda_lib):
    pc = W.paged_case([32768], 32, 8, 128, page_size=16, seed=11, device="cuda")
    o, lse = run_gpu(cuda_lib, pc)
    ro, rl = oracle_decode(pc)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl, "32k")


def test_decode_workload_all_requests(cuda_lib):
    """The full 256-request decode workload (kv U{512..32768}, 16-token pages in random
    order, 32/8 heads) in the benchmark's launch configuration: every one of its 256 x 32
    output rows is compared with the oracle (pages gathered to the host 32 requests at a
    time)."""
    pc = W.config("decode", device="cuda")
    o, lse = run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    check_paged_decode_all_rows(pc, o, lse, oracle_decode, "decode workload")


def test_page_table_padding_is_bitwise_invisible(cuda_lib):
    outs = []
    for pad in (-1, 0, 77):
        pc = W.paged_case([40, 1500, 7], 16, 4, 128, page_size=16, pad=pad, stride=130,
                          seed=13, device="cuda")
        outs.append(run_gpu(cuda_lib, pc))
        assert cuda_lib.device_status() == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_nan_in_unused_tail_slots_is_invisible(cuda_lib):
    pc = W.paged_case([20, 1030], 8, 2, 128, page_size=16, seed=17, device="cuda")
    o1, l1 = run_gpu(cuda_lib, pc)
    for b, n in enumerate(pc.kv_lens):
        last = int(pc.page_table[b, (n - 1) // 16])
        pc.k_pages[last, n % 16:] = float("nan")
        pc.v_pages[last, n % 16:] = float("nan")
    o2, l2 = run_gpu(cuda_lib, pc)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_zero_length_rows_are_exact_zeros(cuda_lib):
    pc = W.paged_case([0, 5, 0], 8, 2, 128, page_size=16, seed=19, device="cuda")
    o, l = run_gpu(cuda_lib, pc)
    assert torch.all(o[0] == 0) and torch.all(o[2] == 0)
    assert torch.all(torch.isneginf(l[0])) and torch.all(torch.isneginf(l[2]))


@pytest.mark.parametrize("stride", [None, 16384])
def test_batch_composition_is_bitwise_invariant(cuda_lib, stride):
    """A 188-page table puts the batch and each single request under 128-key chunks (few
    work items); a 16384-page table (256k keys of capacity) puts both under 1024-key
    chunks.  For a given chunk length a request's result does not depend on the batch."""
    pc = W.paged_case([3000, 64, 1025], 32, 8, 128, page_size=16, seed=23, stride=stride,
                      device="cuda")
    o, l = run_gpu(cuda_lib, pc)
    for b in range(3):
        sub_o, sub_l = cuda_lib.paged_decode(pc.q[b:b + 1].contiguous(), pc.k_pages, pc.v_pages,
                                             pc.page_table[b:b + 1].contiguous(),
                                             pc.kv_lens_t[b:b + 1].contiguous(),
                                             sm_scale=pc.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(sub_o[0], o[b]) and torch.equal(sub_l[0], l[b])


def test_bad_page_id_reports_bounds_status(cuda_lib):
    pc = W.paged_case([40], 8, 2, 128, page_size=16, seed=29, device="cuda")
    pc.page_table[0, 1] = pc.num_pages + 5
    run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == -6
    pc.page_table[0, 1] = 0
    run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0


def test_merge_modes_give_the_same_bits(cuda_lib):
    """The chunk merge runs one CTA per (request, head) when a call has few rows and one
    warp per row otherwise, with the same arithmetic in the same order.  A request's
    result must not depend on which mode its batch size picked.  A 16384-page table
    (256k keys of capacity) keeps both calls under 1024-key chunks."""
    kv = [5000] + [int(x) for x in np.random.default_rng(7).integers(1, 9000, 39)]
    pc = W.paged_case(kv, 32, 8, 128, page_size=16, seed=31, stride=16384, device="cuda")
    o, l = run_gpu(cuda_lib, pc)  # 40 x 32 = 1280 rows: a warp per row
    o1, l1 = cuda_lib.paged_decode(pc.q[:1].contiguous(), pc.k_pages, pc.v_pages,
                                   pc.page_table[:1].contiguous(), pc.kv_lens_t[:1].contiguous(),
                                   sm_scale=pc.sm_scale)  # 32 rows: a CTA per row
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    assert torch.equal(o1[0], o[0]) and torch.equal(l1[0], l[0])
    ro, rl = oracle_decode(W.PagedCase("r0", pc.q[:1], torch.tensor([0, 1], dtype=torch.int32),
                                       pc.k_pages, pc.v_pages, pc.page_table[:1],
                                       pc.kv_lens_t[:1], kv[:1], [1], 16, 32, 8, 128, True,
                                       pc.sm_scale))
    check_rows(o1[0].float().cpu(), l1[0].cpu(), ro, rl, "request 0")


def test_pending_status_survives_workspace_growth(cuda_lib):
    """A device error left unread by one call is still reported after a later call made
    the library grow its workspace (the status word moves to the new buffer)."""
    pc = W.paged_case([40], 8, 2, 128, page_size=16, seed=37, device="cuda")
    pc.page_table[0, 1] = pc.num_pages + 5  # a page id outside the pool
    run_gpu(cuda_lib, pc)  # leaves PGQA_DEV_BOUNDS pending
    # 2048 requests with 32k-key tables: about 1 GB of split-KV partial results, more than
    # the default workspace, so this call reallocates it
    big = W.paged_case([1] * 2048, 32, 8, 128, page_size=16, stride=2048, seed=38,
                       device="cuda")
    run_gpu(cuda_lib, big)
    assert cuda_lib.device_status() == -6
    assert cuda_lib.device_status() == 0


@pytest.mark.parametrize("e4m3", [False, True], ids=["bf16", "e4m3"])
def test_pool_without_pages(cuda_lib, e4m3):
    """Requests with no keys over a pool with no pages: every row is zeros, lse = -inf."""
    make = W.paged_case_e4m3 if e4m3 else W.paged_case
    pc = make([0, 0, 0], 8, 2, 128, seed=10, device="cuda")
    pc.k_pages, pc.v_pages = pc.k_pages[:0], pc.v_pages[:0]
    kw = dict(k_scale=pc.meta["k_scale"], v_scale=pc.meta["v_scale"]) if e4m3 else {}
    o, lse = run_gpu(cuda_lib, pc, **kw)
    assert cuda_lib.device_status() == 0
    assert torch.equal(o, torch.zeros_like(o))
    assert torch.equal(lse, torch.full_like(lse, -float("inf")))
