"""GPU parity of the paged prefill / append (pgqa_paged_prefill_bf16) against the oracle.

Ragged query rows attend over a paged NHD KV cache addressed by a page table (FlashInfer
documentation, flashinfer.prefill, BatchPrefillWithPagedKVCacheWrapper; page-table rules
of the vllm-rlt pull request "feat: add FlashInfer attention backend for SM120 decode").
Small cases are compared on every row; the cached-prefix hd256 serving shape and a
4-token-per-request decode (speculative verification) are compared on sampled rows.
Invariants: the result equals the ragged prefill over the same keys laid out
contiguously (bit for bit), and page-table padding and NaN in unused key slots of a
request's last page are invisible.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows, gather_rows, sample_prefill_rows

pytestmark = pytest.mark.gpu


def run_gpu(api, pc, **kw):
    o, lse = api.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                               pc.kv_lens_t, causal=pc.causal, sm_scale=pc.sm_scale, **kw)
    torch.cuda.synchronize()
    return o, lse


def oracle_paged(pc, rows=None):
    return oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                  pc.kv_lens_t, pc.num_qo_heads, pc.num_kv_heads, pc.causal,
                                  pc.sm_scale, rows=rows)


def full_check(api, pc, what):
    o, lse = run_gpu(api, pc)
    assert api.device_status() == 0
    ro, rl = oracle_paged(pc)
    return check_rows(o.reshape(-1, o.shape[-1]).float().cpu(), lse.reshape(-1).cpu(), ro, rl,
                      what)


SMALL = [
    # qo_lens, kv_lens, Hq, Hk, d, causal, page_size
    ([17, 64], [17, 64], 4, 2, 128, True, 16),
    ([200, 77], [500, 1000], 8, 1, 128, True, 16),       # cached prefix
    ([200, 77], [500, 1000], 8, 1, 128, False, 32),
    ([90, 40], [30, 40], 4, 4, 128, True, 64),           # kv < qo: leading rows see no key
    ([0, 33, 0, 70], [10, 33, 0, 0], 16, 1, 128, True, 16),  # empty q / empty kv requests
    ([513], [700], 16, 16, 128, True, 128),              # G = 1, one page per K/V tile
    ([260, 31], [300, 31], 32, 2, 128, True, 16),        # G = 16
    ([129, 200], [129, 700], 8, 2, 256, True, 16),       # hd256
    ([64, 300], [64, 333], 4, 1, 256, False, 64),
    ([4] * 8, [1000, 17, 129, 4096, 5, 2048, 3000, 64], 32, 8, 128, True, 16),  # 4-token decode
    ([1] * 5, [1, 16, 17, 300, 1029], 8, 2, 128, True, 32),  # one-token decode shape
    ([3, 7], [2000, 131], 16, 4, 256, True, 32),         # hd256 multi-token decode
    ([37, 5, 130], [200, 90, 130], 64, 1, 128, True, 16),  # G = 64
    ([9, 40], [300, 41], 128, 1, 256, True, 32),         # G = 128, hd256
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"p{i}" for i in range(len(SMALL))])
def test_small_shapes(cuda_lib, shape):
    qo, kv, hq, hk, d, causal, ps = shape
    pc = W.paged_case(kv, hq, hk, d, page_size=ps, qo_lens=qo, causal=causal,
                      seed=len(qo) * 37 + hq + d + ps, device="cuda")
    full_check(cuda_lib, pc, f"paged {shape}")


@pytest.mark.parametrize("d,ps", [(128, 16), (128, 64), (256, 16), (256, 32), (256, 128)])
def test_matches_ragged_prefill_bitwise(cuda_lib, d, ps):
    """The paged kernel and the ragged kernel see the same keys in the same tiles, so
    their results agree bit for bit."""
    qo, kv = [300, 45, 1], [1000, 45, 777]
    pc = W.paged_case(kv, 16, 4, d, page_size=ps, qo_lens=qo, seed=41 + d + ps, device="cuda")
    o_p, l_p = run_gpu(cuda_lib, pc)
    ks, vs = [], []
    for b, n in enumerate(kv):
        pages = pc.page_table[b, :(n + ps - 1) // ps].long()
        ks.append(pc.k_pages[pages].reshape(-1, 4, d)[:n])
        vs.append(pc.v_pages[pages].reshape(-1, 4, d)[:n])
    k = torch.cat(ks).contiguous()
    v = torch.cat(vs).contiguous()
    kv_indptr = torch.tensor(np.concatenate([[0], np.cumsum(kv)]), dtype=torch.int32,
                             device="cuda")
    o_r, l_r = cuda_lib.ragged_prefill(pc.q, k, v, pc.q_indptr, kv_indptr, causal=True,
                                       sm_scale=pc.sm_scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    assert torch.equal(o_p, o_r) and torch.equal(l_p, l_r)


@pytest.mark.parametrize("d", [128, 256])
def test_nan_in_unused_tail_slots_is_invisible(cuda_lib, d):
    ps = 16
    kv = [20, 1030, 130]
    pc = W.paged_case(kv, 8, 2, d, page_size=ps, qo_lens=[20, 70, 3], seed=43 + d,
                      device="cuda")
    o1, l1 = run_gpu(cuda_lib, pc)
    for b, n in enumerate(kv):
        last = int(pc.page_table[b, (n - 1) // ps])
        pc.k_pages[last, n % ps:] = float("nan")
        pc.v_pages[last, n % ps:] = float("nan")
    o2, l2 = run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    assert torch.isfinite(o2).all()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_page_table_padding_is_bitwise_invisible(cuda_lib):
    outs = []
    for pad in (-1, 0, 55):
        pc = W.paged_case([40, 1500, 7], 16, 4, 128, page_size=32, qo_lens=[40, 100, 7],
                          pad=pad, stride=70, seed=47, device="cuda")
        outs.append(run_gpu(cuda_lib, pc))
        assert cuda_lib.device_status() == 0
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


def test_prefix_hd256_shape_sampled(cuda_lib):
    """The cached-prefix hd256 serving shape (8 requests, qo U{256..2048}, prefix
    U{0..8192}, 16/4 heads) with its keys in a paged cache of 16-token pages."""
    qo, kv = W.config_lengths("prefix_hd256")
    pc = W.paged_case(kv, 16, 4, 256, page_size=16, qo_lens=qo, seed=0, device="cuda")
    o, lse = run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    rows = sample_prefill_rows(qo, 16, 4, seed=3, per_request_random=16)
    og, lg = gather_rows(o, lse, rows, 16)
    ro, rl = oracle_paged(pc, rows=rows)
    check_rows(og, lg, ro, rl, "paged prefix_hd256")


def test_prefill_hd128_shape_many_items_per_cta(cuda_lib):
    """The 16-request hd128 serving shape in 16-token pages: about 33 work items per CTA,
    which exercises the K/V stage hand-off across many steps and item boundaries (a
    stage-release race once timed out here); sampled rows against the oracle."""
    qo, kv = W.config_lengths("prefill_hd128")
    pc = W.paged_case(kv, 32, 8, 128, page_size=16, qo_lens=qo, seed=0, device="cuda")
    for _ in range(3):
        o, lse = run_gpu(cuda_lib, pc)
        assert cuda_lib.device_status() == 0
    rows = sample_prefill_rows(qo, 32, 4, seed=5, per_request_random=8)
    og, lg = gather_rows(o, lse, rows, 32)
    ro, rl = oracle_paged(pc, rows=rows)
    check_rows(og, lg, ro, rl, "paged prefill_hd128")


def test_multi_token_decode_sampled(cuda_lib):
    """Four query tokens per request (speculative verification) over the first 48
    requests of the paged decode workload's lengths, 32/8 heads, 16-token pages."""
    kv = W.config_lengths("decode")[1][:48]
    pc = W.paged_case(kv, 32, 8, 128, page_size=16, qo_lens=[4] * len(kv), seed=5,
                      device="cuda")
    o, lse = run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(4 * len(kv) * 32, 600, replace=False)).astype(np.int64)
    og, lg = gather_rows(o, lse, rows, 32)
    ro, rl = oracle_paged(pc, rows=rows)
    check_rows(og, lg, ro, rl, "4-token decode")


def test_bad_kv_len_reports_bounds_and_writes_nothing(cuda_lib):
    pc = W.paged_case([40, 50], 8, 2, 128, page_size=16, qo_lens=[5, 6], seed=53,
                      device="cuda")
    pc.kv_lens_t[1] = pc.page_table.shape[1] * 16 + 1
    o = torch.full_like(pc.q, 7.0)
    run_gpu(cuda_lib, pc, out=o)
    assert cuda_lib.device_status() == -6
    assert torch.all(o == 7.0)


def test_bad_page_id_reports_bounds_status(cuda_lib):
    pc = W.paged_case([300], 8, 2, 128, page_size=16, qo_lens=[10], seed=59, device="cuda")
    pc.page_table[0, 3] = pc.num_pages + 5
    run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == -6
    pc.page_table[0, 3] = 0
    run_gpu(cuda_lib, pc)
    assert cuda_lib.device_status() == 0


# ---------------------------------------------------------------- split-KV (short work lists)
# A work list shorter than two items per SM has its requests cut into chunks of 2048 keys
# (head_dim 128; 4096 keys for head_dim 256);
# the chunks' partial results are merged by their LSE weights (FlashInfer documentation,
# flashinfer.cascade "Merge Attention States").

@pytest.mark.parametrize("batch", [1, 4])
def test_split_kv_multi_token_decode_long_context(cuda_lib, batch):
    kv = [32768 - 77 * b for b in range(batch)]
    pc = W.paged_case(kv, 32, 8, 128, page_size=16, qo_lens=[4] * batch, seed=101 + batch,
                      device="cuda")
    full_check(cuda_lib, pc, f"split-KV 4-token decode, batch {batch}")


def test_split_kv_ragged_long_prefix_prefill(cuda_lib):
    """One request, 300 query rows over 20000 keys, 8 query heads on one kv head: 10
    q-tile items cut into 10 chunks each; causal masking across chunk boundaries."""
    case = W.ragged_case([300], [20000], 8, 1, 128, causal=True, seed=103, device="cuda")
    o, lse = cuda_lib.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    rows = sample_prefill_rows([300], 8, 8, seed=7, per_request_random=40)
    og, lg = gather_rows(o, lse, rows, 8)
    ro, rl = oracle.ragged_attention(case.q, case.k, case.v, case.q_indptr, case.kv_indptr, 8, 1,
                                     True, case.sm_scale, rows=rows)
    check_rows(og, lg, ro, rl, "split-KV ragged prefill")


def test_split_kv_non_causal_and_short_requests(cuda_lib):
    """Split regime with a mix: non-causal long request, requests shorter than a chunk, an
    empty request, and a request with fewer keys than queries."""
    qo = [7, 3, 0, 40, 1]
    kv = [9000, 100, 500, 20, 4100]
    pc = W.paged_case(kv, 16, 4, 128, page_size=32, qo_lens=qo, causal=False, seed=107,
                      device="cuda")
    full_check(cuda_lib, pc, "split-KV non-causal mix")
    pc2 = W.paged_case(kv, 16, 4, 128, page_size=32, qo_lens=qo, causal=True, seed=107,
                       device="cuda")
    full_check(cuda_lib, pc2, "split-KV causal mix")


# head_dim 256 in the split regime: the hd256 kernel processes each chunk's tile range and
# writes fp32 partial rows; the merge kernel combines 256-column rows.

@pytest.mark.parametrize("ps", [16, 64])
def test_split_kv_hd256_paged_short_list(cuda_lib, ps):
    """Two requests with long cached prefixes (qo 200 / 37 over 9000 / 4100 keys), 16/4
    heads: 12 q-tile items per kv head, cut into 4096-key chunks; all rows checked."""
    pc = W.paged_case([9000, 4100], 16, 4, 256, page_size=ps, qo_lens=[200, 37], seed=111 + ps,
                      device="cuda")
    full_check(cuda_lib, pc, f"split-KV hd256 paged, page {ps}")


def test_split_kv_hd256_ragged_and_paged_agree_bitwise(cuda_lib):
    """The same split work in the ragged and the paged kernel: same chunks, tiles and
    merge, so the same bits; plus a multi-token decode mix and the oracle."""
    qo, kv = [4, 4, 1, 0, 9], [20000, 5000, 300, 700, 30]
    pc = W.paged_case(kv, 16, 4, 256, page_size=16, qo_lens=qo, seed=117, device="cuda")
    o_p, l_p = run_gpu(cuda_lib, pc)
    ks, vs = [], []
    for b, n in enumerate(kv):
        pages = pc.page_table[b, :(n + 15) // 16].long()
        ks.append(pc.k_pages[pages].reshape(-1, 4, 256)[:n])
        vs.append(pc.v_pages[pages].reshape(-1, 4, 256)[:n])
    kv_indptr = torch.tensor(np.concatenate([[0], np.cumsum(kv)]), dtype=torch.int32,
                             device="cuda")
    o_r, l_r = cuda_lib.ragged_prefill(pc.q, torch.cat(ks).contiguous(), torch.cat(vs).contiguous(),
                                       pc.q_indptr, kv_indptr, causal=True, sm_scale=pc.sm_scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    assert torch.equal(o_p, o_r) and torch.equal(l_p, l_r)
    ro, rl = oracle_paged(pc)
    check_rows(o_p.reshape(-1, 256).float().cpu(), l_p.reshape(-1).cpu(), ro, rl,
               "split-KV hd256 decode mix")


@pytest.mark.parametrize("e4m3", [False, True], ids=["bf16", "e4m3"])
def test_calls_with_no_query_rows_or_no_pages(cuda_lib, e4m3):
    """A call whose requests hold no query rows returns the empty outputs; over a pool with
    no pages and requests with no keys, every row is zeros with lse = -inf."""
    make = W.paged_case_e4m3 if e4m3 else W.paged_case
    pc = make([37, 0], 8, 2, 128, qo_lens=[0, 0], seed=8, device="cuda")
    kw = dict(k_scale=pc.meta["k_scale"], v_scale=pc.meta["v_scale"]) if e4m3 else {}
    o, lse = run_gpu(cuda_lib, pc, **kw)
    assert cuda_lib.device_status() == 0
    assert o.shape == (0, 8, 128) and lse.shape == (0, 8)
    for max_qo in ([None, 4] if e4m3 else [None]):  # E4M3: conversion and tensor-core forms
        pc = make([0, 0], 8, 2, 128, qo_lens=[3, 4], seed=9, device="cuda")
        pc.k_pages, pc.v_pages = pc.k_pages[:0], pc.v_pages[:0]
        o, lse = run_gpu(cuda_lib, pc, **kw, **({} if max_qo is None else
                                                 dict(max_qo_len=max_qo)))
        assert cuda_lib.device_status() == 0
        assert torch.equal(o, torch.zeros_like(o))
        assert torch.equal(lse, torch.full_like(lse, -float("inf")))
