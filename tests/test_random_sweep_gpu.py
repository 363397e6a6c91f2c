"""Seeded random sweep of shapes through every compute entry point, each case compared
with the float64 oracle on all rows.

Every case draws its own shapes from a fixed seed:
- batch size; per-request lengths, including empty requests and kv_len < qo_len;
- query and kv head counts, head_dim, causal or not, sm_scale;
- page size, KV layout (NHD / HND) and FP8 scales; for the E4M3 paged prefill, short
  or long query runs (its two paths).

The sweep reaches combinations that the hand-written cases do not list: long and short
requests mixed in one batch, several KV heads with large groups, and both split regimes
of the paged prefill and the decode.  The tolerance is the path's: |o - oracle| <=
1e-2 + 1e-2 |oracle| and |lse - oracle| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows

pytestmark = pytest.mark.gpu

N_CASES = 12


def _lens(rng, batch, lo, hi, p_zero=0.1):
    out = []
    for _ in range(batch):
        out.append(0 if rng.random() < p_zero else int(rng.integers(lo, hi + 1)))
    return out


def _scale(rng, d):
    r = rng.random()
    if r < 0.1:
        return 0.0
    if r < 0.2:
        return -1.0 / math.sqrt(d)
    return float(rng.uniform(0.3, 2.0) / math.sqrt(d))


def _heads(rng, groups):
    g = int(rng.choice(groups))
    hk = int(rng.choice([1, 2, 3]))
    return g * hk, hk


def _hnd(t):
    return t.permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("case", range(N_CASES))
def test_ragged_prefill_sweep(cuda_lib, case):
    rng = np.random.default_rng(5000 + case)
    batch = int(rng.integers(1, 6))
    d = int(rng.choice([128, 256]))
    hq, hk = _heads(rng, [1, 2, 4, 8, 16])
    causal = bool(rng.random() < 0.75)
    qo = _lens(rng, batch, 1, 300)
    kv = [max(0, q + int(rng.integers(-40, 700))) for q in qo]
    c = W.ragged_case(qo, kv, hq, hk, d, causal=causal, sm_scale=_scale(rng, d),
                      seed=6000 + case, device="cuda")
    o, lse = cuda_lib.ragged_prefill(c.q, c.k, c.v, c.q_indptr, c.kv_indptr, causal=causal,
                                     sm_scale=c.sm_scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.ragged_attention(c.q, c.k, c.v, c.q_indptr, c.kv_indptr, hq, hk, causal,
                                     c.sm_scale)
    check_rows(o.reshape(-1, d), lse.reshape(-1), ro, rl,
               f"ragged case {case}: qo {qo} kv {kv} heads {hq}/{hk} d {d} causal {causal}")


@pytest.mark.parametrize("case", range(N_CASES))
def test_paged_prefill_sweep(cuda_lib, case):
    rng = np.random.default_rng(7000 + case)
    batch = int(rng.integers(1, 6))
    d = int(rng.choice([128, 256]))
    hq, hk = _heads(rng, [1, 2, 4, 8])
    ps = int(rng.choice([16, 32, 64, 128]))
    layout = str(rng.choice(["NHD", "HND"]))
    # short query runs (speculative verification) or longer appends
    short = rng.random() < 0.5
    qo = _lens(rng, batch, 1, 8 if short else 250, p_zero=0.05)
    kv = [q + int(rng.integers(0, 3000 if short else 600)) for q in qo]
    pc = W.paged_case(kv, hq, hk, d, page_size=ps, qo_lens=qo, sm_scale=_scale(rng, d),
                      seed=8000 + case, device="cuda", extra_pages=int(rng.integers(0, 5)))
    k, v = (pc.k_pages, pc.v_pages) if layout == "NHD" else (_hnd(pc.k_pages), _hnd(pc.v_pages))
    o, lse = cuda_lib.paged_prefill(pc.q, k, v, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                    causal=True, sm_scale=pc.sm_scale, kv_layout=layout)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                    pc.kv_lens_t, hq, hk, True, pc.sm_scale)
    check_rows(o.reshape(-1, d), lse.reshape(-1), ro, rl,
               f"paged case {case}: qo {qo} kv {kv} heads {hq}/{hk} d {d} page {ps} {layout}")


@pytest.mark.parametrize("case", range(N_CASES))
def test_paged_decode_sweep(cuda_lib, case):
    rng = np.random.default_rng(9000 + case)
    batch = int(rng.integers(1, 9))
    hq, hk = _heads(rng, [1, 2, 4, 8])
    ps = int(rng.choice([16, 32, 64, 128]))
    layout = str(rng.choice(["NHD", "HND"]))
    kv = _lens(rng, batch, 1, 5000)
    # a wide page table gives small batches longer chunks (the chunk length follows the
    # table's key capacity)
    stride = None if rng.random() < 0.5 else 70000 // ps
    pc = W.paged_case(kv, hq, hk, 128, page_size=ps, sm_scale=_scale(rng, 128), stride=stride,
                      seed=10000 + case, device="cuda")
    k, v = (pc.k_pages, pc.v_pages) if layout == "NHD" else (_hnd(pc.k_pages), _hnd(pc.v_pages))
    o, lse = cuda_lib.paged_decode(pc.q, k, v, pc.page_table, pc.kv_lens_t,
                                   sm_scale=pc.sm_scale, kv_layout=layout)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                    pc.kv_lens_t, hq, hk, True, pc.sm_scale)
    check_rows(o.reshape(-1, 128), lse.reshape(-1), ro, rl,
               f"decode case {case}: kv {kv} heads {hq}/{hk} page {ps} {layout} stride {stride}")


@pytest.mark.parametrize("case", range(N_CASES))
def test_e4m3_decode_sweep(cuda_lib, case):
    rng = np.random.default_rng(11000 + case)
    batch = int(rng.integers(1, 9))
    hq, hk = _heads(rng, [1, 2, 4, 8])
    ps = int(rng.choice([16, 32, 64, 128]))
    kv = _lens(rng, batch, 1, 5000)
    ks, vs = float(rng.uniform(0.1, 4.0)), float(rng.uniform(0.1, 4.0))
    pc = W.paged_case_e4m3(kv, hq, hk, 128, page_size=ps, sm_scale=_scale(rng, 128),
                           seed=12000 + case, device="cuda", k_scale=ks, v_scale=vs)
    o, lse = cuda_lib.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens_t,
                                   sm_scale=pc.sm_scale, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, ks, vs,
                                         pc.page_table, pc.kv_lens_t, hq, hk, True,
                                         pc.sm_scale)
    check_rows(o.reshape(-1, 128), lse.reshape(-1), ro, rl,
               f"e4m3 case {case}: kv {kv} heads {hq}/{hk} page {ps} scales {ks:.2f}/{vs:.2f}")


@pytest.mark.parametrize("case", range(N_CASES))
def test_e4m3_prefill_sweep(cuda_lib, case):
    """The E4M3 paged prefill on both of its paths: few query rows per request (the
    tensor-core path, max_qo_len * G <= 16) or longer runs and head_dim 256 (the pages
    converted first, K to bf16 and V to f16); causal or not, both layouts, random scales."""
    rng = np.random.default_rng(13000 + case)
    batch = int(rng.integers(1, 6))
    hq, hk = _heads(rng, [1, 2, 4, 8])
    g = hq // hk
    short = rng.random() < 0.5
    d = 128 if short else int(rng.choice([128, 256]))
    ps = int(rng.choice([16, 32, 64, 128]))
    layout = str(rng.choice(["NHD", "HND"]))
    causal = bool(rng.random() < 0.75)
    qmax = max(1, 16 // g) if short else 200
    qo = _lens(rng, batch, 1, qmax, p_zero=0.05)
    kv = [max(0, q + int(rng.integers(-3, 3000 if short else 500))) for q in qo]
    ks, vs = float(rng.uniform(0.1, 4.0)), float(rng.uniform(0.1, 4.0))
    pc = W.paged_case_e4m3(kv, hq, hk, d, page_size=ps, qo_lens=qo, sm_scale=_scale(rng, d),
                           seed=14000 + case, device="cuda", k_scale=ks, v_scale=vs,
                           extra_pages=int(rng.integers(0, 5)))
    k, v = (pc.k_pages, pc.v_pages) if layout == "NHD" else (_hnd(pc.k_pages), _hnd(pc.v_pages))
    o, lse = cuda_lib.paged_prefill(pc.q, k, v, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                    causal=causal, sm_scale=pc.sm_scale, kv_layout=layout,
                                    k_scale=ks, v_scale=vs, max_qo_len=max(max(qo), 1))
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, ks, vs,
                                         pc.page_table, pc.kv_lens_t, hq, hk, causal,
                                         pc.sm_scale)
    check_rows(o.reshape(-1, d), lse.reshape(-1), ro, rl,
               f"e4m3 prefill case {case}: qo {qo} kv {kv} heads {hq}/{hk} d {d} page {ps} "
               f"{layout} causal {causal} scales {ks:.2f}/{vs:.2f}")
