"""GPU parity of the ragged prefill (pgqa_ragged_prefill_bf16) against the float64 oracle.

Small cases are compared element by element on every row; the large serving workloads
(16 x U{128..4096} hd128, the cached-prefix hd256 batch, one 32k-token request) are run
in full on the GPU, in the launch configuration the benchmark times, and compared on
sampled rows, which the oracle computes one by one (rows are independent).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows, gather_rows, sample_prefill_rows

pytestmark = pytest.mark.gpu


def run_gpu(api, case):
    o, lse = api.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                causal=case.causal, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    return o, lse


def full_check(api, case, what):
    o, lse = run_gpu(api, case)
    ro, rl = oracle.ragged_attention(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                     case.num_qo_heads, case.num_kv_heads, case.causal,
                                     case.sm_scale)
    return check_rows(o.reshape(-1, o.shape[-1]).float().cpu(), lse.reshape(-1).cpu(), ro, rl,
                      what)


def test_tiny_workload(cuda_lib):
    case = W.config("tiny", device="cuda")
    full_check(cuda_lib, case, "tiny")


SMALL = [
    # qo_lens, kv_lens, Hq, Hk, d, causal
    ([17, 64], [17, 64], 4, 2, 128, True),
    ([1], [1], 1, 1, 128, True),
    ([300, 5, 129, 128], [300, 5, 129, 128], 8, 2, 128, True),
    ([200, 77], [500, 1000], 8, 1, 128, True),       # cached prefix (kv > qo)
    ([200, 77], [500, 1000], 8, 1, 128, False),
    ([90, 40], [30, 40], 4, 4, 128, True),           # kv < qo: leading rows see no key
    ([0, 33, 0, 70], [10, 33, 0, 0], 16, 1, 128, True),  # empty q / empty kv requests
    ([513], [513], 16, 16, 128, True),               # G = 1
    ([260, 31], [260, 31], 32, 2, 128, True),        # G = 16
    ([129, 200], [129, 700], 8, 2, 256, True),       # hd256
    ([64, 300], [64, 300], 4, 1, 256, False),
    ([37, 5, 130], [200, 5, 130], 64, 2, 128, True),    # G = 32: 4 tokens per q tile
    ([37, 5, 130], [200, 90, 130], 64, 1, 128, False),  # G = 64: 2 tokens per q tile
    ([9, 3, 40], [300, 3, 41], 128, 1, 128, True),      # G = 128: one token per q tile
    ([21, 6], [150, 6], 128, 1, 256, True),             # G = 128, hd256
    ([33, 70], [400, 70], 64, 2, 256, False),           # G = 32, hd256
]


@pytest.mark.parametrize("shape", SMALL, ids=[f"s{i}" for i in range(len(SMALL))])
def test_small_shapes(cuda_lib, shape):
    qo, kv, hq, hk, d, causal = shape
    case = W.ragged_case(qo, kv, hq, hk, d, causal=causal, seed=len(qo) * 31 + hq + d,
                         device="cuda")
    full_check(cuda_lib, case, f"shape {shape}")


@pytest.mark.parametrize("scale", [0.0, -0.2, 0.5])
def test_unusual_scales(cuda_lib, scale):
    case = W.ragged_case([150, 40], [150, 90], 8, 2, 128, causal=True, sm_scale=scale,
                         seed=5, device="cuda")
    full_check(cuda_lib, case, f"scale {scale}")


def test_large_logits_stay_stable(cuda_lib):
    case = W.ragged_case([300], [300], 8, 1, 128, causal=True, seed=9, device="cuda",
                         k_scale=6.0)
    full_check(cuda_lib, case, "K x 6")


@pytest.mark.parametrize("name", ["prefill_hd128", "prefix_hd256", "long"])
def test_serving_workloads_sampled(cuda_lib, name):
    case = W.config(name, device="cuda")
    o, lse = run_gpu(cuda_lib, case)
    G = case.num_qo_heads // case.num_kv_heads
    rows = sample_prefill_rows(case.qo_lens, case.num_qo_heads, G, seed=1)
    og, lg = gather_rows(o, lse, rows, case.num_qo_heads)
    ro, rl = oracle.ragged_attention(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                     case.num_qo_heads, case.num_kv_heads, case.causal,
                                     case.sm_scale, rows=rows)
    check_rows(og, lg, ro, rl, name)
    assert torch.isfinite(o.float()).all()


def test_repeat_is_bitwise_identical(cuda_lib):
    case = W.ragged_case([700, 33, 1200], [700, 500, 1200], 16, 4, 128, seed=3, device="cuda")
    o1, l1 = run_gpu(cuda_lib, case)
    o2, l2 = run_gpu(cuda_lib, case)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_request_order_is_bitwise_invariant(cuda_lib):
    case = W.ragged_case([333, 70, 901], [333, 400, 901], 8, 2, 128, seed=4, device="cuda")
    o, l = run_gpu(cuda_lib, case)
    qs, ks = case.q_indptr.tolist(), case.kv_indptr.tolist()
    order = [2, 0, 1]
    rq = torch.cat([case.q[qs[b]:qs[b + 1]] for b in order])
    rk = torch.cat([case.k[ks[b]:ks[b + 1]] for b in order])
    rv = torch.cat([case.v[ks[b]:ks[b + 1]] for b in order])
    qo2 = [case.qo_lens[b] for b in order]
    kv2 = [case.kv_lens[b] for b in order]
    o2, l2 = cuda_lib.ragged_prefill(rq, rk, rv, W._indptr(qo2, "cuda"), W._indptr(kv2, "cuda"),
                                     causal=True, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    start = 0
    for nb, b in enumerate(order):
        n = qo2[nb]
        assert torch.equal(o2[start:start + n], o[qs[b]:qs[b + 1]])
        assert torch.equal(l2[start:start + n], l[qs[b]:qs[b + 1]])
        start += n


def test_causal_never_reads_future_keys(cuda_lib):
    case = W.ragged_case([256], [256], 8, 2, 128, seed=6, device="cuda")
    o, l = run_gpu(cuda_lib, case)
    k2, v2 = case.k.clone(), case.v.clone()
    k2[200:] = 3.0
    v2[200:] = -9.0
    o2, l2 = cuda_lib.ragged_prefill(case.q, k2, v2, case.q_indptr, case.kv_indptr,
                                     causal=True, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    assert torch.equal(o2[:200], o[:200]) and torch.equal(l2[:200], l[:200])
    assert not torch.equal(o2[200:], o[200:])


def test_lse_optional(cuda_lib):
    case = W.ragged_case([100], [100], 4, 1, 128, seed=8, device="cuda")
    o, _ = run_gpu(cuda_lib, case)
    o2, l2 = cuda_lib.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                     causal=True, return_lse=False)
    torch.cuda.synchronize()
    assert l2 is None and torch.equal(o, o2)


def test_bad_indptr_reports_bounds_status(cuda_lib):
    case = W.ragged_case([10, 20], [10, 20], 4, 1, 128, seed=2, device="cuda")
    bad = torch.tensor([0, 10, 5], dtype=torch.int32, device="cuda")  # decreasing
    out = torch.full_like(case.q, 7.0)
    cuda_lib.ragged_prefill(case.q, case.k, case.v, bad, case.kv_indptr, out=out)
    assert cuda_lib.device_status() == -6
    assert bool((out == 7.0).all())                      # nothing written
    run_gpu(cuda_lib, case)                              # library still usable


def test_calls_with_no_query_rows_or_no_keys(cuda_lib):
    """A call whose requests hold no query rows returns the empty outputs; a call whose
    requests hold no keys (K/V without rows) gives every row zeros and lse = -inf."""
    case = W.ragged_case([0], [37], 8, 2, 128, seed=6, device="cuda")
    o, lse = run_gpu(cuda_lib, case)
    assert o.shape == (0, 8, 128) and lse.shape == (0, 8)
    case = W.ragged_case([5, 70], [0, 0], 8, 2, 128, seed=7, device="cuda")
    assert case.k.shape[0] == 0
    o, lse = run_gpu(cuda_lib, case)
    assert torch.equal(o, torch.zeros_like(o))
    assert torch.equal(lse, torch.full_like(lse, -float("inf")))
