"""K/V page pools in other layouts (pgqa_paged_prefill_bf16_strided,
pgqa_paged_decode_bf16_strided): HND [num_pages, Hk, page_size, d] (FlashInfer
documentation, flashinfer_benchmark.py "Attention Flags", --kv_layout NHD / HND) and a
per-layer slice of a layer-interleaved cache [num_pages, layers, page_size, Hk, d] (the
vllm-rlt pull request's GPU tests run its decode on non-contiguous layer slices).  The
same keys in any layout give the packed-NHD result bit for bit: only the TMA addressing
differs.  One case is also checked against the oracle directly."""
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows

pytestmark = pytest.mark.gpu


def layouts(pc, layers=3, layer=1):
    """(name, kv_layout, k, v) views of pc's pools in other layouts, same contents."""
    hnd_k = pc.k_pages.permute(0, 2, 1, 3).contiguous()
    hnd_v = pc.v_pages.permute(0, 2, 1, 3).contiguous()
    out = [("hnd", "HND", hnd_k, hnd_v)]
    stk = torch.randn((pc.num_pages, layers) + tuple(pc.k_pages.shape[1:]), device="cuda",
                      dtype=torch.float32).to(torch.bfloat16)
    stv = torch.randn_like(stk, dtype=torch.float32).to(torch.bfloat16)
    stk[:, layer] = pc.k_pages
    stv[:, layer] = pc.v_pages
    out.append(("layer-slice", "NHD", stk[:, layer], stv[:, layer]))
    # an HND view of a permuted (non-contiguous) tensor: strides differ from a packed HND
    out.append(("hnd-view", "HND", pc.k_pages.permute(0, 2, 1, 3), pc.v_pages.permute(0, 2, 1, 3)))
    # pages padded by 8 elements: the page stride is not a multiple of the head stride
    n, ps, hk, d = pc.k_pages.shape
    padded = []
    for src in (pc.k_pages, pc.v_pages):
        flat = torch.zeros((n, ps * hk * d + 8), device="cuda", dtype=torch.bfloat16)
        view = flat.as_strided((n, ps, hk, d), (ps * hk * d + 8, hk * d, d, 1))
        view.copy_(src)
        padded.append(view)
    out.append(("padded-pages", "NHD", padded[0], padded[1]))
    return out


@pytest.mark.parametrize("d,ps", [(128, 16), (128, 64), (256, 16), (256, 32)])
def test_paged_prefill_layouts_match_nhd_bitwise(cuda_lib, d, ps):
    pc = W.paged_case([500, 45, 1300], 16, 4, d, page_size=ps, qo_lens=[200, 45, 7],
                      seed=81 + d + ps, device="cuda")
    o, lse = cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                                    pc.kv_lens_t)
    for name, lay, k, v in layouts(pc):
        assert not (lay == "NHD" and k.is_contiguous())
        o2, l2 = cuda_lib.paged_prefill(pc.q, k, v, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                        kv_layout=lay)
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        assert torch.equal(o2, o) and torch.equal(l2, lse), name


@pytest.mark.parametrize("ps", [16, 128])
def test_paged_decode_layouts_match_nhd_bitwise(cuda_lib, ps):
    pc = W.paged_case([1, 700, 3000, 1025], 32, 8, 128, page_size=ps, seed=83 + ps,
                      device="cuda")
    o, lse = cuda_lib.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens_t)
    for name, lay, k, v in layouts(pc):
        o2, l2 = cuda_lib.paged_decode(pc.q, k, v, pc.page_table, pc.kv_lens_t, kv_layout=lay)
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        assert torch.equal(o2, o) and torch.equal(l2, lse), name


def test_hnd_paged_prefill_against_oracle(cuda_lib):
    pc = W.paged_case([333, 64], 8, 2, 128, page_size=32, qo_lens=[100, 64], seed=87,
                      device="cuda")
    k = pc.k_pages.permute(0, 2, 1, 3).contiguous()
    v = pc.v_pages.permute(0, 2, 1, 3).contiguous()
    o, lse = cuda_lib.paged_prefill(pc.q, k, v, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                    kv_layout="HND")
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                    pc.kv_lens_t, 8, 2, True, pc.sm_scale)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl, "HND prefill")


def test_mismatched_k_v_strides_are_refused(cuda_lib):
    pc = W.paged_case([40], 8, 2, 128, page_size=16, seed=89, device="cuda")
    k = pc.k_pages.permute(0, 2, 1, 3).contiguous()
    with pytest.raises(ValueError):
        cuda_lib.paged_decode(pc.q, k, pc.v_pages.permute(0, 2, 1, 3), pc.page_table,
                              pc.kv_lens_t, kv_layout="HND")
