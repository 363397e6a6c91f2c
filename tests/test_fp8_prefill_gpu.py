"""GPU parity of the paged prefill over an FP8 E4M3 KV cache (pgqa_paged_prefill_e4m3)
against the float64 oracle's E4M3 path, on both of its paths: few query rows per request
(multi-token decode: the tensor-core E4M3 decode with the rows as MMA columns) and longer
query runs or head_dim 256 (the pages converted in the workspace, K to bf16 and V to f16,
then the paged prefill's converted-page instances).  Ragged queries over a paged cache with bottom-right causal masking are
FlashInfer documentation, flashinfer.prefill (BatchPrefillWithPagedKVCacheWrapper); the
E4M3 cache is flashinfer_benchmark.py "Attention Flags" (--kv_dtype fp8_e4m3)."""
import numpy as np
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows

pytestmark = pytest.mark.gpu

PGQA_ERR_DEVICE_BOUNDS = -6


def run(api, pc, max_qo, causal=True, **kw):
    o, lse = api.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                               pc.kv_lens_t, causal=causal, sm_scale=pc.sm_scale,
                               k_scale=pc.meta["k_scale"], v_scale=pc.meta["v_scale"],
                               max_qo_len=max_qo, **kw)
    torch.cuda.synchronize()
    return o, lse


def oracle_e4m3(pc, causal=True, rows=None):
    return oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages,
                                       pc.meta["k_scale"], pc.meta["v_scale"], pc.page_table,
                                       pc.kv_lens_t, pc.num_qo_heads, pc.num_kv_heads, causal,
                                       pc.sm_scale, rows=rows)


def mixed_lens(G, n=10, seed=0):
    """kv lengths over several chunks and a ragged page tail, query rows 0 .. 16 / G with a
    few requests holding fewer keys than query rows."""
    rng = np.random.default_rng(seed)
    qmax = 16 // G
    kv = [0, 1, 5, 16, 100, 1023, 1025, 3000, 4097, 2] + [int(x) for x in
                                                          rng.integers(1, 2500, n - 10)]
    qo = [int(x) for x in rng.integers(1, qmax + 1, len(kv))]
    qo[0] = qmax            # rows with no key at all
    qo[1] = qmax            # one key, seen by the last row only (causal)
    qo[9] = qmax            # two keys: the first rows see none (causal, qmax > 2)
    qo[3] = 0               # a request without query rows
    return kv, qo


@pytest.mark.parametrize("G,ps,causal", [(1, 16, True), (2, 64, True), (4, 16, True),
                                         (8, 32, True), (4, 128, False), (1, 32, False)])
def test_e4m3_prefill_against_oracle(cuda_lib, G, ps, causal):
    hk = 8 // G if G < 8 else 2
    kv, qo = mixed_lens(G, 12, seed=G + ps)
    pc = W.paged_case_e4m3(kv, G * hk, hk, 128, page_size=ps, qo_lens=qo, seed=301 + G + ps,
                           device="cuda", k_scale=0.5, v_scale=2.0)
    o, lse = run(cuda_lib, pc, 16 // G, causal)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc, causal)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl,
               f"e4m3 prefill G={G} ps={ps} causal={causal}")


@pytest.mark.parametrize("G,max_qo", [(4, 1), (4, 4), (8, 2), (1, 16)])
def test_one_row_per_request_matches_e4m3_decode(cuda_lib, G, max_qo):
    """One query row per request: declared as one row per request, the call is the decode,
    bit for bit.  Declared with room for more rows it runs the 16-column form, whose MMAs
    accumulate a product's hi and lo E4M3 parts in one fp32 column where the one-row form
    keeps them in two columns added at the end: the same values up to fp32 rounding, both
    within the oracle's tolerance."""
    hk = 8 // G if G < 8 else 2
    pc = W.paged_case_e4m3([0, 1, 17, 1024, 3000, 4097, 60], G * hk, hk, 128, page_size=16,
                           seed=311 + G, device="cuda")
    od, ld = cuda_lib.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens_t,
                                   sm_scale=pc.sm_scale, k_scale=pc.meta["k_scale"],
                                   v_scale=pc.meta["v_scale"])
    o, lse = run(cuda_lib, pc, max_qo)
    assert cuda_lib.device_status() == 0
    if max_qo == 1:
        assert torch.equal(o, od) and torch.equal(lse, ld)
        return
    ro, rl = oracle_e4m3(pc)
    for a, b in ((o, lse), (od, ld)):
        check_rows(a.reshape(-1, 128).float().cpu(), b.reshape(-1).cpu(), ro, rl,
                   f"one row per request G={G} max_qo={max_qo}")
    assert (o.float() - od.float()).abs().max().item() <= 2e-2
    fin = torch.isfinite(ld)
    assert torch.equal(fin, torch.isfinite(lse))
    assert (lse[fin] - ld[fin]).abs().max().item() <= 1e-4


def test_multi_row_form_with_896_key_chunks(cuda_lib):
    """Several query rows per request over a call large enough for the longest chunks: the
    multi-row tensor-core form caps them at 896 keys (7 tiles), so requests end just
    before, at and just after multiples of 896 here, with 128-token pages split across
    chunk boundaries."""
    rng = np.random.default_rng(5)
    kv = [895, 896, 897, 1791, 1792, 1793, 2688, 2689, 0, 1, 3, 127, 128, 129]
    kv += [int(x) for x in rng.integers(1, 4000, 64 - len(kv))]
    qo = [int(x) for x in rng.integers(1, 5, len(kv))]
    qo[8] = 4  # no keys at all
    # 256 pages of 128 keys per table row: with 64 requests and one kv head the chunk
    # ladder stays at its top (1024 keys, 896 for this form)
    pc = W.paged_case_e4m3(kv, 4, 1, 128, page_size=128, qo_lens=qo, seed=331, device="cuda",
                           k_scale=0.75, v_scale=1.5, stride=256)
    o, lse = run(cuda_lib, pc, 4)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl,
               "multi-row e4m3, 896-key chunks")


def test_e4m3_prefill_hnd_and_float8_dtype_match_packed_bitwise(cuda_lib):
    pc = W.paged_case_e4m3([700, 5, 2100, 33], 32, 8, 128, page_size=32, qo_lens=[4, 3, 1, 4],
                           seed=321, device="cuda")
    o, lse = run(cuda_lib, pc, 4)
    kw = dict(causal=True, sm_scale=pc.sm_scale, k_scale=pc.meta["k_scale"],
              v_scale=pc.meta["v_scale"], max_qo_len=4)
    o2, l2 = cuda_lib.paged_prefill(pc.q, pc.k_pages.view(torch.float8_e4m3fn),
                                    pc.v_pages.view(torch.float8_e4m3fn), pc.q_indptr,
                                    pc.page_table, pc.kv_lens_t, **kw)
    kh = pc.k_pages.permute(0, 2, 1, 3).contiguous()
    vh = pc.v_pages.permute(0, 2, 1, 3).contiguous()
    o3, l3 = cuda_lib.paged_prefill(pc.q, kh, vh, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                    kv_layout="HND", **kw)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    for a, b in ((o2, l2), (o3, l3)):
        assert torch.equal(a, o) and torch.equal(b, lse)


def test_multi_token_workload_sampled_rows(cuda_lib):
    """The 256-request decode workload's cache as FP8 E4M3 (scales 1) with 4 query rows per
    request, the last 4 positions of each request's keys (the multi-token decode the
    benchmark times): every request's first and last rows of two heads, and random rows,
    against the oracle."""
    pc = W.config("decode", device="cuda")
    k8 = pc.k_pages.to(torch.float8_e4m3fn).view(torch.uint8)
    v8 = pc.v_pages.to(torch.float8_e4m3fn).view(torch.uint8)
    mt = W.multi_token_case(pc, 4, k8, v8, seed=331)
    o, lse = run(cuda_lib, mt, 4)
    assert cuda_lib.device_status() == 0
    rng = np.random.default_rng(333)
    hq = mt.num_qo_heads
    rows = set()
    for b in range(mt.batch):
        for t in (4 * b, 4 * b + 3):
            rows.update({t * hq, t * hq + int(rng.integers(0, hq))})
    rows.update(rng.integers(0, 4 * mt.batch * hq, 512).tolist())
    rows = np.array(sorted(rows), dtype=np.int64)
    ro, rl = oracle_e4m3(mt, True, rows=rows)
    idx = torch.as_tensor(rows, device="cuda")
    check_rows(o.reshape(-1, 128).index_select(0, idx).float().cpu(),
               lse.reshape(-1).index_select(0, idx).cpu(), ro, rl, "multi-token workload")


def test_rows_beyond_the_declared_maximum_are_refused(cuda_lib):
    """A request with more query rows than max_qo_len: PGQA_ERR_DEVICE_BOUNDS and none of its
    rows written; the other requests are computed."""
    pc = W.paged_case_e4m3([300, 500, 40], 32, 8, 128, page_size=16, qo_lens=[2, 5, 3],
                           seed=341, device="cuda")
    o = torch.full_like(pc.q, 7.0)
    lse = torch.full(pc.q.shape[:2], 9.0, dtype=torch.float32, device="cuda")
    run(cuda_lib, pc, 4, out=o, lse=lse)
    assert cuda_lib.device_status() == PGQA_ERR_DEVICE_BOUNDS
    assert cuda_lib.device_status() == 0
    assert bool((o[2:7] == 7.0).all()) and bool((lse[2:7] == 9.0).all())
    keep = np.array([t * 32 + h for t in (0, 1, 7, 8, 9) for h in range(32)], dtype=np.int64)
    ro, rl = oracle_e4m3(pc, True, rows=keep)
    idx = torch.as_tensor(keep, device="cuda")
    check_rows(o.reshape(-1, 128).index_select(0, idx).float().cpu(),
               lse.reshape(-1).index_select(0, idx).cpu(), ro, rl, "other requests")


@pytest.mark.parametrize("d,G,ps,causal", [(128, 4, 16, True), (128, 1, 64, True),
                                           (128, 8, 32, False), (128, 16, 16, True),
                                           (256, 4, 16, True), (256, 2, 128, False),
                                           (128, 64, 16, True), (256, 32, 32, True)])
def test_e4m3_long_prefill_against_oracle(cuda_lib, d, G, ps, causal):
    """Query runs longer than 16 / G rows (and head_dim 256): the pages are converted in
    the workspace (K to bf16, V to f16) and the paged prefill runs over them."""
    hk = 2 if G >= 8 else 4
    qo, kv = [300, 45, 7, 0, 129], [700, 45, 1300, 20, 129]
    pc = W.paged_case_e4m3(kv, G * hk, hk, d, page_size=ps, qo_lens=qo, seed=361 + G + d + ps,
                           device="cuda", k_scale=0.5, v_scale=2.0)
    o, lse = run(cuda_lib, pc, max(qo), causal)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc, causal)
    check_rows(o.reshape(-1, d).float().cpu(), lse.reshape(-1).cpu(), ro, rl,
               f"e4m3 long prefill d={d} G={G} ps={ps} causal={causal}")


# Three draws of the random sweep's conversion-path cases with large scales (a sharp softmax
# over values up to ~20): with P rounded to bf16 a few outputs fall outside the tolerance.
SHARP_CASES = [
    dict(qo=[168, 60, 36], kv=[382, 497, 394], hq=24, hk=3, d=256, ps=128, ks=2.4796,
         vs=3.5294, sm=0.082759, seed=14111),
    dict(qo=[147, 68, 177, 0, 154], kv=[260, 217, 465, 241, 322], hq=8, hk=2, d=128, ps=64,
         ks=1.5529, vs=3.5720, sm=0.168655, seed=14118),
    dict(qo=[196, 177, 22, 157, 68], kv=[384, 422, 216, 203, 190], hq=8, hk=1, d=128, ps=128,
         ks=3.3333, vs=2.4256, sm=0.123823, seed=14126),
]


@pytest.mark.parametrize("c", SHARP_CASES, ids=["hd256", "hd128_ps64", "hd128_ps128"])
def test_conversion_path_keeps_weights_to_f16_precision(cuda_lib, c):
    """The converted pages hold K in bf16 and V in f16 (both exact), and P.V takes P rounded
    to f16 (11 bits) where the bf16 prefill rounds it to bf16 (8 bits).  On sharp softmaxes
    over values near 20 the conversion path stays inside the tolerance, and its worst error
    relative to the tolerance is below that of the bf16 prefill over the same values."""
    d = c["d"]
    pc = W.paged_case_e4m3(c["kv"], c["hq"], c["hk"], d, page_size=c["ps"], qo_lens=c["qo"],
                           sm_scale=c["sm"], seed=c["seed"], device="cuda", k_scale=c["ks"],
                           v_scale=c["vs"])
    o8, l8 = run(cuda_lib, pc, max(c["qo"]))
    kb = pc.k_pages.view(torch.float8_e4m3fn).to(torch.bfloat16)
    vb = pc.v_pages.view(torch.float8_e4m3fn).to(torch.bfloat16)
    ob, lb = cuda_lib.paged_prefill(pc.q, kb, vb, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                    causal=True, sm_scale=pc.sm_scale * c["ks"])
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc, True)
    check_rows(o8.reshape(-1, d).float().cpu(), l8.reshape(-1).cpu(), ro, rl,
               f"conversion path, sharp softmax {c['seed']}")
    band = 1e-2 + 1e-2 * np.abs(ro)
    r8 = (np.abs(o8.reshape(-1, d).double().cpu().numpy() - ro) / band).max()
    rb = (np.abs(ob.reshape(-1, d).double().cpu().numpy() * c["vs"] - ro) / band).max()
    assert r8 < rb, (r8, rb)


def test_pool_by_page_and_by_table_slot_agree_bitwise(cuda_lib):
    """The converted pool is indexed by page when the caller's pool is no larger than
    batch x page_table_stride pages, else by table slot with a rewritten table: same bits."""
    pc = W.paged_case_e4m3([700], 16, 4, 128, page_size=16, qo_lens=[300], seed=373,
                           device="cuda", extra_pages=10)  # 54 pages > 1 x 44 slots: by slot
    o1, l1 = run(cuda_lib, pc, 300)
    wide = torch.cat([pc.page_table, torch.full((1, 16), -1, dtype=torch.int32, device="cuda")],
                     dim=1)  # 60 slots >= 54 pages: by page
    o2, l2 = cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, wide,
                                    pc.kv_lens_t, causal=True, sm_scale=pc.sm_scale,
                                    k_scale=pc.meta["k_scale"], v_scale=pc.meta["v_scale"],
                                    max_qo_len=300)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    ro, rl = oracle_e4m3(pc, True)
    check_rows(o1.reshape(-1, 128).float().cpu(), lse_cpu(l1), ro, rl, "by table slot")


def lse_cpu(lse):
    return lse.reshape(-1).cpu()


def test_bad_page_id_on_the_conversion_path_is_reported(cuda_lib):
    pc = W.paged_case_e4m3([300, 500], 32, 8, 128, page_size=16, qo_lens=[100, 50], seed=381,
                           device="cuda")
    pc.page_table[1, 3] = pc.num_pages + 3
    run(cuda_lib, pc, 100)
    assert cuda_lib.device_status() == PGQA_ERR_DEVICE_BOUNDS
    assert cuda_lib.device_status() == 0


def test_default_max_qo_len_is_the_total_row_count(cuda_lib):
    """Without max_qo_len the binding passes total_q, an upper bound: here 7 rows x 4 heads
    > 16 columns, so the conversion path runs; it agrees with the tensor-core path (which
    the true maximum, 4, selects) to the parity tolerance."""
    pc = W.paged_case_e4m3([100, 2000], 32, 8, 128, page_size=16, qo_lens=[3, 4], seed=391,
                           device="cuda")
    o1, l1 = cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                                    pc.kv_lens_t, sm_scale=pc.sm_scale,
                                    k_scale=pc.meta["k_scale"], v_scale=pc.meta["v_scale"])
    o2, l2 = run(cuda_lib, pc, 4)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc, True)
    for o, l, what in ((o1, l1, "conversion path"), (o2, l2, "tensor-core path")):
        check_rows(o.reshape(-1, 128).float().cpu(), l.reshape(-1).cpu(), ro, rl, what)


def test_conversion_path_hnd_and_float8_dtype_match_packed_bitwise(cuda_lib):
    pc = W.paged_case_e4m3([700, 5, 1300], 16, 4, 128, page_size=32, qo_lens=[200, 5, 64],
                           seed=395, device="cuda")
    o, lse = run(cuda_lib, pc, 200)
    kw = dict(causal=True, sm_scale=pc.sm_scale, k_scale=pc.meta["k_scale"],
              v_scale=pc.meta["v_scale"], max_qo_len=200)
    o2, l2 = cuda_lib.paged_prefill(pc.q, pc.k_pages.view(torch.float8_e4m3fn),
                                    pc.v_pages.view(torch.float8_e4m3fn), pc.q_indptr,
                                    pc.page_table, pc.kv_lens_t, **kw)
    kh = pc.k_pages.permute(0, 2, 1, 3).contiguous()
    vh = pc.v_pages.permute(0, 2, 1, 3).contiguous()
    o3, l3 = cuda_lib.paged_prefill(pc.q, kh, vh, pc.q_indptr, pc.page_table, pc.kv_lens_t,
                                    kv_layout="HND", **kw)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    for a, b in ((o2, l2), (o3, l3)):
        assert torch.equal(a, o) and torch.equal(b, lse)


def test_conversion_path_short_list_splits_after_conversion(cuda_lib):
    """One request of 20 query rows (80 columns at G 4: the conversion path) over 20k keys:
    a work list short enough for the bf16 prefill to split it into chunks, merged by LSE;
    every row against the oracle."""
    pc = W.paged_case_e4m3([20000, 0], 32, 8, 128, page_size=16, qo_lens=[20, 3], seed=397,
                           device="cuda")
    o, lse = run(cuda_lib, pc, 20)
    assert cuda_lib.device_status() == 0
    ro, rl = oracle_e4m3(pc, True)
    check_rows(o.reshape(-1, 128).float().cpu(), lse.reshape(-1).cpu(), ro, rl,
               "conversion path, split-KV")


@pytest.mark.parametrize("max_qo", [4, 64])
def test_e4m3_layer_slice_matches_packed_bitwise(cuda_lib, max_qo):
    """A per-layer slice of a layer-interleaved E4M3 cache [pages, layers, slots, heads, d]
    (non-contiguous pages) gives the packed result bit for bit on both paths."""
    qo = [4, 3] if max_qo == 4 else [64, 17]
    pc = W.paged_case_e4m3([900, 2500], 16, 4, 128, page_size=16, qo_lens=qo, seed=399,
                           device="cuda")
    o, lse = run(cuda_lib, pc, max_qo)
    layers = 3
    shape = (pc.num_pages, layers) + tuple(pc.k_pages.shape[1:])
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    kst = torch.randint(0, 256, shape, generator=gen, device="cuda", dtype=torch.int32)
    vst = torch.randint(0, 256, shape, generator=gen, device="cuda", dtype=torch.int32)
    kst, vst = kst.to(torch.uint8), vst.to(torch.uint8)
    kst[:, 1] = pc.k_pages
    vst[:, 1] = pc.v_pages
    o2, l2 = cuda_lib.paged_prefill(pc.q, kst[:, 1], vst[:, 1], pc.q_indptr, pc.page_table,
                                    pc.kv_lens_t, causal=True, sm_scale=pc.sm_scale,
                                    k_scale=pc.meta["k_scale"], v_scale=pc.meta["v_scale"],
                                    max_qo_len=max_qo)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("max_qo", [4, None], ids=["tensor-core", "conversion"])
def test_nan_bytes_in_unused_tail_slots_are_invisible(cuda_lib, max_qo):
    """E4M3 NaN bytes in the key slots past each request's last key (its last page's tail)
    change nothing: the scores of those slots are masked and their V rows never reach
    P.V (0 * NaN would be NaN)."""
    kv, qo = [20, 1030, 3, 901], [4, 3, 2, 4]
    pc = W.paged_case_e4m3(kv, 16, 4, 128, page_size=16, qo_lens=qo, seed=131, device="cuda")
    mq = max_qo if max_qo is not None else sum(qo)
    o1, l1 = run(cuda_lib, pc, mq)
    for b, n in enumerate(pc.kv_lens):
        last = int(pc.page_table[b, (n - 1) // 16])
        pc.k_pages[last, n % 16:] = 0x7F   # E4M3 NaN
        pc.v_pages[last, n % 16:] = 0xFF
    o2, l2 = run(cuda_lib, pc, mq)
    assert cuda_lib.device_status() == 0
    assert torch.isfinite(o2.float()).all()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
