"""Serving guarantees of the C ABI on the GPU.

- Batch-composition invariance: a request's output and lse do not depend on which other
  requests share the launch or on their order, bit for bit, among launches that take the
  same chunking regime.  The work list cuts every request into (kv head, q tile) items
  with a fixed K/V tiling, and split-KV chunks are request-local (2048 keys in the
  prefill; 1024, 512, 256 or 128 keys in the decode), so each row's arithmetic is the
  same in any such batch (the vllm-rlt pull request "feat: add FlashInfer attention
  backend for SM120 decode" asks the same of its decode kernel, Design notes).
- CUDA-graph replay: once a call has run (so the workspace exists), the prefills and the
  decode can be captured into a CUDA graph; replaying it after rewriting the captured
  input buffers (new contents and new per-request lengths within the same buffer sizes)
  gives the eager results for the new inputs, bit for bit, because the plan kernels read
  the lengths and patch the tensor maps on the device.
"""
import numpy as np
import pytest
import torch

from paged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _indptr(lens):
    return torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")


def test_ragged_prefill_batch_composition_is_bitwise_invariant(cuda_lib):
    qo = [300, 1, 129, 700]
    kv = [300, 900, 129, 1500]
    case = W.ragged_case(qo, kv, 16, 4, 128, causal=True, seed=61, device="cuda")
    o, lse = cuda_lib.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr)
    qi = case.q_indptr.tolist()
    ki = case.kv_indptr.tolist()
    for order in ([3, 1], [2], [0, 3, 2, 1]):
        q = torch.cat([case.q[qi[b]:qi[b + 1]] for b in order]).contiguous()
        k = torch.cat([case.k[ki[b]:ki[b + 1]] for b in order]).contiguous()
        v = torch.cat([case.v[ki[b]:ki[b + 1]] for b in order]).contiguous()
        o2, l2 = cuda_lib.ragged_prefill(q, k, v, _indptr([qo[b] for b in order]),
                                         _indptr([kv[b] for b in order]))
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        at = 0
        for b in order:
            n = qo[b]
            assert torch.equal(o2[at:at + n], o[qi[b]:qi[b + 1]]), (order, b)
            assert torch.equal(l2[at:at + n], lse[qi[b]:qi[b + 1]]), (order, b)
            at += n


def test_paged_prefill_batch_composition_is_bitwise_invariant(cuda_lib):
    qo = [4, 64, 1, 200]
    kv = [1000, 64, 3000, 700]
    pc = W.paged_case(kv, 32, 8, 128, page_size=16, qo_lens=qo, seed=67, device="cuda")
    o, lse = cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                                    pc.kv_lens_t)
    qi = pc.q_indptr.tolist()
    for order in ([2, 0], [3, 2, 1, 0]):
        q = torch.cat([pc.q[qi[b]:qi[b + 1]] for b in order]).contiguous()
        o2, l2 = cuda_lib.paged_prefill(q, pc.k_pages, pc.v_pages, _indptr([qo[b] for b in order]),
                                        pc.page_table[order].contiguous(),
                                        pc.kv_lens_t[order].contiguous())
        torch.cuda.synchronize()
        assert cuda_lib.device_status() == 0
        at = 0
        for b in order:
            n = qo[b]
            assert torch.equal(o2[at:at + n], o[qi[b]:qi[b + 1]]), (order, b)
            assert torch.equal(l2[at:at + n], lse[qi[b]:qi[b + 1]]), (order, b)
            at += n


def test_cuda_graph_replay_with_rewritten_inputs(cuda_lib):
    api = cuda_lib
    dev = torch.device("cuda")
    # buffers sized for the largest step; lengths change between replays
    qo_a, kv_a = [100, 37, 300], [100, 500, 300]
    qo_b, kv_b = [50, 80, 250], [900, 80, 260]
    case_a = W.ragged_case(qo_a, kv_a, 16, 4, 128, seed=71, device=dev)
    case_b = W.ragged_case(qo_b, kv_b, 16, 4, 128, seed=72, device=dev)
    tq = max(case_a.total_q, case_b.total_q)
    tk = max(sum(kv_a), sum(kv_b))
    q = torch.zeros((tq, 16, 128), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((tk, 4, 128), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    qi = torch.zeros(4, dtype=torch.int32, device=dev)
    ki = torch.zeros(4, dtype=torch.int32, device=dev)
    o = torch.zeros_like(q)
    lse = torch.zeros((tq, 16), dtype=torch.float32, device=dev)

    dec_a = W.paged_case([40, 2100, 1025], 32, 8, 128, page_size=16, seed=73, extra_pages=200,
                         device=dev)
    dec_b = W.paged_case([1500, 7, 3000], 32, 8, 128, page_size=16, seed=74, device=dev)
    npages = max(dec_a.num_pages, dec_b.num_pages)
    stride = max(dec_a.page_table.shape[1], dec_b.page_table.shape[1])
    kp = torch.zeros((npages, 16, 8, 128), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    pt = torch.full((3, stride), -1, dtype=torch.int32, device=dev)
    kl = torch.zeros(3, dtype=torch.int32, device=dev)
    dq = torch.zeros((3, 32, 128), dtype=torch.bfloat16, device=dev)
    do = torch.zeros_like(dq)
    dl = torch.zeros((3, 32), dtype=torch.float32, device=dev)
    pq = torch.zeros((12, 32, 128), dtype=torch.bfloat16, device=dev)  # 4 rows per request
    pqi = torch.arange(0, 13, 4, dtype=torch.int32, device=dev)
    po = torch.zeros_like(pq)
    pl = torch.zeros((12, 32), dtype=torch.float32, device=dev)

    def load(case, dec, pqv):
        q.zero_(); k.zero_(); v.zero_()
        q[:case.total_q].copy_(case.q)
        k[:sum(case.kv_lens)].copy_(case.k)
        v[:sum(case.kv_lens)].copy_(case.v)
        qi.copy_(case.q_indptr)
        ki.copy_(case.kv_indptr)
        kp.zero_(); vp.zero_(); pt.fill_(-1)
        kp[:dec.num_pages].copy_(dec.k_pages)
        vp[:dec.num_pages].copy_(dec.v_pages)
        pt[:, :dec.page_table.shape[1]].copy_(dec.page_table)
        kl.copy_(dec.kv_lens_t)
        dq.copy_(dec.q)
        pq.copy_(pqv)

    def step():
        api.ragged_prefill(q, k, v, qi, ki, out=o, lse=lse)
        api.paged_decode(dq, kp, vp, pt, kl, out=do, lse=dl)
        api.paged_prefill(pq, kp, vp, pqi, pt, kl, out=po, lse=pl)

    g = torch.Generator(device=dev)
    g.manual_seed(75)
    pq_a = torch.randn((12, 32, 128), generator=g, device=dev).to(torch.bfloat16)
    pq_b = torch.randn((12, 32, 128), generator=g, device=dev).to(torch.bfloat16)

    # eager references
    refs = []
    for case, dec, pqv in ((case_a, dec_a, pq_a), (case_b, dec_b, pq_b)):
        load(case, dec, pqv)
        step()
        torch.cuda.synchronize()
        assert api.device_status() == 0
        refs.append([t.clone() for t in (o, lse, do, dl, po, pl)])

    load(case_a, dec_a, pq_a)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(graph):
        step()
    for idx, (case, dec, pqv) in enumerate(((case_b, dec_b, pq_b), (case_a, dec_a, pq_a),
                                            (case_b, dec_b, pq_b))):
        for t in (o, lse, do, dl, po, pl):
            t.zero_()
        load(case, dec, pqv)
        graph.replay()
        torch.cuda.synchronize()
        assert api.device_status() == 0
        ref = refs[1] if case is case_b else refs[0]
        nq = case.total_q
        assert torch.equal(o[:nq], ref[0][:nq]) and torch.equal(lse[:nq], ref[1][:nq]), idx
        for got, want in zip((do, dl, po, pl), ref[2:]):
            assert torch.equal(got, want), idx


def test_calls_on_a_side_stream_match_the_default_stream(cuda_lib):
    """Every entry point enqueues on the stream it is given (here a second stream of the
    tensors' device) and gives the same bits as on the current stream."""
    case = W.ragged_case([300, 77], [300, 900], 16, 4, 128, seed=77, device="cuda")
    pc = W.paged_case([1000, 20], 32, 8, 128, page_size=16, qo_lens=[4, 3], seed=78,
                      device="cuda")
    dc = W.paged_case([1000, 20, 4000], 32, 8, 128, page_size=16, seed=79, device="cuda")

    def run(stream):
        return (cuda_lib.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                        stream=stream),
                cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                                       pc.kv_lens_t, stream=stream),
                cuda_lib.paged_decode(dc.q, dc.k_pages, dc.v_pages, dc.page_table, dc.kv_lens_t,
                                      stream=stream))

    ref = run(None)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    got = run(side)
    side.synchronize()
    assert cuda_lib.device_status(side) == 0
    for (o1, l1), (o2, l2) in zip(ref, got):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_batches_beyond_the_plans_shared_memory_path(cuda_lib):
    """Batches of more than 2048 requests make the prefill plan keep its per-request
    arrays in global memory instead of shared memory; 3000 short requests go through the
    ragged prefill, the paged prefill and the decode, checked against the oracle on a
    sample of requests."""
    import oracle
    from gpu_util import check_rows
    rng = np.random.default_rng(91)
    batch = 3000
    qo = rng.integers(1, 4, batch).tolist()
    kv = [q + int(x) for q, x in zip(qo, rng.integers(0, 60, batch))]
    case = W.ragged_case(qo, kv, 8, 2, 128, causal=True, seed=92, device="cuda")
    o, lse = cuda_lib.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr)
    pc = W.paged_case(kv, 8, 2, 128, page_size=16, qo_lens=qo, seed=93, device="cuda")
    po, pl = cuda_lib.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                                    pc.kv_lens_t)
    dc = W.paged_case(kv, 8, 2, 128, page_size=16, seed=94, device="cuda")
    do, dl = cuda_lib.paged_decode(dc.q, dc.k_pages, dc.v_pages, dc.page_table, dc.kv_lens_t)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    qi = case.q_indptr.tolist()
    pick = sorted(set([0, batch - 1] + rng.choice(batch, 40, replace=False).tolist()))
    rows = np.array([(t * 8 + h) for b in pick for t in range(qi[b], qi[b + 1])
                     for h in range(8)], dtype=np.int64)
    ro, rl = oracle.ragged_attention(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                     8, 2, True, case.sm_scale, rows=rows)
    idx = torch.as_tensor(rows, device="cuda")
    check_rows(o.reshape(-1, 128)[idx], lse.reshape(-1)[idx], ro, rl, "ragged, 3000 requests")
    ro, rl = oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                    pc.kv_lens_t, 8, 2, True, pc.sm_scale, rows=rows)
    check_rows(po.reshape(-1, 128)[idx], pl.reshape(-1)[idx], ro, rl, "paged, 3000 requests")
    drows = np.array([b * 8 + h for b in pick for h in range(8)], dtype=np.int64)
    ro, rl = oracle.paged_attention(dc.q, dc.q_indptr, dc.k_pages, dc.v_pages, dc.page_table,
                                    dc.kv_lens_t, 8, 2, True, dc.sm_scale, rows=drows)
    didx = torch.as_tensor(drows, device="cuda")
    check_rows(do.reshape(-1, 128)[didx], dl.reshape(-1)[didx], ro, rl, "decode, 3000 requests")


@pytest.mark.parametrize("rows", [4, 48], ids=["tensor-core", "conversion"])
def test_cuda_graph_replay_e4m3_paged_prefill(cuda_lib, rows):
    """The E4M3 paged prefill captured once and replayed over rewritten inputs (pages,
    page table, kv_lens and queries of two different calls, alternating) gives the eager
    results bit for bit, on both of its paths (rows query rows per request: 4 x G = 16 is
    the tensor-core form, 48 the conversion of the pages the call reads)."""
    api = cuda_lib
    dev = torch.device("cuda")
    qo = [rows] * 3
    ca = W.paged_case_e4m3([900, 40, 2100], 16, 4, 128, page_size=16, qo_lens=qo, seed=81,
                           extra_pages=30, device=dev)
    cb = W.paged_case_e4m3([3000, 700, 9], 16, 4, 128, page_size=16, qo_lens=qo, seed=82,
                           device=dev)
    npages = max(ca.num_pages, cb.num_pages)
    stride = max(ca.page_table.shape[1], cb.page_table.shape[1])
    kp = torch.zeros((npages, 16, 4, 128), dtype=torch.uint8, device=dev)
    vp = torch.zeros_like(kp)
    pt = torch.full((3, stride), -1, dtype=torch.int32, device=dev)
    kl = torch.zeros(3, dtype=torch.int32, device=dev)
    q = torch.zeros_like(ca.q)
    o = torch.zeros_like(q)
    lse = torch.zeros(q.shape[:2], dtype=torch.float32, device=dev)
    qi = ca.q_indptr.clone()

    def load(c):
        kp.zero_(); vp.zero_(); pt.fill_(-1)
        kp[:c.num_pages].copy_(c.k_pages)
        vp[:c.num_pages].copy_(c.v_pages)
        pt[:, :c.page_table.shape[1]].copy_(c.page_table)
        kl.copy_(c.kv_lens_t)
        q.copy_(c.q)

    def step():
        api.paged_prefill(q, kp, vp, qi, pt, kl, causal=True, sm_scale=ca.sm_scale,
                          k_scale=ca.meta["k_scale"], v_scale=ca.meta["v_scale"],
                          max_qo_len=rows, out=o, lse=lse)

    refs = {}
    for name, c in (("a", ca), ("b", cb)):
        load(c)
        step()
        torch.cuda.synchronize()
        assert api.device_status() == 0
        refs[name] = (o.clone(), lse.clone())

    load(ca)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(graph):
        step()
    for idx, (name, c) in enumerate((("b", cb), ("a", ca), ("b", cb), ("a", ca))):
        o.zero_(); lse.zero_()
        load(c)
        graph.replay()
        torch.cuda.synchronize()
        assert api.device_status() == 0
        assert torch.equal(o, refs[name][0]) and torch.equal(lse, refs[name][1]), (idx, name)
