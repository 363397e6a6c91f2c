"""Helpers shared by the GPU parity tests: tolerance checks and row sampling."""
import numpy as np
import torch

# Tolerance of the path (bf16 output, fp32 LSE): |o - oracle| <= 1e-2 + 1e-2 |oracle|,
# |lse - oracle_lse| <= 1e-3, LSE of rows with no visible key exactly -inf.
O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 1e-3


def check_rows(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """o_gpu [n, d] (any float tensor/array), lse_gpu [n]; refs float64 arrays."""
    og = np.asarray(o_gpu.float().cpu() if isinstance(o_gpu, torch.Tensor) else o_gpu,
                    dtype=np.float64)
    lg = np.asarray(lse_gpu.float().cpu() if isinstance(lse_gpu, torch.Tensor) else lse_gpu,
                    dtype=np.float64)
    assert og.shape == o_ref.shape, (og.shape, o_ref.shape)
    assert np.all(np.isfinite(og)), f"{what}: non-finite output"
    err = np.abs(og - o_ref)
    bound = O_ATOL + O_RTOL * np.abs(o_ref)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of tolerance; first at row {i[0]} "
                             f"col {i[1]}: gpu {og[tuple(i)]} oracle {o_ref[tuple(i)]}; "
                             f"max err {err.max():.3e}")
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), ninf_ref), f"{what}: -inf LSE rows differ"
    fin = ~ninf_ref
    if fin.any():
        lerr = np.abs(lg[fin] - lse_ref[fin])
        assert lerr.max() <= LSE_ATOL, f"{what}: max LSE err {lerr.max():.3e}"
    assert np.all(og[ninf_ref] == 0.0), f"{what}: rows without keys must be exact zeros"
    max_err = float(err.max()) if err.size else 0.0  # a call may hold no query rows
    return max_err, float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0


def sample_prefill_rows(qo_lens, num_qo_heads, group, seed=0, per_request_random=24):
    """Rows t * Hq + h to compare on a large ragged case: each request's first and last
    rows, rows on both sides of every few q-tile boundaries, and random rows; heads cover
    the first, last and random heads of the packing group."""
    rng = np.random.default_rng(seed)
    tpt = 128 // group
    rows = []
    start = 0
    for qo in qo_lens:
        if qo == 0:
            continue
        toks = {0, 1, qo - 1, qo // 2}
        for b in range(tpt, qo, max(tpt, (qo // 6) // tpt * tpt)):
            toks.update({b - 1, b})
        toks.update(rng.integers(0, qo, per_request_random).tolist())
        for t in sorted(x for x in toks if 0 <= x < qo):
            heads = {0, num_qo_heads - 1, int(rng.integers(0, num_qo_heads))}
            for h in heads:
                rows.append((start + t) * num_qo_heads + h)
        start += qo
    return np.array(sorted(set(rows)), dtype=np.int64)


def gather_rows(o, lse, rows, num_qo_heads):
    """Pick rows t * Hq + h out of o [T, Hq, d] / lse [T, Hq] (device tensors)."""
    idx = torch.as_tensor(rows, device=o.device)
    o2 = o.reshape(-1, o.shape[-1]).index_select(0, idx)
    l2 = lse.reshape(-1).index_select(0, idx)
    return o2.float().cpu(), l2.float().cpu()


def check_paged_decode_all_rows(pc, o, lse, oracle_fn, what="", requests_per_pass=32):
    """Compare every output row of a one-row-per-request paged call with the oracle.

    pc is a workloads.PagedCase on the GPU (bf16 or E4M3 pages), o [batch, Hq, d] and
    lse [batch, Hq] the GPU results.  The requests' pages are gathered to the host
    `requests_per_pass` requests at a time (a few GB of host memory at most), renumbered
    0..n-1 with a page table of their own, and oracle_fn(sub_case) computes all of their
    rows.
    """
    from paged_gqa_attention_varlen_gb300 import workloads as W
    ps, d = pc.page_size, pc.head_dim
    worst = 0.0
    for b0 in range(0, pc.batch, requests_per_pass):
        b1 = min(pc.batch, b0 + requests_per_pass)
        lens = pc.kv_lens[b0:b1]
        npg = [(n + ps - 1) // ps for n in lens]
        ids = [pc.page_table[b, :n] for b, n in zip(range(b0, b1), npg) if n]
        if ids:
            idx = torch.cat(ids).long()
            kp = pc.k_pages.index_select(0, idx).cpu()
            vp = pc.v_pages.index_select(0, idx).cpu()
        else:
            kp = pc.k_pages[:1].cpu()
            vp = pc.v_pages[:1].cpu()
        table = torch.full((b1 - b0, max(1, max(npg))), -1, dtype=torch.int32)
        off = 0
        for i, n in enumerate(npg):
            table[i, :n] = torch.arange(off, off + n, dtype=torch.int32)
            off += n
        sub = W.PagedCase(f"{pc.name}[{b0}:{b1}]", pc.q[b0:b1].cpu(),
                          torch.arange(0, b1 - b0 + 1, dtype=torch.int32), kp, vp, table,
                          torch.tensor(lens, dtype=torch.int32), list(lens), [1] * (b1 - b0), ps,
                          pc.num_qo_heads, pc.num_kv_heads, d, True, pc.sm_scale, dict(pc.meta))
        ro, rl = oracle_fn(sub)
        err, _ = check_rows(o[b0:b1].reshape(-1, d).float().cpu(), lse[b0:b1].reshape(-1).cpu(),
                            ro, rl, f"{what} requests {b0}..{b1 - 1}")
        worst = max(worst, err)
    return worst
