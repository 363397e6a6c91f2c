"""Pins for the float64 CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * a dense-matrix formulation in numpy/scipy (K/V heads expanded with np.repeat, an
    explicit mask matrix, scipy.special.logsumexp) on many tiny shapes;
  * hand-derived worked examples in tests/golden/closed_form_cases.json;
  * closed forms (single key, constant V, zero scale, identical keys, dominant key,
    empty rows) and invariants (GQA = MHA with repeated KV heads, request order,
    causal never reads the future, decode = ragged prefill, split + merge = whole,
    page-table padding is never read).
A dropped term, a wrong sign, a wrong head mapping or a transposed operand in the
oracle fails at least one of these.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")


def f64(t):
    return t.to(torch.float64).numpy()


def brute_ragged(case):
    """Dense numpy attention: explicit mask matrix, library logsumexp."""
    q, k, v = f64(case.q), f64(case.k), f64(case.v)
    G = case.num_qo_heads // case.num_kv_heads
    k = np.repeat(k, G, axis=1)
    v = np.repeat(v, G, axis=1)
    qi = case.q_indptr.numpy()
    ki = case.kv_indptr.numpy()
    o_all = np.zeros(q.shape)
    lse_all = np.full(q.shape[:2], -np.inf)
    for b in range(case.batch):
        Q = q[qi[b]:qi[b + 1]]
        K = k[ki[b]:ki[b + 1]]
        V = v[ki[b]:ki[b + 1]]
        qo, kv = Q.shape[0], K.shape[0]
        if qo == 0:
            continue
        S = np.einsum("ihd,jhd->hij", Q, K) * case.sm_scale
        ii = np.arange(qo)[:, None]
        jj = np.arange(kv)[None, :]
        mask = (jj <= ii + kv - qo) if case.causal else np.ones((qo, kv), bool)
        S = np.where(mask[None], S, -np.inf)
        if kv == 0:
            continue
        lse = logsumexp(S, axis=-1)
        with np.errstate(invalid="ignore"):
            P = np.exp(S - lse[..., None])
        P = np.nan_to_num(P, nan=0.0)
        O = np.einsum("hij,jhd->ihd", P, V)
        o_all[qi[b]:qi[b + 1]] = O
        lse_all[qi[b]:qi[b + 1]] = lse.T
    return o_all.reshape(-1, q.shape[-1]), lse_all.reshape(-1)


def run_oracle(case, rows=None):
    return oracle.ragged_attention(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                   case.num_qo_heads, case.num_kv_heads, case.causal,
                                   case.sm_scale, rows=rows)


def assert_lse_close(a, b, tol):
    a, b = np.asarray(a), np.asarray(b)
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    assert np.all(np.abs(a[fin] - b[fin]) <= tol)


SHAPES = [
    # qo_lens, kv_lens, Hq, Hk, d
    ([5], [5], 1, 1, 16),
    ([7, 3], [7, 9], 2, 1, 16),
    ([4, 9, 1], [12, 9, 30], 4, 1, 32),
    ([6], [2], 8, 1, 16),          # kv shorter than qo: empty leading rows when causal
    ([33, 17], [40, 64], 8, 2, 16),
    ([3, 8], [3, 8], 4, 4, 16),
    ([17, 64], [17, 64], 4, 2, 128),
    ([9, 20], [30, 20], 2, 1, 256),
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", SHAPES)
def test_oracle_matches_dense_brute_force(shape, causal):
    qo, kv, hq, hk, d = shape
    case = W.ragged_case(qo, kv, hq, hk, d, causal=causal, seed=sum(qo) + 7 * hq + d)
    o, lse = run_oracle(case)
    bo, blse = brute_ragged(case)
    assert np.max(np.abs(o - bo)) <= 1e-12
    assert_lse_close(lse, blse, 1e-12)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _bf16(x):
    t = torch.tensor(x, dtype=torch.float64)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.to(torch.float64), t), "golden input not exactly representable"
    return b


def _lse_values(xs):
    return np.array([-np.inf if x == "-inf" else float(x) for x in xs])


@pytest.mark.parametrize("idx", range(4))
def test_oracle_golden_ragged(idx):
    c = _golden()["ragged"][idx]
    o, lse = oracle.ragged_attention(_bf16(c["q"]), _bf16(c["k"]), _bf16(c["v"]),
                                     torch.tensor(c["q_indptr"], dtype=torch.int32),
                                     torch.tensor(c["kv_indptr"], dtype=torch.int32),
                                     c["num_qo_heads"], c["num_kv_heads"], c["causal"],
                                     c["sm_scale"])
    assert np.max(np.abs(o - np.array(c["o"], dtype=np.float64))) <= 1e-12, c["name"]
    assert_lse_close(lse, _lse_values(c["lse"]), 1e-12)


def test_oracle_golden_paged():
    c = _golden()["paged"][0]
    o, lse = oracle.paged_attention(_bf16(c["q"]), torch.tensor([0, 1], dtype=torch.int32),
                                    _bf16(c["k_pages"]), _bf16(c["v_pages"]),
                                    torch.tensor(c["page_table"], dtype=torch.int32),
                                    torch.tensor(c["kv_lens"], dtype=torch.int32),
                                    c["num_qo_heads"], c["num_kv_heads"], c["causal"],
                                    c["sm_scale"])
    assert np.max(np.abs(o - np.array(c["o"]))) <= 1e-12
    assert_lse_close(lse, _lse_values(c["lse"]), 1e-12)


def test_single_key_returns_value_and_score():
    case = W.ragged_case([1], [1], 4, 2, 128, causal=True, seed=3)
    o, lse = run_oracle(case)
    v = f64(case.v)[0]           # [Hk, d]
    q, k = f64(case.q)[0], f64(case.k)[0]
    for h in range(4):
        g = h // 2
        assert np.array_equal(o[h], v[g])             # exact: one weight of 1
        assert abs(lse[h] - case.sm_scale * float(q[h] @ k[g])) <= 1e-12


def test_constant_value_rows_return_that_value():
    case = W.ragged_case([10, 5], [12, 5], 2, 1, 32, causal=True, seed=5)
    const = torch.linspace(-3, 3, 32).to(torch.bfloat16)
    case.v[:] = const
    o, _ = run_oracle(case)
    assert np.max(np.abs(o - f64(const)[None, :])) <= 1e-12


def test_zero_scale_is_mean_of_allowed_values():
    case = W.ragged_case([6], [9], 2, 1, 16, causal=True, sm_scale=0.0, seed=9)
    o, lse = run_oracle(case)
    v = f64(case.v)[:, 0, :]
    for i in range(6):
        n = i + 9 - 6 + 1
        for h in range(2):
            r = i * 2 + h
            assert np.max(np.abs(o[r] - v[:n].mean(0))) <= 1e-12
            assert abs(lse[r] - math.log(n)) <= 1e-12


def test_identical_keys_give_uniform_weights():
    case = W.ragged_case([1], [8], 1, 1, 16, causal=False, seed=11)
    case.k[:] = case.k[0]
    o, lse = run_oracle(case)
    q, k, v = f64(case.q)[0, 0], f64(case.k)[0, 0], f64(case.v)[:, 0]
    assert np.max(np.abs(o[0] - v.mean(0))) <= 1e-12
    assert abs(lse[0] - (case.sm_scale * float(q @ k) + math.log(8))) <= 1e-12


def test_dominant_key_selects_its_value():
    case = W.ragged_case([1], [6], 1, 1, 16, causal=False, sm_scale=1.0, seed=13)
    case.q[:] = 0
    case.q[0, 0, 0] = 8.0
    case.k[:] = 0
    case.k[4, 0, 0] = 16.0      # s = 128 for key 4, 0 for the rest
    o, lse = run_oracle(case)
    v = f64(case.v)[:, 0]
    w_other = math.exp(-128.0)
    expect = (v[4] + w_other * (v.sum(0) - v[4])) / (1 + 5 * w_other)
    assert np.max(np.abs(o[0] - expect)) <= 1e-12
    assert abs(lse[0] - (128.0 + math.log1p(5 * w_other))) <= 1e-12


def test_empty_kv_gives_zero_and_neg_inf():
    case = W.ragged_case([3, 2], [0, 4], 2, 1, 16, causal=False, seed=1)
    o, lse = run_oracle(case)
    assert np.all(o[:6] == 0.0) and np.all(np.isneginf(lse[:6]))
    assert np.all(np.isfinite(lse[6:]))


def test_gqa_equals_mha_with_repeated_kv_heads():
    case = W.ragged_case([7, 12], [9, 12], 8, 2, 32, causal=True, seed=21)
    o, lse = run_oracle(case)
    mha = W.RaggedCase("mha", case.q, case.k.repeat_interleave(4, dim=1),
                       case.v.repeat_interleave(4, dim=1), case.q_indptr, case.kv_indptr,
                       case.qo_lens, case.kv_lens, 8, 8, 32, True, case.sm_scale)
    o2, lse2 = run_oracle(mha)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_request_order_does_not_change_results():
    case = W.ragged_case([5, 11, 3], [8, 11, 20], 4, 2, 16, causal=True, seed=23)
    o, lse = run_oracle(case)
    # reverse the request order
    qs, ks = case.q_indptr.tolist(), case.kv_indptr.tolist()
    order = [2, 1, 0]
    q2 = torch.cat([case.q[qs[b]:qs[b + 1]] for b in order])
    k2 = torch.cat([case.k[ks[b]:ks[b + 1]] for b in order])
    v2 = torch.cat([case.v[ks[b]:ks[b + 1]] for b in order])
    qo2 = [case.qo_lens[b] for b in order]
    kv2 = [case.kv_lens[b] for b in order]
    rev = W.RaggedCase("rev", q2, k2, v2, W._indptr(qo2, "cpu"), W._indptr(kv2, "cpu"), qo2,
                       kv2, 4, 2, 16, True, case.sm_scale)
    o2, lse2 = run_oracle(rev)
    H = 4
    for nb, b in enumerate(order):
        a = slice(qs[b] * H, qs[b + 1] * H)
        start = sum(qo2[:nb]) * H
        c = slice(start, start + qo2[nb] * H)
        assert np.array_equal(o[a], o2[c]) and np.array_equal(lse[a], lse2[c])


def test_causal_never_reads_future_keys():
    case = W.ragged_case([6], [10], 2, 1, 16, causal=True, seed=29)
    o, lse = run_oracle(case)
    qo, kv = 6, 10
    for i in range(qo):
        pert = W.RaggedCase("p", case.q, case.k.clone(), case.v.clone(), case.q_indptr,
                            case.kv_indptr, case.qo_lens, case.kv_lens, 2, 1, 16, True,
                            case.sm_scale)
        first_future = i + kv - qo + 1
        pert.k[first_future:] = 5.0
        pert.v[first_future:] = -7.0
        rows = np.array([i * 2, i * 2 + 1], dtype=np.int64)
        o2, lse2 = run_oracle(pert, rows)
        assert np.array_equal(o[rows], o2) and np.array_equal(lse[rows], lse2)
    # and the perturbation is visible to a row that may read it (the test has teeth)
    pert.k[kv - 1:] = 5.0
    o3, _ = run_oracle(pert, np.array([(qo - 1) * 2], dtype=np.int64))
    assert not np.array_equal(o[(qo - 1) * 2], o3[0])


def test_decode_equals_ragged_prefill_on_contiguous_kv():
    pc = W.paged_case([37, 5, 16, 64], 8, 2, 32, page_size=16, seed=31)
    o, lse = oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                                    pc.kv_lens_t, 8, 2, True, pc.sm_scale)
    ks, vs = [], []
    for b, n in enumerate(pc.kv_lens):
        pages = pc.page_table[b, :(n + 15) // 16].long()
        ks.append(pc.k_pages[pages].reshape(-1, 2, 32)[:n])
        vs.append(pc.v_pages[pages].reshape(-1, 2, 32)[:n])
    rc = W.RaggedCase("c", pc.q, torch.cat(ks), torch.cat(vs), pc.q_indptr,
                      W._indptr(pc.kv_lens, "cpu"), pc.qo_lens, pc.kv_lens, 8, 2, 32, True,
                      pc.sm_scale)
    o2, lse2 = run_oracle(rc)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_page_table_padding_is_never_read():
    outs = []
    for pad in (-1, 0, 12345):
        pc = W.paged_case([20, 33], 4, 1, 16, page_size=16, pad=pad, stride=6, seed=37)
        outs.append(oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages,
                                           pc.page_table, pc.kv_lens_t, 4, 1, True,
                                           pc.sm_scale))
    for o, lse in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(lse, outs[0][1])


def test_paged_rejects_out_of_range_page():
    pc = W.paged_case([20], 2, 1, 16, page_size=16, seed=41)
    pc.page_table[0, 1] = pc.num_pages
    with pytest.raises(ValueError):
        oracle.paged_attention(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, pc.page_table,
                               pc.kv_lens_t, 2, 1, True, pc.sm_scale)


@pytest.mark.parametrize("cuts", [[0, 13, 40], [0, 1, 2, 40], [0, 40], [0, 0, 40]])
def test_split_then_merge_equals_whole(cuts):
    """Attention over keys A u B equals the merge of attention over A and over B."""
    kv = 40
    case = W.ragged_case([1], [kv], 4, 1, 16, causal=False, seed=43)
    o, lse = run_oracle(case)
    vs, ss = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        part = W.RaggedCase("part", case.q, case.k[a:b], case.v[a:b], case.q_indptr,
                            W._indptr([b - a], "cpu"), [1], [b - a], 4, 1, 16, False,
                            case.sm_scale)
        po, pl = run_oracle(part)
        vs.append(po)
        ss.append(pl)
    mo, ml = oracle.merge_states(np.stack(vs), np.stack(ss))
    assert np.max(np.abs(mo - o)) <= 1e-12
    assert np.max(np.abs(ml - lse)) <= 1e-12


def test_merge_is_associative_and_handles_empty_states():
    rng = np.random.default_rng(0)
    v = rng.standard_normal((4, 5, 8))
    s = rng.standard_normal((4, 5)) * 3
    s[1, 2] = -np.inf
    whole_v, whole_s = oracle.merge_states(v, s)
    av, as_ = oracle.merge_states(v[:2], s[:2])
    bv, bs = oracle.merge_states(v[2:], s[2:])
    tv, ts = oracle.merge_states(np.stack([av, bv]), np.stack([as_, bs]))
    assert np.max(np.abs(tv - whole_v)) <= 1e-12 and np.max(np.abs(ts - whole_s)) <= 1e-12
    ev, es = oracle.merge_states(np.zeros((2, 1, 3)), np.full((2, 1), -np.inf))
    assert np.all(ev == 0) and np.isneginf(es[0])


def test_bf16_widening_matches_torch():
    """The oracle reads bf16 bit patterns; a single-key row returns V exactly, so its
    output pins the decoding against torch's own bf16 -> float64 conversion."""
    x = torch.tensor([0.0, -0.0, 1.0, -2.5, 3.140625, 1e-38, 6.5e4, -1e30,
                      2 ** -133], dtype=torch.float32).to(torch.bfloat16)
    n = x.numel()
    case = W.ragged_case([1], [1], 1, 1, n, causal=False, seed=0)
    case.v[0, 0] = x
    o, _ = run_oracle(case)
    assert np.array_equal(o[0], x.to(torch.float64).numpy())


# ---------------------------------------------------------------- FP8 E4M3 KV cache
def test_e4m3_decoder_matches_torch_float8_for_every_byte():
    b = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])
    assert np.array_equal(np.signbit(ours[ok]), np.signbit(ref[ok]))


def test_e4m3_closed_forms():
    vals = oracle.e4m3_decode(np.array([0x38, 0x7E, 0x01, 0x08, 0x07, 0xB8, 0x00, 0x80, 0x7F],
                                       dtype=np.uint8))
    assert vals[0] == 1.0                      # exponent 7 (= bias), mantissa 0
    assert vals[1] == 448.0                    # largest finite: 2^8 * 1.75
    assert vals[2] == 2.0 ** -9                # smallest subnormal: 1/8 * 2^-6
    assert vals[3] == 2.0 ** -6                # smallest normal
    assert vals[4] == 7 / 8 * 2.0 ** -6        # largest subnormal
    assert vals[5] == -1.0
    assert vals[6] == 0.0 and not np.signbit(vals[6])
    assert vals[7] == 0.0 and np.signbit(vals[7])
    assert np.isnan(vals[8])


def _dense_paged(q, k, v, qo, kv, G, causal, scale):
    """Dense numpy attention over contiguous per-request K/V (float64 inputs)."""
    qi = np.concatenate([[0], np.cumsum(qo)])
    ki = np.concatenate([[0], np.cumsum(kv)])
    k = np.repeat(k, G, axis=1)
    v = np.repeat(v, G, axis=1)
    o_all = np.zeros(q.shape)
    lse_all = np.full(q.shape[:2], -np.inf)
    for b in range(len(qo)):
        Q, K, V = q[qi[b]:qi[b + 1]], k[ki[b]:ki[b + 1]], v[ki[b]:ki[b + 1]]
        if len(Q) == 0 or len(K) == 0:
            continue
        S = np.einsum("ihd,jhd->hij", Q, K) * scale
        ii = np.arange(len(Q))[:, None]
        jj = np.arange(len(K))[None, :]
        mask = (jj <= ii + len(K) - len(Q)) if causal else np.ones((len(Q), len(K)), bool)
        S = np.where(mask[None], S, -np.inf)
        lse = logsumexp(S, axis=-1)
        with np.errstate(invalid="ignore"):
            P = np.nan_to_num(np.exp(S - lse[..., None]), nan=0.0)
        o_all[qi[b]:qi[b + 1]] = np.einsum("hij,jhd->ihd", P, V)
        lse_all[qi[b]:qi[b + 1]] = lse.T
    return o_all.reshape(-1, q.shape[-1]), lse_all.reshape(-1)


def _contiguous_kv(pc, pages_f64):
    out = []
    for b, n in enumerate(pc.kv_lens):
        npg = (n + pc.page_size - 1) // pc.page_size
        rows = pages_f64[pc.page_table[b, :npg].numpy()].reshape(-1, pc.num_kv_heads, pc.head_dim)
        out.append(rows[:n])
    return np.concatenate(out)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("qo,kv,hq,hk,d,ps", [
    ([1, 1, 1], [5, 40, 17], 4, 1, 16, 16),
    ([3, 9], [30, 9], 8, 2, 32, 16),
    ([4], [100], 4, 4, 128, 32),
])
def test_e4m3_oracle_matches_dense_brute_force(causal, qo, kv, hq, hk, d, ps):
    pc = W.paged_case_e4m3(kv, hq, hk, d, page_size=ps, qo_lens=qo, causal=causal, seed=d + ps)
    ks, vs = pc.meta["k_scale"], pc.meta["v_scale"]
    o, lse = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, ks, vs,
                                         pc.page_table, pc.kv_lens_t, hq, hk, causal, pc.sm_scale)
    kf = pc.k_pages.view(torch.float8_e4m3fn).to(torch.float64).numpy() * ks
    vf = pc.v_pages.view(torch.float8_e4m3fn).to(torch.float64).numpy() * vs
    bo, blse = _dense_paged(f64(pc.q), _contiguous_kv(pc, kf), _contiguous_kv(pc, vf), qo, kv,
                            hq // hk, causal, pc.sm_scale)
    assert np.max(np.abs(o - bo)) <= 1e-12
    assert_lse_close(lse, blse, 1e-12)


def test_e4m3_oracle_equals_bf16_oracle_on_representable_values():
    """E4M3 values times a power-of-two scale are exact in bf16, so the bf16 oracle over
    those values must give the very same float64 results."""
    pc = W.paged_case_e4m3([70, 3, 129], 8, 2, 64, page_size=16, qo_lens=[5, 3, 2], seed=3,
                           k_scale=0.25, v_scale=4.0)
    kb = (pc.k_pages.view(torch.float8_e4m3fn).float() * 0.25).to(torch.bfloat16)
    vb = (pc.v_pages.view(torch.float8_e4m3fn).float() * 4.0).to(torch.bfloat16)
    o8, l8 = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, 0.25, 4.0,
                                         pc.page_table, pc.kv_lens_t, 8, 2, True, pc.sm_scale)
    o16, l16 = oracle.paged_attention(pc.q, pc.q_indptr, kb, vb, pc.page_table, pc.kv_lens_t, 8,
                                      2, True, pc.sm_scale)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)


def test_e4m3_scales_fold_into_score_scale_and_output():
    pc = W.paged_case_e4m3([50, 200], 4, 2, 32, page_size=16, qo_lens=[1, 1], seed=5)
    base_o, base_l = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, 1.0,
                                                 1.0, pc.page_table, pc.kv_lens_t, 4, 2, True,
                                                 pc.sm_scale)
    o, l = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, 3.0, 1.0,
                                       pc.page_table, pc.kv_lens_t, 4, 2, True, pc.sm_scale / 3.0)
    assert np.max(np.abs(o - base_o)) <= 1e-12 and np.max(np.abs(l - base_l)) <= 1e-12
    o, l = oracle.paged_attention_e4m3(pc.q, pc.q_indptr, pc.k_pages, pc.v_pages, 1.0, 2.5,
                                       pc.page_table, pc.kv_lens_t, 4, 2, True, pc.sm_scale)
    assert np.max(np.abs(o - 2.5 * base_o)) <= 1e-12 and np.array_equal(l, base_l)
