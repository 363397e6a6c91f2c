"""Seeded synthetic inputs for ragged prefill and paged decode.

This module holds input generation only -- no attention arithmetic -- so that both the
CUDA path and the CPU oracle can be fed the same tensors.  Every workload is drawn in a
fixed order from seed 0 unless a seed is given:

    lengths (CPU generator) -> cached-prefix lengths -> Q -> K -> V -> page permutation

Lengths come from a CPU ``torch.Generator`` so they do not depend on the device; the
tensors come from a generator on the target device (i.i.d. N(0, 1) drawn in float32,
then rounded to bf16).  Comparisons always read back the stored bf16 tensors, so the
generator choice never affects parity.

The named workloads mirror the serving shapes of the ragged-prefill and paged-decode
paths (Atlas "Module flashinfer" ragged_prefill_bf16_hd128 / _hd256; vllm-rlt PR
"feat: add FlashInfer attention backend for SM120 decode", block_size 16, NHD):

    tiny            batch 2, qo = kv = {17, 64}, 4 qo / 2 kv heads, d 128, causal
    prefill_hd128   batch 16, qo = kv ~ U{128..4096}, 32 / 8 heads, d 128, causal
    prefix_hd256    batch 8, qo ~ U{256..2048}, kv = qo + U{0..8192}, 16 / 4 heads, d 256,
                    causal (bottom-right)
    decode          batch 256, kv ~ U{512..32768}, page 16 NHD, random page permutation,
                    32 / 8 heads, d 128
    long            batch 1, qo = kv = 32768, 64 / 8 heads, d 128, causal, K scaled by 3
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_CHUNK = 1 << 26  # elements drawn per randn call, bounds the float32 staging buffer


def _randn_bf16(shape, gen, device, scale=1.0):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:e].copy_(x)
    return out


def _indptr(lens, device):
    ip = [0]
    for n in lens:
        ip.append(ip[-1] + int(n))
    return torch.tensor(ip, dtype=torch.int32, device=device)


@dataclass
class RaggedCase:
    name: str
    q: torch.Tensor            # [total_q, Hq, d] bf16
    k: torch.Tensor            # [total_kv, Hk, d] bf16
    v: torch.Tensor            # [total_kv, Hk, d] bf16
    q_indptr: torch.Tensor     # [batch + 1] int32
    kv_indptr: torch.Tensor    # [batch + 1] int32
    qo_lens: list
    kv_lens: list
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    causal: bool
    sm_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def batch(self):
        return len(self.qo_lens)

    @property
    def total_q(self):
        return int(sum(self.qo_lens))


@dataclass
class PagedCase:
    name: str
    q: torch.Tensor            # [total_q, Hq, d] bf16 (decode: [batch, Hq, d])
    q_indptr: torch.Tensor     # [batch + 1] int32 (decode: 0..batch)
    k_pages: torch.Tensor      # [num_pages, page_size, Hk, d] bf16
    v_pages: torch.Tensor      # [num_pages, page_size, Hk, d] bf16
    page_table: torch.Tensor   # [batch, stride] int32, padded with `pad`
    kv_lens_t: torch.Tensor    # [batch] int32
    kv_lens: list
    qo_lens: list
    page_size: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    causal: bool
    sm_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def batch(self):
        return len(self.kv_lens)

    @property
    def num_pages(self):
        return int(self.k_pages.shape[0])


def ragged_case(qo_lens, kv_lens, num_qo_heads, num_kv_heads, head_dim, causal=True,
                sm_scale=None, seed=0, device="cpu", k_scale=1.0, name="custom"):
    """Packed NHD Q/K/V for the given per-request lengths."""
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tq, tk = int(sum(qo_lens)), int(sum(kv_lens))
    q = _randn_bf16((tq, num_qo_heads, head_dim), gen, device)
    k = _randn_bf16((tk, num_kv_heads, head_dim), gen, device, scale=k_scale)
    v = _randn_bf16((tk, num_kv_heads, head_dim), gen, device)
    return RaggedCase(name, q, k, v, _indptr(qo_lens, device), _indptr(kv_lens, device),
                      [int(x) for x in qo_lens], [int(x) for x in kv_lens], num_qo_heads,
                      num_kv_heads, head_dim, bool(causal), float(sm_scale))


def paged_case(kv_lens, num_qo_heads, num_kv_heads, head_dim, page_size=16, qo_lens=None,
               causal=True, sm_scale=None, seed=0, device="cpu", pad=-1, extra_pages=0,
               stride=None, name="custom"):
    """Q plus a paged NHD K/V cache whose pages are a seeded random permutation.

    qo_lens=None gives decode (one query row per request).  Page-table slots past a
    request's last page hold `pad`.  `extra_pages` adds unreferenced pages.
    """
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    batch = len(kv_lens)
    if qo_lens is None:
        qo_lens = [1] * batch
    n_pages_req = [(int(n) + page_size - 1) // page_size for n in kv_lens]
    num_pages = sum(n_pages_req) + extra_pages
    if stride is None:
        stride = max(1, max(n_pages_req) if n_pages_req else 1)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    q = _randn_bf16((int(sum(qo_lens)), num_qo_heads, head_dim), gen, device)
    kp = _randn_bf16((max(num_pages, 1), page_size, num_kv_heads, head_dim), gen, device)
    vp = _randn_bf16((max(num_pages, 1), page_size, num_kv_heads, head_dim), gen, device)
    perm = torch.randperm(max(num_pages, 1), generator=gen, device=device).to(torch.int32)
    table = torch.full((batch, stride), pad, dtype=torch.int32, device=device)
    off = 0
    for b, n in enumerate(n_pages_req):
        if n:
            table[b, :n] = perm[off:off + n]
        off += n
    return PagedCase(name, q, _indptr(qo_lens, device), kp, vp, table,
                     torch.tensor([int(x) for x in kv_lens], dtype=torch.int32, device=device),
                     [int(x) for x in kv_lens], [int(x) for x in qo_lens], page_size,
                     num_qo_heads, num_kv_heads, head_dim, bool(causal), float(sm_scale))


def paged_case_e4m3(kv_lens, num_qo_heads, num_kv_heads, head_dim, page_size=16, qo_lens=None,
                    causal=True, sm_scale=None, seed=0, device="cpu", k_scale=0.5, v_scale=2.0,
                    extra_pages=0, stride=None, name="custom_e4m3"):
    """paged_case() with the K/V pages stored as FP8 E4M3 bytes (uint8 tensors): the
    seeded bf16 draws rounded to the nearest E4M3 value by torch's float8_e4m3fn cast.
    The element values are byte value x k_scale / v_scale (stored in meta)."""
    pc = paged_case(kv_lens, num_qo_heads, num_kv_heads, head_dim, page_size, qo_lens, causal,
                    sm_scale, seed, device, extra_pages=extra_pages, stride=stride, name=name)
    pc.k_pages = pc.k_pages.float().to(torch.float8_e4m3fn).view(torch.uint8)
    pc.v_pages = pc.v_pages.float().to(torch.float8_e4m3fn).view(torch.uint8)
    pc.meta.update(k_scale=float(k_scale), v_scale=float(v_scale))
    return pc


def multi_token_case(pc, qo_len, k_pages=None, v_pages=None, seed=0, k_scale=1.0,
                     v_scale=1.0, name=None):
    """pc's paged cache (or the given pools, e.g. an E4M3 copy) with qo_len query rows per
    request: the last qo_len positions of each request's keys, as in multi-token decode.
    Q is drawn from `seed`; the page table and kv lengths are pc's."""
    device = pc.q.device
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    qo = [int(qo_len)] * pc.batch
    q = _randn_bf16((qo_len * pc.batch, pc.num_qo_heads, pc.head_dim), gen, device)
    return PagedCase(name or f"{pc.name}_x{qo_len}", q, _indptr(qo, device),
                     pc.k_pages if k_pages is None else k_pages,
                     pc.v_pages if v_pages is None else v_pages, pc.page_table, pc.kv_lens_t,
                     list(pc.kv_lens), qo, pc.page_size, pc.num_qo_heads, pc.num_kv_heads,
                     pc.head_dim, True, pc.sm_scale,
                     dict(pc.meta, k_scale=float(k_scale), v_scale=float(v_scale)))


def _lens(gen, n, lo, hi):
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


CONFIG_SHAPES = {  # heads, head_dim, page size (0: ragged K/V) and causality of each workload
    "tiny": dict(num_qo_heads=4, num_kv_heads=2, head_dim=128, page_size=0, causal=True),
    "prefill_hd128": dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=0, causal=True),
    "prefix_hd256": dict(num_qo_heads=16, num_kv_heads=4, head_dim=256, page_size=0, causal=True),
    "decode": dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, causal=True),
    "long": dict(num_qo_heads=64, num_kv_heads=8, head_dim=128, page_size=0, causal=True),
}


def config(name: str, device="cpu", seed=0):
    """One of the named serving workloads (see the module docstring)."""
    shape = CONFIG_SHAPES[name]
    hq, hk, d = shape["num_qo_heads"], shape["num_kv_heads"], shape["head_dim"]
    qo, kv = config_lengths(name, seed)
    if name == "decode":
        return paged_case(kv, hq, hk, d, page_size=shape["page_size"], seed=seed, device=device,
                          name=name)
    return ragged_case(qo, kv, hq, hk, d, shape["causal"], seed=seed, device=device,
                       k_scale=3.0 if name == "long" else 1.0, name=name)


CONFIG_NAMES = ("tiny", "prefill_hd128", "prefix_hd256", "decode", "long")


def config_lengths(name: str, seed=0):
    """Per-request (qo_lens, kv_lens) of a named workload without drawing any tensor."""
    cg = torch.Generator()
    cg.manual_seed(seed)
    if name == "tiny":
        return [17, 64], [17, 64]
    if name == "prefill_hd128":
        lens = _lens(cg, 16, 128, 4096)
        return lens, lens
    if name == "prefix_hd256":
        qo = _lens(cg, 8, 256, 2048)
        prefix = _lens(cg, 8, 0, 8192)
        return qo, [a + b for a, b in zip(qo, prefix)]
    if name == "decode":
        kv = _lens(cg, 256, 512, 32768)
        return [1] * 256, kv
    if name == "long":
        return [32768], [32768]
    raise KeyError(name)
