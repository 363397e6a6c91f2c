"""The C ABI without a GPU: the library builds, loads, exports every function the public
header declares, and its host-side argument checks return the documented status codes
before any CUDA call is made (pointers below are never dereferenced)."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADERS = sorted((ROOT / "include").glob("*.h"))


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(([^;{}]*)\)\s*;", text):
            if m.group(1) not in ("if", "while", "return", "sizeof"):
                names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from paged_gqa_attention_varlen_gb300 import build
    path = build.build()
    return ctypes.CDLL(str(path))


@pytest.fixture(scope="module")
def api():
    from paged_gqa_attention_varlen_gb300 import api
    return api


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pgqa_ragged_prefill_bf16", "pgqa_paged_prefill_bf16", "pgqa_paged_decode_bf16",
              "ragged_prefill_bf16", "paged_prefill_bf16", "paged_decode_bf16",
              "pgqa_set_workspace", "pgqa_get_device_status"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_declared_function(api):
    assert set(declared_functions()) <= set(api.ABI_FUNCTIONS)


def test_version_and_status_strings(api):
    assert api.lib.pgqa_version() >= 10000
    for code in range(-8, 1):
        assert api.lib.pgqa_status_string(code).decode() != "unknown status"
        assert code in api.STATUS_NAMES
    assert api.lib.pgqa_status_string(123) == b"unknown status"


A = 1 << 20  # a 16-byte aligned fake device address (never dereferenced)


def prefill(api, **kw):
    args = dict(q=A, k=A, v=A, o=A, lse=A, qi=A, ki=A, batch=2, hq=8, hk=2, d=128, causal=1,
                scale=0.1)
    args.update(kw)
    p = ctypes.c_void_p
    return api.lib.pgqa_ragged_prefill_bf16(
        p(args["q"]), p(args["k"]), p(args["v"]), p(args["o"]), p(args["lse"]), p(args["qi"]),
        p(args["ki"]), args["batch"], args["hq"], args["hk"], args["d"], args["causal"],
        args["scale"], None)


def decode(api, **kw):
    args = dict(q=A, kp=A, vp=A, pt=A, kl=A, ps=16, stride=8, npages=100, o=A, lse=A, batch=4,
                hq=32, hk=8, d=128, scale=0.1)
    args.update(kw)
    p = ctypes.c_void_p
    return api.lib.pgqa_paged_decode_bf16(
        p(args["q"]), p(args["kp"]), p(args["vp"]), p(args["pt"]), p(args["kl"]), args["ps"],
        args["stride"], args["npages"], p(args["o"]), p(args["lse"]), args["batch"], args["hq"],
        args["hk"], args["d"], args["scale"], None)


def paged_prefill(api, **kw):
    args = dict(q=A, kp=A, vp=A, o=A, lse=A, qi=A, pt=A, stride=8, kl=A, ps=16, npages=100,
                batch=2, hq=8, hk=2, d=128, causal=1, scale=0.1)
    args.update(kw)
    p = ctypes.c_void_p
    return api.lib.pgqa_paged_prefill_bf16(
        p(args["q"]), p(args["kp"]), p(args["vp"]), p(args["o"]), p(args["lse"]), p(args["qi"]),
        p(args["pt"]), args["stride"], p(args["kl"]), args["ps"], args["npages"], args["batch"],
        args["hq"], args["hk"], args["d"], args["causal"], args["scale"], None)


def test_paged_prefill_host_validation(api):
    assert paged_prefill(api, batch=0) == 0
    assert paged_prefill(api, batch=-2) == -1
    assert paged_prefill(api, kl=0) == -1
    assert paged_prefill(api, qi=0) == -1
    assert paged_prefill(api, pt=A + 2) == -1               # misaligned page table
    assert paged_prefill(api, kp=A + 8) == -1
    assert paged_prefill(api, ps=8) == -2
    assert paged_prefill(api, ps=48) == -2
    assert paged_prefill(api, ps=256) == -2
    assert paged_prefill(api, d=64) == -2
    assert paged_prefill(api, hq=24, hk=8) == -2
    assert paged_prefill(api, scale=float("inf")) == -1
    assert paged_prefill(api, npages=-1) == -1
    assert paged_prefill(api, stride=1 << 28, ps=128) == -2  # keys per request overflow int32


def test_strided_page_pool_validation(api):
    p = ctypes.c_void_p
    lib = api.lib

    def pf(page_s, slot_s, head_s, batch=2):
        return lib.pgqa_paged_prefill_bf16_strided(p(A), p(A), p(A), p(A), p(A), p(A), p(A), 8,
                                                   p(A), 16, 100, page_s, slot_s, head_s, batch,
                                                   8, 2, 128, 1, 0.1, None)

    def dc(page_s, slot_s, head_s, batch=2):
        return lib.pgqa_paged_decode_bf16_strided(p(A), p(A), p(A), p(A), p(A), 16, 8, 100,
                                                  page_s, slot_s, head_s, p(A), p(A), batch, 8, 2,
                                                  128, 0.1, None)

    nhd = (16 * 2 * 128, 2 * 128, 128)
    hnd = (2 * 16 * 128, 128, 16 * 128)
    for fn in (pf, dc):
        assert fn(*nhd, batch=0) == 0
        assert fn(0, 256, 128) == -1                # zero stride
        assert fn(4096, 256, 4) == -1               # not a multiple of 8 elements
        assert fn(-4096, 256, 128) == -1
        assert fn(1 << 36, 256, 128) == -1
    import torch
    if not torch.cuda.is_available():
        for fn in (pf, dc):
            assert fn(*nhd) == -7 and fn(*hnd) == -7


def test_e4m3_decode_validation(api):
    p = ctypes.c_void_p
    lib = api.lib

    def dc(page_s=16 * 8 * 128, slot_s=8 * 128, head_s=128, ks=0.5, vs=2.0, batch=2, ps=16, d=128):
        return lib.pgqa_paged_decode_e4m3(p(A), p(A), p(A), p(A), p(A), ps, 8, 100, page_s, slot_s,
                                          head_s, ks, vs, p(A), p(A), batch, 32, 8, d, 0.1, None)

    assert dc(batch=0) == 0
    assert dc(head_s=8) == -1                      # 8 bytes: not a multiple of 16
    assert dc(ks=float("nan")) == -1
    assert dc(vs=float("inf")) == -1
    assert dc(ps=24) == -2
    assert dc(d=256) == -2
    import torch
    if not torch.cuda.is_available():
        assert dc() == -7


def test_e4m3_prefill_validation(api):
    """pgqa_paged_prefill_e4m3: argument checks before any CUDA call, on both of its
    paths (the tensor-core path for max_qo_len * G <= 16 at head_dim 128, the conversion
    path otherwise)."""
    p = ctypes.c_void_p
    lib = api.lib

    def pf(page_s=16 * 8 * 128, slot_s=8 * 128, head_s=128, ks=0.5, vs=2.0, batch=2, ps=16,
           d=128, max_qo=4, hq=32, hk=8, qi=A, pt=A):
        if d == 256:
            page_s, slot_s, head_s = 16 * hk * 256, hk * 256, 256
        return lib.pgqa_paged_prefill_e4m3(p(A), p(A), p(A), p(A), p(A), p(qi), p(pt), 8, p(A),
                                           ps, 100, page_s, slot_s, head_s, ks, vs, batch,
                                           max_qo, hq, hk, d, 1, 0.1, None)

    assert pf(batch=0) == 0
    assert pf(max_qo=0) == -1                      # max_qo_len < 1
    assert pf(qi=0) == -1                          # no q_indptr
    assert pf(qi=A + 2) == -1                      # misaligned q_indptr
    assert pf(ks=float("nan")) == -1
    assert pf(vs=float("-inf")) == -1
    for max_qo in (4, 5, 300):                     # tensor-core path, conversion path
        assert pf(max_qo=max_qo, head_s=8) == -1   # 8 bytes: not a multiple of 16
        assert pf(max_qo=max_qo, ps=24) == -2
        assert pf(max_qo=max_qo, hq=24, hk=8) == -2  # group 3
    assert pf(d=64, max_qo=300) == -2
    import torch
    if not torch.cuda.is_available():
        # valid on each path: no device here
        assert pf(max_qo=4) == -7                  # 4 rows x G 4 = 16 columns
        assert pf(max_qo=5) == -7                  # conversion path
        assert pf(d=256, max_qo=1) == -7           # head_dim 256: conversion path
        assert pf(hq=128, hk=8, max_qo=1) == -7    # group 16: conversion path


def test_prefill_host_validation(api):
    assert prefill(api, batch=0) == 0                       # empty batch: early return
    assert prefill(api, batch=-1) == -1
    assert prefill(api, q=0) == -1
    assert prefill(api, o=A + 8) == -1                      # misaligned output
    assert prefill(api, d=64) == -2
    assert prefill(api, d=192) == -2
    assert prefill(api, hq=6, hk=4) == -2                   # not a multiple
    assert prefill(api, hq=24, hk=8) == -2                  # group 3 does not divide 128
    assert prefill(api, scale=float("nan")) == -1


def test_decode_host_validation(api):
    assert decode(api, batch=0) == 0
    assert decode(api, batch=-3) == -1
    assert decode(api, kl=0) == -1
    assert decode(api, ps=8) == -2
    assert decode(api, ps=48) == -2
    assert decode(api, ps=256) == -2
    assert decode(api, d=256) == -2
    assert decode(api, hq=48, hk=8) == -2                   # group 6
    assert decode(api, hq=128, hk=8) == -2                  # group 16
    assert decode(api, q=A + 4) == -1


def test_valid_calls_without_a_gpu_report_no_device(api):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert prefill(api) == -7
    assert decode(api) == -7
    for ps in (32, 64, 128):
        assert decode(api, ps=ps) == -7
    for ps in (16, 32, 64, 128):
        assert paged_prefill(api, ps=ps) == -7
    assert paged_prefill(api, d=256) == -7


def test_workspace_size_queries(api):
    lib = api.lib
    n = lib.pgqa_workspace_bytes_decode(256, 2048, 16, 32, 128)
    # 256 requests x 32 chunks x 32 heads x (128 + 1) floats of partial results
    assert n >= 256 * 32 * 32 * 129 * 4
    assert lib.pgqa_workspace_bytes_decode(-1, 1, 16, 1, 128) == 0
    m = lib.pgqa_workspace_bytes_prefill(16, 33_000, 32, 8)
    assert m >= (33_000 * 4 // 128) * 8 * 16
    assert lib.pgqa_workspace_bytes_prefill(1, -5, 32, 8) == 0


def _chunk_keys(batch, max_kv, hk):
    """The decode's chunk rule restated: the longest of 1024, 512, 256, 128 keys for which
    batch * ceil(max_kv / chunk) * hk >= 2048, else 128."""
    chunk = 1024
    while chunk > 128 and batch * max(1, -(-max_kv // chunk)) * hk < 2048:
        chunk //= 2
    return chunk


def test_decode_chunk_rule_through_the_workspace_query(api):
    """pgqa_workspace_bytes_decode sizes the partial results for one kv head, the case with
    the most chunks; its growth with the table's key capacity follows the chunk rule."""
    lib = api.lib
    hq, d = 32, 128

    def partial_bytes(batch, stride, ps):
        chunks = batch * -(-(stride * ps) // _chunk_keys(batch, stride * ps, 1))
        return chunks * hq * d * 4

    assert _chunk_keys(1, 32768, 8) == 128 and _chunk_keys(4, 32768, 8) == 512
    assert _chunk_keys(16, 32768, 8) == 1024 and _chunk_keys(256, 512, 8) == 1024
    for batch, stride, ps in ((1, 2048, 16), (3, 188, 16), (4, 2048, 16), (40, 16384, 16),
                              (256, 2048, 16), (2, 100, 128)):
        n = lib.pgqa_workspace_bytes_decode(batch, stride, ps, hq, d)
        want = partial_bytes(batch, stride, ps)
        # the fp32 partial rows plus lse, int arrays and headers of at most a few KB per
        # request and 1 MiB of fixed arrays
        assert want <= n <= want * 1.01 + (1 << 20) + 4096 * batch, (batch, stride, ps, n, want)


def test_binding_refuses_cpu_tensors(api):
    import torch
    q = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    ip = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises((ValueError, TypeError, RuntimeError, AssertionError)):
        api.ragged_prefill(q, q[:, :1].contiguous(), q[:, :1].contiguous(), ip, ip)


def test_the_product_package_never_imports_the_oracle():
    """The oracle is test infrastructure: nothing in the package (binding, build, inputs)
    may import it, so the product path has no CPU route to an answer."""
    import ast
    from pathlib import Path
    pkg = Path(__file__).resolve().parents[1] / "paged_gqa_attention_varlen_gb300"
    for path in pkg.rglob("*.py"):
        tree = ast.parse(path.read_text())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom):
                names = [node.module or ""]
            assert not any(n == "oracle" or n.startswith("oracle.") for n in names), path


def test_empty_tensor_stand_ins(api):
    """Tensors without rows get a device address from a stand-in: one row of the same
    shape, or (a page pool without pages) a zeroed span that covers one page under the
    pool's strides; tensors with rows are passed as they are."""
    import torch
    k = torch.zeros(0, 4, 128, dtype=torch.bfloat16)
    s = api._with_rows(k)
    assert s.shape == (1, 4, 128) and s.dtype == k.dtype and bool((s == 0).all())
    full = torch.ones(3, 4, 128, dtype=torch.bfloat16)
    assert api._with_rows(full) is full
    # an HND pool slice with padded strides: slot stride 160, head stride 16 * 160
    pool = torch.zeros(0, 8, 16, 160, dtype=torch.uint8)[..., :128]
    strides = (pool.stride(0), pool.stride(2), pool.stride(1))  # page, slot, head
    st = api._pool_with_page(pool, 16, 8, 128, strides)
    assert st.dim() == 1 and st.numel() == 15 * strides[1] + 7 * strides[2] + 128
    pages = torch.zeros(2, 16, 8, 128, dtype=torch.bfloat16)
    assert api._pool_with_page(pages, 16, 8, 128, (16 * 8 * 128, 8 * 128, 128)) is pages
