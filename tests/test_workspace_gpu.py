"""The library's workspace at the C ABI, on the GPU.

Every call needs device scratch: the prefills for their work list and tensor maps, the
decode for its split-KV partial results.  By default the library allocates it lazily
(128 MiB, grown when a call needs more), as the lazily allocated kernel workspace of the
vllm-rlt pull request "feat: add FlashInfer attention backend for SM120 decode" (Design
notes).  A caller may hand it a buffer of its own instead (pgqa_set_workspace).

- A caller buffer gives the same results as the lazy workspace, bit for bit.
- A caller buffer too small for a call's fixed arrays makes the call return
  PGQA_ERR_WORKSPACE with nothing enqueued.
- An E4M3 paged prefill whose converted pages do not fit a caller buffer returns
  PGQA_ERR_WORKSPACE with nothing enqueued.
- A prefill whose work list outgrows a (small) caller buffer reports
  PGQA_ERR_DEVICE_CAPACITY through the device status and writes nothing.
- A device status left unread by a call on a non-blocking stream survives a later call
  that grows the workspace.
Each test returns the library to its lazy workspace before it ends.
"""
import pytest
import torch

from paged_gqa_attention_varlen_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PGQA_ERR_WORKSPACE = -3
PGQA_ERR_DEVICE_BOUNDS = -6
PGQA_ERR_DEVICE_CAPACITY = -8


@pytest.fixture
def lazy_after(cuda_lib):
    yield cuda_lib
    torch.cuda.synchronize()
    cuda_lib.set_workspace(None)


def _prefill(api, case, **kw):
    return api.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                              causal=True, sm_scale=case.sm_scale, **kw)


def _decode(api, pc, **kw):
    return api.paged_decode(pc.q, pc.k_pages, pc.v_pages, pc.page_table, pc.kv_lens_t,
                            sm_scale=pc.sm_scale, **kw)


def test_caller_workspace_gives_the_lazy_results_bitwise(lazy_after):
    api = lazy_after
    case = W.ragged_case([300, 1, 129, 700], [300, 900, 129, 1500], 16, 4, 128, seed=201,
                         device="cuda")
    c256 = W.ragged_case([40, 300], [500, 300], 8, 2, 256, seed=202, device="cuda")
    pc = W.paged_case([1, 700, 3000, 33], 32, 8, 128, page_size=16, seed=203, device="cuda")
    short = W.paged_case([5000, 300], 32, 8, 128, page_size=16, qo_lens=[3, 2], seed=204,
                         device="cuda")  # a short work list: split-KV + merge
    runs = []
    for buf in (None, torch.empty(64 << 20, dtype=torch.uint8, device="cuda")):
        api.set_workspace(buf)
        r = [_prefill(api, case), _prefill(api, c256), _decode(api, pc),
             api.paged_prefill(short.q, short.k_pages, short.v_pages, short.q_indptr,
                               short.page_table, short.kv_lens_t, causal=True,
                               sm_scale=short.sm_scale)]
        torch.cuda.synchronize()
        assert api.device_status() == 0
        runs.append(r)
    api.set_workspace(None)  # before the caller buffer goes out of scope
    for (o0, l0), (o1, l1) in zip(*runs):
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_too_small_caller_workspace_is_refused_before_anything_runs(lazy_after):
    api = lazy_after
    case = W.ragged_case([100, 50], [100, 50], 8, 2, 128, seed=205, device="cuda")
    pc = W.paged_case([3000, 64, 1025], 32, 8, 128, page_size=16, seed=206, device="cuda")
    buf = torch.empty(100 << 10, dtype=torch.uint8, device="cuda")  # 100 KiB
    api.set_workspace(buf)
    o = torch.full_like(case.q, 7.0)
    with pytest.raises(api.PgqaError) as e:
        _prefill(api, case, out=o)
    assert e.value.code == PGQA_ERR_WORKSPACE
    od = torch.full_like(pc.q, 7.0)
    with pytest.raises(api.PgqaError) as e:
        _decode(api, pc, out=od)
    assert e.value.code == PGQA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((od == 7.0).all())
    assert api.device_status() == 0
    api.set_workspace(None)


def test_work_list_overflow_reports_capacity_and_writes_nothing(lazy_after):
    api = lazy_after
    # 600 one-token requests with 8 kv heads: 4800 work items, more than the 4096 a
    # 256 KiB buffer holds once the per-request arrays are carved out
    lens = [1] * 600
    case = W.ragged_case(lens, lens, 8, 8, 128, seed=207, device="cuda")
    buf = torch.empty(256 << 10, dtype=torch.uint8, device="cuda")  # kept alive while in use
    api.set_workspace(buf)
    o = torch.full_like(case.q, 7.0)
    lse = torch.full(case.q.shape[:2], 9.0, dtype=torch.float32, device="cuda")
    _prefill(api, case, out=o, lse=lse)
    torch.cuda.synchronize()
    assert api.device_status() == PGQA_ERR_DEVICE_CAPACITY
    assert api.device_status() == 0
    assert bool((o == 7.0).all()) and bool((lse == 9.0).all())
    # the same call with the lazy workspace runs
    api.set_workspace(None)
    o2, l2 = _prefill(api, case)
    torch.cuda.synchronize()
    assert api.device_status() == 0
    assert torch.isfinite(l2).all()


def test_pending_status_survives_growth_on_a_non_blocking_stream(lazy_after):
    """The bad call runs on a torch side stream (non-blocking); the growing call follows on
    the default stream with no synchronisation in between."""
    api = lazy_after
    api.set_workspace(None)  # start from a fresh 128 MiB lazy workspace
    pc = W.paged_case([40, 30000], 8, 2, 128, page_size=16, seed=208, device="cuda")
    pc.page_table[0, 1] = pc.num_pages + 5  # a page id outside the pool
    big = W.paged_case([1] * 2048, 32, 8, 128, page_size=16, stride=2048, seed=209,
                       device="cuda")  # about 1 GB of partial results: the workspace grows
    _decode(api, W.paged_case([4], 8, 2, 128, page_size=16, seed=210, device="cuda"))
    torch.cuda.synchronize()  # the 128 MiB workspace exists
    assert api.device_status() == 0
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _decode(api, pc, stream=side)  # leaves PGQA_DEV_BOUNDS pending
    _decode(api, big)  # grows the workspace while the side stream may still run
    torch.cuda.synchronize()
    assert api.device_status() == PGQA_ERR_DEVICE_BOUNDS
    assert api.device_status() == 0


def test_e4m3_conversion_pool_larger_than_the_caller_buffer_is_refused(lazy_after):
    api = lazy_after
    # 1875 pages of 16 x 8 x 128: about 123 MB of bf16 K and V besides the prefill's part
    pc = W.paged_case_e4m3([30000], 32, 8, 128, page_size=16, qo_lens=[300], seed=211,
                           device="cuda")
    buf = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    api.set_workspace(buf)
    o = torch.full_like(pc.q, 7.0)
    with pytest.raises(api.PgqaError) as e:
        api.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr, pc.page_table,
                          pc.kv_lens_t, sm_scale=pc.sm_scale, k_scale=0.5, v_scale=2.0,
                          max_qo_len=300, out=o)
    assert e.value.code == PGQA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())
    assert api.device_status() == 0
    api.set_workspace(None)
