"""The device-side failure path, run on the GPU without a fault.

Every mbarrier wait in this library's kernels is bounded: when it runs out it records
PGQA_DEV_TIMEOUT in the device status word and the kernel returns, so that the host
reads an error instead of meeting a hung GPU.  pgqa_selftest_expired_wait makes one such
wait run out on purpose (it waits on a barrier that nothing arrives at; the limit is two
seconds).  The status call must report it once, and the same context must go on computing
correct results.  The other failure cases (bad indptr, kv_len or page id) are in the
prefill and decode tests.
"""
import pytest
import torch

import oracle
from paged_gqa_attention_varlen_gb300 import workloads as W
from gpu_util import check_rows

pytestmark = pytest.mark.gpu

PGQA_ERR_DEVICE_TIMEOUT = -5


def test_expired_wait_is_reported_once_and_the_context_stays_usable(cuda_lib):
    assert cuda_lib.device_status() == 0
    cuda_lib.selftest_expired_wait()
    assert cuda_lib.device_status() == PGQA_ERR_DEVICE_TIMEOUT
    assert cuda_lib.device_status() == 0  # the status call cleared it
    case = W.config("tiny", device="cuda")
    o, lse = cuda_lib.ragged_prefill(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                     causal=True, sm_scale=case.sm_scale)
    torch.cuda.synchronize()
    assert cuda_lib.device_status() == 0
    ro, rl = oracle.ragged_attention(case.q, case.k, case.v, case.q_indptr, case.kv_indptr,
                                     case.num_qo_heads, case.num_kv_heads, True, case.sm_scale)
    check_rows(o.reshape(-1, 128), lse.reshape(-1), ro, rl, "after the expired wait")


def test_expired_wait_on_a_side_stream(cuda_lib):
    side = torch.cuda.Stream()
    cuda_lib.selftest_expired_wait(stream=side)
    assert cuda_lib.device_status(side) == PGQA_ERR_DEVICE_TIMEOUT
    assert cuda_lib.device_status(side) == 0
