"""Host-side logic of bench.py without a GPU: work accounting, and the multi-rank
reduction (max over ranks) under a world-size-2 gloo process group."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def test_visible_pairs_closed_forms():
    # causal, kv >= qo: qo * (kv - qo) + qo (qo + 1) / 2
    for qo, kv in [(1, 1), (5, 5), (7, 20), (128, 4096)]:
        assert bench.visible_pairs(qo, kv) == qo * (kv - qo) + qo * (qo + 1) // 2
    assert bench.visible_pairs(4, 9, causal=False) == 36
    # kv < qo: only the last kv rows see keys (1 + 2 + ... + kv)
    assert bench.visible_pairs(10, 3) == 6
    assert bench.visible_pairs(3, 0) == 0


def test_flops_and_bytes():
    assert bench.prefill_flops([2], [2], 4, 128) == 4 * 128 * 4 * 3
    assert bench.decode_kv_bytes([100, 28], 8, 128) == 128 * 8 * 128 * 4


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=2)
    try:
        got = bench.reduce_max(10.0 + rank * 5.0, torch.device("cpu"))
        bench.barrier(torch.device("cpu"))
        ws, r, local = bench.dist_env()
        q.put((rank, got, ws, r, local))
    finally:
        torch.distributed.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert [(r[2], r[3], r[4]) for r in res] == [(2, 0, 0), (2, 1, 1)]


def test_reference_arm_skips_non_zero_ranks(capsys):
    class A:
        gpus, steps, warmup, ref_rows = 2, 1, 0, 10
    assert bench.bench_reference(A, 2, 1) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_one_line(capsys):
    import json

    class A:
        gpus, steps, warmup, ref_rows = 1, 1, 0, 20
    assert bench.bench_reference(A, 1, 0) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["value"] > 0
    # the same workload description as the GPU arm's line, plus the sample
    cfg = dict(line["config"])
    assert cfg.pop("sample")
    assert cfg == bench.bench_config()
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True


def test_config_shapes_match_the_workload_generator():
    from paged_gqa_attention_varlen_gb300 import workloads as W
    c = W.config("tiny")
    shape = W.CONFIG_SHAPES["tiny"]
    assert (c.num_qo_heads, c.num_kv_heads, c.head_dim, c.causal) == (
        shape["num_qo_heads"], shape["num_kv_heads"], shape["head_dim"], shape["causal"])
    cfg = bench.bench_config()
    qo, kv = W.config_lengths("prefill_hd128")
    assert cfg["prefill"]["total_q"] == sum(qo) == 39332
    assert cfg["decode"]["kv_bytes"] == sum(W.config_lengths("decode")[1]) * 8 * 128 * 2 * 2


def test_source_code_md5_ignores_comments_but_not_code(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("// header\nint f(int x) { return x + 1; }  // one\n/* block\n comment */\n")
    b = tmp_path / "b.cu"
    b.write_text("// other header\nint f(int x) {\n    return x + 1;\n}\n")
    c = tmp_path / "c.cu"
    c.write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_code_md5(a) == bench.source_code_md5(b)
    assert bench.source_code_md5(a) != bench.source_code_md5(c)
