"""Benchmark of the hot path: ragged GQA prefill + paged GQA decode on GB300.

One step = one ragged prefill over the 16-request hd128 workload (16 requests, lengths
U{128..4096}, 32 qo / 8 kv heads, causal) followed by one paged decode over the
256-request workload (kv U{512..32768}, page 16, 32 / 8 heads, split-KV + merge), both
through the C ABI (libpgqa) on inputs already resident in HBM.  Both exceed the 129 MB
L2 (the prefill moves 0.81 GB of Q, K, V, O and lse for the seed-0 draw of 39,332 query
tokens; the decode reads 16.3 GB of K/V), so no flush is needed between steps.

Printed (rank 0, one JSON line): value = prefill TFLOP/s (causal-visible pairs only,
4 * d flops per pair and query head), with the prefill's tok/s (query tokens / s) beside
it; the decode KV GB/s sits under "secondary".  Each carries its roofline against
MEASURED_PEAKS.json, with the algorithmic bytes per launch next to the measured DRAM
traffic.  `e2e` repeats the measurement with
host-resident inputs copied in (pinned memory) and outputs copied out every step.
`cpu_baseline` times the float64 oracle on a bounded row sample on the host cores.
The e2e steps run pipelined, as a serving loop would: step s + 1's inputs are copied in on
a second stream while step s computes and copies out (`serial_value`: one stream).
`median_ms_per_launch` gives the median over the timed steps; `cuda_graph` times the same
two calls captured in CUDA graphs and replayed back to back (after the timed region).

--impl reference times that oracle as the reference arm on the same workload and metric.
Multi-GPU (torchrun): every rank runs the same per-GPU workload (requests are
independent; replicas, no data-path collective), value = all ranks' work / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ragged prefill TFLOP/s (% BF16 peak); paged decode KV GB/s (% HBM peak)"
PREFILL_WORKLOAD = "prefill_hd128"
DECODE_WORKLOAD = "decode"


# ------------------------------------------------------------------ work accounting
def visible_pairs(qo, kv, causal=True):
    """Number of (query row, key) pairs a request attends to (per query head)."""
    if not causal:
        return qo * kv
    tot = 0
    for i in range(qo):
        tot += min(kv, max(0, i + kv - qo + 1))
    return tot


def prefill_flops(qo_lens, kv_lens, hq, d, causal=True):
    return sum(4 * d * hq * visible_pairs(a, b, causal) for a, b in zip(qo_lens, kv_lens))


def decode_kv_bytes(kv_lens, hk, d):
    return sum(kv_lens) * hk * d * 2 * 2


def prefill_algorithmic_bytes(qo_lens, kv_lens, hq, hk, d):
    """Bytes a prefill must move at least once: Q, K, V and O (bf16) and lse (fp32)."""
    tq, tk = sum(qo_lens), sum(kv_lens)
    return tq * hq * d * 2 * 2 + tk * hk * d * 2 * 2 + tq * hq * 4


def decode_algorithmic_bytes(kv_lens, hq, hk, d, max_pages):
    """K/V plus q, o (bf16), lse (fp32), the page table and the lengths (int32)."""
    b = len(kv_lens)
    return decode_kv_bytes(kv_lens, hk, d) + b * hq * d * 2 * 2 + b * hq * 4 + \
        b * max_pages * 4 + b * 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


KERNEL_SOURCES = {"prefill_attention": "paged_gqa_attention_varlen_gb300/csrc/prefill.cu",
                  "decode": "paged_gqa_attention_varlen_gb300/csrc/decode.cu"}


def source_code_md5(path):
    """md5 of a CUDA source with its comments and whitespace removed: it changes when the
    code changes, not when only a comment does."""
    import hashlib
    import re
    with open(path) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.md5(" ".join(src.split()).encode()).hexdigest()


def load_traffic():
    """Per-launch DRAM bytes (ncu dram__bytes_read.sum + dram__bytes_write.sum) of each
    kernel from profiles/traffic.json -- None for a kernel whose source code changed since
    the counters were taken (the file records source_code_md5 of the source)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for key, src in KERNEL_SOURCES.items():
        r = rec.get(key)
        try:
            md5 = source_code_md5(os.path.join(ROOT, src))
        except OSError:
            md5 = None
        out[key] = r["bytes_per_launch"] if r and r.get("source_md5") == md5 else None
    return out


# ------------------------------------------------------------------ distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def reduce_max(x: float, device) -> float:
    """Max of a scalar over ranks (identity without a process group)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(device):
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        reduce_max(0.0, device)


# ------------------------------------------------------------------ clocks
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.gpu_index = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU baseline
def oracle_sample_prefill(case, budget_rows, seed=0):
    """A bounded row sample of the prefill workload and its flops."""
    rng = np.random.default_rng(seed)
    total_rows = case.total_q * case.num_qo_heads
    rows = np.sort(rng.choice(total_rows, size=min(budget_rows, total_rows), replace=False))
    qi = case.q_indptr.cpu().numpy()
    flops = 0
    for r in rows:
        t = r // case.num_qo_heads
        b = int(np.searchsorted(qi, t, side="right") - 1)
        i = t - qi[b]
        qo, kv = case.qo_lens[b], case.kv_lens[b]
        n = kv if not case.causal else min(kv, max(0, i + kv - qo + 1))
        flops += 4 * case.head_dim * n
    return rows.astype(np.int64), flops


def run_oracle_sample(case, host, rows):
    import oracle
    t0 = time.perf_counter()
    oracle.ragged_attention(host["q"], host["k"], host["v"], host["qi"], host["ki"],
                            case.num_qo_heads, case.num_kv_heads, case.causal, case.sm_scale,
                            rows=rows)
    return time.perf_counter() - t0


def host_copies(case):
    return {"q": case.q.cpu(), "k": case.k.cpu(), "v": case.v.cpu(),
            "qi": case.q_indptr.cpu(), "ki": case.kv_indptr.cpu()}


# ------------------------------------------------------------------ main arms
def bench_config():
    """The `config` object of the bench line, from the workloads' lengths and shapes alone
    (no tensor is drawn), so that both arms report the same one."""
    from paged_gqa_attention_varlen_gb300 import workloads as W
    qo, kv = W.config_lengths(PREFILL_WORKLOAD)
    ps = W.CONFIG_SHAPES[PREFILL_WORKLOAD]
    _, dkv = W.config_lengths(DECODE_WORKLOAD)
    ds = W.CONFIG_SHAPES[DECODE_WORKLOAD]
    return {"workload": f"{PREFILL_WORKLOAD} + {DECODE_WORKLOAD}",
            "prefill": {"batch": len(qo), "total_q": int(sum(qo)),
                        "num_qo_heads": ps["num_qo_heads"], "num_kv_heads": ps["num_kv_heads"],
                        "head_dim": ps["head_dim"], "causal": ps["causal"],
                        "flops": prefill_flops(qo, kv, ps["num_qo_heads"], ps["head_dim"],
                                               ps["causal"])},
            "decode": {"batch": len(dkv), "sum_kv": int(sum(dkv)), "page_size": ds["page_size"],
                       "num_qo_heads": ds["num_qo_heads"], "num_kv_heads": ds["num_kv_heads"],
                       "head_dim": ds["head_dim"],
                       "kv_bytes": decode_kv_bytes(dkv, ds["num_kv_heads"], ds["head_dim"])},
            "l2": "inputs larger than L2 (0.81 GB prefill Q/K/V/O/lse, 16.3 GB decode K/V), "
                  "no flush"}


def bench_reference(args, ws, rank):
    """The float64 oracle, timed on the host cores, on a row sample per step."""
    if rank != 0:
        return 0
    import oracle
    from paged_gqa_attention_varlen_gb300 import workloads as W
    case = W.config(PREFILL_WORKLOAD, device="cpu")
    host = host_copies(case)
    rows, flops = oracle_sample_prefill(case, args.ref_rows, seed=1)
    for _ in range(args.warmup):
        run_oracle_sample(case, host, rows[: max(1, len(rows) // 8)])
    times = [run_oracle_sample(case, host, rows) for _ in range(args.steps)]
    total = sum(times)
    value = flops * args.steps / total / 1e12
    sample = (f"{len(rows)} random (token, head) rows of the {PREFILL_WORKLOAD} workload per "
              f"step ({flops / 1e9:.2f} GFLOP of visible pairs)")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": dict(bench_config(), sample=sample),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_gpu(args, ws, rank, local):
    from paged_gqa_attention_varlen_gb300 import api
    from paged_gqa_attention_varlen_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    traffic = load_traffic()

    pf = W.config(PREFILL_WORKLOAD, device=dev)
    dc = W.config(DECODE_WORKLOAD, device=dev)
    pf_flops = prefill_flops(pf.qo_lens, pf.kv_lens, pf.num_qo_heads, pf.head_dim)
    pf_tokens = sum(pf.qo_lens)
    pf_alg_bytes = prefill_algorithmic_bytes(pf.qo_lens, pf.kv_lens, pf.num_qo_heads,
                                             pf.num_kv_heads, pf.head_dim)
    dc_bytes = decode_kv_bytes(dc.kv_lens, dc.num_kv_heads, dc.head_dim)
    dc_alg_bytes = decode_algorithmic_bytes(dc.kv_lens, dc.num_qo_heads, dc.num_kv_heads,
                                            dc.head_dim, dc.page_table.shape[1])
    o_pf = torch.empty_like(pf.q)
    l_pf = torch.empty(pf.q.shape[:2], dtype=torch.float32, device=dev)
    o_dc = torch.empty_like(dc.q)
    l_dc = torch.empty(dc.q.shape[:2], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def prefill(st=stream):
        api.ragged_prefill(pf.q, pf.k, pf.v, pf.q_indptr, pf.kv_indptr, causal=True,
                           sm_scale=pf.sm_scale, out=o_pf, lse=l_pf, stream=st)

    def decode(st=stream):
        api.paged_decode(dc.q, dc.k_pages, dc.v_pages, dc.page_table, dc.kv_lens_t,
                         sm_scale=dc.sm_scale, out=o_dc, lse=l_dc, stream=st)

    for _ in range(max(args.warmup, 3)):
        prefill()
        decode()
    torch.cuda.synchronize(dev)
    if api.device_status() != 0:
        raise RuntimeError("device status after warm-up is not ok")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(dev)
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        prefill()
        ev[s][1].record(stream)
        decode()
        ev[s][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dev)
    clk = clocks.stop()
    total_ms = reduce_max(t_begin.elapsed_time(t_end), dev)
    pf_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dc_ms = [e[1].elapsed_time(e[2]) for e in ev]
    pf_total = reduce_max(sum(pf_ms), dev)
    dc_total = reduce_max(sum(dc_ms), dev)
    status = api.device_status()

    value = pf_flops * ws * args.steps / (pf_total / 1e3) / 1e12
    dc_gbs = dc_bytes * ws * args.steps / (dc_total / 1e3) / 1e9
    pf_launch_ms = pf_total / args.steps
    dc_launch_ms = dc_total / args.steps
    pf_achieved = pf_flops / (pf_launch_ms / 1e3) / 1e12
    dc_achieved = dc_bytes / (dc_launch_ms / 1e3) / 1e9

    # end to end: pinned host inputs copied in and outputs copied out every step
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    hq = {k: v.cpu().pin_memory() for k, v in
          (("q", pf.q), ("k", pf.k), ("v", pf.v), ("qi", pf.q_indptr), ("ki", pf.kv_indptr))}
    ho = torch.empty(o_pf.shape, dtype=o_pf.dtype).pin_memory()
    hl = torch.empty(l_pf.shape, dtype=l_pf.dtype).pin_memory()
    dq = {k: torch.empty_like(v, device=dev) for k, v in hq.items()}
    h2d = sum(v.numel() * v.element_size() for v in hq.values())
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for _ in range(e2e_steps):
        for k in hq:
            dq[k].copy_(hq[k], non_blocking=True)
        api.ragged_prefill(dq["q"], dq["k"], dq["v"], dq["qi"], dq["ki"], causal=True,
                           sm_scale=pf.sm_scale, out=o_pf, lse=l_pf, stream=stream)
        ho.copy_(o_pf, non_blocking=True)
        hl.copy_(l_pf, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    serial_ms = reduce_max(e0.elapsed_time(e1), dev)
    serial_value = pf_flops * ws * e2e_steps / (serial_ms / 1e3) / 1e12

    # the same steps pipelined as a serving loop runs them: step s + 1's inputs are copied
    # in on a second stream (into the other of two device buffers) while step s computes
    # and copies its output out; every step still moves its full inputs and outputs
    copy_in = torch.cuda.Stream(dev)
    dq2 = [dq, {k: torch.empty_like(v) for k, v in dq.items()}]
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    in_free = [torch.cuda.Event(), torch.cuda.Event()]
    torch.cuda.synchronize(dev)
    e0.record(stream)
    copy_in.wait_stream(stream)
    for s in range(e2e_steps):
        i = s % 2
        with torch.cuda.stream(copy_in):
            if s >= 2:
                copy_in.wait_event(in_free[i])
            for k in hq:
                dq2[i][k].copy_(hq[k], non_blocking=True)
            in_ready[i].record(copy_in)
        stream.wait_event(in_ready[i])
        api.ragged_prefill(dq2[i]["q"], dq2[i]["k"], dq2[i]["v"], dq2[i]["qi"], dq2[i]["ki"],
                           causal=True, sm_scale=pf.sm_scale, out=o_pf, lse=l_pf, stream=stream)
        in_free[i].record(stream)
        ho.copy_(o_pf, non_blocking=True)
        hl.copy_(l_pf, non_blocking=True)
    stream.wait_stream(copy_in)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1), dev)
    e2e_value = pf_flops * ws * e2e_steps / (e2e_ms / 1e3) / 1e12
    del dq2

    # decode end to end: per-step inputs (q, page table, lengths) in, output out; the
    # paged KV cache is serving state that stays resident in HBM
    dh = {k: v.cpu().pin_memory() for k, v in
          (("q", dc.q), ("pt", dc.page_table), ("kl", dc.kv_lens_t))}
    dd = {k: torch.empty_like(v, device=dev) for k, v in dh.items()}
    dho = torch.empty(o_dc.shape, dtype=o_dc.dtype).pin_memory()
    dhl = torch.empty(l_dc.shape, dtype=l_dc.dtype).pin_memory()
    d_h2d = sum(v.numel() * v.element_size() for v in dh.values())
    d_d2h = dho.numel() * dho.element_size() + dhl.numel() * dhl.element_size()
    e0.record(stream)
    for _ in range(e2e_steps):
        for k in dh:
            dd[k].copy_(dh[k], non_blocking=True)
        api.paged_decode(dd["q"], dc.k_pages, dc.v_pages, dd["pt"], dd["kl"],
                         sm_scale=dc.sm_scale, out=o_dc, lse=l_dc, stream=stream)
        dho.copy_(o_dc, non_blocking=True)
        dhl.copy_(l_dc, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    d_e2e_ms = reduce_max(e0.elapsed_time(e1), dev)
    d_e2e_value = dc_bytes * ws * e2e_steps / (d_e2e_ms / 1e3) / 1e9

    # the same calls replayed from CUDA graphs (after the timed region; reported beside it)
    graph = None
    if args.graph_reps > 0:
        graph = {"prefill_ms_per_launch": graph_ms(prefill, dev, args.graph_reps),
                 "decode_ms_per_launch": graph_ms(decode, dev, args.graph_reps),
                 "reps": args.graph_reps}
        graph["prefill_tflops"] = pf_flops / (graph["prefill_ms_per_launch"] / 1e3) / 1e12
        graph["prefill_tok_s"] = pf_tokens / (graph["prefill_ms_per_launch"] / 1e3)
        graph["decode_gbs"] = dc_bytes / (graph["decode_ms_per_launch"] / 1e3) / 1e9
        if api.device_status() != 0:
            raise RuntimeError("device status after the graph replays is not ok")

    extra = None if args.no_extra else bench_extra(api, W, dev, stream, dc, peaks)

    if rank != 0:
        return 0

    # CPU baseline: the oracle on a bounded row sample of the same prefill workload
    cpu = None
    if not args.no_cpu_baseline and ws == 1:
        import oracle
        case_h = W.RaggedCase(pf.name, pf.q, pf.k, pf.v, pf.q_indptr.cpu(), pf.kv_indptr.cpu(),
                              pf.qo_lens, pf.kv_lens, pf.num_qo_heads, pf.num_kv_heads,
                              pf.head_dim, True, pf.sm_scale)
        host = host_copies(case_h)
        rows, flops = oracle_sample_prefill(case_h, args.cpu_rows, seed=1)
        secs = run_oracle_sample(case_h, host, rows)
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.threads(),
               "kind": "oracle",
               "sample": f"{len(rows)} random (token, head) rows of {PREFILL_WORKLOAD} "
                         f"({flops / 1e9:.2f} GFLOP, {secs:.1f} s)"}

    pf_tr = traffic.get("prefill_attention")
    dc_tr = traffic.get("decode")
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(),
        "tok_s": pf_tokens * ws * args.steps / (pf_total / 1e3),
        "roofline": {"bound": "tensor", "kernel": "prefill (plan + attention launch pair)",
                     "achieved": pf_achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": pf_achieved / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " burst bf16",
                     "traffic": pf_tr, "algorithmic_bytes": pf_alg_bytes,
                     "traffic_over_algorithmic": (pf_tr / pf_alg_bytes) if pf_tr else None},
        "secondary": {
            "metric": "paged decode KV GB/s", "value": dc_gbs, "unit": "GB/s",
            "ms_per_launch": dc_launch_ms,
            "roofline": {"bound": "hbm", "kernel": "decode (plan + split-KV + merge)",
                         "achieved": dc_achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": dc_achieved / peaks["hbm_gbs"],
                         "peak_source": peaks["source"] + " copy bandwidth",
                         "traffic": dc_tr, "algorithmic_bytes": dc_alg_bytes,
                         "traffic_over_algorithmic": (dc_tr / dc_alg_bytes) if dc_tr else None},
            "e2e": {"value": d_e2e_value, "unit": "GB/s", "h2d_bytes_per_step": d_h2d,
                    "d2h_bytes_per_step": d_d2h,
                    "note": "KV cache resident (serving state); q, page table, lengths in"}},
        "prefill_ms_per_launch": pf_launch_ms,
        "median_ms_per_launch": {"prefill": statistics.median(pf_ms),
                                 "decode": statistics.median(dc_ms)},
        "cuda_graph": graph,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "tok_s": pf_tokens * ws * e2e_steps / (e2e_ms / 1e3),
                "note": "pipelined: step s+1's inputs copied in on a second stream while step s "
                        "computes and copies out",
                "serial_value": serial_value},
        "gpu_launches": args.steps * (3 + 3),
        "clocks": clk,
        "device_status": status,
        "cpu_baseline": cpu,
        "extra": extra,
    }
    print(json.dumps(line), flush=True)
    return 0


def graph_ms(fn, dev, reps):
    """Milliseconds per call of fn(stream) captured once in a CUDA graph and replayed
    `reps` times back to back between CUDA events."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        fn(side)  # a call on the capture stream first, as graph capture wants
    torch.cuda.current_stream(dev).wait_stream(side)
    with torch.cuda.graph(g):
        fn(torch.cuda.current_stream(dev))
    for _ in range(3):
        g.replay()
    st = torch.cuda.current_stream(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(st)
    for _ in range(reps):
        g.replay()
    e1.record(st)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / reps


def time_calls(fn, stream, reps=20, warmup=3):
    """Milliseconds per call of fn(): back-to-back launches between CUDA events on `stream`."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps


def bench_extra(api, W, dev, stream, dc, peaks):
    """The paged prefill (ragged queries over a paged KV cache) on the prefill_hd128 and
    prefix_hd256 shapes with 16-token pages, the ragged prefix_hd256 beside it, the ragged
    prefill of one 32k-token request,
    4-token-per-request decode (speculative verification) over the resident 256-request
    decode cache, and the decode and the 4-token decode over that cache stored as FP8 E4M3;
    each timed on its own (inputs resident in HBM)."""
    out = {}

    def tensor_line(flops, ms, what):
        tf = flops / (ms / 1e3) / 1e12
        return {"what": what, "ms_per_launch": ms, "value": tf, "unit": "TFLOP/s",
                "roofline": {"bound": "tensor", "peak": peaks["bf16_tflops"],
                             "frac": tf / peaks["bf16_tflops"]}}

    for name in ("prefill_hd128", "prefix_hd256"):
        qo, kv = W.config_lengths(name)
        rc = W.config(name, device=dev)
        pc = W.paged_case(kv, rc.num_qo_heads, rc.num_kv_heads, rc.head_dim, page_size=16,
                          qo_lens=qo, seed=0, device=dev)
        flops = prefill_flops(qo, kv, rc.num_qo_heads, rc.head_dim)
        o = torch.empty_like(pc.q)
        lse = torch.empty(pc.q.shape[:2], dtype=torch.float32, device=dev)
        ms = time_calls(lambda: api.paged_prefill(pc.q, pc.k_pages, pc.v_pages, pc.q_indptr,
                                                  pc.page_table, pc.kv_lens_t, causal=True,
                                                  sm_scale=pc.sm_scale, out=o, lse=lse,
                                                  stream=stream), stream)
        out[f"paged_prefill_{name}"] = tensor_line(flops, ms, f"{name} shape, keys in 16-token "
                                                   "pages (random page order)")
        if name == "prefill_hd128":
            # the same pages as an FP8 E4M3 cache: converted to bf16 in the workspace, then
            # the bf16 paged prefill (the conversion is inside the timed call)
            k8 = pc.k_pages.to(torch.float8_e4m3fn)
            v8 = pc.v_pages.to(torch.float8_e4m3fn)
            mq = max(qo)
            ms = time_calls(lambda: api.paged_prefill(pc.q, k8, v8, pc.q_indptr, pc.page_table,
                                                      pc.kv_lens_t, causal=True,
                                                      sm_scale=pc.sm_scale, k_scale=1.0,
                                                      v_scale=1.0, max_qo_len=mq, out=o,
                                                      lse=lse, stream=stream), stream)
            out["paged_prefill_e4m3_prefill_hd128"] = tensor_line(
                flops, ms, "prefill_hd128 shape over an FP8 E4M3 cache of 16-token pages "
                "(pages converted to bf16 in the call)")
            del k8, v8
        if name == "prefix_hd256":
            o2 = torch.empty_like(rc.q)
            l2 = torch.empty(rc.q.shape[:2], dtype=torch.float32, device=dev)
            ms = time_calls(lambda: api.ragged_prefill(rc.q, rc.k, rc.v, rc.q_indptr,
                                                       rc.kv_indptr, causal=True,
                                                       sm_scale=rc.sm_scale, out=o2, lse=l2,
                                                       stream=stream), stream)
            out["ragged_prefill_prefix_hd256"] = tensor_line(flops, ms, "prefix_hd256, ragged K/V")
        del pc, rc, o, lse
    # head_dim 256 with a short work list: 2 requests of 256 query rows over 16k-key cached
    # prefixes (16 / 4 heads): 16 q-tile items per kv head, split into 2048-key chunks
    sqo, skv = [256, 256], [256 + 16384, 256 + 16384]
    sc = W.ragged_case(sqo, skv, 16, 4, 256, causal=True, seed=5, device=dev)
    so = torch.empty_like(sc.q)
    sl = torch.empty(sc.q.shape[:2], dtype=torch.float32, device=dev)
    ms = time_calls(lambda: api.ragged_prefill(sc.q, sc.k, sc.v, sc.q_indptr, sc.kv_indptr,
                                               causal=True, sm_scale=sc.sm_scale, out=so, lse=sl,
                                               stream=stream), stream, reps=20)
    out["ragged_prefill_hd256_short_list"] = tensor_line(
        prefill_flops(sqo, skv, 16, 256), ms,
        "batch 2, qo 256 over 16k-key prefixes, 16/4 heads, d 256 (split-KV regime)")
    del sc, so, sl
    # one 32k-token request, 64 / 8 heads (G = 8), K scaled by 3: long items, few boundaries
    lc = W.config("long", device=dev)
    lo = torch.empty_like(lc.q)
    ll = torch.empty(lc.q.shape[:2], dtype=torch.float32, device=dev)
    ms = time_calls(lambda: api.ragged_prefill(lc.q, lc.k, lc.v, lc.q_indptr, lc.kv_indptr,
                                               causal=True, sm_scale=lc.sm_scale, out=lo, lse=ll,
                                               stream=stream), stream, reps=5)
    out["ragged_prefill_long"] = tensor_line(
        prefill_flops(lc.qo_lens, lc.kv_lens, lc.num_qo_heads, lc.head_dim), ms,
        "one 32768-token request, 64/8 heads, d 128, causal, K x 3")
    del lc, lo, ll
    # 4 query tokens per request over the decode workload's paged cache
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    q4 = torch.randn((dc.batch * 4, dc.num_qo_heads, dc.head_dim), generator=g, device=dev,
                     dtype=torch.float32).to(torch.bfloat16)
    qi4 = torch.arange(0, 4 * dc.batch + 1, 4, dtype=torch.int32, device=dev)
    o4 = torch.empty_like(q4)
    l4 = torch.empty(q4.shape[:2], dtype=torch.float32, device=dev)
    ms = time_calls(lambda: api.paged_prefill(q4, dc.k_pages, dc.v_pages, qi4, dc.page_table,
                                              dc.kv_lens_t, causal=True, sm_scale=dc.sm_scale,
                                              out=o4, lse=l4, stream=stream), stream, reps=10)
    kv_bytes = decode_kv_bytes(dc.kv_lens, dc.num_kv_heads, dc.head_dim)
    gbs = kv_bytes / (ms / 1e3) / 1e9
    out["multi_token_decode_q4"] = {
        "what": "256 requests x 4 query tokens (decode workload's cache, causal)",
        "ms_per_launch": ms, "value": gbs, "unit": "GB/s",
        "roofline": {"bound": "hbm", "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"]}}
    # the decode workload's cache as FP8 E4M3 (per-tensor scales), same requests
    k8 = dc.k_pages.to(torch.float8_e4m3fn)
    v8 = dc.v_pages.to(torch.float8_e4m3fn)
    o8 = torch.empty_like(dc.q)
    l8 = torch.empty(dc.q.shape[:2], dtype=torch.float32, device=dev)
    ms = time_calls(lambda: api.paged_decode(dc.q, k8, v8, dc.page_table, dc.kv_lens_t,
                                             sm_scale=dc.sm_scale, k_scale=1.0, v_scale=1.0,
                                             out=o8, lse=l8, stream=stream), stream, reps=20)
    gbs8 = kv_bytes / 2 / (ms / 1e3) / 1e9
    out["decode_e4m3"] = {
        "what": "decode workload (256 requests) with an FP8 E4M3 KV cache; GB/s of E4M3 K/V",
        "ms_per_launch": ms, "value": gbs8, "unit": "GB/s",
        "roofline": {"bound": "hbm", "peak": peaks["hbm_gbs"], "frac": gbs8 / peaks["hbm_gbs"]}}
    # 4 query tokens per request over the E4M3 cache (the same q4 rows)
    ms = time_calls(lambda: api.paged_prefill(q4, k8, v8, qi4, dc.page_table, dc.kv_lens_t,
                                              causal=True, sm_scale=dc.sm_scale, k_scale=1.0,
                                              v_scale=1.0, max_qo_len=4, out=o4, lse=l4,
                                              stream=stream), stream, reps=20)
    gbs84 = kv_bytes / 2 / (ms / 1e3) / 1e9
    out["multi_token_decode_q4_e4m3"] = {
        "what": "256 requests x 4 query tokens over the FP8 E4M3 cache (causal); GB/s of E4M3 K/V",
        "ms_per_launch": ms, "value": gbs84, "unit": "GB/s",
        "roofline": {"bound": "hbm", "peak": peaks["hbm_gbs"], "frac": gbs84 / peaks["hbm_gbs"]}}
    del k8, v8, q4, o4, l4
    out["device_status"] = api.device_status()
    torch.cuda.empty_cache()
    return out


def profile_case(args):
    """Run one bounded case of a hot-path kernel `--reps` times (for ncu captures)."""
    from paged_gqa_attention_varlen_gb300 import api
    from paged_gqa_attention_varlen_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    if args.profile in ("prefill_hd128", "prefix_hd256", "long", "tiny"):
        c = W.config(args.profile, device=dev)
        o = torch.empty_like(c.q)
        lse = torch.empty(c.q.shape[:2], dtype=torch.float32, device=dev)
        for _ in range(args.reps):
            api.ragged_prefill(c.q, c.k, c.v, c.q_indptr, c.kv_indptr, causal=c.causal,
                               sm_scale=c.sm_scale, out=o, lse=lse)
    elif args.profile in ("paged_prefill_hd128", "paged_prefix_hd256", "decode_q4",
                          "decode_q4_e4m3", "paged_prefill_e4m3_hd128"):
        # paged prefill: the named shape in 16-token pages; decode_q4: 4 query tokens per
        # request over the first --decode-batch requests of the decode workload; the _e4m3
        # cases store the same pages as FP8 E4M3 (scales 1)
        e4m3 = args.profile.endswith("e4m3") or "_e4m3_" in args.profile
        if args.profile.startswith("decode_q4"):
            kv = W.config_lengths("decode")[1][:args.decode_batch]
            c = W.paged_case(kv, 32, 8, 128, page_size=16, qo_lens=[4] * len(kv), seed=0,
                             device=dev)
        else:
            name = "prefill_hd128" if e4m3 else args.profile[len("paged_"):]
            qo, kv = W.config_lengths(name)
            hq, hk, d = (32, 8, 128) if name == "prefill_hd128" else (16, 4, 256)
            c = W.paged_case(kv, hq, hk, d, page_size=16, qo_lens=qo, seed=0, device=dev)
        kp, vp, extra = c.k_pages, c.v_pages, {}
        if e4m3:
            kp, vp = kp.to(torch.float8_e4m3fn), vp.to(torch.float8_e4m3fn)
            extra = dict(k_scale=1.0, v_scale=1.0, max_qo_len=max(c.qo_lens))
        o = torch.empty_like(c.q)
        lse = torch.empty(c.q.shape[:2], dtype=torch.float32, device=dev)
        for _ in range(args.reps):
            api.paged_prefill(c.q, kp, vp, c.q_indptr, c.page_table, c.kv_lens_t,
                              causal=True, sm_scale=c.sm_scale, out=o, lse=lse, **extra)
    else:  # decode slice: the first --decode-batch requests of the decode workload
        kv = W.config_lengths("decode")[1][:args.decode_batch]
        if args.profile == "decode_e4m3":
            c = W.paged_case_e4m3(kv, 32, 8, 128, page_size=16, seed=0, device=dev)
            scales = dict(k_scale=c.meta["k_scale"], v_scale=c.meta["v_scale"])
        else:
            c = W.paged_case(kv, 32, 8, 128, page_size=16, seed=0, device=dev)
            scales = {}
        o = torch.empty_like(c.q)
        lse = torch.empty(c.q.shape[:2], dtype=torch.float32, device=dev)
        for _ in range(args.reps):
            api.paged_decode(c.q, c.k_pages, c.v_pages, c.page_table, c.kv_lens_t,
                             sm_scale=c.sm_scale, out=o, lse=lse, **scales)
    torch.cuda.synchronize(dev)
    st = api.device_status()
    print(json.dumps({"profile": args.profile, "reps": args.reps, "status": st,
                      "max_mem_gb": torch.cuda.max_memory_allocated(dev) / 1e9}))
    return 0 if st == 0 else 1


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--ref-rows", type=int, default=3000,
                    help="oracle rows per CPU-baseline / reference step")
    ap.add_argument("--cpu-rows", type=int, default=800000,
                    help="oracle rows timed for the cpu_baseline object (about 10-30 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph-reps", type=int, default=20,
                    help="CUDA-graph replays per kernel timed after the main region (0: skip)")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the paged-prefill and multi-token-decode measurements")
    ap.add_argument("--profile", choices=["prefill_hd128", "prefix_hd256", "long", "tiny",
                                          "decode", "paged_prefill_hd128", "paged_prefix_hd256",
                                          "decode_q4", "decode_e4m3", "decode_q4_e4m3",
                                          "paged_prefill_e4m3_hd128"], default=None,
                    help="run one bounded case --reps times and exit (ncu captures)")
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--decode-batch", type=int, default=32)
    args = ap.parse_args(argv)
    if args.profile:
        return profile_case(args)
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return bench_reference(args, ws, rank)
    init_dist(ws, "nccl")
    try:
        return bench_gpu(args, ws, rank, local)
    finally:
        if torch.distributed.is_available() and torch.distributed.is_initialized():
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
