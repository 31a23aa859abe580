"""Benchmark: paged decode attention at the Llama-3-8B attention shape on GB300.

One step = one zl_decode_attn call (attention kernel + merge kernel) over the
whole batch: 64 sequences, 32 query / 8 KV heads, head dim 128, context
lengths U[512, 4096], page size 16, pages scattered over a pool 1.25x the
total. The KV working set (~0.6 GB) is larger than L2 (129 MB), so no flush
is needed between steps.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]

Prints one JSON line. ``value`` is KV read bandwidth (algorithmic bytes: every
visible token's K and V rows, once) over all GPUs; ``--impl reference`` times
the CPU oracle on the host cores instead. Multi-GPU runs are independent
replicas (the path has no exchange step).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV read GB/s (Llama-3-8B shape)"
UNIT = "GB/s"
WORKLOAD = "llama3_8b_decode"
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
CSRC = os.path.join(ROOT, "paged_decode_attention_gqa_gb300", "csrc")
# the sources whose hash must match the one an ncu traffic figure was taken with
KERNEL_SRC = {"gqa": [os.path.join(CSRC, "gqa_kernel.cuh"), os.path.join(CSRC, "gqa_decode.cu")],
              "mla": [os.path.join(CSRC, "mla_decode.cu")]}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash(kind):
    """Hash of the kernel sources with // comments and blank space removed, so
    that editing a comment does not void a traffic figure but any code change
    does."""
    import re
    h = hashlib.sha256()
    for path in KERNEL_SRC[kind]:
        with open(path, encoding="utf-8") as f:
            text = f.read()
        code = re.sub(r"//[^\n]*", "", text)
        h.update("".join(code.split()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(workload, kind):
    """DRAM bytes per attention launch from the committed ncu summary, if the
    kernel source has not changed since it was captured; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_sha256_16") != kernel_hash(kind):
        return None
    return e.get("dram_bytes_per_launch")


def kv_bytes(w):
    """Algorithmic bytes: the K and V rows of every visible token, once (MLA:
    the one latent row, V being part of it)."""
    tokens = int(np.asarray(w.seq_lens, dtype=np.int64).sum())
    if w.mla:
        return tokens * w.D_qk * 2
    return tokens * w.Hkv * 2 * w.D_qk * 2


def unique_kv_bytes(w):
    """The same bytes over distinct cache rows: a page that several sequences
    map (a shared prefix) counts once, with the most slots any of them sees.
    This is what has to come from HBM; it equals kv_bytes when no page is
    shared."""
    P = w.page_size
    L = np.asarray(w.seq_lens, dtype=np.int64)
    n = (L + P - 1) // P
    if n.sum() == 0:
        return 0
    seq = np.repeat(np.arange(w.B), n)
    j = np.arange(int(n.sum())) - np.repeat(np.cumsum(n) - n, n)
    pages = np.asarray(w.block_table)[seq, j].astype(np.int64)
    slots = np.minimum(P, L[seq] - j * P)
    most = np.zeros(int(pages.max()) + 1, dtype=np.int64)
    np.maximum.at(most, pages, slots)
    tokens = int(most.sum())
    return tokens * w.D_qk * 2 if w.mla else tokens * w.Hkv * 2 * w.D_qk * 2


def io_bytes(w):
    """Q read + out written + block table and seq_lens read (per launch)."""
    pages = int(((w.seq_lens.astype(np.int64) + w.page_size - 1) // w.page_size).sum())
    return w.B * w.q_len * w.Hq * (w.D_qk + w.D_v) * 2 + pages * 4 + w.B * 4


def metric_name(workload, q_len=1):
    if q_len != 1:
        return f"decode-attn KV read GB/s ({workload}, {q_len} query tokens)"
    return METRIC if workload == WORKLOAD else f"decode-attn KV read GB/s ({workload})"


def make_workload(name, batch=None, q_len=1):
    from paged_decode_attention_gqa_gb300 import workloads
    fn = workloads.WORKLOADS[name]
    kw = {}
    if batch:
        kw["B"] = batch
    if q_len != 1:
        kw["q_len"] = q_len
    return fn(**kw)


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the raw samples go to $ZL_CLOCKS_DIR when it is set (to keep them),
        # else to a temporary directory
        out_dir = os.environ.get("ZL_CLOCKS_DIR") or tempfile.mkdtemp(prefix="zl_clocks_")
        self.path = os.path.join(out_dir, f"clocks_gpu{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def max_over_ranks(x, world, device):
    """The largest value of x over all ranks (the job's time is its slowest rank's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(w, min_seconds=10.0, max_calls=50):
    """The oracle as it stands, on all host cores: (seconds per call, calls, threads)."""
    import oracle
    orc = oracle.load()
    threads = cpu_cores()
    q, k = w.bits(w.q), w.bits(w.k_pool)
    v = None if w.mla else w.bits(w.v_pool)
    times = []
    res = None
    t_start = time.perf_counter()
    while len(times) < max_calls and (time.perf_counter() - t_start) < min_seconds:
        t0 = time.perf_counter()
        res = orc.decode_attn(q, k, v, w.strides, w.block_table, w.seq_lens, Hkv=w.Hkv,
                              page_size=w.page_size, num_pages=w.num_pages, scale=w.scale,
                              D_v=w.D_v, num_threads=threads)
        times.append(time.perf_counter() - t0)
    return statistics.median(times), len(times), threads, res


def parity_summary(out_gpu, lse_gpu, res):
    """Element-wise errors of the measured call's output against the oracle's."""
    ref, ref_lse, status = res
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    diff = np.abs(got - ref)
    big = np.abs(ref) >= 1e-2
    ratio = diff / (1e-2 + 1e-2 * np.abs(ref))
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    return {"max_abs_err": float(diff.max()),
            "max_rel_err": float((diff[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
            "worst_err_over_tolerance": float(ratio.max()),
            "lse_max_abs_err": float(np.abs(lse[fin] - ref_lse[fin]).max()) if fin.any() else 0.0,
            "within_tolerance": bool((ratio <= 1.0).all()), "oracle_status": int(status),
            "tolerance": "|gpu - oracle| <= 1e-2 + 1e-2 |oracle| per element (bf16 out, fp64 "
                         "oracle), the whole output of the last timed call"}


def run_reference(args, world, rank, budget_s=120.0):
    """CPU oracle arm: rank 0 only; other ranks exit without work.

    Each step runs the oracle on the first n sequences of the workload, n sized
    so that warm-up plus timed steps take about ``budget_s`` seconds (the whole
    batch when that fits).
    """
    if rank != 0:
        return
    from paged_decode_attention_gqa_gb300 import workloads
    w = make_workload(args.workload, args.batch, args.q_len)
    import oracle
    orc = oracle.load()
    threads = cpu_cores()
    q, k = w.bits(w.q), w.bits(w.k_pool)
    v = None if w.mla else w.bits(w.v_pool)

    def run(n):
        orc.decode_attn(q[:n], k, v, w.strides, w.block_table[:n], w.seq_lens[:n], Hkv=w.Hkv,
                        page_size=w.page_size, num_pages=w.num_pages, scale=w.scale,
                        D_v=w.D_v, num_threads=threads)

    t0 = time.perf_counter()
    run(8)
    per_seq = (time.perf_counter() - t0) / 8
    per_step = budget_s / max(1, args.steps + args.warmup)
    n = int(max(1, min(w.B, per_step // max(per_seq, 1e-9))))
    for _ in range(args.warmup):
        run(n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(n)
    dt = (time.perf_counter() - t0) / args.steps
    sample_bytes = kv_bytes(w) * int(w.seq_lens[:n].astype(np.int64).sum()) // int(
        w.seq_lens.astype(np.int64).sum())
    gbs = sample_bytes / dt / 1e9
    sample = (f"first {n} of {w.B} sequences per step (all heads), "
              f"{int(w.seq_lens[:n].sum())} tokens")
    line = {
        "impl": "reference", "metric": metric_name(args.workload, args.q_len), "value": gbs, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_of(w, world),
        "cpu_baseline": {"value": gbs, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w, world):
    lens = w.seq_lens
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "D_qk": w.D_qk,
            "D_v": w.D_v, "page_size": w.page_size,
            "seq_len": f"{int(lens.min())}..{int(lens.max())} (sum {int(lens.sum())})",
            "q_len": w.q_len, "kv_bytes_per_step": kv_bytes(w), "seed": w.seed,
            "l2": ("no flush: KV working set per step exceeds the 129 MB L2"
                   if kv_bytes(w) > 4 * 129e6 else "L2 flushed between steps (a 2 x L2 write, outside"
                   " the per-step events)"),
            "parallelism": f"replicas x{world}"}


def run_ours(args, world, rank, local):
    import paged_decode_attention_gqa_gb300 as zl

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        zl.build()
    if world > 1:
        dist.barrier()
    zl.lib()

    w = make_workload(args.workload, args.batch, args.q_len)
    kind = "mla" if w.mla else "gqa"
    q, k = w.q.to(dev), w.k_pool.to(dev)
    v = None if w.mla else w.v_pool.to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty(w.B, w.q_len, w.Hq, w.D_v, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(w.B, w.q_len, w.Hq, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    npref = 0
    if args.shared_prefix:
        npref = int(w.notes.get("shared_prefix_tokens", 0)) // w.page_size
        assert npref > 0, "--shared-prefix needs a workload with a shared prefix"
    p = zl.make_params(q, k, v, bt, sl, out, page_size=w.page_size, scale=w.scale, Hkv=w.Hkv,
                       D_v=w.D_v, lse=lse, err_flags=err, max_seq_len=w.max_seq_len,
                       single_launch=args.single_launch and not w.mla,
                       shared_prefix_pages=npref)
    need = zl.workspace_size_mla(p) if w.mla else zl.workspace_size(p)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    stream = torch.cuda.current_stream()
    # Small working sets are flushed from L2 between steps (a 2x L2 write).
    flush = None
    if kv_bytes(w) <= 4 * 129e6:
        flush = torch.empty(int(2 * 129e6) // 4, dtype=torch.int32, device=dev)

    # --with-append: each step first writes the q_len new tokens' K/V rows into
    # their page slots (zl_kv_append), then attends, as a decode step does.
    ap = None
    if args.with_append:
        from paged_decode_attention_gqa_gb300 import workloads as _wl
        k_new, v_new = _wl.new_token_rows(w.seed, w.B, w.q_len, w.Hkv, w.D_qk,
                                          None if w.mla else w.D_v)
        k_new = k_new.to(dev)
        v_new = None if v_new is None else v_new.to(dev)
        ap = zl.make_append_params(k_new, v_new, k, v, bt, sl, page_size=w.page_size,
                                   layout=w.layout, err_flags=err)
    stream_ptr = ctypes.c_void_p(stream.cuda_stream)

    def call():
        if ap is not None:
            rc = zl.lib().zl_kv_append(ctypes.byref(ap), stream_ptr)
            assert rc == zl.OK, rc
        zl.call(p, mla=w.mla, stream=stream)

    def step():
        if flush is not None:
            flush.zero_()
        call()

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"

    # ---- timed region: K steps, CUDA events on the launching stream, clocks sampled
    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.4)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # With an L2 flush between steps, each step's call is timed on its own
    # (events after the flush, around the call) and the flush is left out.
    step_evs = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)] if flush is not None else None)
    t_begin.record(stream)
    for i in range(args.steps):
        if flush is None:
            call()
        else:
            flush.zero_()
            step_evs[i][0].record(stream)
            call()
            step_evs[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if flush is None:
        ms = t_begin.elapsed_time(t_end) / args.steps
    else:
        ms = sum(a.elapsed_time(b) for a, b in step_evs) / args.steps
    ms = max_over_ranks(ms, world, dev)
    # the library's own count per call: attention (+ merge) per token group
    launches = args.steps * (2 if w.mla else zl.launches(p))
    if ap is not None:
        launches += args.steps                              # the KV append
    if flush is not None:
        launches += args.steps                              # the L2 flush memset

    # ---- per-kernel timing, after the timed region: the library records
    # events around the attention kernel alone, the bench around the call.
    # (Events between the two launches would keep the merge from starting
    # early, so the headline steps above carry none.)
    n_ev = max(10, min(args.steps, 1000))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_ev)]
    # torch only reports elapsed time for events it has recorded itself; record
    # each once here, the library re-records them around the attention kernel.
    for a, b in evs:
        a.record(stream)
        b.record(stream)
    call_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(n_ev)]
    for i in range(n_ev):
        p.attn_begin, p.attn_end = evs[i][0].cuda_event, evs[i][1].cuda_event
        if flush is not None:
            flush.zero_()
        call_evs[i][0].record(stream)
        call()
        call_evs[i][1].record(stream)
    torch.cuda.synchronize()
    p.attn_begin = p.attn_end = None
    # Host time to issue one call: a burst short enough that the launch queue
    # never fills (a long loop would pace the host at the GPU's rate).
    n_host = 32
    h0 = time.perf_counter()
    for _ in range(n_host):
        call()
    host_us = (time.perf_counter() - h0) / n_host * 1e6
    torch.cuda.synchronize()
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in call_evs)
    append = None
    if ap is not None:
        app_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_ev)]
        for a, b in app_evs:
            if flush is not None:
                flush.zero_()
            a.record(stream)
            zl.lib().zl_kv_append(ctypes.byref(ap), stream_ptr)
            b.record(stream)
        torch.cuda.synchronize()
        app_ms = statistics.mean(a.elapsed_time(b) for a, b in app_evs)
        # new rows read once, written once into the pools
        app_bytes = 2 * w.B * w.q_len * w.Hkv * (w.D_qk + (0 if w.mla else w.D_v)) * 2
        append = {"us_per_launch": app_ms * 1e3, "bytes_per_launch": app_bytes,
                  "GBs": app_bytes / (app_ms * 1e-3) / 1e9,
                  "note": "zl_kv_append alone, L2 flushed first when the step flushes"}
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"

    # ---- end to end through the public API: host inputs in, host result out.
    # Every step copies its inputs (q, block table, seq_lens) in from pinned host
    # memory and its output back; steps are pipelined the way a serving loop
    # overlaps them: two device buffer sets, inputs copied on one stream, the
    # call on another, the output copied out on a third, ordered by events.
    e2e = None
    if not args.no_e2e:
        pin_q = w.q.pin_memory()
        pin_bt = torch.from_numpy(w.block_table).pin_memory()
        pin_sl = torch.from_numpy(w.seq_lens).pin_memory()
        pin_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        dq = [q, torch.empty_like(q)]
        dbt = [bt, torch.empty_like(bt)]
        dsl = [sl, torch.empty_like(sl)]
        dout = [out, torch.empty_like(out)]
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        e2e_steps = max(10, min(args.steps, 2000))
        h2d = pin_q.numel() * 2 + pin_bt.numel() * 4 + pin_sl.numel() * 4
        d2h = pin_out[0].numel() * 2
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        torch.cuda.synchronize()
        for e in ev_comp + ev_out:
            e.record(s_comp)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            j = i & 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_comp[j])          # set j no longer read by step i - 2
                dq[j].copy_(pin_q, non_blocking=True)
                dbt[j].copy_(pin_bt, non_blocking=True)
                dsl[j].copy_(pin_sl, non_blocking=True)
                ev_in[j].record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(ev_in[j])
                s_comp.wait_event(ev_out[j])         # out j copied out by step i - 2
                if flush is not None:
                    flush.zero_()
                if w.mla:
                    zl.decode_attn_mla(dq[j], k, dbt[j], dsl[j], page_size=w.page_size,
                                       scale=w.scale, D_v=w.D_v, out=dout[j], workspace=ws,
                                       max_seq_len=w.max_seq_len, stream=s_comp)
                else:
                    zl.decode_attn(dq[j], k, v, dbt[j], dsl[j], page_size=w.page_size,
                                   scale=w.scale, out=dout[j], workspace=ws,
                                   max_seq_len=w.max_seq_len, single_launch=args.single_launch,
                                   shared_prefix_pages=npref, stream=s_comp)
                ev_comp[j].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[j])
                pin_out[j].copy_(dout[j], non_blocking=True)
                ev_out[j].record(s_out)
        torch.cuda.synchronize()
        e2e_s = (time.perf_counter() - t0) / e2e_steps
        e2e = {"value": kv_bytes(w) * world / e2e_s / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "us_per_step": e2e_s * 1e6,
               "note": "every step copies q, block table and seq_lens in from pinned host memory "
                       "and its output back (host wall clock); steps pipelined over two buffer "
                       "sets and three streams; the KV cache is device-resident state"
                       + ("; includes the L2 flush" if flush is not None else "")}

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    kvb = kv_bytes(w)
    peak, peak_kind = measured_peaks()
    # the roofline counts the bytes HBM has to deliver: a shared page once
    algo = unique_kv_bytes(w) + io_bytes(w)
    logical = kvb + io_bytes(w)
    achieved = algo / (attn_ms * 1e-3) / 1e9
    cpu = None
    parity = None
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline is an N = 1 figure
        cpu_s, cpu_calls, cores, res = time_oracle(w)
        cpu = {"value": kvb / cpu_s / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"the whole workload per call, {cpu_calls} calls (median)"}
        if ap is None:  # (with the append the device pools hold the new rows)
            parity = parity_summary(out, lse, res)
    line = {
        "metric": metric_name(args.workload, args.q_len),
        "value": kvb * world / (ms * 1e-3) / 1e9,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "us_per_call": call_ms * 1e3,
        "host_enqueue_us_per_call": host_us,
        "us_per_step": ms * 1e3,
        "pct_hbm_roofline": {"of_measured": achieved / peak, "of_nominal_8TBs": achieved / 8000.0},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": dict(config_of(w, world), split_merge=(
            "in the attention kernel (single launch)" if kind == "gqa" and args.single_launch
            else "second launch (programmatic dependent launch)"),
            step="kv append + attention" if ap is not None else "attention",
            shared_prefix_pages=npref),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "kernel": f"{kind}_decode_kernel", "attn_us_per_launch": attn_ms * 1e3,
                     "algorithmic_bytes_per_launch": algo,
                     **({"logical_bytes_per_launch": logical,
                         "bytes_note": "algorithmic bytes count each shared page once; "
                                       "value counts every sequence's reads"}
                        if logical != algo else {}),
                     "traffic": traffic_per_launch(w.name, kind)},
        "cpu_baseline": cpu,
        "parity": parity,
        "e2e": e2e,
        "gpu_launches": launches,
        "kv_append": append,
        "clocks": clocks,
    }
    if w.mla:
        flops = 2.0 * int(w.seq_lens.astype(np.int64).sum()) * w.q_len * w.Hq * (w.D_qk + w.D_v)
        line["tensor"] = {"tflops": flops / (attn_ms * 1e-3) / 1e12, "flops_per_launch": flops}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload to time (the bench line is the default one; others are "
                         "for per-workload tables and profiling)")
    ap.add_argument("--batch", type=int, default=None, help="override the batch size")
    ap.add_argument("--with-append", action="store_true",
                    help="each step writes the new tokens' K/V (zl_kv_append) before attending")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="pass the workload's shared prefix pages (read once per group)")
    ap.add_argument("--single-launch", action="store_true",
                    help="GQA: merge split-KV partials inside the attention kernel")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence (llama3_8b_decode, mla_decode)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        args.steps = 5 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        run_reference(args, world, rank)
    else:
        args.steps = 10000 if args.steps is None else args.steps
        args.warmup = 20 if args.warmup is None else args.warmup
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
