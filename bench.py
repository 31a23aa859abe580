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


def time_oracle(w, min_seconds=10.0, max_calls=50, threads=None):
    """The oracle as it stands, on all host cores (or `threads` of them):
    (seconds per call, calls, threads, the last call's result)."""
    import oracle
    orc = oracle.load()
    threads = cpu_cores() if threads is None else threads
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


class Case:
    """One workload on the device, ready to call: inputs, output buffers, the
    C-ABI params and workspace, the optional KV append and L2 flush."""

    def __init__(self, w, dev, *, single_launch=False, shared_prefix=False, with_append=False,
                 hint=True, fused_append=False):
        import paged_decode_attention_gqa_gb300 as zl
        self.zl, self.w, self.dev = zl, w, dev
        self.kind = "mla" if w.mla else "gqa"
        self.q, self.k = w.q.to(dev), w.k_pool.to(dev)
        self.v = None if w.mla else w.v_pool.to(dev)
        self.bt = torch.from_numpy(w.block_table).to(dev)
        self.sl = torch.from_numpy(w.seq_lens).to(dev)
        self.out = torch.empty(w.B, w.q_len, w.Hq, w.D_v, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(w.B, w.q_len, w.Hq, dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.npref = 0
        if shared_prefix:
            self.npref = int(w.notes.get("shared_prefix_tokens", 0)) // w.page_size
            assert self.npref > 0, "--shared-prefix needs a workload with a shared prefix"
        self.single_launch = single_launch and not w.mla
        self.max_seq_len = w.max_seq_len if hint else 0
        # fused_append: each step's decode call itself first stores the q_len new
        # tokens' K/V rows (k_new / v_new in the params): one launch less.
        self.k_new = self.v_new = None
        if fused_append:
            from paged_decode_attention_gqa_gb300 import workloads as _wl
            k_new, v_new = _wl.new_token_rows(w.seed, w.B, w.q_len, w.Hkv, w.D_qk,
                                              None if w.mla else w.D_v)
            self.k_new = k_new.to(dev)
            self.v_new = None if v_new is None else v_new.to(dev)
        self.fused_append = fused_append
        self.p = zl.make_params(self.q, self.k, self.v, self.bt, self.sl, self.out,
                                page_size=w.page_size, scale=w.scale, Hkv=w.Hkv, D_v=w.D_v,
                                lse=self.lse, err_flags=self.err, max_seq_len=self.max_seq_len,
                                single_launch=self.single_launch, shared_prefix_pages=self.npref,
                                k_new=self.k_new, v_new=self.v_new)
        need = zl.workspace_size_mla(self.p) if w.mla else zl.workspace_size(self.p)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        self.p.workspace, self.p.workspace_bytes = self.ws.data_ptr(), self.ws.numel()
        self.stream = torch.cuda.current_stream()
        self.stream_ptr = ctypes.c_void_p(self.stream.cuda_stream)
        # Small working sets are flushed from L2 between steps (a 2x L2 write).
        self.flush = None
        if kv_bytes(w) <= 4 * 129e6:
            self.flush = torch.empty(int(2 * 129e6) // 4, dtype=torch.int32, device=dev)
        # with_append: each step first writes the q_len new tokens' K/V rows
        # into their page slots (zl_kv_append), then attends, as a decode step does.
        self.ap = None
        if with_append:
            from paged_decode_attention_gqa_gb300 import workloads as _wl
            k_new, v_new = _wl.new_token_rows(w.seed, w.B, w.q_len, w.Hkv, w.D_qk,
                                              None if w.mla else w.D_v)
            self.k_new = k_new.to(dev)
            self.v_new = None if v_new is None else v_new.to(dev)
            self.ap = zl.make_append_params(self.k_new, self.v_new, self.k, self.v, self.bt,
                                            self.sl, page_size=w.page_size, layout=w.layout,
                                            err_flags=self.err)

    def call(self):
        if self.ap is not None:
            rc = self.zl.lib().zl_kv_append(ctypes.byref(self.ap), self.stream_ptr)
            assert rc == self.zl.OK, rc
        self.zl.call(self.p, mla=self.w.mla, stream=self.stream)

    def step(self):
        if self.flush is not None:
            self.flush.zero_()
        self.call()

    def check_errors(self):
        assert int(self.err.item()) == 0, f"device error flags {int(self.err.item())}"

    def launches_per_step(self):
        n = 2 if self.w.mla else self.zl.launches(self.p)
        if self.ap is not None:
            n += 1  # the KV append
        if self.flush is not None:
            n += 1  # the L2 flush memset
        return n

    def time_steps(self, steps):
        """Mean ms per step over `steps` steps, CUDA events on the launching
        stream. With an L2 flush between steps, each step's call is timed on
        its own (events after the flush, around the call)."""
        stream = self.stream
        t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        step_evs = ([(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                     for _ in range(steps)] if self.flush is not None else None)
        t_begin.record(stream)
        for i in range(steps):
            if self.flush is None:
                self.call()
            else:
                self.flush.zero_()
                step_evs[i][0].record(stream)
                self.call()
                step_evs[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if self.flush is None:
            return t_begin.elapsed_time(t_end) / steps
        return sum(a.elapsed_time(b) for a, b in step_evs) / steps

    def time_kernel(self, n_ev):
        """(attention-kernel ms, whole-call ms): the library records events
        around the attention kernel alone, the bench around the call. Events
        between the two launches would keep the merge from starting early, so
        the timed steps carry none; this is a separate pass."""
        stream = self.stream
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_ev)]
        # torch only reports elapsed time for events it has recorded itself;
        # record each once here, the library re-records them around the kernel.
        for a, b in evs:
            a.record(stream)
            b.record(stream)
        call_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(n_ev)]
        for i in range(n_ev):
            self.p.attn_begin, self.p.attn_end = evs[i][0].cuda_event, evs[i][1].cuda_event
            if self.flush is not None:
                self.flush.zero_()
            call_evs[i][0].record(stream)
            self.call()
            call_evs[i][1].record(stream)
        torch.cuda.synchronize()
        self.p.attn_begin = self.p.attn_end = None
        return (statistics.mean(a.elapsed_time(b) for a, b in evs),
                statistics.mean(a.elapsed_time(b) for a, b in call_evs))

    def host_enqueue_us(self, n_host=32):
        """Host time to issue one call: a burst short enough that the launch
        queue never fills (a long loop would pace the host at the GPU's rate)."""
        h0 = time.perf_counter()
        for _ in range(n_host):
            self.call()
        us = (time.perf_counter() - h0) / n_host * 1e6
        torch.cuda.synchronize()
        return us

    def time_append(self, n_ev):
        w = self.w
        app_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n_ev)]
        for a, b in app_evs:
            if self.flush is not None:
                self.flush.zero_()
            a.record(self.stream)
            self.zl.lib().zl_kv_append(ctypes.byref(self.ap), self.stream_ptr)
            b.record(self.stream)
        torch.cuda.synchronize()
        app_ms = statistics.mean(a.elapsed_time(b) for a, b in app_evs)
        # new rows read once, written once into the pools
        app_bytes = 2 * w.B * w.q_len * w.Hkv * (w.D_qk + (0 if w.mla else w.D_v)) * 2
        return {"us_per_launch": app_ms * 1e3, "bytes_per_launch": app_bytes,
                "GBs": app_bytes / (app_ms * 1e-3) / 1e9,
                "note": "zl_kv_append alone, L2 flushed first when the step flushes"}

    def e2e(self, steps, warm, world):
        """End to end through the public API: host inputs in, host result out.
        Every step copies its inputs (q, block table, seq_lens) in from pinned
        host memory and its output back; steps are pipelined the way a serving
        loop overlaps them: two device buffer sets, inputs copied on one stream,
        the call on another, the output copied out on a third, ordered by
        events. `warm` pipelined steps run first, untimed, so that the
        pipeline is full and the streams and events are warm."""
        zl, w = self.zl, self.w
        pin_q = w.q.pin_memory()
        pin_bt = torch.from_numpy(w.block_table).pin_memory()
        pin_sl = torch.from_numpy(w.seq_lens).pin_memory()
        pin_out = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
                   for _ in range(2)]
        dq = [self.q, torch.empty_like(self.q)]
        dbt = [self.bt, torch.empty_like(self.bt)]
        dsl = [self.sl, torch.empty_like(self.sl)]
        dout = [self.out, torch.empty_like(self.out)]
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        h2d = pin_q.numel() * 2 + pin_bt.numel() * 4 + pin_sl.numel() * 4
        d2h = pin_out[0].numel() * 2
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        torch.cuda.synchronize()
        for e in ev_comp + ev_out:
            e.record(s_comp)

        def one(i):
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
                if self.flush is not None:
                    self.flush.zero_()
                if w.mla:
                    zl.decode_attn_mla(dq[j], self.k, dbt[j], dsl[j], page_size=w.page_size,
                                       scale=w.scale, D_v=w.D_v, out=dout[j], workspace=self.ws,
                                       max_seq_len=self.max_seq_len, stream=s_comp)
                else:
                    zl.decode_attn(dq[j], self.k, self.v, dbt[j], dsl[j], page_size=w.page_size,
                                   scale=w.scale, out=dout[j], workspace=self.ws,
                                   max_seq_len=self.max_seq_len,
                                   single_launch=self.single_launch,
                                   shared_prefix_pages=self.npref, stream=s_comp)
                ev_comp[j].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[j])
                pin_out[j].copy_(dout[j], non_blocking=True)
                ev_out[j].record(s_out)

        for i in range(warm):
            one(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(warm, warm + steps):
            one(i)
        torch.cuda.synchronize()
        e2e_s = (time.perf_counter() - t0) / steps
        return {"value": kv_bytes(w) * world / e2e_s / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": e2e_s * 1e6, "steps": steps, "warmup_steps": warm,
                "note": "every step copies q, block table and seq_lens in from pinned host memory "
                        "and its output back (host wall clock, after the warm-up steps); steps "
                        "pipelined over two buffer sets and three streams; the KV cache is "
                        "device-resident state"
                        + ("; includes the L2 flush" if self.flush is not None else "")}


def roofline_bytes(w):
    """(algorithmic bytes per launch, logical bytes per launch): the bytes HBM
    has to deliver count a shared page once; logical counts every sequence's
    reads."""
    return unique_kv_bytes(w) + io_bytes(w), kv_bytes(w) + io_bytes(w)


def mla_flops(w):
    return 2.0 * int(w.seq_lens.astype(np.int64).sum()) * w.q_len * w.Hq * (w.D_qk + w.D_v)


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    return 1900.0, "fallback (burst)"


# Every other seeded configuration, timed in the same process after the
# headline (each entry: name, workload, Case options).
EXTRA_WORKLOADS = [
    ("tiny_gqa", "tiny_gqa", {}),
    ("tiny_gqa (no max_seq_len)", "tiny_gqa", {"hint": False}),
    ("llama70b_prefix_decode", "llama70b_prefix_decode", {}),
    ("llama70b_prefix_decode (shared prefix)", "llama70b_prefix_decode",
     {"shared_prefix": True}),
    ("long_context_decode", "long_context_decode", {}),
    ("mla_decode", "mla_decode", {}),
    ("mqa32_decode", "mqa32_decode", {}),
    ("mqa32_decode (no max_seq_len)", "mqa32_decode", {"hint": False}),
]


def measure_extra(dev, steps, warmup, oracle_seconds):
    """The other seeded configurations at full size: per call and per
    attention kernel, algorithmic bytes and roofline fraction, parity of the
    whole output against the oracle, and the oracle's own rate on the host."""
    peak, peak_kind = measured_peaks()
    tpeak, tpeak_kind = bf16_peak()
    entries = {}
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    cache = {}
    for label, name, opts in EXTRA_WORKLOADS:
        w = cache.get(name) or make_workload(name)
        cache = {name: w}  # keep one workload's host copy at a time
        c = Case(w, dev, **opts)
        for _ in range(warmup):
            c.step()
        torch.cuda.synchronize()
        c.check_errors()
        ms = c.time_steps(steps)
        attn_ms, call_ms = c.time_kernel(max(10, min(steps, 200)))
        c.check_errors()
        algo, logical = roofline_bytes(w)
        cpu_s, cpu_calls, cores, res = time_oracle(w, min_seconds=oracle_seconds, max_calls=3)
        e = {"us_per_step": ms * 1e3, "us_per_call": call_ms * 1e3,
             "attn_us_per_launch": attn_ms * 1e3,
             "kv_GBs_per_step": kv_bytes(w) / (ms * 1e-3) / 1e9,
             "algorithmic_bytes_per_launch": algo,
             "roofline_frac": (algo / (attn_ms * 1e-3) / 1e9) / peak,
             "launches_per_step": c.launches_per_step(),
             "config": config_of(w, 1),
             "parity": parity_summary(c.out, c.lse, res),
             "oracle": {"GBs": kv_bytes(w) / cpu_s / 1e9, "us_per_call": cpu_s * 1e6,
                        "cores": cores, "calls": cpu_calls, "kind": "oracle",
                        "sample": "the whole workload per call"}}
        if logical != algo:
            e["logical_bytes_per_launch"] = logical
            e["logical_GBs_attn"] = logical / (attn_ms * 1e-3) / 1e9
            e["roofline_note"] = ("roofline_frac counts each distinct cache row once (the bytes "
                                  "HBM must deliver); the shared prefix is served from L2, so "
                                  "logical_GBs_attn is the rate the kernel consumes K/V at")
        if opts.get("shared_prefix"):
            e["shared_prefix_pages"] = c.npref
        if not opts.get("hint", True):
            e["max_seq_len"] = "not given (split plan decided on the device)"
        if w.mla:
            fl = mla_flops(w)
            e["tensor"] = {"tflops": fl / (attn_ms * 1e-3) / 1e12, "flops_per_launch": fl,
                           "frac_of_bf16_peak": fl / (attn_ms * 1e-3) / 1e12 / tpeak,
                           "peak_tflops": tpeak, "peak_kind": tpeak_kind}
        entries[label] = e
        del c
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    return {"entries": entries, "peak_GBs": peak, "peak_kind": peak_kind, "clocks": clocks,
            "steps": steps, "warmup": warmup,
            "note": "each entry timed in this process after the headline, full-size inputs; "
                    "us_per_step over the timed steps (L2 flushed between steps when the KV "
                    "working set is under 4 x L2), attn_us_per_launch from events the library "
                    "records around the attention kernel; parity is the whole output of the "
                    "last call against the fp64 oracle"}


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
    c = Case(w, dev, single_launch=args.single_launch, shared_prefix=args.shared_prefix,
             with_append=args.with_append, hint=not args.no_hint,
             fused_append=args.fused_append)
    kind = c.kind

    for _ in range(max(args.warmup, 3)):
        c.step()
    torch.cuda.synchronize()
    c.check_errors()

    # ---- timed region: K steps, CUDA events on the launching stream, clocks sampled
    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.4)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms = c.time_steps(args.steps)
    clocks = sampler.stop()
    ms = max_over_ranks(ms, world, dev)
    # the library's own count per call: attention (+ merge) per token group
    launches = args.steps * c.launches_per_step()

    # ---- per-kernel timing, after the timed region
    attn_ms, call_ms = c.time_kernel(max(10, min(args.steps, 1000)))
    host_us = c.host_enqueue_us()
    append = c.time_append(max(10, min(args.steps, 1000))) if c.ap is not None else None
    c.check_errors()

    # ---- end to end through the public API (steady state: the pipeline is
    # warmed up first, then at least 200 steps are timed)
    e2e = None
    if not args.no_e2e:
        e2e = c.e2e(max(200, min(args.steps, 2000)), 20, world)

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    kvb = kv_bytes(w)
    peak, peak_kind = measured_peaks()
    algo, logical = roofline_bytes(w)
    achieved = algo / (attn_ms * 1e-3) / 1e9
    cpu = None
    parity = None
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline is an N = 1 figure
        cpu_s, cpu_calls, cores, res = time_oracle(w)
        cpu = {"value": kvb / cpu_s / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"the whole workload per call, {cpu_calls} calls (median)"}
        # the same oracle on one core, for the scaling of the host baseline
        one_s, one_calls, _, _ = time_oracle(w, min_seconds=3.0, max_calls=3, threads=1)
        cpu["single_core"] = {"value": kvb / one_s / 1e9, "unit": UNIT, "cores": 1,
                              "sample": f"the whole workload per call, {one_calls} calls "
                                        "(median)"}
        if c.ap is None and not c.fused_append:  # (an append puts the new rows in the pools)
            parity = parity_summary(c.out, c.lse, res)
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
        "config": config_of(w, world),
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
        "clocks": clocks,
    }
    # options that change what a step is are named only when used
    if kind == "gqa" and args.single_launch:
        line["config"]["split_merge"] = "in the attention kernel (single launch)"
    if c.ap is not None:
        line["config"]["step"] = "kv append + attention"
        line["kv_append"] = append
    if c.fused_append:
        line["config"]["step"] = "kv append fused into the attention launch + attention"

    if c.npref:
        line["config"]["shared_prefix_pages"] = c.npref
    if args.no_hint:
        line["config"]["max_seq_len"] = "not given"
    if w.mla:
        fl = mla_flops(w)
        tpeak, tpeak_kind = bf16_peak()
        line["tensor"] = {"tflops": fl / (attn_ms * 1e-3) / 1e12, "flops_per_launch": fl,
                          "frac_of_bf16_peak": fl / (attn_ms * 1e-3) / 1e12 / tpeak,
                          "peak_kind": tpeak_kind}
    if not args.no_workloads and world == 1 and args.workload == WORKLOAD and args.q_len == 1 \
            and not (args.single_launch or args.with_append or args.shared_prefix or args.no_hint
                     or args.batch or args.fused_append):
        del c
        torch.cuda.empty_cache()
        line["workloads"] = measure_extra(dev, 200, 5, oracle_seconds=3.0)
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
    ap.add_argument("--fused-append", action="store_true",
                    help="each step's decode call stores the new tokens' K/V itself (k_new / "
                         "v_new), then attends, in one launch")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="pass the workload's shared prefix pages (read once per group)")
    ap.add_argument("--single-launch", action="store_true",
                    help="GQA: merge split-KV partials inside the attention kernel")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence (llama3_8b_decode, mla_decode)")
    ap.add_argument("--no-hint", action="store_true",
                    help="pass no max_seq_len (the split plan is then decided on the device)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="headline only: skip timing the other seeded configurations")
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
