"""Benchmark of the NVFP4 lightning indexer step on GB300.

One step = the whole hot path over one batch: NVFP4 insert of the step's new
keys, the decode indexer over every decode request, the prefill indexer over
every prefill chunk.  Default workload: the long-context mixed step (16
decode requests at a 131072-token context with 8 queries each, plus 2 prefill
chunks of 8192 new tokens on 65536-token histories, 8 index heads), the only
named configuration that runs every step of the path; the cache holds all
2.24 M keys, written once before timing.

Metric: indexer pages scored per second = sum over (query row, head) of the
history pages scored, per second of step time.  Timing: CUDA events on the
launching stream around each step (and around each kernel, for the roofline),
L2 flushed (a 2 x L2 write) between steps, W warm-up steps first.

Besides the step, the line carries timings taken apart from it: the
whole-cache inserts, MXFP4-page calls, the block-sparse attend over the
decode rows' selected pages (``kernels.attend_decode``), and a ``workloads``
record with every other named workload's kernels (time, achieved rate,
fraction of the measured peak) beside the oracle's pages/s on a short
sample of it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--sweep] [--no-workloads] [--no-attend]

Prints ONE JSON line on rank 0.  Under torchrun each rank runs its own full
batch (weak scaling, no data-path collective); value = all ranks' pages /
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_INDEX = {"tiny_decode": 0, "decode_batch": 1, "spec_decode": 2, "ragged_prefill": 3, "long_mixed": 4}
KERNEL_SOURCES = ["csrc/prefill.cu", "csrc/decode.cu", "csrc/insert.cu", "csrc/ptx.cuh", "csrc/codec.cuh",
                  "csrc/topk.cuh", "csrc/internal.h"]
# the files each timed kernel is compiled from (its own .cu and the headers it includes)
_HEADERS = ["csrc/ptx.cuh", "csrc/codec.cuh", "csrc/topk.cuh", "csrc/internal.h"]
KERNEL_DEPS = {"prefill": ["csrc/prefill.cu"] + _HEADERS, "decode": ["csrc/decode.cu"] + _HEADERS,
               "insert": ["csrc/insert.cu", "csrc/codec.cuh", "csrc/internal.h"],
               "attend": ["csrc/attend.cu", "csrc/internal.h"]}


# ----------------------------------------------------------------------------- host-side logic
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(kernel: str = None) -> str:
    """Hash of the kernel sources: all of them, or those `kernel` is built from."""
    h = hashlib.sha256()
    for rel in (KERNEL_DEPS[kernel] if kernel else KERNEL_SOURCES):
        h.update(open(os.path.join(ROOT, "sparse_attention_block_nvfp4_gb300", rel), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel's current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == workload and parts[2] == cur:
            return float(parts[3])
    return None


def work_counts(w: workloads.Workload) -> dict:
    """Algorithmic work of one step (history pages only; the local page is not scored)."""
    H = w.num_heads
    out = {}
    # decode
    seq = w.dec_seq_lens.astype(np.int64)
    ql = w.query_len
    if w.num_decode_reqs:
        pos = seq[:, None] - ql + np.arange(ql)[None, :]
        hist_rows = np.where(pos >= 0, pos // 128, 0)                  # pages per (row)
        req_pages = np.where(seq >= 1, (seq - 1) // 128, 0)           # pages read per request
        R = ql * H
        out["dec_pages_scored"] = int(hist_rows.sum()) * H
        out["dec_bytes"] = int(req_pages.sum()) * (9216 + 4) + w.num_decode_reqs * (R * 128 + R * 64 + 4)
        # the same over MXFP4 pages (8704 bytes)
        out["dec_bytes_mx"] = int(req_pages.sum()) * (8704 + 4) + w.num_decode_reqs * (R * 128 + R * 64 + 4)
        out["dec_flops"] = int(req_pages.sum()) * 2 * 128 * 128 * R
    else:
        out.update(dec_pages_scored=0, dec_bytes=0, dec_bytes_mx=0, dec_flops=0)
    # prefill
    if w.num_prefill_reqs:
        tot = 0
        for s, q in zip(w.pre_seq_lens.astype(np.int64), w.pre_query_lens.astype(np.int64)):
            pos = s - q + np.arange(q)
            tot += int(np.where(pos >= 0, pos // 128, 0).sum())
        out["pre_pages_scored"] = tot * H
        out["pre_flops"] = tot * H * 2 * 128 * 128
    else:
        out.update(pre_pages_scored=0, pre_flops=0)
    out["pages_scored"] = out["dec_pages_scored"] + out["pre_pages_scored"]
    return out


def step_new_tokens(w: workloads.Workload) -> np.ndarray:
    """Indices (into w.k_bf16) of the keys a step inserts: the decode queries'
    own tokens and the prefill chunks' new tokens (the rest is history)."""
    seq = w.seq_lens.astype(np.int64)
    start = np.concatenate([[0], np.cumsum(np.maximum(seq, 0))])
    idx = []
    for r in range(w.num_decode_reqs):
        idx.append(np.arange(start[r + 1] - min(w.query_len, seq[r]), start[r + 1]))
    for k in range(w.num_prefill_reqs):
        r = w.num_decode_reqs + k
        idx.append(np.arange(start[r + 1] - w.pre_query_lens[k], start[r + 1]))
    return np.concatenate(idx) if idx else np.zeros(0, np.int64)


def aggregate(per_rank_pages, per_rank_seconds) -> float:
    """Whole-job throughput: all ranks' work over the slowest rank's time."""
    return float(sum(per_rank_pages)) / float(max(per_rank_seconds))


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's value (all ranks get it); identity for one rank."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as tdist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle samples every 100 ms while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm
def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class GpuStep:
    """Device-resident inputs of one workload and the three library calls."""

    def __init__(self, w, device):
        import torch
        import sparse_attention_block_nvfp4_gb300 as idx
        self.idx, self.torch, self.w, self.dev = idx, torch, w, device
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
        self.kv = torch.zeros((w.num_blocks, 128, 72), dtype=torch.uint8, device=device)
        # the history: every cached key inserted once, outside the timed region
        # (kept on the device: the full-cache fill is also timed on its own)
        self.k_all, self.slot_all = up(w.k_bf16.view(np.int16)), up(w.slot_mapping)
        idx.insert(self.k_all, self.slot_all, self.kv)
        new = step_new_tokens(w)
        self.h_k_new = w.k_bf16[new].view(np.int16)
        self.h_slot_new = w.slot_mapping[new]
        self.k_new, self.slot_new = up(self.h_k_new), up(self.h_slot_new)
        self.plan = idx.Plan(num_heads=w.num_heads, max_reqs=max(1, w.num_decode_reqs),
                             max_query_len=max(1, w.query_len), max_pages_per_req=w.page_table.shape[1],
                             max_prefill_tokens=max(1, w.total_prefill_q),
                             max_prefill_reqs=max(1, w.num_prefill_reqs))
        self.h = dict(q_dec=w.q_decode, q_pre=w.q_prefill, dec_table=w.dec_page_table,
                      pre_table=w.pre_page_table, dec_seq=w.dec_seq_lens, pre_seq=w.pre_seq_lens,
                      cu=w.cu_seqlens_q)
        self.d = {k: up(v) for k, v in self.h.items()}
        rows = w.num_decode_rows + w.total_prefill_q
        self.out = torch.empty((rows, w.num_heads, 16), dtype=torch.int32, device=device)
        self.nd = w.num_decode_rows
        self.max_q = int(w.pre_query_lens.max()) if w.num_prefill_reqs else 0
        # insert; decode scoring + merge; prefill scoring + merge
        self.launches_per_step = (1 if len(new) else 0) + (2 if w.num_decode_reqs else 0) + \
            (2 if w.num_prefill_reqs else 0)

    def run(self, stream, d=None, events=None, k_new=None, slot_new=None, out=None):
        """Enqueue one step; events: dict name -> (start, end) recorded around each kernel."""
        d = d or self.d
        k_new = self.k_new if k_new is None else k_new
        slot_new = self.slot_new if slot_new is None else slot_new
        out = self.out if out is None else out
        w = self.w

        def rec(name, i):
            if events is not None:
                events[name][i].record(stream)
        if k_new.shape[0]:
            rec("insert", 0)
            self.idx.insert(k_new, slot_new, self.kv, stream=stream)
            rec("insert", 1)
        if w.num_decode_reqs:
            rec("decode", 0)
            self.plan.decode(d["q_dec"], self.kv, d["dec_table"], d["dec_seq"], w.query_len,
                             out=out[: self.nd], stream=stream)
            rec("decode", 1)
        if w.num_prefill_reqs:
            rec("prefill", 0)
            self.plan.prefill(d["q_pre"], d["cu"], self.kv, d["pre_table"], d["pre_seq"], self.max_q,
                              out=out[self.nd:], stream=stream)
            rec("prefill", 1)


def gpu_arm(args, w, rank, world, local):
    import torch
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    st = GpuStep(w, dev)
    work = work_counts(w)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) if args.flush else 1, dtype=torch.uint8, device=dev)
    names = ["insert", "decode", "prefill"]

    def new_events():
        return {n: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for n in names}

    for _ in range(args.warmup):
        flush.fill_(1)
        st.run(stream)
    torch.cuda.synchronize()
    if st.plan.status() != 0:
        raise RuntimeError("device status set during warm-up")

    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize()
    step_ev, kern_ev = [], []
    with ClockSampler(local) as clk:
        for _ in range(args.steps):
            flush.fill_(1)                                   # L2 flush between timed steps
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev = new_events()
            s0.record(stream)
            st.run(stream, events=ev)
            s1.record(stream)
            step_ev.append((s0, s1))
            kern_ev.append(ev)
        torch.cuda.synchronize()
    if world > 1:
        tdist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    ran = {"insert": st.k_new.shape[0] > 0, "decode": w.num_decode_reqs > 0, "prefill": w.num_prefill_reqs > 0}
    kern_ms = {n: [e[n][0].elapsed_time(e[n][1]) for e in kern_ev] for n in names if ran[n]}
    total_s = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    status = st.plan.status()

    # ---- the insert on its own over the whole cache (every key of every
    # request; the same bytes each time), outside the step
    fill_ms = []
    for i in range(4):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st.idx.insert(st.k_all, st.slot_all, st.kv, stream=stream)
        b.record(stream)
        b.synchronize()
        if i > 0:
            fill_ms.append(a.elapsed_time(b))

    # ---- the fused qk-norm + RoPE insert over the whole cache (each
    # request's keys at positions 0 .. seq_len - 1, NeoX RoPE over all 128
    # elements, a seeded synthetic norm weight), into its own pages; outside
    # the step
    nr = None
    if args.norm_rope:
        seq = np.concatenate([w.dec_seq_lens, w.pre_seq_lens]).astype(np.int64)
        h_pos = np.concatenate([np.arange(x, dtype=np.int64) for x in seq])
        max_pos = int(seq.max())
        inv = 10000.0 ** (-np.arange(64, dtype=np.float64) / 64.0)
        ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
        table = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)).to(dev)
        rng_w = np.random.Generator(np.random.PCG64(7))
        wts = torch.from_numpy(rng_w.uniform(0.5, 1.5, 128).astype(np.float32)).to(torch.bfloat16).to(dev)
        pos_d = torch.from_numpy(h_pos).to(dev)
        rope_pages = torch.zeros_like(st.kv)
        nr = {"ms": [], "keys": int(h_pos.size), "table_bytes": max_pos * 128 * 4}
        for i in range(4):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            st.idx.insert_norm_rope(st.k_all, pos_d, st.slot_all, wts, 1e-6, table, 128, True, rope_pages,
                                    stream=stream)
            b.record(stream)
            b.synchronize()
            if i > 0:
                nr["ms"].append(a.elapsed_time(b))
        del rope_pages, table, pos_d

    # ---- MXFP4 pages: the same decode / prefill calls over an MXFP4 copy of
    # the cache (filled by mxfp4_insert, timed like the NVFP4 fill), each
    # call timed alone with the L2 flushed before it; not part of the step
    mx = None
    if args.mxfp4:
        idx = st.idx
        pages = torch.zeros((w.num_blocks, 8704), dtype=torch.uint8, device=dev)
        mx = {"fill": []}

        def timed(fn, key, reps):
            for i in range(reps):
                flush.fill_(1)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                if key is not None and i >= 3:
                    mx.setdefault(key, []).append(a.elapsed_time(b))
        for i in range(4):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            idx.mxfp4_insert(st.k_all, st.slot_all, pages, stream=stream)
            b.record(stream)
            b.synchronize()
            if i > 0:
                mx["fill"].append(a.elapsed_time(b))
        d = st.d
        reps = 3 + max(3, min(args.steps, 50))
        if w.num_decode_reqs:
            timed(lambda: st.plan.decode_mxfp4(d["q_dec"], pages, d["dec_table"], d["dec_seq"], w.query_len,
                                               out=st.out[: st.nd], stream=stream), "decode", reps)
        if w.num_prefill_reqs:
            timed(lambda: st.plan.prefill_mxfp4(d["q_pre"], d["cu"], pages, d["pre_table"], d["pre_seq"],
                                                st.max_q, out=st.out[st.nd:], stream=stream), "prefill", reps)
        torch.cuda.synchronize()
        mx["status"] = st.plan.status()
        del pages

    # ---- end to end: host buffers in, ids out, through the same C ABI calls.
    # Every step copies its inputs from pinned host memory and reads its ids
    # back inside the timed region, pipelined as a serving loop runs it: two
    # device buffer sets; a copy stream uploads step i + 1's inputs and reads
    # step i's ids back while the compute stream runs the next step.  No L2
    # flush inside the pipeline: a step reads more than L2 holds (the decode
    # history alone is larger).
    e2e = None
    if args.e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        hin = {k: pin(v) for k, v in st.h.items()}
        hk, hs = pin(st.h_k_new), pin(st.h_slot_new)
        sets = [dict(d={k: torch.empty_like(v) for k, v in st.d.items()}, k=torch.empty_like(st.k_new),
                     s=torch.empty_like(st.slot_new), out=torch.empty_like(st.out),
                     h_out=torch.empty(st.out.shape, dtype=torch.int32).pin_memory()) for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in hin.values()) + hk.numel() * 2 + hs.numel() * 8
        d2h = st.out.numel() * 4
        copy = torch.cuda.Stream(device=dev)
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]

        def upload(b):
            for k in hin:
                sets[b]["d"][k].copy_(hin[k], non_blocking=True)
            sets[b]["k"].copy_(hk, non_blocking=True)
            sets[b]["s"].copy_(hs, non_blocking=True)
            ev_in[b].record(copy)

        def pipeline(n):
            with torch.cuda.stream(copy):
                upload(0)
            for i in range(n):
                b = i & 1
                stream.wait_event(ev_in[b])
                st.run(stream, d=sets[b]["d"], k_new=sets[b]["k"], slot_new=sets[b]["s"], out=sets[b]["out"])
                ev_done[b].record(stream)
                with torch.cuda.stream(copy):
                    if i + 1 < n:
                        if i >= 1:
                            copy.wait_event(ev_done[b ^ 1])     # step i - 1 is done with that set
                        upload(b ^ 1)
                    copy.wait_event(ev_done[b])
                    sets[b]["h_out"].copy_(sets[b]["out"], non_blocking=True)

        pipeline(max(args.warmup, 2))                            # warm-up, untimed
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(copy)
        pipeline(args.steps)
        stream.wait_stream(copy)
        copy.wait_stream(stream)
        t1.record(copy)
        t1.synchronize()
        e2e_s = max_over_ranks(t0.elapsed_time(t1) / 1e3, world, dev)
        e2e = {"value": work["pages_scored"] * args.steps * world / e2e_s, "unit": "pages/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "pipelined": "step i+1 uploaded and step i read back on a copy stream while the next step runs",
               "l2": "not flushed inside the pipeline (a step reads more than L2 holds)"}
    att = attend_leg(st, w, dev, flush, stream) if getattr(args, "attend", False) else None
    return dict(st=st, work=work, step_ms=step_ms, kern_ms=kern_ms, total_s=total_s, clk=clk.summary(),
                e2e=e2e, status=status, fill_ms=sorted(fill_ms)[len(fill_ms) // 2], mx=mx, nr=nr, att=att,
                num_sms=torch.cuda.get_device_properties(dev).multi_processor_count)


def roofline_block(res, w, wname, peaks, peak_kind):
    work, km = res["work"], res["kern_ms"]
    avg = {n: (sum(v) / len(v) if v else 0.0) for n, v in km.items()}
    avg = {n: avg.get(n, 0.0) for n in ("insert", "decode", "prefill")}
    n_new = res["st"].k_new.shape[0]
    kernels = {}
    if avg.get("prefill"):
        tf = work["pre_flops"] / (avg["prefill"] / 1e3) / 1e12
        kernels["prefill"] = {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                              "frac": tf / peaks["bf16_tflops"], "ms": avg["prefill"],
                              "traffic": recorded_traffic("prefill", wname)}
    if avg.get("decode"):
        gb = work["dec_bytes"] / (avg["decode"] / 1e3) / 1e9
        kernels["decode"] = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gb / peaks["hbm_gbs"], "ms": avg["decode"],
                             "tensor_tflops": work["dec_flops"] / (avg["decode"] / 1e3) / 1e12,
                             "traffic": recorded_traffic("decode", wname)}
    if avg.get("insert"):
        gb = n_new * (256 + 8 + 72) / (avg["insert"] / 1e3) / 1e9
        kernels["insert"] = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": gb / peaks["hbm_gbs"], "ms": avg["insert"],
                             "traffic": recorded_traffic("insert", wname)}
    n_all = res["st"].k_all.shape[0]
    if res.get("fill_ms"):
        gb = n_all * (256 + 8 + 72) / (res["fill_ms"] / 1e3) / 1e9
        kernels["insert_fill"] = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": gb / peaks["hbm_gbs"], "ms": res["fill_ms"], "keys": int(n_all),
                                  "note": "whole-cache insert, timed apart from the step"}
    nr = res.get("nr")
    if nr and nr["ms"]:
        ms = sorted(nr["ms"])[len(nr["ms"]) // 2]
        gb = (nr["keys"] * (256 + 8 + 8 + 72) + nr["table_bytes"]) / (ms / 1e3) / 1e9
        kernels["insert_norm_rope_fill"] = {
            "bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gb / peaks["hbm_gbs"],
            "ms": ms, "keys": nr["keys"],
            "note": "whole-cache fused qk-norm + RoPE (NeoX, rotary_dim 128) + NVFP4 insert; bytes: "
                    "key, slot, position and row per token plus the cos/sin table once"}
    mx = res.get("mx")
    if mx:
        med = lambda v: sorted(v)[len(v) // 2]
        if mx.get("prefill"):
            ms = sum(mx["prefill"]) / len(mx["prefill"])
            tf = work["pre_flops"] / (ms / 1e3) / 1e12
            kernels["prefill_mxfp4"] = {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                                        "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"], "ms": ms,
                                        "note": "MXFP4 pages, bf16 operands; timed alone, not part of the step"}
        if mx.get("decode"):
            ms = sum(mx["decode"]) / len(mx["decode"])
            gb = work["dec_bytes_mx"] / (ms / 1e3) / 1e9
            kernels["decode_mxfp4"] = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": gb / peaks["hbm_gbs"], "ms": ms,
                                       "note": "MXFP4 pages (8704 B); timed alone, not part of the step"}
        if mx.get("fill"):
            ms = med(mx["fill"])
            gb = n_all * (256 + 8 + 68) / (ms / 1e3) / 1e9
            kernels["insert_fill_mxfp4"] = {"bound": "hbm", "achieved": gb, "peak": peaks["hbm_gbs"],
                                            "unit": "GB/s", "frac": gb / peaks["hbm_gbs"], "ms": ms,
                                            "keys": int(n_all), "note": "whole-cache MXFP4 insert"}
    att = res.get("att")
    if att:
        kernels["attend_decode"] = dict(att, peak=peaks["hbm_gbs"], frac=att["achieved"] / peaks["hbm_gbs"])
    # the tensor pipes' own dense rate at the sampled clock, next to the
    # cuBLAS-measured burst (a tuned kernel can exceed what cuBLAS reached)
    tp = tensor_issue_peak((res.get("clk") or {}).get("sm_mhz"), res.get("num_sms", 0))
    for k in ("prefill", "prefill_mxfp4"):
        if k in kernels and tp:
            kernels[k]["peak_issue"] = tp
            kernels[k]["frac_issue"] = kernels[k]["achieved"] / tp
    step_kernels = ("insert", "decode", "prefill")
    dom = max((k for k in kernels if k in step_kernels), key=lambda k: kernels[k]["ms"])
    rl = dict(kernels[dom])
    rl.pop("ms", None)
    rl.pop("tensor_tflops", None)
    rl["kernel"] = dom
    rl["peak_source"] = f"{peak_kind} ({'bf16 dense burst; fp16 has the same dense rate' if rl['unit'] == 'TFLOP/s' else 'copy bandwidth'})"
    if "peak_issue" in rl:
        rl["peak_issue_source"] = ("8192 flop per clock per SM (dense fp16 MMA rate) x SMs x median sampled "
                                   "SM clock; frac_issue = achieved / peak_issue")
    return rl, kernels


# ----------------------------------------------------------------------------- CPU oracle arm
class OracleSampler:
    """Time the CPU oracle on bounded samples of the workload's step.  The
    history of one sampled decode request and one sampled prefill chunk is
    inserted once (the resident cache; not timed); each unit then quantises
    that request's new keys and scores and selects its rows: the decode
    request's query rows, or 32 rows of the prefill chunk."""

    def __init__(self, w, rng_seed: int = 0):
        from oracle import nvfp4 as onvfp4
        self.w = w
        self.rng = np.random.Generator(np.random.PCG64(rng_seed))
        seq = w.seq_lens.astype(np.int64)
        self.seq = seq
        self.start = np.concatenate([[0], np.cumsum(np.maximum(seq, 0))])
        self.kv = np.zeros((w.num_blocks, 128, 72), np.uint8)
        self.dr = int(self.rng.integers(w.num_decode_reqs)) if w.num_decode_reqs else None
        self.pr = int(self.rng.integers(w.num_prefill_reqs)) if w.num_prefill_reqs else None
        for r in ([self.dr] if self.dr is not None else []) + \
                 ([w.num_decode_reqs + self.pr] if self.pr is not None else []):
            a, b = int(self.start[r]), int(self.start[r + 1])
            onvfp4.insert(w.k_bf16[a:b], w.slot_mapping[a:b], self.kv)
        self.turn = 0

    def _unit(self):
        """One unit of oracle work: returns (pages scored, seconds, description)."""
        from oracle import indexer as oidx, nvfp4 as onvfp4
        w, H = self.w, self.w.num_heads
        kinds = [k for k, v in (("decode", self.dr), ("prefill", self.pr)) if v is not None]
        kind = kinds[self.turn % len(kinds)]
        self.turn += 1
        if kind == "decode":
            r = self.dr
            rows = np.arange(r * w.query_len, (r + 1) * w.query_len)
            t0 = time.perf_counter()
            a = int(self.start[r + 1]) - w.query_len
            onvfp4.insert(w.k_bf16[a:int(self.start[r + 1])], w.slot_mapping[a:int(self.start[r + 1])], self.kv)
            res = oidx.decode(w.q_decode, self.kv, w.dec_page_table, w.dec_seq_lens, w.query_len, H, rows=rows)
            return int(np.count_nonzero(~np.isnan(res.S))), time.perf_counter() - t0, \
                f"decode request {r}: {len(rows)} rows x {H} heads"
        k = self.pr
        cu = w.cu_seqlens_q
        rows = np.sort(self.rng.choice(np.arange(cu[k], cu[k + 1]), size=min(32, int(cu[k + 1] - cu[k])),
                                       replace=False))
        t0 = time.perf_counter()
        r = w.num_decode_reqs + k
        toks = int(self.start[r]) + (int(self.seq[r]) - int(w.pre_query_lens[k])) + (rows - cu[k])
        onvfp4.insert(w.k_bf16[toks], w.slot_mapping[toks], self.kv)
        res = oidx.prefill(w.q_prefill, cu, self.kv, w.pre_page_table, w.pre_seq_lens, H, rows=rows)
        return int(np.count_nonzero(~np.isnan(res.S))), time.perf_counter() - t0, \
            f"prefill chunk {k}: {len(rows)} rows x {H} heads"

    def run(self, budget_s: float):
        """Whole units until budget_s of oracle time has passed (at least one)."""
        pages, secs, parts = 0, 0.0, set()
        while True:
            p, s, what = self._unit()
            pages += p
            secs += s
            parts.add(what)
            if secs >= budget_s:
                break
        return pages, secs, "; ".join(sorted(parts))


def cpu_block(w, budget_s):
    pages, secs, what = OracleSampler(w).run(budget_s)
    return {"value": pages / secs if secs else None, "unit": "pages/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": f"{what}; {pages} (row, head, page) scores in {secs:.1f} s, "
                                        f"NumPy float64, BLAS on all host cores"}


def tensor_issue_peak(sm_mhz, num_sms):
    """Dense fp16 / bf16 rate of the tensor pipes at the sampled SM clock:
    8192 flops per clock per SM (one M = 128, N = 256, K = 16 MMA per 128
    clocks; measured 8148 on this GPU with back-to-back MMAs), TFLOP/s."""
    if not sm_mhz:
        return None
    return 8192.0 * num_sms * sm_mhz * 1e6 / 1e12


def workload_record(res, w, wname, peaks, cpu):
    """Per-workload summary: kernel times, achieved rates and fractions of
    the measured peaks, pages scored per second, the oracle's pages/s."""
    work = res["work"]
    _, kernels = roofline_block(res, w, wname, peaks, "measured")
    rec = {"pages_scored_per_step": work["pages_scored"],
           "pages_per_s": work["pages_scored"] * len(res["step_ms"]) / (sum(res["step_ms"]) / 1e3),
           "ms_per_step": sum(res["step_ms"]) / len(res["step_ms"]), "kernels": {}}
    for k in ("decode", "prefill", "insert", "insert_fill"):
        if k in kernels:
            e = kernels[k]
            rec["kernels"][k] = {kk: e[kk] for kk in ("ms", "achieved", "unit", "frac", "bound") if kk in e}
    if cpu is not None:
        rec["oracle_pages_per_s"] = cpu["value"]
        rec["oracle_sample"] = cpu["sample"]
    return rec


def attend_leg(st, w, dev, flush, stream, reps=20):
    """The block-sparse attend over the decode rows' selected pages: bf16
    main cache [num_blocks, 128, H, 128] (K and V, hashed values), one query
    head per KV head, the ids the step's decode just wrote.  Timed alone,
    L2 flushed before each call; not part of the step.  Algorithmic bytes:
    every (request, KV head)'s union of selected pages' visible K and V rows
    once, plus the queries and the fp32 output."""
    import torch
    nd = st.nd
    if nd == 0:
        return None
    H, G = w.num_heads, 1
    req, pos = workloads.attend_rows(w)
    req, pos = req[:nd], pos[:nd]
    kc = workloads.attend_kv_fill(11, 0, w.num_blocks, H, dev)
    vc = workloads.attend_kv_fill(11, 1, w.num_blocks, H, dev)
    q = torch.from_numpy(workloads.attend_q(nd, H * G, np.random.Generator(np.random.PCG64(11))).view(np.int16)).to(dev)
    ids = st.out[:nd].clone()
    d_req, d_pos = torch.from_numpy(req).to(dev), torch.from_numpy(pos).to(dev)
    table = torch.from_numpy(w.page_table).to(dev)
    out = torch.empty((nd, H * G, 128), dtype=torch.float32, device=dev)
    ms = []
    for i in range(3 + reps):
        flush.fill_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        st.idx.sparse_attend(q, kc, vc, table, d_req, d_pos, ids, 128 ** -0.5, out=out, stream=stream)
        b.record(stream)
        b.synchronize()
        if i >= 3:
            ms.append(a.elapsed_time(b))
    ids_np = ids.cpu().numpy()
    uniq, gathered = 0, 0
    for r in range(w.num_decode_reqs):
        rows = np.arange(r * w.query_len, (r + 1) * w.query_len)
        for h in range(H):
            seen = {}
            for t in rows:
                for j in ids_np[t, h]:
                    if j < 0:
                        continue
                    n = min(128, int(pos[t]) - 128 * int(j) + 1)
                    gathered += n
                    seen[int(j)] = max(seen.get(int(j), 0), n)
            uniq += sum(seen.values())
    per_tok = 2 * 128 * 2                                   # K and V rows of one head, bf16
    alg = uniq * per_tok + nd * H * G * 128 * (2 + 4)
    med = sorted(ms)[len(ms) // 2]
    del kc, vc
    return {"bound": "hbm", "ms": med, "achieved": alg / (med / 1e3) / 1e9, "unit": "GB/s",
            "bytes": int(alg), "bytes_gathered_per_unit": int(gathered * per_tok),
            "units": int(nd * H), "q_per_kv": G, "traffic": recorded_traffic("attend", w.name),
            "note": f"the decode rows ({w.num_decode_reqs} requests x {w.query_len} queries, {H} KV heads, "
                    f"one query head each), ids from the step's decode; timed alone, not part of the step"}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long_mixed", choices=list(WORKLOAD_INDEX))
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-mxfp4", dest="mxfp4", action="store_false",
                    help="skip the MXFP4-page timings (kernels decode_mxfp4 / prefill_mxfp4 / insert_fill_mxfp4)")
    ap.add_argument("--no-norm-rope", dest="norm_rope", action="store_false",
                    help="skip the timed whole-cache fused qk-norm + RoPE insert")
    ap.add_argument("--sweep", action="store_true", help="one line per named workload (no e2e / cpu)")
    ap.add_argument("--no-workloads", dest="all_workloads", action="store_false",
                    help="skip the per-workload record of the other named workloads")
    ap.add_argument("--cpu-budget-others", type=float, default=3.0,
                    help="seconds of oracle work per other workload in the per-workload record")
    ap.add_argument("--no-attend", dest="attend", action="store_false",
                    help="skip the timed block-sparse attend over the decode rows")
    ap.add_argument("--no-flush", dest="flush", action="store_false",
                    help="skip the L2 flush (profiling runs only; the timed numbers then see a warm L2)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl" if args.impl == "ours" else "gloo")

    if args.impl == "reference":
        if rank != 0:
            return
        w = workloads.config(WORKLOAD_INDEX[args.workload])
        # each step a bounded sample: whole units (a decode request's rows or
        # 32 rows of a prefill chunk, in turn) until the step's share of about
        # two minutes of oracle time, at most a second, has passed
        per_step = min(1.0, 120.0 / max(1, args.steps + args.warmup))
        sampler = OracleSampler(w)
        for _ in range(args.warmup):
            sampler.run(per_step)
        pages, secs = 0, 0.0
        whats = set()
        for _ in range(args.steps):
            p, s, what = sampler.run(per_step)
            pages += p
            secs += s
            whats.add(what)
        what = "; ".join(sorted(whats))
        v = pages / secs
        line = {"impl": "reference", "metric": "indexer pages scored/s", "value": v, "unit": "pages/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": secs * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": args.workload},
                "cpu_baseline": {"value": v, "unit": "pages/s", "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": f"each step: {what}; NumPy float64 CPU oracle on the host cores"},
                "e2e": {"value": v, "unit": "pages/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    names = list(WORKLOAD_INDEX) if args.sweep else [args.workload]
    peaks, peak_kind = load_peaks()
    for wname in names:
        w = workloads.config(WORKLOAD_INDEX[wname])
        if world > 1:
            # weak scaling: every rank its own batch of the same shape
            w = workloads.config(WORKLOAD_INDEX[wname]) if rank == 0 else _reseeded(wname, rank)
        sweep_args = argparse.Namespace(**vars(args))
        if args.sweep:
            sweep_args.e2e = False
        sweep_args.attend = args.attend and w.num_decode_reqs > 0
        res = gpu_arm(sweep_args, w, rank, world, local)
        work = res["work"]
        value = work["pages_scored"] * args.steps * world / res["total_s"]
        rl, kernels = roofline_block(res, w, wname, peaks, peak_kind)
        line = {
            "metric": "indexer pages scored/s", "value": value, "unit": "pages/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["total_s"] * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16 operands, f32 accumulate", "data": "synthetic",
            "config": {"workload": wname, "shape": w.notes or _describe(w), "num_heads": w.num_heads,
                       "l2": "flushed between timed steps (2 x L2 write)" if args.flush else "not flushed",
                       "pages_scored_per_step": work["pages_scored"]},
            "roofline": rl,
            "kernels": kernels,
            "gpu_launches": res["st"].launches_per_step * args.steps,
            "clocks": res["clk"],
            "device_status": res["status"] | ((res["mx"] or {}).get("status", 0)),
        }
        if res["e2e"] is not None:
            line["e2e"] = res["e2e"]
        if rank == 0 and world == 1 and args.cpu_baseline and not args.sweep:
            line["cpu_baseline"] = cpu_block(w, args.cpu_budget)
        if world == 1 and args.all_workloads and not args.sweep:
            # every named workload: its kernels and the oracle's rate beside them
            recs = {wname: workload_record(res, w, wname, peaks, line.get("cpu_baseline"))}
            del res
            for other in WORKLOAD_INDEX:
                if other == wname:
                    continue
                wo = workloads.config(WORKLOAD_INDEX[other])
                oa = argparse.Namespace(**vars(args))
                oa.e2e = oa.mxfp4 = oa.norm_rope = oa.attend = False
                oa.steps, oa.warmup = min(args.steps, 20), 3
                ro = gpu_arm(oa, wo, rank, world, local)
                line["device_status"] |= ro["status"]
                cpu = cpu_block(wo, args.cpu_budget_others) if args.cpu_baseline else None
                recs[other] = workload_record(ro, wo, other, peaks, cpu)
                del ro
            line["workloads"] = recs
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        tdist.destroy_process_group()


def _describe(w):
    parts = []
    if w.num_decode_reqs:
        parts.append(f"{w.num_decode_reqs} decode req, seq {int(w.dec_seq_lens.min())}..{int(w.dec_seq_lens.max())}, "
                     f"query_len {w.query_len}")
    if w.num_prefill_reqs:
        parts.append(f"{w.num_prefill_reqs} prefill req, new {w.pre_query_lens.tolist()}, "
                     f"seq {w.pre_seq_lens.tolist()}")
    return "; ".join(parts) + f"; H={w.num_heads}, head_dim 128, 128-token NVFP4 pages"


def _reseeded(wname, rank):
    """The same workload shape with another seed (another rank's batch)."""
    import workloads as wl
    w = wl.config(WORKLOAD_INDEX[wname])
    rng = np.random.Generator(np.random.PCG64(1000 + rank))
    q = wl.random_q(w.q_e4m3.shape[0], w.num_heads, rng)
    w.q_e4m3 = q
    return w


if __name__ == "__main__":
    main()
