#!/usr/bin/env python3
"""Benchmark: MLA DCP decode on one GB300 (replicas on N GPUs).

One step = the whole hot path on one batch: the D shard decodes (split-KV
schedule, paged gathers, QK^T + online softmax + PV, split-chunk merge) and the
LSE merge (with the W_UV projection where the workload has one).  The
headline workload is the heaviest one: long context, 32 requests, q_len 2,
128 heads, context U[16384, 32768], DCP D=8 (the D shards are D slices of one
HBM), run as one shard-fused decode launch plus the W_UV projection.  Every
benchmark workload (plain decode D=1 / D=2, MTP, sparse + mixed, long
context; plain decode D=2 and MTP also over an FP8 cache) is measured on both
routes and reported under "configs", each with its own roofline object.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the headline workload.
"""
from __future__ import annotations

import argparse
import json
import math
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

METRIC = "MLA DCP decode query tok/s; KV GB/s & TFLOP/s as % of GB300 roofline"
UNIT = "query tok/s"
FLOPS_PER_KEY_ROW = 2 * (576 + 512)
HEADLINE = "long_context"
CONFIG_NAMES = ("plain_decode_d1", "plain_decode_d2", "mtp", "sparse_mixed", "long_context")
FP8_NAMES = ("plain_decode_d2", "mtp")  # dense workloads also run over an FP8 E4M3 cache
FP8_SCALE = 0.25
DESCR = {
    "tiny": "tiny: 4 requests, context {6,37,130,300}, q_len {4,1,2,2}, H=16, D=2, page 16, merge+W_UV",
    "plain_decode_d1": "plain decode: batch 64, q_len 1, H=16, context 4096, D=1, page 64, merge to 512-wide",
    "plain_decode_d2": "plain decode: batch 64, q_len 1, H=16, context 4096, D=2, page 64, merge to 512-wide",
    "mtp": "MTP decode: batch 128, q_len 2, H=16, context U[1024,8192], D=4, page 64, merge+W_UV",
    "long_context": "long context: batch 32, q_len 2, H=128, context U[16384,32768], D=8, page 64, merge+W_UV",
    "sparse_mixed": "sparse+mixed: 96 requests q_len {1,2,4} + 4x64 prefill, H=64, context U[4096,65536], "
                    "top-k 2048, D=4, page 64, merge+W_UV",
}


_T0 = time.perf_counter()


def log(msg):
    """Progress on stderr (the bench line alone goes to stdout)."""
    print(f"[bench {time.perf_counter() - _T0:8.1f}s] {msg}", file=sys.stderr, flush=True)


def peaks():
    p = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p.update(hbm_gbs=float(m["hbm_gbs"]), bf16_tflops=float(m["bf16_tflops"]),
                 bf16_tflops_sustained=float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), source="measured")
    return p


# ------------------------------------------------------------ algorithmic work


def work_of(w, partial_bytes=4, fused=False, kv_elem_bytes=2):
    """Algorithmic KV bytes, FLOPs and merge bytes of one step of workload w
    (fused: the merge is inside the decode; only the W_UV projection of the
    one merged fp32 result remains).  Each key row the step reads is read
    once: 576 elements of ``kv_elem_bytes`` (2: bf16 cache, 1: FP8 codes)."""
    row_bytes = 576 * kv_elem_bytes
    L = w.seq_lens.cpu().numpy().astype(np.int64)
    qsl = w.query_start_loc.cpu().numpy().astype(np.int64)
    D, H = w.dcp_world, w.num_heads
    q_len = qsl[1:] - qsl[:-1]
    kv_bytes_shard = []
    flops = 0
    if w.topk is None:
        for r in range(D):
            local = np.where(L > r, (L - r - 1) // D + 1, 0)
            kv_bytes_shard.append(int(local.sum()) * row_bytes)
        # every token sees its visible prefix, over all shards together
        vis = 0
        for b in range(len(L)):
            P = L[b] - q_len[b] + np.arange(q_len[b])
            vis += int((P + 1).sum())
        flops = vis * H * FLOPS_PER_KEY_ROW
    else:
        topk = w.topk.cpu().numpy()
        valid = w.topk_valid.cpu().numpy()
        pos = np.empty(w.num_tokens, np.int64)
        for b in range(len(L)):
            pos[qsl[b]:qsl[b + 1]] = L[b] - q_len[b] + np.arange(q_len[b])
        K = topk.shape[1]
        used = (np.arange(K)[None, :] < valid[:, None]) & (topk >= 0) & (topk <= pos[:, None])
        for r in range(D):
            kept = used & (topk % D == r)
            kv_bytes_shard.append(int(kept.sum()) * row_bytes)
        flops = int(used.sum()) * H * FLOPS_PER_KEY_ROW
    T = w.num_tokens
    out_w = 128 if w.w_uv is not None else 512
    if fused:
        merge_bytes = 0 if w.w_uv is None else T * H * (512 * 4 + 4) + T * H * (out_w * 2 + 4)
    else:
        merge_bytes = D * T * H * (512 * partial_bytes + 4) + D * T * 4 + T * H * (out_w * 2 + 4)
    if w.w_uv is not None:
        merge_bytes += H * 512 * 128 * 2
    q_bytes = T * H * 576 * 2
    return dict(kv_bytes=sum(kv_bytes_shard), kv_bytes_shard=kv_bytes_shard, flops=flops, merge_bytes=merge_bytes,
                q_bytes=q_bytes, tokens=T)


# ------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock / throttle samples every 100 ms; the summary keeps
    the samples taken inside the window marked around the timed region
    (which the bench pads with a sustained run of the same replays, so that
    the window holds several samples under load)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.window = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def mark(self, start, end):
        self.window = (start, end)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        import datetime
        if not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons, outside = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 10:
                    continue
                try:
                    ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk, cmax = float(p[2]), float(p[3])
                except ValueError:
                    continue
                if self.window and not (self.window[0] <= ts <= self.window[1]):
                    outside += 1
                    continue
                sm.append(clk)
                mx.append(cmax)
                for n, v in zip(names, p[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "window_s": round(self.window[1] - self.window[0], 3) if self.window else None,
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ our arm


class L2Flush:
    """Empties L2 between timed steps: a 256 MB write, then a 256 MB read of
    another buffer.  The read evicts the lines the write left dirty, so their
    write-back does not land in the next timed step as extra DRAM traffic."""

    def __init__(self, mib=256):
        n = mib * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = torch.ones(n, dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.add_(1)
        self.r.sum()


def flush_l2(flush):
    flush()


def time_workload(name, steps, warmup, with_e2e=False, l2_flush=False, fused=False, clock=None, sustain_s=1.5,
                  fp8=False):
    """Time one workload's decode step.  ``fused``: the step as one
    shard-fused decode launch (all D shards, merge built in; + the W_UV
    projection when the workload has one) instead of D shard calls + the
    merge call.  ``fp8``: the fused step over an FP8 E4M3 copy of the
    workload's cache (codes of cache / FP8_SCALE)."""
    import mla_decode_attention_04_gb300 as mla
    from mla_decode_attention_04_gb300 import pipeline, workloads as wl

    log(f"{name}: building the workload (fused={fused}, fp8={fp8})")
    w = wl.NAMED[name](device="cuda")
    if fp8:
        _, views = wl.fp8_cache(w, FP8_SCALE)
        step = pipeline.fused_step_for_workload(w, fp8_caches=views, kv_scale=FP8_SCALE)
        fused = True
    else:
        step = pipeline.fused_step_for_workload(w) if fused else pipeline.step_for_workload(w)
    work = work_of(w, 4 if fused else step.partials.element_size(), fused=fused, kv_elem_bytes=1 if fp8 else 2)
    flush = L2Flush() if l2_flush else None
    stream = torch.cuda.current_stream()
    log(f"{name}: warm-up")
    for _ in range(warmup):
        step.run()
    torch.cuda.synchronize()
    rc, detail = mla.workspace_status(step.workspace)
    if rc != mla.MLA_OK:
        raise RuntimeError(f"device check {detail} in {name}")
    log(f"{name}: capturing graphs")

    # The step runs as a CUDA graph (how a serving engine replays its decode
    # step): the library launches nothing per replay from the host, so the
    # events time the kernels, not the Python launch path.  One graph for the
    # whole step, and one per decode call and for the merge for the breakdown.
    D = w.dcp_world
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step.run()
    stream.wait_stream(side)
    launches0 = mla.kernel_launch_count()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        step.run()
    launches_per_step = mla.kernel_launch_count() - launches0
    g_dec, g_merge = [], None
    if fused:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fused_decode_only(step)
        g_dec.append(g)
        if step.w_uv is not None:
            g_merge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_merge):
                mla.dcp_lse_merge(step.merged, step.merged_lse, None, step.w_uv, out=step.out, lse_out=step.lse)
    else:
        for r, (cache, bt) in enumerate(step.shards):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step_shard(step, r, cache, bt)
            g_dec.append(g)
        g_merge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_merge):
            step_merge(step)
    torch.cuda.synchronize()

    log(f"{name}: timing")
    if clock is not None:
        # the clock window: a sustained run of the same replays (untimed),
        # then the K timed steps right after it
        t_start = time.time()
        while time.time() - t_start < sustain_s:
            for _ in range(20):
                if flush is not None:
                    flush_l2(flush)
                g_step.replay()
            torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for k in range(steps):
        if flush is not None:
            flush_l2(flush)
        ev[k][0].record(stream)
        g_step.replay()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    if clock is not None:
        clock.mark(t_start, time.time())
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    # breakdown: each decode call and the merge (after an L2 flush when the
    # steps had one)
    parts = g_dec + ([g_merge] if g_merge is not None else [])
    bev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(parts))] for _ in range(steps)]
    for k in range(steps):
        for i, g in enumerate(parts):
            if flush is not None:
                flush_l2(flush)
            bev[k][2 * i].record(stream)
            g.replay()
            bev[k][2 * i + 1].record(stream)
    torch.cuda.synchronize()
    nd = len(g_dec)
    decode_ms = [[e[2 * r].elapsed_time(e[2 * r + 1]) for r in range(nd)] for e in bev]
    merge_ms = [e[2 * nd].elapsed_time(e[2 * nd + 1]) if g_merge is not None else 0.0 for e in bev]
    launches = launches_per_step * steps
    rc, detail = mla.workspace_status(step.workspace)
    if rc != mla.MLA_OK:
        raise RuntimeError(f"device check {detail} in {name} (graph replays)")
    res = dict(name=name, w=w, step=step, work=work, step_ms=step_ms, decode_ms=decode_ms, merge_ms=merge_ms,
               launches=launches, fused=fused, fp8=fp8)
    if with_e2e:
        log(f"{name}: end-to-end timing")
        res["e2e"] = time_e2e(w, step, steps, flush)
    log(f"{name}: done, step {statistics.median(step_ms):.4f} ms")
    return res


def fused_decode_only(step):
    out = step.merged[0] if step.w_uv is not None else step.out
    lse = step.merged_lse[0] if step.w_uv is not None else step.lse
    step.decode(out, lse)


def step_shard(step, r, cache, bt):
    import mla_decode_attention_04_gb300 as mla
    if step.topk is not None:
        mla.mla_sparse_dcp_decode(step.q_nope, step.q_pe, cache, bt, step.seq_lens, step.qsl, step.topk,
                                  step.topk_valid, step.D, r, step.scale, out=step.partials[r], lse=step.lses[r],
                                  local_counts=step.counts[r], workspace=step.workspace)
    else:
        mla.mla_dcp_decode(step.q_nope, step.q_pe, cache, bt, step.seq_lens, step.qsl, step.max_query_len,
                           step.max_seq_len, step.D, r, step.scale, out=step.partials[r], lse=step.lses[r],
                           row_counts=step.counts[r], num_splits=step.num_splits, workspace=step.workspace)


def step_merge(step):
    import mla_decode_attention_04_gb300 as mla
    mla.dcp_lse_merge(step.partials, step.lses, step.counts, step.w_uv, out=step.out, lse_out=step.lse)


def time_e2e(w, step, steps, flush):
    """Same step through the public API with the per-step inputs (queries and
    request metadata) copied from pinned host memory and the output read
    back; the KV cache is device-resident state.  Timed twice: as one CUDA
    graph holding the copies, the library calls and the read-back (how a
    serving engine replays its decode step; the headline e2e), and with
    eager copies and launches from Python."""
    hq_n = w.q_nope.cpu().pin_memory()
    hq_p = w.q_pe.cpu().pin_memory()
    hmeta = [t.cpu().pin_memory() for t in (w.seq_lens, w.query_start_loc)]
    htabs = [s.block_table.cpu().pin_memory() for s in w.shards]
    hsparse = [] if w.topk is None else [w.topk.cpu().pin_memory(), w.topk_valid.cpu().pin_memory()]
    hout = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    dev_meta = [step.seq_lens, step.qsl]
    dev_tabs = list(step.tables) if hasattr(step, "tables") else [s[1] for s in step.shards]
    dev_sparse = [] if w.topk is None else [step.topk, step.topk_valid]
    h2d = sum(t.numel() * t.element_size() for t in [hq_n, hq_p] + hmeta + htabs + hsparse)
    d2h = hout.numel() * hout.element_size()
    stream = torch.cuda.current_stream()

    def one_step():
        step.q_nope.copy_(hq_n, non_blocking=True)
        step.q_pe.copy_(hq_p, non_blocking=True)
        for d, h in zip(dev_meta + dev_tabs + dev_sparse, hmeta + htabs + hsparse):
            d.copy_(h, non_blocking=True)
        step.run()
        hout.copy_(step.out, non_blocking=True)

    def timed(run):
        times = []
        for _ in range(steps):
            if flush is not None:
                flush_l2(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    ms_eager = timed(one_step)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        one_step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        one_step()
    torch.cuda.synchronize()
    ms = timed(g.replay)
    return dict(value=w.num_tokens / (ms * 1e-3), unit=UNIT, ms_per_step=ms, h2d_bytes_per_step=int(h2d),
                d2h_bytes_per_step=int(d2h),
                how="one CUDA graph per step: host-to-device copies of the step's inputs from pinned memory, the "
                    "library calls, the device-to-host copy of the output",
                eager={"value": w.num_tokens / (ms_eager * 1e-3), "ms_per_step": ms_eager,
                       "how": "the same copies and calls issued eagerly from Python each step"})


def route_tag(res):
    """Key of a timed route in profiles/traffic.json."""
    return ("decode_fused_" if res["fused"] else "decode_shards_") + res["name"] + ("_fp8" if res.get("fp8") else "")


def roofline_of(work, dec_ms_total, launches, pk, tag):
    """The decode's roofline object: bound by whichever of its KV bytes at
    HBM bandwidth or its FLOPs at bf16 tensor peak takes longer; achieved =
    that quantity over the decode calls' measured time; per launch of the
    decode kernel (``launches`` per step)."""
    t_hbm = work["kv_bytes"] / (pk["hbm_gbs"] * 1e9)
    t_tc = work["flops"] / (pk["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        bound, unit, peak = "hbm", "GB/s", pk["hbm_gbs"]
        achieved = work["kv_bytes"] / (dec_ms_total * 1e-3) / 1e9
    else:
        bound, unit, peak = "tensor", "TFLOP/s", pk["bf16_tflops"]
        achieved = work["flops"] / (dec_ms_total * 1e-3) / 1e12
    tr = profile_traffic(tag)
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": tr, "algorithmic_bytes": work["kv_bytes"] / launches,
            "algorithmic_flops": work["flops"] / launches, "launches_per_step": launches,
            "roofline_ms": max(t_hbm, t_tc) * 1e3}


def summarize(res, pk):
    work = res["work"]
    step_ms = statistics.median(res["step_ms"])
    dec_ms = [statistics.median([d[r] for d in res["decode_ms"]]) for r in range(len(res["decode_ms"][0]))]
    merge_ms = statistics.median(res["merge_ms"])
    dec_total = sum(dec_ms)
    roof = roofline_of(work, dec_total, len(dec_ms), pk, route_tag(res))
    merge_gbs = work["merge_bytes"] / (merge_ms * 1e-3) / 1e9 if merge_ms > 0 else None
    return dict(
        ms_per_step=step_ms,
        query_tok_s=work["tokens"] / (step_ms * 1e-3),
        decode_ms=dec_ms, merge_ms=merge_ms,
        kv_gbs=work["kv_bytes"] / (dec_total * 1e-3) / 1e9,
        tflops=work["flops"] / (dec_total * 1e-3) / 1e12,
        roofline_bound=roof["bound"],
        roofline_ms=roof["roofline_ms"],
        step_roofline_frac=roof["roofline_ms"] / step_ms,
        decode_roofline_frac=roof["frac"],
        roofline=roof,
        merge_gbs=merge_gbs,
        merge_hbm_frac=merge_gbs / pk["hbm_gbs"] if merge_gbs is not None else None,
        merge_bytes=work["merge_bytes"],
        merge_traffic=profile_traffic(("merge_fused_" if res["fused"] else "merge_shards_") + res["name"]),
        kv_bytes=work["kv_bytes"], flops=work["flops"],
    )


def rounded(d):
    if isinstance(d, dict):
        return {k: rounded(v) for k, v in d.items()}
    if isinstance(d, list):
        return [rounded(v) for v in d]
    if isinstance(d, float):
        return float(f"{d:.6g}")
    return d


def profile_traffic(kernel_tag):
    """DRAM bytes per launch from a committed ncu summary, if it describes the
    current kernel build; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel_tag)
        if not ent:
            return None
        from mla_decode_attention_04_gb300 import build as b
        if ent.get("source_digest") != b.source_digest():
            return None
        return ent.get("dram_bytes_per_launch")
    except Exception:
        return None


def replica_max_ms(step_ms, device):
    """Slowest rank's step time (every rank runs an independent replica of the
    workload; the job is done when the slowest one is)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return step_ms
    t = torch.tensor([step_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_rank, world, step_ms):
    """Query tokens of all ranks per second of the slowest rank's step."""
    return tokens_per_rank * world / (step_ms * 1e-3)


def run_ours(args):
    import mla_decode_attention_04_gb300 as mla
    from mla_decode_attention_04_gb300 import build as mla_build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        torch.cuda.set_device(local)
    mla_build.build()
    mla.load_library()
    pk = peaks()

    with ClockSampler(torch.cuda.current_device()) as clk:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        head = time_workload(HEADLINE, args.steps, args.warmup, with_e2e=True, fused=True, clock=clk)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    clocks = clk.summary()
    s = summarize(head, pk)
    step_ms = replica_max_ms(s["ms_per_step"], "cuda")
    tokens = head["work"]["tokens"]
    value = whole_job_value(tokens, world, step_ms)
    head_line = {k: head[k] for k in ("e2e", "launches")}
    del head
    torch.cuda.empty_cache()

    # every workload on both routes (the headline's fused route is the line
    # itself), and the dense fused route over FP8 caches
    configs = {}
    if args.configs != "headline" and rank == 0:
        names = [n for n in CONFIG_NAMES if args.configs == "all" or n in args.configs.split(",")]
        runs = [(n, False, False) for n in names] + [(n, True, False) for n in names if n != HEADLINE]
        runs += [(n, True, True) for n in FP8_NAMES if args.configs == "all" or n in args.configs.split(",")]
        for n, fused, fp8 in runs:
            r = time_workload(n, max(3, min(args.steps, 10)), max(3, min(args.warmup, 3)), fused=fused, fp8=fp8)
            cs = summarize(r, pk)
            key = n + ("_fp8" if fp8 else "") + ("_fused" if fused else "")
            configs[key] = rounded(cs)
            configs[key]["workload"] = DESCR[n] + (
                "; FP8 E4M3 cache (codes of cache / 0.25, scale 0.25)" if fp8 else "") + (
                "; one shard-fused decode launch" if fused else "; D shard calls + merge call")
            del r
            torch.cuda.empty_cache()
        configs[HEADLINE + "_fused"] = dict(rounded(s), workload=DESCR[HEADLINE] + "; one shard-fused decode launch "
                                                                                 "(the headline line)")

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded torch/numpy draws; no dataset)",
        "config": {"workload": DESCR[HEADLINE],
                   "route": "one shard-fused decode launch over the 8 DCP shards (the online softmax runs over "
                            "each shard's keys in turn: the LSE merge), plus its prep and split-merge kernels, then "
                            "the W_UV projection of the merged rows",
                   "l2": "inputs larger than L2, no flush: every step streams 0.9 GB of KV (> 129 MB L2)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "kv_gbs": s["kv_gbs"],
        "tflops": s["tflops"],
        "step_roofline_frac": s["step_roofline_frac"],
        "decode_roofline_frac": s["decode_roofline_frac"],
        "merge_hbm_frac": s["merge_hbm_frac"],
        "roofline": dict(s["roofline"],
                         kernel="shard-fused decode call (prep + decode + split-merge launches) as a CUDA graph, CUDA "
                                "events around each replay on the launching stream",
                         peak_source=pk["source"] + " (MEASURED_PEAKS.json bf16_tflops, burst cuBLAS GEMM)",
                         frac_of_sustained=s["roofline"]["achieved"] / pk["bf16_tflops_sustained"]
                         if s["roofline"]["unit"] == "TFLOP/s" else None),
        "e2e": head_line["e2e"],
        "clocks": clocks,
        "gpu_launches": head_line["launches"],
        "wall_s": wall,
        "configs": configs,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


# --------------------------------------------------------- oracle (CPU) arm


def oracle_sample_step(w, h, threads):
    """The oracle's whole step (every shard, merge, W_UV) on workload w."""
    import oracle
    D = w.dcp_world
    parts, lses, counts = [], [], []
    for r in range(D):
        o, l, c = oracle.dcp_decode(h["q_nope"], h["q_pe"], h["caches"][r], h["tables"][r], h["seq_lens"], h["qsl"],
                                    D, r, w.scale, threads=threads)
        parts.append(o), lses.append(l), counts.append(c)
    merged, lse = oracle.lse_merge(np.stack(parts), np.stack(lses), np.stack(counts))
    if h["w_uv"] is not None:
        merged = oracle.wuv_project(merged, h["w_uv"])
    return merged, lse


def oracle_sample(batch):
    """``batch`` requests drawn as the headline workload draws its 32
    (lengths U[16384, 32768], q_len 2, 128 heads, D=8, W_UV), on the host."""
    from mla_decode_attention_04_gb300 import workloads as wl
    w = wl.NAMED[HEADLINE](device="cpu", batch=batch)
    h = dict(q_nope=wl.bf16_bits(w.q_nope), q_pe=wl.bf16_bits(w.q_pe), seq_lens=w.seq_lens.numpy(),
             qsl=w.query_start_loc.numpy(), caches=[wl.bf16_bits(s.cache) for s in w.shards],
             tables=[s.block_table.numpy() for s in w.shards],
             w_uv=None if w.w_uv is None else wl.bf16_bits(w.w_uv))
    return w, h


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def time_oracle(batch, threads, budget_s, max_reps):
    w, h = oracle_sample(batch)
    oracle_sample_step(w, h, threads)  # warm (loads the library)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_sample_step(w, h, threads)
        reps += 1
        if time.perf_counter() - t0 > budget_s or reps >= max_reps:
            break
    return w.num_tokens / ((time.perf_counter() - t0) / reps), reps


def cpu_baseline(args, batch=2):
    import oracle
    threads = oracle.default_threads()
    log(f"cpu baseline: {batch} requests on {threads} threads")
    v_all, reps = time_oracle(batch, threads, 10.0, 20)
    log("cpu baseline: 1 request on 1 thread")
    v_one, reps1 = time_oracle(1, 1, 1.0, 1)
    log("cpu baseline: done")
    return {"value": v_all, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{batch} requests drawn as the headline workload draws its 32 (q_len 2, H=128, context "
                      f"U[16384,32768], all 8 shards + merge + W_UV), fp64 C oracle on {threads} threads, "
                      f"{reps} repetitions",
            "one_thread": {"value": v_one, "unit": UNIT, "cores": 1,
                           "sample": f"1 request drawn the same way, 1 thread, {reps1} repetition"},
            "nproc": os.cpu_count(), "cpu_model": cpu_model()}


def oracle_full_step(w, threads):
    """The oracle's whole step on workload w, dense or sparse: every shard's
    attention, the LSE merge (with the sparse counts) and W_UV."""
    import oracle
    from mla_decode_attention_04_gb300 import workloads as wl
    qn, qp = wl.bf16_bits(w.q_nope), wl.bf16_bits(w.q_pe)
    L, qsl = w.seq_lens.numpy(), w.query_start_loc.numpy()
    parts, lses, counts = [], [], []
    for r, sh in enumerate(w.shards):
        cache, table = wl.bf16_bits(sh.cache), sh.block_table.numpy()
        if w.topk is None:
            o, l, c = oracle.dcp_decode(qn, qp, cache, table, L, qsl, w.dcp_world, r, w.scale, threads=threads)
        else:
            o, l, c = oracle.sparse_dcp_decode(qn, qp, cache, table, L, qsl, w.topk.numpy(), w.topk_valid.numpy(),
                                               w.dcp_world, r, w.scale, threads=threads)
        parts.append(o), lses.append(l), counts.append(c)
    merged, lse = oracle.lse_merge(np.stack(parts), np.stack(lses), np.stack(counts))
    if w.w_uv is not None:
        merged = oracle.wuv_project(merged, wl.bf16_bits(w.w_uv))
    return merged, lse


def run_cpu_full(args):
    """The fp64 oracle's step on every benchmark workload at full size, on all
    host cores (one step each), and on one thread over the first requests
    of each (a bounded sample): one JSON line per workload."""
    import oracle
    from mla_decode_attention_04_gb300 import workloads as wl
    threads = oracle.default_threads()
    for name in CONFIG_NAMES:
        w = wl.NAMED[name](device="cpu")
        t0 = time.perf_counter()
        oracle_full_step(w, threads)
        dt = time.perf_counter() - t0
        n1 = {"long_context": 1, "sparse_mixed": 4}.get(name, 8)
        w1 = wl.NAMED[name](device="cpu", **({"batch": n1} if name != "sparse_mixed" else {"n_decode": n1, "n_prefill": 0}))
        t0 = time.perf_counter()
        oracle_full_step(w1, 1)
        dt1 = time.perf_counter() - t0
        print(json.dumps({"cpu_full": name, "workload": DESCR[name], "threads": threads, "nproc": os.cpu_count(),
                          "cpu_model": cpu_model(), "seconds_per_step": dt, "query_tok_s": w.num_tokens / dt,
                          "one_thread": {"requests": n1, "query_tokens": w1.num_tokens, "seconds": dt1,
                                         "query_tok_s": w1.num_tokens / dt1,
                                         "sample": f"the first {n1} requests drawn the same way, 1 thread"}}),
              flush=True)
        del w, w1


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    import oracle
    threads = oracle.default_threads()
    w, h = oracle_sample(2)
    for _ in range(args.warmup):
        oracle_sample_step(w, h, threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample_step(w, h, threads)
        times.append(time.perf_counter() - t0)
    ms = statistics.median(times) * 1e3
    value = w.num_tokens / (ms * 1e-3)
    sample = ("2 requests per step, drawn as the headline workload draws its 32 (q_len 2, H=128, context "
              "U[16384,32768], all 8 shards + merge + W_UV), fp64 C oracle")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": DESCR[HEADLINE], "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample,
                         "nproc": os.cpu_count(), "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(name, repeat, route="fused"):
    """Run the step of one benchmark workload ``repeat`` times, untimed: the
    command the ncu summaries under profiles/ are captured from."""
    from mla_decode_attention_04_gb300 import pipeline, workloads as wl
    w = wl.NAMED[name](device="cuda")
    fused = route in ("fused", "fp8")
    if route == "fp8":
        _, views = wl.fp8_cache(w, FP8_SCALE)
        step = pipeline.fused_step_for_workload(w, fp8_caches=views, kv_scale=FP8_SCALE)
    else:
        step = pipeline.fused_step_for_workload(w) if fused else pipeline.step_for_workload(w)
    for _ in range(repeat):
        step.run()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": name, "repeat": repeat, "route": route}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--configs", default="all", help="all | headline | comma list of workload names")
    ap.add_argument("--profile-case", default=None, help="run one workload's step untimed (for ncu), print no bench line")
    ap.add_argument("--repeat", type=int, default=3, help="steps of --profile-case")
    ap.add_argument("--cpu-full", action="store_true",
                    help="time the fp64 oracle on every workload at full size (all cores) and on a one-thread sample")
    ap.add_argument("--route", default="fused", choices=["fused", "shards", "fp8"],
                    help="--profile-case: one shard-fused decode launch, D shard calls + merge, or the fused launch "
                         "over an FP8 copy of the cache")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case, args.repeat, args.route)
        return
    if args.cpu_full:
        run_cpu_full(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
