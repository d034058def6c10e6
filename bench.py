#!/usr/bin/env python
"""Benchmark of the paged-KV attention hot path on one GB300 (or N replicas).

One step = one pass of the whole hot path over one flat batch: the slot-mapped
write of the step's new K/V (``pkv_write``) followed by attention over the
paged cache (``pkv_attention_varlen``: split-KV decode + log-sum-exp combine,
or the tiled prefill).  The headline workload is batch-1 decode at context
8192 (GQA 32/8, D = 128, bf16; 512 blocks of a shuffled 4096-block pool); the
metric is KV bytes read per second.  Successive steps rotate over 8 disjoint
block tables that tile the 268 MB pool, so every step reads its 33.5 MB of K/V
from HBM, not from the 129 MB L2.  Steps are captured in a CUDA graph and
replayed, the way a serving engine runs decode.

Printed: one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead, on bounded samples of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode KV GB/s (% HBM peak); prefill attention TFLOP/s (% bf16 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEADLINE = "decode_8k"
WORKLOAD_TEXT = {
    "decode_8k": "batch-1 decode, 1 query token at context 8192, GQA 32/8, head_dim 128, bf16, "
                 "16-token blocks: 512-block table from a shuffled 4096-block pool",
    "prefill_8k": "causal prefill of T=8192 tokens, GQA 32/8, head_dim 128, bf16, K/V written "
                  "through slot_mapping into 512 shuffled 16-token blocks",
    "batched_decode_64": "64 decodes, context U[512,4096], GQA 32/8, head_dim 128, bf16",
    "mixed_chunked": "flat batch: 2048-token prefill chunk + 3-token tail on 1000 + 62 decodes "
                     "U[256,2048], GQA 32/8, head_dim 128, bf16",
    "cascade_64x4k": "64 decodes sharing a 4096-token prefix (256 blocks), U[0,511] own cached "
                     "keys + 1 new token each, GQA 32/8, head_dim 128, bf16; shared-prefix "
                     "(cascade) attention, 4 replicas of 84 MB",
    "batched_decode_64_e4m3": "batched_decode_64 over an 8-bit E4M3 KV cache (k_scale = "
                              "v_scale = 0.5; q, new K/V and out bf16)",
    "decode_8k_e4m3": "decode_8k over an 8-bit E4M3 KV cache (k_scale = v_scale = 0.5; q, new "
                      "K/V and out bf16): 512-block table from a shuffled 8192-block pool",
    "prefill_8k_e4m3": "prefill_8k over an 8-bit E4M3 KV cache (k_scale = v_scale = 0.5; q, new "
                       "K/V and out bf16): the write quantises the 8192 tokens into 512 "
                       "shuffled blocks",
    "tiny_mixed_f32": "fp32, 2 q heads / 1 KV head, head_dim 64, 32-block pool: a 32-token "
                      "prefill, a decode at context 40 and a 3-token tail on a 45-token prefix "
                      "(a correctness case: the time is reported, the roofline fraction means "
                      "nothing at this size)",
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=8000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOAD_TEXT))
    p.add_argument("--no-secondary", action="store_true", help="skip the secondary workload lines")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# Distributed plumbing (one process per GPU; replicas, no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over ranks (identity on one process)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# Accounting (algorithmic work, counted as the method defines it)
# ---------------------------------------------------------------------------

def kv_bytes(requests, hkv, d, esize) -> int:
    """K and V bytes the step must read: each kv head once, seq_len tokens."""
    return sum((r.computed + r.scheduled) * hkv * d * 2 * esize for r in requests)


def causal_flops(requests, hq, d) -> int:
    """2 FLOPs per multiply-add of QK^T and of PV over visible (key <= query) pairs."""
    total = 0
    for r in requests:
        L, n = r.computed + r.scheduled, r.scheduled
        visible = sum(L - n + i + 1 for i in range(n))
        total += visible * 4 * d * hq
    return total


def write_bytes(num_tokens, hkv, d, esize) -> int:
    return num_tokens * hkv * d * esize * 2 * 2      # K and V, read + write


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured (MEASURED_PEAKS.json)"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel_file: str, workload: str):
    """DRAM bytes per launch of `workload` from the committed ncu summary, if
    it was taken on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    src = os.path.join(ROOT, "paged_kv_attention_17_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    for line in text.splitlines():
        m = re.match(r"\|\s*(\S+)\s*\|\s*(\S+)\s*\|\s*(\d+)\s*\|\s*([0-9a-f]{16})\s*\|", line)
        if m and m.group(1) == kernel_file and m.group(2) == workload and m.group(4) == digest:
            return {"workload": m.group(2), "bytes": int(m.group(3))}
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.proc, self.t0, self.t1 = index, None, None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside or rows[-3:]
        mhz = sorted(r[1] for r in use)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_region": bool(inside)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _device_replicas(w, device):
    import numpy as np
    import torch
    from paged_kv_attention_17_gb300 import metadata

    def tt(x):
        if w.dtype == "bf16":
            return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)

    def cache(x):
        # E4M3 caches hold their uint8 codes
        if w.kv_dtype == "e4m3":
            return torch.from_numpy(np.ascontiguousarray(x)).to(device)
        return tt(x)

    common = {"q": tt(w.q), "k_new": tt(w.k_new), "v_new": tt(w.v_new),
              "k_cache": cache(w.k_pool), "v_cache": cache(w.v_pool)}
    reps = []
    for reqs in w.replicas:
        m = metadata.build(reqs, w.block_size)
        reps.append({"meta": m, "requests": reqs,
                     "qsl": torch.from_numpy(m["query_start_loc"]).to(device),
                     "seq_lens": torch.from_numpy(m["seq_lens"]).to(device),
                     "block_table": torch.from_numpy(m["block_table"]).to(device),
                     "slot_mapping": torch.from_numpy(m["slot_mapping"]).to(device)})
    return common, reps


def _cascade_tensors(w, reps, device):
    """Shared table, own-key tables and lengths of each replica of a cascade."""
    import numpy as np
    import torch
    P = w.shared_blocks * w.block_size
    for rep in reps:
        reqs = rep["requests"]
        own = [r.blocks[w.shared_blocks:] for r in reqs]
        width = max(max(len(b) for b in own), 1)
        table = np.zeros((len(own), width), dtype=np.int32)
        for i, b in enumerate(own):
            table[i, :len(b)] = b
        lens = [r.computed + r.scheduled - P for r in reqs]
        rep["shared_table"] = torch.tensor(reqs[0].blocks[:w.shared_blocks], dtype=torch.int32,
                                           device=device)
        rep["suffix_table"] = torch.from_numpy(table).to(device)
        rep["suffix_lens"] = torch.tensor(lens, dtype=torch.int32, device=device)
        rep["max_suffix_len"] = max(lens)


def run_e2e_cascade(args, w, reps, common, csplits, cws, flag, bytes_step):
    """Per step: pinned host -> device copies of Q, new K/V and the metadata
    (slot mapping, query_start_loc, own-key lengths and tables, shared table),
    pkv_write + pkv_cascade_attention, device -> host copy of the output."""
    import torch

    import paged_kv_attention_17_gb300 as pkv
    keys = ("qsl", "slot_mapping", "suffix_lens", "suffix_table", "shared_table")
    host = {k: common[k].cpu().pin_memory() for k in ("q", "k_new", "v_new")}
    hreps = [{k: r[k].cpu().pin_memory() for k in keys} for r in reps]
    dev = {k: torch.empty_like(common[k]) for k in ("q", "k_new", "v_new")}
    dmeta = {k: torch.empty_like(reps[0][k]) for k in keys}
    out = torch.empty_like(common["q"])
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def one(i):
        hr, rep = hreps[i % len(hreps)], reps[i % len(reps)]
        for k in dev:
            dev[k].copy_(host[k], non_blocking=True)
        for k in dmeta:
            dmeta[k].copy_(hr[k], non_blocking=True)
        pkv.pkv_write(dev["k_new"], dev["v_new"], dmeta["slot_mapping"], common["k_cache"],
                      common["v_cache"], error_flag=flag)
        pkv.pkv_cascade_attention(dev["q"], common["k_cache"], common["v_cache"], out,
                                  dmeta["qsl"], dmeta["suffix_lens"], dmeta["suffix_table"],
                                  dmeta["shared_table"], rep["meta"]["max_query_len"],
                                  rep["max_suffix_len"], w.softmax_scale, prefix_splits=csplits,
                                  workspace=cws, error_flag=flag)
        hout.copy_(out, non_blocking=True)

    k = min(args.steps, 500)
    for i in range(min(20, k)):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(k):
        one(i)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / k
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + \
        sum(t.numel() * t.element_size() for t in hreps[0].values())
    d2h = hout.numel() * hout.element_size()
    return {"value": round((bytes_step / 1e9) / (ms / 1e3), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
            "ms_per_step": round(ms, 6), "mode": "eager API calls, pinned host buffers"}


def _launches_per_step(splits, meta):
    n = 2                                             # write + decode
    if splits > 1:
        n += 1                                        # combine
    if meta["max_query_len"] > 4:
        n += 1                                        # prefill tiles
    return n


def graph_sizes(k: int, group: int) -> list[int]:
    """Graph lengths a run of k steps replays: k // group replays of a graph
    of `group` steps, then one graph of the remaining k % group."""
    full, rest = divmod(k, group)
    return ([group] if full else []) + ([rest] if rest else [])


def precapture_sizes(warmup: int, steps: int, group: int) -> list[int]:
    """Every graph length the warm-up, the timed steps and the percentile
    replays (graphs of `group` steps) use: captured before any timing."""
    return sorted(set(graph_sizes(warmup, group) + graph_sizes(steps, group) + [group]))


def gpu_lead_in():
    """Keep the GPU busy (a bounded spin of ~0.25 ms at full clock) while the
    host enqueues the start event and the first steps, so the timed region
    starts on a busy, clocked-up GPU instead of including the host's launch
    latency and the clock ramp after an idle gap."""
    import torch
    torch.cuda._sleep(500_000)


def step_percentiles(run_steps, per_rep, device, reps=60):
    """p10 / p50 / p90 of the per-step time over individually timed replays of
    `per_rep` steps each (outside the main timed region)."""
    import torch
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        gpu_lead_in()
        a.record()
        run_steps(per_rep)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / per_rep)
    times.sort()
    pick = lambda q: round(times[min(len(times) - 1, int(q * len(times)))], 6)  # noqa: E731
    return [pick(0.1), pick(0.5), pick(0.9)]


def mixed_roofline(w, hq, hkv, d, esize, ms_step, peaks):
    """A mixed step is bound by the slower of its two classes: t* = max(KV bytes
    of the decode-class requests / HBM peak, causal FLOPs of the long requests /
    bf16 peak); the fraction is t* over the measured step, with each class's
    rate over the whole step beside it."""
    dec = [r for r in w.requests if r.scheduled <= 4]
    pre = [r for r in w.requests if r.scheduled > 4]
    b = kv_bytes(dec, hkv, d, esize)
    f = causal_flops(pre, hq, d)
    t_b = b / (float(peaks["hbm_gbs"]) * 1e9)
    t_f = f / (float(peaks["bf16_tflops"]) * 1e12)
    t_star = max(t_b, t_f)
    return {"t_star_ms": round(t_star * 1e3, 6), "frac": round(t_star / (ms_step / 1e3), 4),
            "bound": "hbm" if t_b >= t_f else "tensor",
            "decode_kv_bytes": b, "chunk_flops": f,
            "decode_gbs_over_step": round(b / 1e9 / (ms_step / 1e3), 1),
            "chunk_tflops_over_step": round(f / 1e12 / (ms_step / 1e3), 1)}


def run_gpu(args, rank, world, local_rank):
    import numpy as np
    import torch

    import paged_kv_attention_17_gb300 as pkv
    import workloads

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    name = args.workload
    reps_wanted = {"decode_8k": 8, "decode_8k_e4m3": 16, "cascade_64x4k": 4}.get(name, 1)
    w = workloads.NAMED[name](replicas=reps_wanted) if name != "tiny_mixed_f32" else workloads.NAMED[name]()
    common, reps = _device_replicas(w, device)
    e4m3 = w.kv_dtype == "e4m3"
    esize = 1 if e4m3 else (2 if w.dtype == "bf16" else 4)     # cache bytes per element
    m0 = reps[0]["meta"]
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    splits = pkv.pkv_num_splits(w.num_seqs, m0["max_query_len"], m0["max_seq_len"], hq, hkv, d,
                                local_rank)
    ws_bytes = pkv.pkv_workspace_bytes(w.num_seqs, hq, d, splits)
    workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(common["q"])
    flag = torch.zeros(1, dtype=torch.int32, device=device)

    cascade = w.shared_blocks > 0
    if cascade:
        _cascade_tensors(w, reps, device)
        csplits = pkv.pkv_cascade_splits(w.num_tokens, w.shared_blocks, hq, hkv, d,
                                         common["q"].dtype, local_rank)
        cws = torch.empty(pkv.pkv_cascade_workspace_bytes(w.num_tokens, hq, d, csplits),
                          dtype=torch.uint8, device=device)

    def write(rep):
        if e4m3:
            pkv.pkv_write_e4m3(common["k_new"], common["v_new"], rep["slot_mapping"],
                               common["k_cache"], common["v_cache"], w.k_scale, w.v_scale,
                               error_flag=flag)
            return
        pkv.pkv_write(common["k_new"], common["v_new"], rep["slot_mapping"], common["k_cache"],
                      common["v_cache"], error_flag=flag)

    def attend(rep):
        m = rep["meta"]
        if cascade:
            pkv.pkv_cascade_attention(
                common["q"], common["k_cache"], common["v_cache"], out, rep["qsl"],
                rep["suffix_lens"], rep["suffix_table"], rep["shared_table"], m["max_query_len"],
                rep["max_suffix_len"], w.softmax_scale, prefix_splits=csplits, workspace=cws,
                error_flag=flag)
            return
        if e4m3:
            pkv.pkv_attention_varlen_e4m3(
                common["q"], common["k_cache"], common["v_cache"], out, rep["qsl"],
                rep["seq_lens"], rep["block_table"], m["max_query_len"], m["max_seq_len"],
                w.softmax_scale, w.k_scale, w.v_scale, causal=w.causal, num_splits=splits,
                workspace=workspace, error_flag=flag)
            return
        pkv.pkv_attention_varlen(common["q"], common["k_cache"], common["v_cache"], out, rep["qsl"],
                                 rep["seq_lens"], rep["block_table"], m["max_query_len"],
                                 m["max_seq_len"], w.softmax_scale, causal=w.causal,
                                 num_splits=splits, workspace=workspace, error_flag=flag)

    # decode-class steps: the write rides in the decode kernel
    # (pkv_write_attention_varlen, and its E4M3 form)
    fused = m0["max_query_len"] <= 4 and not cascade

    def fused_step(rep):
        m = rep["meta"]
        if e4m3:
            pkv.pkv_write_attention_varlen_e4m3(
                common["k_new"], common["v_new"], rep["slot_mapping"], common["q"],
                common["k_cache"], common["v_cache"], out, rep["qsl"], rep["seq_lens"],
                rep["block_table"], m["max_query_len"], m["max_seq_len"], w.softmax_scale,
                w.k_scale, w.v_scale, causal=w.causal, num_splits=splits, workspace=workspace,
                error_flag=flag)
            return
        pkv.pkv_write_attention_varlen(common["k_new"], common["v_new"], rep["slot_mapping"],
                                       common["q"], common["k_cache"], common["v_cache"], out,
                                       rep["qsl"], rep["seq_lens"], rep["block_table"],
                                       m["max_query_len"], m["max_seq_len"], w.softmax_scale,
                                       causal=w.causal, num_splits=splits, workspace=workspace,
                                       error_flag=flag)

    def step(i):
        rep = reps[i % len(reps)]
        if fused:
            fused_step(rep)
            return
        write(rep)
        attend(rep)

    # eager warm-up (sets kernel attributes, resolves the TMA encoder) before capture
    for i in range(len(reps)):
        step(i)
    torch.cuda.synchronize()

    G = len(reps)
    use_graph = m0["max_query_len"] <= 4               # decode steps: graph, as a server runs them
    graphs = {}
    timed = {"active": False, "captures": 0}

    def graph_of(nsteps, body):
        if nsteps in graphs:
            return graphs[nsteps]
        if timed["active"]:
            timed["captures"] += 1                    # never expected: checked below
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for i in range(nsteps):
                    body(i)
        torch.cuda.current_stream().wait_stream(s)
        graphs[nsteps] = g
        return g

    def run_steps(k):
        if not use_graph:
            for i in range(k):
                step(i)
            return
        full, rest = divmod(k, G)
        if full:
            g = graph_of(G, step)
            for _ in range(full):
                g.replay()
        if rest:
            graph_of(rest, step).replay()

    # ---- every graph the warm-up and the timed steps replay is captured (and
    #      replayed once) here, so the timed region holds replays only ----
    if use_graph:
        for n in precapture_sizes(args.warmup, args.steps, G):
            graph_of(n, step).replay()
        torch.cuda.synchronize()

    # ---- warm-up, then exactly K timed steps ----
    run_steps(args.warmup)
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks.mark(True)
    timed["active"] = True
    gpu_lead_in()
    start.record()
    run_steps(args.steps)
    end.record()
    torch.cuda.synchronize()
    timed["active"] = False
    clocks.mark(False)
    barrier(world)
    if timed["captures"]:
        raise RuntimeError("a CUDA graph was captured inside the timed region")
    ms_total = reduce_max(start.elapsed_time(end), world, device)
    clk = clocks.stop() if rank == 0 else None
    if int(flag.item()) != 0:
        raise RuntimeError(f"device error flag {int(flag.item())}")
    ms_step = ms_total / args.steps
    pct = step_percentiles(run_steps, G if use_graph else 4, device)
    bytes_step = kv_bytes(w.requests, hkv, d, esize)
    flops_step = causal_flops(w.requests, hq, d)
    decode_like = m0["max_query_len"] <= 4
    per_rank_value = (bytes_step / 1e9) / (ms_step / 1e3) if decode_like else (flops_step / 1e12) / (ms_step / 1e3)
    value = per_rank_value * world

    # ---- the dominant kernel alone: attention calls back to back, events around ----
    nat = 400 if decode_like else 20
    att_body = lambda i: attend(reps[i % len(reps)])  # noqa: E731
    if use_graph:
        ga = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(ga, stream=s):
                for i in range(G):
                    att_body(i)
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(20):
            ga.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_lead_in()
    a0.record()
    if use_graph:
        for _ in range(nat):
            ga.replay()
        calls = nat * G
    else:
        for i in range(nat):
            att_body(i)
        calls = nat
    a1.record()
    torch.cuda.synchronize()
    att_ms = a0.elapsed_time(a1) / calls
    cascade_info = None
    if cascade:
        # the same batch through the plain call (full tables), and the bytes a
        # cascade must read from HBM: the shared prefix once, every own part
        def plain(i):
            rep = reps[i % len(reps)]
            mm = rep["meta"]
            pkv.pkv_attention_varlen(common["q"], common["k_cache"], common["v_cache"], out,
                                     rep["qsl"], rep["seq_lens"], rep["block_table"],
                                     mm["max_query_len"], mm["max_seq_len"], w.softmax_scale,
                                     num_splits=splits, workspace=workspace, error_flag=flag)
        for i in range(20):
            plain(i)
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        for i in range(nat):
            plain(i)
        p1.record()
        torch.cuda.synchronize()
        plain_ms = p0.elapsed_time(p1) / nat
        P = w.shared_blocks * w.block_size
        unique = (P + sum(r.computed + r.scheduled - P for r in w.requests)) * hkv * d * 2 * esize
        cascade_info = {"prefix_splits": csplits, "plain_call_ms": round(plain_ms, 6),
                        "cascade_call_ms": round(att_ms, 6),
                        "speedup_vs_plain": round(plain_ms / att_ms, 3),
                        "unique_kv_bytes": unique,
                        "logical_kv_bytes": bytes_step}
    if decode_like and cascade:
        # roofline on the bytes a cascade has to move (prefix once + own parts)
        achieved = (cascade_info["unique_kv_bytes"] / 1e9) / (att_ms / 1e3)
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4)}
        kernel_file = "decode.cu"
    elif decode_like:
        achieved = (bytes_step / 1e9) / (att_ms / 1e3)
        peak = float(peaks["hbm_gbs"])
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4)}
        kernel_file = "decode.cu"
    elif any(r.scheduled <= 4 for r in w.requests):
        # a mixed step (decode rows and long chunks in one call): bound by the
        # slower of its classes, t* = max(decode KV bytes / HBM peak, chunk
        # FLOPs / bf16 peak); reported in the binding class's unit as the rate
        # that would finish t*'s work in the measured call time, so that
        # frac = t* / call time
        mr = mixed_roofline(w, hq, hkv, d, esize, att_ms, peaks)
        if mr["bound"] == "hbm":
            peak, unit = float(peaks["hbm_gbs"]), "GB/s"
        else:
            peak, unit = float(peaks["bf16_tflops"]), "TFLOP/s"
        roof = {"bound": mr["bound"], "achieved": round(mr["frac"] * peak, 1), "peak": peak,
                "unit": unit, "frac": mr["frac"], "t_star_ms": mr["t_star_ms"]}
        kernel_file = "decode.cu" if mr["bound"] == "hbm" else "prefill.cu"
    else:
        achieved = (flops_step / 1e12) / (att_ms / 1e3)
        peak = float(peaks["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4)}
        kernel_file = "prefill.cu"
    tr = traffic_record(kernel_file, name)
    roof["traffic"] = tr["bytes"] if tr else None
    roof["kernel"] = ("pkv_attention_varlen call (split-KV decode kernel + LSE combine), "
                      f"{splits} splits" if decode_like else "pkv_attention_varlen call (prefill)")
    if not decode_like and "t_star_ms" in roof:
        roof["kernel"] = ("pkv_attention_varlen call over the mixed batch (decode rows + prefill "
                          "chunk): frac = t* / call time")
    if cascade:
        roof["kernel"] = (f"pkv_cascade_attention call (prefix pass, {csplits} splits; own-key "
                          "pass; merge)")
    roof["peak_source"] = peak_src
    roof["ms_per_launch"] = round(att_ms, 6)

    # ---- the KV scatter alone (pkv_write / pkv_write_e4m3, steps that run it
    #      as its own launch): GB/s on 2 x (read + write) bytes, K and V, each
    #      call timed with events after an L2 flush ----
    scatter = None
    if not fused:
        n_written = int((reps[0]["slot_mapping"] >= 0).sum().item())
        src_es = common["k_new"].element_size()
        moved = 2 * n_written * hkv * d * (src_es + esize)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(20)]
        for i in range(3):
            write(reps[i % len(reps)])
        for i, (e0, e1) in enumerate(ev):
            flush.fill_(i & 0xFF)
            e0.record()
            write(reps[i % len(reps)])
            e1.record()
        torch.cuda.synchronize()
        us = sum(e0.elapsed_time(e1) for e0, e1 in ev) / len(ev) * 1e3
        del flush
        scatter = {"value": round(moved / 1e3 / us, 1), "unit": "GB/s", "us_per_call": round(us, 3),
                   "bytes_per_call": moved, "tokens": n_written,
                   "frac_of_hbm_peak": round(moved / 1e3 / us / float(peaks["hbm_gbs"]), 4),
                   "timing": "20 calls, each after a 256 MB L2 flush, CUDA events around the call",
                   "kernel": "kv_write_e4m3_kernel" if e4m3 else "kv_write_kernel"}

    # ---- end to end through the public API with host buffers ----
    if cascade:
        e2e = run_e2e_cascade(args, w, reps, common, csplits, cws, flag, bytes_step)
    else:
        e2e = run_e2e(args, w, reps, common, splits, workspace, flag, device, bytes_step,
                      flops_step, decode_like)

    result = {
        "metric": METRIC, "value": round(value, 2),
        "unit": "GB/s" if decode_like else "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if e4m3 else w.dtype,
        "data": "synthetic: seeded N(0,1) PCG64(0), cast to bf16 (RNE)" + (
            "; cache codes drawn as E4M3 bit fields (exponent 4..8)" if e4m3 else ""),
        "config": {"workload": f"{name}: {WORKLOAD_TEXT[name]}", "num_splits": splits,
                   "step": ("pkv_write_attention_varlen (write fused into the decode kernel)"
                            if fused else "pkv_write + attention call"),
                   "kv_bytes_per_step": bytes_step, "flops_per_step": flops_step,
                   "l2": (f"cold: steps rotate over {len(reps)} disjoint 512-block tables of a "
                          "268 MB pool" if name.startswith("decode_8k") else
                          "inputs larger than L2"),
                   "cuda_graph": use_graph, "parallelism": f"replicas x{world}"},
        "roofline": roof, "e2e": e2e,
        "gpu_launches": (4 if cascade else _launches_per_step(splits, m0) - (1 if fused else 0))
                        * args.steps,
        "ms_per_step_p10_p50_p90": pct,
    }
    if name == "mixed_chunked":
        result["mixed_roofline"] = mixed_roofline(w, hq, hkv, d, esize, ms_step, peaks)
    if cascade_info is not None:
        result["cascade"] = cascade_info
    if scatter is not None:
        result["scatter"] = scatter
    if clk is not None:
        result["clocks"] = clk
    return result, w


def run_e2e_graphs(args, w, reps, common, bytes_step):
    """Decode steps through the package's CUDA-graph runner: per step the
    packed inputs (Q, new K/V, metadata) are staged in pinned host memory and
    one graph replay copies them to the device (pkv_stage_inputs), writes and
    attends, the output rows written into pinned host memory."""
    import torch

    from paged_kv_attention_17_gb300.graphs import DecodeGraphRunner
    m0 = reps[0]["meta"]
    width = int(reps[0]["block_table"].shape[1])
    n = w.num_seqs
    scales = (w.k_scale, w.v_scale) if w.kv_dtype == "e4m3" else None
    runner = DecodeGraphRunner(common["k_cache"], common["v_cache"], w.num_q_heads,
                               w.softmax_scale, width, m0["max_seq_len"], max_batch=n,
                               kv_scales=scales)
    hq = common["q"].cpu()
    hk, hv = common["k_new"].cpu(), common["v_new"].cpu()
    packed = [runner.pack(n, hq, hk, hv, r["slot_mapping"].cpu(), r["seq_lens"].cpu(),
                          r["block_table"].cpu()) for r in reps]
    steps = []

    def one(i):
        st = runner.begin(n)
        runner.stage(st, packed[i % len(packed)])
        runner.launch(st)
        steps.append(st)

    k = min(args.steps, 2000)
    for i in range(min(20, k)):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(k):
        one(i)
    e1.record()
    _, fl = runner.result(steps[-1])
    torch.cuda.synchronize()
    if fl != 0:
        raise RuntimeError(f"device error flag {fl} in the graph runner")
    ms = e0.elapsed_time(e1) / k
    b = runner.layouts[runner.sizes[-1]].b
    h2d = runner.layouts[b].nbytes
    d2h = b * w.num_q_heads * w.head_dim * common["q"].element_size() + 4
    return {"value": round((bytes_step / 1e9) / (ms / 1e3), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
            "ms_per_step": round(ms, 6),
            "mode": "CUDA-graph runner: per step the packed inputs are staged in pinned host "
                    "memory; one replay copies them to the device with a library kernel over "
                    "NVLink-C2C, then writes and attends, writing the output rows into pinned "
                    "host memory"}


def run_e2e(args, w, reps, common, splits, workspace, flag, device, bytes_step, flops_step,
            decode_like):
    """Per step: pinned host -> device copies of the step's inputs (Q, new K/V,
    metadata), the two API calls, device -> host copy of the output.  Decode
    steps go through the CUDA-graph runner instead (run_e2e_graphs)."""
    import torch

    import paged_kv_attention_17_gb300 as pkv
    if decode_like and w.num_seqs <= 512:
        return run_e2e_graphs(args, w, reps, common, bytes_step)
    host = {k: common[k].cpu().pin_memory() for k in ("q", "k_new", "v_new")}
    hreps = [{k: r[k].cpu().pin_memory() for k in ("qsl", "seq_lens", "block_table", "slot_mapping")}
             for r in reps]
    dq = torch.empty_like(common["q"])
    dk, dv = torch.empty_like(common["k_new"]), torch.empty_like(common["v_new"])
    dmeta = {k: torch.empty_like(reps[0][k]) for k in ("qsl", "seq_lens", "block_table", "slot_mapping")}
    out = torch.empty_like(common["q"])
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def one(i):
        hr, m = hreps[i % len(hreps)], reps[i % len(reps)]["meta"]
        dq.copy_(host["q"], non_blocking=True)
        dk.copy_(host["k_new"], non_blocking=True)
        dv.copy_(host["v_new"], non_blocking=True)
        for k in dmeta:
            dmeta[k].copy_(hr[k], non_blocking=True)
        if w.kv_dtype == "e4m3":
            pkv.pkv_write_e4m3(dk, dv, dmeta["slot_mapping"], common["k_cache"],
                               common["v_cache"], w.k_scale, w.v_scale, error_flag=flag)
            pkv.pkv_attention_varlen_e4m3(
                dq, common["k_cache"], common["v_cache"], out, dmeta["qsl"], dmeta["seq_lens"],
                dmeta["block_table"], m["max_query_len"], m["max_seq_len"], w.softmax_scale,
                w.k_scale, w.v_scale, causal=w.causal, num_splits=splits, workspace=workspace,
                error_flag=flag)
        else:
            pkv.pkv_write(dk, dv, dmeta["slot_mapping"], common["k_cache"], common["v_cache"],
                          error_flag=flag)
            pkv.pkv_attention_varlen(dq, common["k_cache"], common["v_cache"], out,
                                     dmeta["qsl"], dmeta["seq_lens"], dmeta["block_table"],
                                     m["max_query_len"], m["max_seq_len"], w.softmax_scale,
                                     causal=w.causal, num_splits=splits, workspace=workspace,
                                     error_flag=flag)
        hout.copy_(out, non_blocking=True)

    k = min(args.steps, 2000) if decode_like else max(1, min(args.steps, 5))
    for i in range(min(20, k)):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(k):
        one(i)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / k
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + \
        sum(t.numel() * t.element_size() for t in hreps[0].values())
    d2h = hout.numel() * hout.element_size()
    val = (bytes_step / 1e9) / (ms / 1e3) if decode_like else (flops_step / 1e12) / (ms / 1e3)
    return {"value": round(val, 2), "unit": "GB/s" if decode_like else "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k,
            "ms_per_step": round(ms, 6), "mode": "eager API calls, pinned host buffers"}


SECONDARY = ("batched_decode_64", "mixed_chunked", "prefill_8k", "prefill_8k_e4m3")
# workloads whose CPU baseline also reports a one-thread figure (the small and
# decode configurations of the measurement plan)
ONE_THREAD_TOO = ("tiny_mixed_f32", "decode_8k", "batched_decode_64")


def run_secondary(name, local_rank, steps, warmup, cpu_seconds):
    """One more workload of the headline run, timed the same way (its own
    warm-up, timed steps, roofline, clocks, end-to-end figure and CPU oracle
    baseline)."""
    import torch
    args = parse_args(["--workload", name, "--steps", str(steps), "--warmup", str(warmup)])
    res, _ = run_gpu(args, 0, 1, local_rank)
    torch.cuda.synchronize()
    keep = ("value", "unit", "steps", "warmup", "ms_per_step", "ms_per_step_p10_p50_p90",
            "roofline", "e2e", "clocks", "mixed_roofline", "gpu_launches", "dtype", "scatter")
    out = {"workload": res["config"]["workload"], "num_splits": res["config"]["num_splits"],
           "step": res["config"]["step"], "l2": res["config"]["l2"]}
    out.update({k: res[k] for k in keep if k in res})
    if cpu_seconds > 0:
        out["cpu_baseline"] = cpu_baseline(name, cpu_seconds)
        if name in ONE_THREAD_TOO:
            one = cpu_baseline_one_thread(name, cpu_seconds / 2)
            if one is not None:
                out["cpu_baseline"]["one_thread"] = one
    return out


# ---------------------------------------------------------------------------
# CPU oracle: the reference arm and the cpu_baseline
# ---------------------------------------------------------------------------

def oracle_sampler(name):
    """Return (w, cache, run(sample_keys) -> bytes) for timing the oracle on
    a bounded sample: its two-pass attention of the workload's decode rows over
    the first `sample_keys` keys of each context (cache already written by the
    oracle's scatter, which is not timed)."""
    import workloads
    from oracle import flatten as ofl
    from oracle import ref
    w = workloads.NAMED[name]()
    _, _, kc, vc, _ = ref.paged_step(w, tokens=[])      # the oracle's write only
    esize = 1 if w.kv_dtype == "e4m3" else (2 if w.dtype == "bf16" else 4)

    def run(sample_keys):
        import numpy as np
        from types import SimpleNamespace
        reqs = []
        for r in w.requests:
            L = min(r.computed + r.scheduled, max(sample_keys, r.scheduled))
            reqs.append(SimpleNamespace(computed=L - r.scheduled, scheduled=r.scheduled,
                                        blocks=r.blocks))
        m = ofl.flatten(reqs)
        ref.attention(w.q, kc, vc, m["query_start_loc"], m["seq_lens"], m["block_table"],
                      num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads,
                      softmax_scale=w.softmax_scale, causal=w.causal, dtype=w.dtype,
                      kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale)
        return kv_bytes(reqs, w.num_kv_heads, w.head_dim, esize), causal_flops(
            reqs, w.num_q_heads, w.head_dim)
    full_keys = max(r.computed + r.scheduled for r in w.requests)
    return w, run, full_keys


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(name, seconds):
    w, run, full = oracle_sampler(name)
    t = time.perf_counter()
    run(full)
    t_full = time.perf_counter() - t
    reps = max(1, int(seconds / max(t_full, 1e-3)))
    t = time.perf_counter()
    tot_b = tot_f = 0
    for _ in range(reps):
        b, f = run(full)
        tot_b, tot_f = tot_b + b, tot_f + f
    dt = time.perf_counter() - t
    decode_like = max(r.scheduled for r in w.requests) <= 4
    val = (tot_b / 1e9) / dt if decode_like else (tot_f / 1e12) / dt
    return {"value": round(val, 4), "unit": "GB/s" if decode_like else "TFLOP/s",
            "cores": cores_used(), "kind": "oracle",
            "sample": f"{reps} x full {name} step of oracle.ref.attention (float64 numpy, default "
                      f"BLAS threads) over the cache the oracle scatter wrote; scatter untimed"}


def cpu_baseline_one_thread(name, seconds):
    """The same oracle timing with one BLAS/OpenMP thread, in a child process
    (thread pools are fixed when numpy loads)."""
    import subprocess
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = (f"import json, bench; r = bench.cpu_baseline({name!r}, {seconds!r}); "
            f"print(json.dumps({{'value': r['value'], 'unit': r['unit']}}))")
    try:
        out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                             text=True, timeout=120 + 4 * seconds)
        res = json.loads(out.stdout.strip().splitlines()[-1])
        res["cores"] = 1
        return res
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None


def run_reference(args, rank, world):
    if rank != 0:
        return None
    name = args.workload
    w, run, full = oracle_sampler(name)
    t = time.perf_counter()
    run(full)
    t_full = time.perf_counter() - t
    budget = 150.0 / max(1, args.steps + args.warmup)   # whole run within a few minutes
    keys = full if t_full <= budget else max(16, int(full * budget / t_full) // 16 * 16)
    for _ in range(args.warmup):
        run(keys)
    t = time.perf_counter()
    tot_b = tot_f = 0
    for _ in range(args.steps):
        b, f = run(keys)
        tot_b, tot_f = tot_b + b, tot_f + f
    dt = time.perf_counter() - t
    decode_like = max(r.scheduled for r in w.requests) <= 4
    val = (tot_b / 1e9) / dt if decode_like else (tot_f / 1e12) / dt
    unit = "GB/s" if decode_like else "TFLOP/s"
    sample = (f"each step: oracle.ref.attention of {name}'s rows over the first {keys} of "
              f"{full} context keys (float64 numpy), cache written once by the oracle scatter")
    return {"impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{name}: {WORKLOAD_TEXT[name]}"},
            "cpu_baseline": {"value": round(val, 4), "unit": unit, "cores": cores_used(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, 4), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            res = run_reference(args, rank, world)
            if res is not None:
                print(json.dumps(res), flush=True)
            return 0
        result, w = run_gpu(args, rank, world, local_rank)
        if rank == 0 and world == 1 and not args.no_secondary and args.workload == HEADLINE:
            # the other configurations of the pages' workloads, each timed with
            # at least 20 steps after at least 3 warm-up steps
            cs = 0.0 if args.no_cpu_baseline else min(args.cpu_seconds, 8.0)
            result["secondary"] = {
                n: run_secondary(n, local_rank, max(args.steps, 20), max(args.warmup, 3), cs)
                for n in SECONDARY}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
            if args.workload in ONE_THREAD_TOO:
                one = cpu_baseline_one_thread(args.workload, args.cpu_seconds / 2)
                if one is not None:
                    result["cpu_baseline"]["one_thread"] = one
        if rank == 0:
            print(json.dumps(result), flush=True)
        return 0
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
