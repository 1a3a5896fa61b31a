#!/usr/bin/env python3
"""Benchmark of the paged-attention hot path: one step = kv_append of the step's
new tokens + batch_attention over the whole mixed batch.

Headline workload (N=1, default ``--workload long_prefill``): the long-prompt
prefill batch -- 4 prompts of 16384 tokens processed as their second chunk
(8192 new tokens over 8192 cached) plus 64 decode requests with kv_len ~
U[2048, 16384]; 64 query / 8 kv heads, head_dim 128, page_size 16, random page
permutation.  Its time is dominated by the prefill chunks' tensor-core work, so
the headline unit is prefill TFLOP/s ("Chunked prefill" (k4i.top), #flops:
4 d per attended (query, key) pair and query head, the causally masked pairs not
counted).  Workloads whose time is dominated by streaming the KV cache report
algorithmic GB/s (K/V pages read once per request, q, out, page ids, append
read + write).

Prints ONE JSON line (rank 0):
* ``value`` -- the headline workload's work per second of device time with
  inputs resident in HBM;
* ``e2e`` -- the same work per second of a step that also copies its inputs
  from pinned host memory and reads the output back;
* ``roofline`` -- the dominant kernel's algorithmic FLOPs (or bytes) per launch
  over its mean CUDA-event duration, against the measured burst peak;
* ``cpu_baseline`` -- the CPU oracle on a bounded sample of the workload;
* ``per_config`` -- the other four workloads (tiny mixed batch, 7B-class MHA
  decode, chunked-prefill mixed batch, large-model GQA decode shard), each timed
  the same way, with its own unit, roofline and end-to-end rate.

``--impl reference`` times the CPU oracle (the only reference this method has)
on the same workload, metric and unit.  Multi-GPU (torchrun): independent
replicas, one per GPU, no collective on the data path (``scaling: weak``).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import shutil
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "mixed-batch paged attention: decode KV GB/s, prefill TFLOP/s, % of roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
HEADLINE = "long_prefill"
# the five workloads of the method's cases, in order (tiny mixed batch, 7B-class
# MHA decode, chunked-prefill mixed batch, large-model GQA decode shard,
# long-prompt prefill); the ones not chosen as headline go to ``per_config``
CONFIGS = ["tiny_mixed", "mha_decode", "chunked_prefill_mixed", "gqa_decode_shard", "long_prefill"]


# ----------------------------------------------------------------- accounting
# Decode requests whose kv head serves at least this many query heads run in
# the tensor-core kernel (as key-split work items); the others in the CUDA-core
# split-KV kernel.  Mirrors the library planner's routing rule.
TC_DECODE_MIN_GROUP = 4
# Requests with 2 <= qo_len <= min(this, 128 / g) run as key-split items of the
# tensor-core decode kernel (the planner's verify routing).
VERIFY_MAX_TOKENS = 16


def step_accounting(wl, k=0):
    """Algorithmic bytes / FLOPs of one step, split by kernel class.  K/V bytes
    count each request's keys once; keys of a prefix shared by several requests
    (pages read in place) count once per step, under the first request."""
    Hq, Hkv, d, P = wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
    dec_bytes = pre_flops = pre_bytes = 0
    nnz_new = 0
    seen_prefix = set()
    verify_max = min(VERIFY_MAX_TOKENS, 128 // wl.group_size)
    # requests that fit two 128-row Q tiles run in their own kernel where
    # prefill runs on CTA pairs (head_dim 128)
    short_max = 2 * (128 // wl.group_size) if wl.head_dim == 128 else verify_max
    ver_flops = ver_bytes = sh_flops = sh_bytes = 0
    # rows the append kernel itself writes when the prefill kernels append
    # their chunks' own key tiles (requests with qo_len > two Q tiles' tokens:
    # new tokens from the first 128-aligned key at or after the cached prefix)
    fuse_min = 2 * (128 // wl.group_size) + 1
    app_rows_fused = 0
    tree = False
    for r in wl.steps[k].requests:
        nnz_new += r.qo_len
        tree = tree or r.parents is not None
        keep = r.qo_len
        if r.qo_len >= fuse_min:
            cached = r.kv_len - r.qo_len
            keep = min(r.qo_len, max(0, -(-cached // 128) * 128 - cached))
        app_rows_fused += keep
        sq = wl.seqs[r.seq]
        kv_read = r.kv_len
        if sq.prefix >= 0:
            if sq.prefix in seen_prefix:
                kv_read -= sq.prefix_len
            seen_prefix.add(sq.prefix)
        npages = -(-r.kv_len // P)
        if r.qo_len == 1:
            dec_bytes += kv_read * Hkv * d * 2 * 2 + 2 * Hq * d * 2 + npages * 4
        elif r.qo_len > 1:
            cached = r.kv_len - r.qo_len
            if r.parents is not None:
                # draft tree: each node sees the cached keys and its branch
                depth = np.zeros(r.qo_len, np.int64)
                for i, p in enumerate(r.parents):
                    depth[i] = 1 + (depth[p] if p >= 0 else 0)
                pairs = r.qo_len * cached + int(depth.sum())
            elif wl.causal:
                pairs = r.qo_len * cached + r.qo_len * (r.qo_len + 1) // 2
            else:
                pairs = r.qo_len * r.kv_len
            fl = 4 * d * Hq * pairs
            by = kv_read * Hkv * d * 2 * 2 + 2 * r.qo_len * Hq * d * 2 + npages * 4
            pre_flops += fl
            pre_bytes += by
            if r.qo_len <= verify_max:  # key-split items of the tensor-core decode kernel
                ver_flops += fl
                ver_bytes += by
            elif r.qo_len <= short_max:
                sh_flops += fl
                sh_bytes += by
    app_bytes = nnz_new * Hkv * d * 2 * 2 * 2
    tc_decode = wl.group_size >= TC_DECODE_MIN_GROUP
    return dict(decode_bytes=dec_bytes, append_bytes=app_bytes, prefill_flops=pre_flops,
                prefill_bytes=pre_bytes, nnz_new=nnz_new,
                # the append kernel's own bytes in a fused call (the tree call
                # never fuses)
                append_kernel_bytes_fused=app_bytes if tree else app_rows_fused * Hkv * d * 2 * 2 * 2,
                # work per kernel
                tc_flops=pre_flops - ver_flops - sh_flops, tc_bytes=pre_bytes - ver_bytes - sh_bytes,
                short_flops=sh_flops, short_bytes=sh_bytes,
                tc_decode_bytes=(dec_bytes if tc_decode else 0) + ver_bytes,
                cuda_decode_bytes=0 if tc_decode else dec_bytes)


def kernel_source_hash(name):
    """Hash of a kernel's source file and of the device headers (.cuh) it
    includes, directly or through another of them, in that order."""
    import re
    csrc = os.path.join(ROOT, "decode_attention_append_gb300", "csrc")
    files, todo = [], [name]
    while todo:
        f = todo.pop(0)
        if f in files:
            continue
        files.append(f)
        with open(os.path.join(csrc, f)) as fh:
            todo += re.findall(r'#include "([\w.]+\.cuh)"', fh.read())
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload, kernel_file):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source is unchanged since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            tab = json.load(f)
        ent = tab.get(workload)
        if ent and ent.get("source_hash") == kernel_source_hash(kernel_file):
            return ent.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        """Start sampling (query only: nothing about the GPU is changed).  The
        samples go to a temporary file that stop() reads and removes."""
        if not shutil.which("nvidia-smi"):
            return
        try:
            fd, self.path = tempfile.mkstemp(prefix="daa_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # wait for the first sample so the window is covered
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            self.fh.flush()
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        try:
            os.remove(self.path)
        except OSError:
            pass
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


# --------------------------------------------------------------- GPU setup
class GpuStep:
    """Device-resident workload: pool with the cached prefixes, page table,
    the step's q / k_new / v_new, outputs and workspace."""

    def __init__(self, wl, device, k=0, fused=True, prefix_groups=True):
        import decode_attention_append_gb300 as daa
        self.daa = daa
        self.fused = fused
        self.wl, self.dev = wl, device
        self.pool = torch.full(wl.pool_shape(), 0x7FC1, dtype=torch.int16, device=device).view(torch.bfloat16)
        it = wl.initial_table()
        k0, v0 = wl.initial_kv()
        if k0.shape[0]:
            t0 = daa.PageTable.from_host(it["qo_indptr"], it["kv_indptr"], it["page_indices"],
                                         it["last_page_len"], device)
            daa.kv_append(k0.to(device), v0.to(device), self.pool, t0.qo_indptr, t0.page_indices,
                          t0.kv_indptr, t0.last_page_len)
        del k0, v0
        st = wl.step_table(k)
        self.host_table = st
        self.table = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                             st["last_page_len"], device)
        q, kn, vn = wl.step_inputs(k)
        self.h_q, self.h_k, self.h_v = (x.pin_memory() for x in (q, kn, vn))
        self.q, self.k_new, self.v_new = (x.to(device) for x in (q, kn, vn))
        # requests that share a cached prefix: the shared-prefix calls attend it
        # once per group (off with --no-prefix-groups)
        groups = wl.prefix_groups(k)
        self.groups = groups if prefix_groups and int(groups[1].max(initial=0)) > 0 else None
        self.runner = daa.BatchAttention(self.table, wl.num_qo_heads, self.pool, causal=wl.causal,
                                         sm_scale=wl.sm_scale, prefix_groups=self.groups)
        # draft-tree verification: the step's mask rows (int32 view of the bits)
        self.tree = wl.has_tree(k)
        self.h_mask = self.mask = None
        if self.tree:
            self.h_mask = torch.from_numpy(wl.tree_mask(k).view(np.int32)).pin_memory()
            self.mask = self.h_mask.to(device)
        self.out = torch.empty_like(self.q)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        # pinned host copies of the int32 page table (re-sent every e2e step)
        self.h_ints = [torch.from_numpy(st[n]).pin_memory() for n in
                       ("qo_indptr", "kv_indptr", "page_indices", "last_page_len")]
        self.d_ints = [torch.empty_like(x, device=device) for x in self.h_ints]
        torch.cuda.synchronize()

    def step(self):
        if self.tree:
            self.runner.append(self.k_new, self.v_new)
            self.runner.run(self.q, out=self.out, tree_mask=self.mask)
        elif self.fused:
            self.runner.step(self.k_new, self.v_new, self.q, out=self.out)
        else:
            self.runner.append(self.k_new, self.v_new)
            self.runner.run(self.q, out=self.out)

    def step_plain(self):
        """The same step without its tree mask (plain causal attention)."""
        self.runner.append(self.k_new, self.v_new)
        self.runner.run(self.q, out=self.out)

    def step_e2e(self, stream):
        """Public API call with host buffers: H2D inputs, append + attention, D2H out."""
        for d, h in zip(self.d_ints, self.h_ints):
            d.copy_(h, non_blocking=True)
        if self.tree:
            self.mask.copy_(self.h_mask, non_blocking=True)
        self.q.copy_(self.h_q, non_blocking=True)
        self.k_new.copy_(self.h_k, non_blocking=True)
        self.v_new.copy_(self.h_v, non_blocking=True)
        qo, kv, pi, ll = self.d_ints
        hosts = (self.host_table["qo_indptr"], self.host_table["kv_indptr"],
                 self.host_table["last_page_len"])
        if self.tree:
            self.daa.kv_append(self.k_new, self.v_new, self.pool, qo, pi, kv, ll)
            self.daa.batch_attention_tree(self.q, self.pool, qo, kv, pi, ll, self.mask,
                                          self.wl.sm_scale, out=self.out,
                                          workspace=self.runner.workspace, host_indptr=hosts)
        elif self.fused:
            self.daa.append_attention(self.k_new, self.v_new, self.q, self.pool, qo, kv, pi, ll,
                                      self.wl.causal, self.wl.sm_scale, out=self.out,
                                      workspace=self.runner.workspace, host_indptr=hosts,
                                      prefix_groups=self.groups)
        else:
            self.daa.kv_append(self.k_new, self.v_new, self.pool, qo, pi, kv, ll)
            self.daa.batch_attention(self.q, self.pool, qo, kv, pi, ll, self.wl.causal,
                                     self.wl.sm_scale, out=self.out,
                                     workspace=self.runner.workspace, host_indptr=hosts,
                                     prefix_groups=self.groups)
        self.h_out.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        h2d = sum(x.numel() * x.element_size() for x in self.h_ints)
        h2d += sum(x.numel() * x.element_size() for x in (self.h_q, self.h_k, self.h_v))
        if self.tree:
            h2d += self.h_mask.numel() * self.h_mask.element_size()
        d2h = self.h_out.numel() * self.h_out.element_size()
        return h2d, d2h

    # ---- pipelined end-to-end steps: the way a serving loop feeds the library
    def setup_pipeline(self):
        """One pinned host buffer packs a step's inputs (page table, q, k_new,
        v_new, tree mask; 256-byte aligned sections), so each step uploads them
        with one copy.  Two device copies of it and of the output let step
        i + 1's upload and step i's download run on a copy stream while step i
        computes."""
        parts = list(self.h_ints) + [self.h_q, self.h_k, self.h_v]
        if self.tree:
            parts.append(self.h_mask)
        offs, at = [], 0
        for x in parts:
            offs.append(at)
            at += (x.numel() * x.element_size() + 255) // 256 * 256
        self.h_pack = torch.empty(at, dtype=torch.uint8, pin_memory=True)
        for x, o in zip(parts, offs):
            n = x.numel() * x.element_size()
            self.h_pack[o:o + n].copy_(x.reshape(-1).view(torch.uint8))
        self.pack_bytes = at
        self.d_pack, self.views, self.d_outs, self.h_outs = [], [], [], []
        for _ in range(2):
            d = torch.empty(at, dtype=torch.uint8, device=self.dev)
            v = [d[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) for x, o in zip(parts, offs)]
            self.d_pack.append(d)
            self.views.append(v)
            self.d_outs.append(torch.empty_like(self.out))
            self.h_outs.append(torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True))
        # uploads and downloads on streams of their own: one in-order copy
        # stream would queue step i + 1's upload behind step i's download
        self.up_stream = torch.cuda.Stream(device=self.dev)
        self.down_stream = torch.cuda.Stream(device=self.dev)
        self.ev_h2d = [torch.cuda.Event() for _ in range(2)]
        self.ev_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_d2h = [torch.cuda.Event() for _ in range(2)]

    # ---- the same loop through the one-call host step of the library
    def use_host_step(self):
        """Plain fused steps (no tree mask, no prefix groups) run end to end
        through daa_append_attention_host: one library call per step."""
        return self.fused and not self.tree and self.groups is None

    def setup_host_step(self):
        st = self.host_table
        sections = {n: torch.from_numpy(st[n]) for n in ("qo_indptr", "kv_indptr", "page_indices",
                                                         "last_page_len")}
        sections.update(q=self.h_q, k_new=self.h_k, v_new=self.h_v)
        self.hs = self.daa.HostStep(sections, self.pool, self.wl.num_qo_heads, causal=self.wl.causal,
                                    sm_scale=self.wl.sm_scale, workspace=self.runner.workspace)
        self.pack_bytes = self.hs.layout.total

    def run_host_steps(self, steps):
        """`steps` host steps, timed on the compute stream from before the
        first upload until the last read-back has landed (ms)."""
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        self.hs.up.wait_event(e0)
        self.hs.down.wait_event(e0)
        for i in range(steps):
            self.hs.step(i)
        for i in range(max(0, steps - 2), steps):
            s.wait_event(self.hs.done(i))
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def _call_api(self, v, out, stream):
        qo, kv, pi, ll, q, kn, vn = v[:7]
        hosts = (self.host_table["qo_indptr"], self.host_table["kv_indptr"],
                 self.host_table["last_page_len"])
        if self.tree:
            self.daa.kv_append(kn, vn, self.pool, qo, pi, kv, ll, stream=stream)
            self.daa.batch_attention_tree(q, self.pool, qo, kv, pi, ll, v[7], self.wl.sm_scale, out=out,
                                          workspace=self.runner.workspace, host_indptr=hosts,
                                          stream=stream)
        elif self.fused:
            self.daa.append_attention(kn, vn, q, self.pool, qo, kv, pi, ll, self.wl.causal,
                                      self.wl.sm_scale, out=out, workspace=self.runner.workspace,
                                      host_indptr=hosts, stream=stream, prefix_groups=self.groups)
        else:
            self.daa.kv_append(kn, vn, self.pool, qo, pi, kv, ll, stream=stream)
            self.daa.batch_attention(q, self.pool, qo, kv, pi, ll, self.wl.causal, self.wl.sm_scale,
                                     out=out, workspace=self.runner.workspace, host_indptr=hosts,
                                     stream=stream, prefix_groups=self.groups)

    def run_pipeline(self, steps):
        """`steps` end-to-end steps, timed on the compute stream by CUDA events
        from before the first upload until the last download has landed (ms)."""
        s, us, ds = torch.cuda.current_stream(), self.up_stream, self.down_stream
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        us.wait_event(e0)
        ds.wait_event(e0)
        for i in range(steps):
            k = i & 1
            us.wait_event(self.ev_done[k])     # step i - 2 has read this input slot
            with torch.cuda.stream(us):
                self.d_pack[k].copy_(self.h_pack, non_blocking=True)
            self.ev_h2d[k].record(us)
            s.wait_event(self.ev_h2d[k])
            s.wait_event(self.ev_d2h[k])       # step i - 2's output has been read back
            self._call_api(self.views[k], self.d_outs[k], s)
            self.ev_done[k].record(s)
            ds.wait_event(self.ev_done[k])
            with torch.cuda.stream(ds):
                self.h_outs[k].copy_(self.d_outs[k], non_blocking=True)
            self.ev_d2h[k].record(ds)
        s.wait_event(self.ev_d2h[0])
        s.wait_event(self.ev_d2h[1])
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)


def max_over_ranks(values, dist, device):
    """Element-wise MAX of per-rank timings over all ranks (every rank gets it):
    the job is as slow as its slowest replica."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(units_per_step, steps, world, ms):
    """Whole-job throughput (G units/s): every one of `world` replicas processed
    `units_per_step` per step for `steps` steps within `ms` milliseconds."""
    return units_per_step * steps * world / (ms * 1e-3) / 1e9


def soak(fn, seconds):
    """Run fn back to back for about `seconds` of wall time (untimed)."""
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < seconds:
        fn()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()


def timed(fn, steps, flush=None):
    """Device time (ms) of `steps` calls of fn on the current stream, by CUDA
    events: one pair around the back-to-back steps when no flush is needed
    (inputs larger than L2), else a pair per step with the L2 flush between."""
    s = torch.cuda.current_stream()
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            fn()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        evs[i][0].record(s)
        fn()
        evs[i][1].record(s)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


# --------------------------------------------------------------- CPU oracle
class OracleSample:
    """The CPU oracle on a bounded sample of step 0: whole requests (decodes
    first, then prefill requests) until the estimated fp64 work reaches the
    budget.  Inputs are generated once; each run() appends the step's new
    tokens and attends, and is timed."""

    def __init__(self, wl, budget_s=12.0):
        import copy

        import oracle
        from synth import SENTINEL_BF16, Request, Step
        self.oracle = oracle
        reqs = wl.steps[0].requests
        P = wl.page_size
        threads = max(1, oracle.num_threads())
        order = ([i for i, r in enumerate(reqs) if r.qo_len == 1] +
                 [i for i, r in enumerate(reqs) if r.qo_len > 1])
        picked, est = [], 0.0
        for i in order:
            r = reqs[i]
            # ~0.5 GFLOP/s per thread for the fp64 loops (4 d flops per pair and head)
            cost = r.kv_len * max(1, r.qo_len) * wl.num_qo_heads * wl.head_dim * 4 / 0.5e9 / threads
            if picked and est + cost > budget_s:
                break
            picked.append(i)
            est += cost
        sw = copy.copy(wl)
        seqs, sreqs, nxt, orig, owners = [], [], 0, [], {}
        for i in picked:
            r = reqs[i]
            src = wl.seqs[r.seq]
            shared, head = 0, np.zeros(0, np.int32)
            if src.prefix >= 0:
                # a shared prefix keeps one copy, read by every sampled request
                if src.prefix not in owners:
                    n = src.prefix_len // P
                    owners[src.prefix] = len(seqs)
                    seqs.append(type(src)(src.prefix_len, np.arange(nxt, nxt + n, dtype=np.int32)))
                    orig.append(src.prefix)
                    nxt += n
                shared, head = src.prefix_len, seqs[owners[src.prefix]].pages
            n = -(-r.kv_len // P) - shared // P
            pages = np.concatenate([head, np.arange(nxt, nxt + n, dtype=np.int32)])
            sreqs.append(Request(len(seqs), r.qo_len, r.kv_len, r.parents))
            seqs.append(type(src)(src.length, pages, owners.get(src.prefix, -1), shared))
            orig.append(r.seq)
            nxt += n
        sw.seqs, sw.steps, sw.num_pages = seqs, [Step(sreqs)], max(1, nxt)
        # the sampled sequences keep their original values
        sw._block = lambda seq, kind, block, _w=wl, _o=orig: _w._block(_o[seq], kind, block)
        self.sw = sw
        self.pool = oracle.new_pool(sw.pool_shape(), SENTINEL_BF16)
        it = sw.initial_table()
        k0, v0 = sw.initial_kv()
        oracle.kv_append(self.pool, k0, v0, it["qo_indptr"], it["page_indices"], it["kv_indptr"],
                         it["last_page_len"])
        self.table = sw.step_table(0)
        self.q, self.kn, self.vn = sw.step_inputs(0)
        self.mask = sw.tree_mask(0) if sw.has_tree(0) else None
        acc = step_accounting(sw)
        self.nbytes = acc["decode_bytes"] + acc["append_bytes"] + acc["prefill_bytes"]
        self.sample = (f"{len(picked)} of {len(reqs)} requests of step 0 (whole requests, decodes "
                       f"first); fp64 oracle on {threads} host threads")
        self.cores = threads

    def run(self):
        o, st = self.oracle, self.table
        t0 = time.perf_counter()
        o.kv_append(self.pool, self.kn, self.vn, st["qo_indptr"], st["page_indices"], st["kv_indptr"],
                    st["last_page_len"])
        o.attention(self.q, self.pool, st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                    st["last_page_len"], self.sw.causal, self.sw.sm_scale, self.sw.num_qo_heads,
                    tree_mask=self.mask)
        return time.perf_counter() - t0


class OracleRowSample:
    """The CPU oracle on sampled query rows of the step's first prefill request
    (for workloads measured in prefill TFLOP/s, whose whole prefill would take
    the fp64 oracle hours).  The request's cached prefix is appended once;
    each run() appends the request's new tokens and attends the sampled rows:
    the chunk's first and last rows, the first and last row of every 16th
    128-key tile boundary, and seeded random rows, until the estimated work
    reaches the budget.  Work = 4 d Hq per attended (query, key) pair
    ("Chunked prefill", #flops), counted by the oracle itself."""

    def __init__(self, wl, budget_s=12.0):
        import copy

        import oracle
        from synth import SENTINEL_BF16, Request, Step
        self.oracle = oracle
        reqs = wl.steps[0].requests
        ri = next(i for i, r in enumerate(reqs) if r.qo_len > 1)
        r = reqs[ri]
        src = wl.seqs[r.seq]
        P = wl.page_size
        sw = copy.copy(wl)
        n = -(-r.kv_len // P)
        sw.seqs = [type(src)(src.length, np.arange(n, dtype=np.int32))]
        sw.steps, sw.num_pages = [Step([Request(0, r.qo_len, r.kv_len, r.parents)])], n
        sw._block = lambda seq, kind, block, _w=wl, _s=r.seq: _w._block(_s, kind, block)
        self.sw = sw
        self.pool = oracle.new_pool(sw.pool_shape(), SENTINEL_BF16)
        it = sw.initial_table()
        k0, v0 = sw.initial_kv()
        oracle.kv_append(self.pool, k0, v0, it["qo_indptr"], it["page_indices"], it["kv_indptr"],
                         it["last_page_len"])
        self.table = sw.step_table(0)
        self.q, self.kn, self.vn = sw.step_inputs(0)
        threads = max(1, oracle.num_threads())
        cached = r.kv_len - r.qo_len
        # rows in order of priority: chunk edges, key-tile boundaries, random
        rng = np.random.default_rng(wl.seed)
        edges = [0, r.qo_len - 1]
        for kb in range(0, r.kv_len, 16 * 128):
            for t in (kb - cached - 1, kb - cached):
                if 0 <= t < r.qo_len:
                    edges.append(t)
        order = list(dict.fromkeys(edges)) + [int(x) for x in rng.permutation(r.qo_len)]
        order = list(dict.fromkeys(order))
        # calibrate the oracle's rate on the first rows, then fill the budget
        probe = order[:8]
        st = self.table
        t0 = time.perf_counter()
        _, _, pairs = oracle.attention(self.q, self.pool, st["qo_indptr"], st["kv_indptr"],
                                       st["page_indices"], st["last_page_len"], sw.causal,
                                       sw.sm_scale, sw.num_qo_heads, sel_rows=probe)
        rate = pairs / max(time.perf_counter() - t0, 1e-6)  # pairs per second
        picked, est = [], 0.0
        for t in order:
            cost = (cached + t + 1 if wl.causal else r.kv_len) / rate
            if picked and est + cost > budget_s:
                break
            picked.append(t)
            est += cost
        self.rows = sorted(picked)
        self.flops_per_pair = 4 * wl.head_dim * wl.num_qo_heads
        self.cores = threads
        self.sample = (f"{len(self.rows)} of {r.qo_len} query rows of prefill request {ri} "
                       f"({r.qo_len} new over {cached} cached: chunk edges, rows at 128-key tile "
                       f"boundaries, seeded random rows) plus its append; fp64 oracle on {threads} "
                       f"host threads")

    def run(self):
        """Seconds for one pass; sets self.flops to the pass's algorithmic work."""
        o, st = self.oracle, self.table
        t0 = time.perf_counter()
        o.kv_append(self.pool, self.kn, self.vn, st["qo_indptr"], st["page_indices"], st["kv_indptr"],
                    st["last_page_len"])
        _, _, pairs = o.attention(self.q, self.pool, st["qo_indptr"], st["kv_indptr"],
                                  st["page_indices"], st["last_page_len"], self.sw.causal,
                                  self.sw.sm_scale, self.sw.num_qo_heads, sel_rows=self.rows)
        dt = time.perf_counter() - t0
        self.flops = self.flops_per_pair * pairs
        return dt


def oracle_sample(wl, unit, budget_s):
    """The oracle sample that measures `unit` on this workload."""
    return OracleRowSample(wl, budget_s) if unit == "TFLOP/s" else OracleSample(wl, budget_s)


def sample_work(s, unit):
    """Work of one run of a sample, in the unit's base (FLOP or bytes)."""
    return s.flops if unit == "TFLOP/s" else s.nbytes


def cpu_baseline(wl, unit, step_work, budget_s=12.0, reps=None):
    """The oracle, as it stands, on a bounded sample of the workload; `value`
    in the headline's unit.  `step_work` (the whole step's work in that unit's
    base) gives the extrapolated time of a full step for the record."""
    s = oracle_sample(wl, unit, budget_s)
    dt = s.run()
    reps = reps or max(1, min(20, int(budget_s / max(dt, 1e-3))))
    times = [dt] + [s.run() for _ in range(reps - 1)]
    t = float(np.median(times))
    scale = 1e12 if unit == "TFLOP/s" else 1e9
    rate = sample_work(s, unit) / t
    return dict(value=rate / scale, unit=unit, cores=s.cores, kind="oracle",
                sample=s.sample + f", median of {len(times)} runs of {t:.3f} s; a whole step at "
                                  f"this rate: {step_work / rate:.1f} s (extrapolated)")


def compact_pool(wl):
    """Same workload with pages renumbered 0..n-1 in order of first use (a page
    shared by several sequences stays shared)."""
    import copy
    w = copy.copy(wl)
    mapping, seqs = {}, []
    for s in wl.seqs:
        for a in s.pages:
            mapping.setdefault(int(a), len(mapping))
        seqs.append(type(s)(s.length, np.asarray([mapping[int(a)] for a in s.pages], np.int32),
                            s.prefix, s.prefix_len))
    w.seqs, w.num_pages = seqs, max(1, len(mapping))
    return w


# ---------------------------------------------------------------------- main
def headline_unit(acc, hbm, bf16):
    """TFLOP/s when the step's ideal tensor-core time (its prefill FLOPs at the
    bf16 peak) exceeds its ideal memory time (decode + append bytes at the HBM
    peak); GB/s of algorithmic bytes otherwise."""
    t_tensor = acc["prefill_flops"] / (bf16 * 1e12)
    t_hbm = (acc["decode_bytes"] + acc["append_bytes"]) / (hbm * 1e9)
    return "TFLOP/s" if t_tensor > t_hbm else "GB/s"


def step_work(acc, unit):
    """Work of one step in the unit's base: prefill FLOPs, or algorithmic bytes."""
    if unit == "TFLOP/s":
        return acc["prefill_flops"]
    return acc["decode_bytes"] + acc["append_bytes"] + acc["prefill_bytes"]


def rate(work, steps, world, ms, unit):
    """Whole-job rate: every replica did `work` per step for `steps` steps."""
    return job_rate(work, steps, world, ms) / (1e3 if unit == "TFLOP/s" else 1.0)


def measure(wl, dev, args, full, clocks=None):
    """Time one workload on this GPU.  Returns the raw timings (ms over
    args.steps steps): device-resident steps, per-kernel CUDA-event records,
    end-to-end steps through the public API with host buffers, and steps on a
    stored plan.  `full` adds the clock window (back-to-back steps around the
    timed region, sampled by `clocks`)."""
    import decode_attention_append_gb300 as daa
    acc = step_accounting(wl)
    algo_bytes = acc["decode_bytes"] + acc["append_bytes"] + acc["prefill_bytes"]
    g = GpuStep(wl, dev, fused=args.api == "fused", prefix_groups=not args.no_prefix_groups)
    flush_buf = None
    need_flush = algo_bytes < 2 * L2_BYTES
    if need_flush:
        flush_buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    flush = (lambda: flush_buf.fill_(1.0)) if need_flush else None
    l2 = ("flushed between steps (256 MB write)" if need_flush
          else f"inputs larger than L2 ({algo_bytes / 1e9:.2f} GB per step)")
    for _ in range(max(3, args.warmup)):
        g.step()
    torch.cuda.synchronize()

    # ---- main timed region: device-resident inputs.  With a clock window,
    # nvidia-smi samples (100 ms period) cover ~1 s of identical steps before
    # the timed region and ~0.5 s after it.
    if full and clocks is not None:
        clocks.start()
        soak(g.step, 1.0)
    args.barrier()
    ms = timed(g.step, args.steps, flush)
    args.barrier()
    # ---- per-kernel roofline pass: CUDA events around each launch
    recs, clk = [], None
    if not args.quick:
        daa.trace_enable(8 * args.steps + 64)
        timed(g.step, args.steps, flush)
        recs = daa.trace_read()
        daa.trace_disable()
        args.barrier()
    if full and clocks is not None:
        soak(g.step, 0.5)
        clk = clocks.stop()
        if clk is not None:
            clk["window"] = "nvidia-smi samples over back-to-back steps around the timed region"

    # ---- e2e: host buffers through the public API.  Inputs larger than L2:
    # a pipelined serving loop (one packed upload per step on a copy stream,
    # overlapping the previous step's compute; the output read back behind
    # it).  L2-flushed small batches: serial steps with the flush between.
    ms_e2e = float("nan")
    e2e_mode = None
    h2d, d2h = g.e2e_bytes()
    if not args.quick:
        if flush is None and g.use_host_step():
            g.setup_host_step()
            g.run_host_steps(3)
            args.barrier()
            ms_e2e = g.run_host_steps(args.steps)
            h2d = g.pack_bytes
            e2e_mode = ("one daa_append_attention_host call per step: the packed inputs' H2D upload on "
                        "an upload stream overlapping the previous step's kernels, the output's D2H on a "
                        "download stream behind them, two device buffer sets alternating; all copies "
                        "inside the timed region")
        elif flush is None:
            g.setup_pipeline()
            g.run_pipeline(3)
            args.barrier()
            ms_e2e = g.run_pipeline(args.steps)
            h2d = g.pack_bytes
            e2e_mode = ("pipelined: one packed H2D upload per step on an upload stream overlapping the "
                        "previous step's compute, the output's D2H on a download stream behind it; all "
                        "copies inside the timed region")
        else:
            for _ in range(2):
                g.step_e2e(torch.cuda.current_stream())
            args.barrier()
            ms_e2e = timed(lambda: g.step_e2e(torch.cuda.current_stream()), args.steps, flush)
            e2e_mode = "serial: H2D inputs, the call, D2H output per step, L2 flushed between steps"
        args.barrier()
    # draft-tree batches: the same steps without the mask, for the mask's cost
    ms_plain = None
    if g.tree and not args.quick:
        for _ in range(3):
            g.step_plain()
        args.barrier()
        ms_plain = timed(g.step_plain, args.steps, flush)
        args.barrier()
    # the same steps on a plan uploaded once (in a model one plan serves every
    # layer of a step): each call launches the kernels only
    ms_planned = float("nan")
    if not g.tree and not args.quick:
        g.runner.plan()
        for _ in range(3):
            g.step()
        args.barrier()
        ms_planned = timed(g.step, args.steps, flush)
        args.barrier()
        g.runner.info = None
    err = daa.device_error(reset=True)
    res = dict(acc=acc, ms=ms, ms_e2e=ms_e2e, ms_planned=ms_planned, ms_plain=ms_plain, recs=recs,
               clk=clk, err=err, h2d=h2d, d2h=d2h, e2e_mode=e2e_mode, l2=l2,
               prefix_groups=g.groups is not None)
    del g, flush_buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def roofline(wl, name, acc, recs, steps, hbm, bf16, bf16_sus, peak_src):
    """The dominant kernel (largest share of traced time): its algorithmic
    FLOPs or bytes per launch over its mean CUDA-event duration, against the
    measured burst peak (each launch runs for microseconds to milliseconds
    inside a step, not back to back for seconds)."""
    per_kernel = {}
    for kname, kms in recs:
        per_kernel.setdefault(kname, []).append(kms)
    tot = {k: sum(v) for k, v in per_kernel.items()}
    if not tot:
        return None, per_kernel
    dom = max(tot, key=tot.get)
    mean_ms = float(np.mean(per_kernel[dom]))
    n_launch = len(per_kernel[dom]) / steps
    t = mean_ms * 1e-3
    if dom in ("prefill_tc", "short_tc"):
        # the tensor-core prefill kernels: bound by whichever ideal time is larger
        key = "tc" if dom == "prefill_tc" else "short"
        fl, by = acc[key + "_flops"] / n_launch, acc[key + "_bytes"] / n_launch
        t_tensor, t_hbm = fl / (bf16 * 1e12), by / (hbm * 1e9)
        if t_tensor >= t_hbm:
            roof = {"bound": "tensor", "achieved": fl / t / 1e12, "peak": bf16, "unit": "TFLOP/s",
                    "peak_source": f"{peak_src} bf16 dense GEMM, burst",
                    "frac_of_sustained": fl / t / 1e12 / bf16_sus,
                    "sustained_peak": bf16_sus}
        else:
            roof = {"bound": "hbm", "achieved": by / t / 1e9, "peak": hbm, "unit": "GB/s",
                    "peak_source": f"{peak_src} HBM copy"}
        roof["ideal_fraction"] = (t_tensor + t_hbm) / t
        kfile = "prefill_pair.cu" if wl.head_dim == 128 and dom == "prefill_tc" else "prefill.cu"
    else:
        kb = {"decode_splitkv": acc["cuda_decode_bytes"], "decode_tc": acc["tc_decode_bytes"],
              "kv_append": acc["append_bytes"]}.get(dom, 0)
        roof = {"bound": "hbm", "achieved": kb / n_launch / t / 1e9, "peak": hbm, "unit": "GB/s",
                "peak_source": f"{peak_src} HBM copy"}
        kfile = {"decode_splitkv": "decode.cu", "decode_tc": "prefill.cu",
                 "kv_append": "append.cu"}.get(dom, "decode.cu")
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["mean_ms"] = mean_ms
    roof["traffic"] = measured_traffic(name, kfile)
    roof["share"] = {k: round(v / sum(tot.values()), 4) for k, v in tot.items()}
    return roof, per_kernel


def make_entry(wl, name, m, args, world, unit):
    """Rates, roofline and per-kernel figures of one measured workload."""
    hbm, bf16, bf16_sus, peak_src = peaks()
    acc = m["acc"]
    work = step_work(acc, unit)
    roof, per_kernel = roofline(wl, name, acc, m["recs"], args.steps, hbm, bf16, bf16_sus, peak_src)
    summary = wl.summary()
    e = {"workload": name, "description": wl.description,
         "value": rate(work, args.steps, world, m["ms"], unit), "unit": unit,
         "ms_per_step": m["ms"] / args.steps,
         "e2e": {"value": rate(work, args.steps, world, m["ms_e2e"], unit), "unit": unit,
                 "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                 "ms_per_step": m["ms_e2e"] / args.steps, "mode": m["e2e_mode"]},
         "gpu_launches": int(round(len(m["recs"]))),
         "roofline": roof,
         "algorithmic": {"bytes_per_step": acc["decode_bytes"] + acc["append_bytes"] + acc["prefill_bytes"],
                         "decode_bytes": acc["decode_bytes"], "append_bytes": acc["append_bytes"],
                         "prefill_flops": acc["prefill_flops"]},
         "config": {"requests": summary["requests"], "decode_requests": summary["decode_requests"],
                    "prefill_requests": summary["prefill_requests"], "kv_tokens": summary["kv_tokens"],
                    "Hq": wl.num_qo_heads, "Hkv": wl.num_kv_heads, "head_dim": wl.head_dim,
                    "page_size": wl.page_size, "num_pages": wl.num_pages,
                    "prefix_groups": m["prefix_groups"], "l2": m["l2"]},
         "device_error": m["err"]}
    e["kernels_ms"] = {k: round(float(np.mean(v)), 5) for k, v in per_kernel.items()}
    if m["ms_planned"] == m["ms_planned"]:  # not NaN
        e["planned"] = {"value": rate(work, args.steps, world, m["ms_planned"], unit), "unit": unit,
                        "ms_per_step": m["ms_planned"] / args.steps,
                        "note": "plan uploaded once (batch_attention_plan), each step runs the "
                                "kernels only; the headline value includes the plan"}
    if m["ms_plain"] is not None:
        e["tree_mask"] = {"ms_per_step_masked": m["ms"] / args.steps,
                          "ms_per_step_unmasked": m["ms_plain"] / args.steps,
                          "overhead": m["ms"] / m["ms_plain"] - 1.0,
                          "note": "same batch and kernels, plain causal attention without the mask"}
    if acc["prefill_flops"] and "prefill_tc" in per_kernel:
        # conservative: the kernel time also covers any decode splits it ran
        pm = float(np.mean(per_kernel["prefill_tc"]))
        e["prefill_tflops"] = acc["prefill_flops"] / (pm * 1e-3) / 1e12
        e["prefill_frac_of_bf16"] = e["prefill_tflops"] / bf16
    if acc["decode_bytes"]:
        kern = "decode_splitkv" if acc["cuda_decode_bytes"] else "decode_tc"
        if kern in per_kernel:
            dm = float(np.mean(per_kernel[kern]))
            e["decode_gbs"] = acc["decode_bytes"] / (dm * 1e-3) / 1e9
            e["decode_frac_of_hbm"] = e["decode_gbs"] / hbm
            e["decode_kernel"] = kern
    if acc["append_bytes"] and "kv_append" in per_kernel:
        # the append kernel's own rate (latency bound for a few tokens per
        # request), over the rows it writes: with the prefill append fused,
        # the prefill kernels write the long chunks' own key tiles
        fused = args.api == "fused" and not args.no_fused_prefill_append
        ab = acc["append_kernel_bytes_fused"] if fused else acc["append_bytes"]
        am = float(np.mean(per_kernel["kv_append"]))
        e["append_kernel_bytes"] = ab
        e["append_gbs"] = ab / (am * 1e-3) / 1e9
        e["append_frac_of_hbm"] = e["append_gbs"] / hbm
    return e


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--api", default="fused", choices=["fused", "two-call"],
                    help="fused: one append_attention call per step; two-call: kv_append then "
                         "batch_attention")
    ap.add_argument("--no-prefix-groups", action="store_true",
                    help="requests that share a cached prefix: plain calls (each request reads "
                         "the prefix) instead of the shared-prefix calls")
    ap.add_argument("--no-fused-prefill-append", action="store_true",
                    help="fused calls: append every row with the append kernel instead of letting "
                         "the prefill kernels write their chunks' own key tiles")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the headline workload only (no per_config map)")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: timed steps only (no clock window, no traced, e2e or "
                         "planned pass, no per_config map)")
    ap.add_argument("--compact-pool", action="store_true",
                    help="renumber pages densely so the pool holds only the pages used "
                         "(same work; smaller device footprint for profiler captures)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from synth import make_workload

    def load(name):
        w = make_workload(name)
        return compact_pool(w) if args.compact_pool else w

    wl = load(args.workload)
    acc = step_accounting(wl)
    hbm, bf16, bf16_sus, _ = peaks()
    unit = headline_unit(acc, hbm, bf16)
    work = step_work(acc, unit)
    config = {"workload": args.workload, "description": wl.description,
              "parallelism": f"replicas{args.gpus}", "compact_pool": bool(args.compact_pool),
              "api": ("append_attention" if args.api == "fused"
                      else "kv_append + batch_attention")}

    if args.impl == "reference":
        if rank != 0:
            return 0
        sample = oracle_sample(wl, unit, budget_s=6.0)
        for _ in range(args.warmup):
            sample.run()
        secs = [sample.run() for _ in range(args.steps)]
        scale = 1e12 if unit == "TFLOP/s" else 1e9
        v = sample_work(sample, unit) * len(secs) / sum(secs) / scale
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(secs) / len(secs),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": unit, "cores": sample.cores, "kind": "oracle",
                                 "sample": sample.sample},
                "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return 0

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
        if rank != 0:
            __graft_entry__.build()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
    args.barrier = barrier
    import decode_attention_append_gb300 as daa
    daa.set_prefill_append_fusion(not args.no_fused_prefill_append)
    config["prefill_append"] = ("append kernel (every row)" if args.no_fused_prefill_append else
                                "fused into the prefill kernels for long chunks")

    # ---- the headline workload, with its clock window
    clocks = ClockSampler(local)
    m = measure(wl, dev, args, full=not args.quick, clocks=clocks)
    ms, ms_e2e, ms_planned = max_over_ranks([m["ms"], m["ms_e2e"], m["ms_planned"]], dist, dev)
    m.update(ms=ms, ms_e2e=ms_e2e, ms_planned=ms_planned)

    # ---- the other configurations, each timed the same way (no clock window)
    per_config = {}
    if not args.quick and not args.no_per_config:
        for name in CONFIGS:
            if name == args.workload:
                continue
            w2 = load(name)
            a2 = step_accounting(w2)
            u2 = headline_unit(a2, hbm, bf16)
            m2 = measure(w2, dev, args, full=False)
            t = max_over_ranks([m2["ms"], m2["ms_e2e"], m2["ms_planned"]], dist, dev)
            m2.update(ms=t[0], ms_e2e=t[1], ms_planned=t[2])
            if rank == 0:
                per_config[name] = make_entry(w2, name, m2, args, world, u2)

    if rank != 0:
        dist.destroy_process_group()
        return 0

    e = make_entry(wl, args.workload, m, args, world, unit)
    config.update(e["config"])
    line = {"metric": METRIC, "value": e["value"], "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": e["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config, "e2e": e["e2e"],
            "gpu_launches": e["gpu_launches"], "roofline": e["roofline"],
            "algorithmic": e["algorithmic"], "clocks": m["clk"], "device_error": e["device_error"],
            "kernels_ms": e["kernels_ms"]}
    for k in ("planned", "tree_mask", "prefill_tflops", "prefill_frac_of_bf16", "decode_gbs",
              "decode_frac_of_hbm", "decode_kernel", "append_gbs", "append_frac_of_hbm"):
        if k in e:
            line[k] = e[k]
    if per_config:
        line["per_config"] = per_config
    if world == 1 and not args.no_cpu_baseline and not args.quick:
        line["cpu_baseline"] = cpu_baseline(wl, unit, work)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
