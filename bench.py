#!/usr/bin/env python3
"""Benchmark of the tiled / top-k / sparse attention hot path on GB300.

One step = one pass of the whole hot path over synthetic inputs shaped like the
pages' workloads, every part through the C ABI of libtts.so:
  vision  dense attention, N = 8547, 16 heads, d = 80, non-causal      (tensor cores)
  varlen  causal GQA prefill, 8 sequences <= 32768 tokens, 32/8 heads, d = 128
  topk    top-2048 of (323, 2590) indexer logits                        (HBM)
  sparse  323 queries x 128 heads, 576/512, 2048 paged indices          (gather)

Prints one JSON line (rank 0). `value` = attention TFLOP/s of the whole step
(dense + sparse FLOPs / step time); per-part figures are under `components`.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--shard [--gather]]

Under torchrun with N ranks the default runs one whole step per GPU (weak scaling);
--shard splits one step's units over the ranks instead (strong scaling: dense attention
by (sequence, KV-head group), top-k by rows, sparse attention by queries; no exchange
while computing, and with --gather one all-gather of the results at the end).

`--impl reference` times the float64 CPU oracle (the only reference there is:
the pages ship no code) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "attn TFLOP/s & % bf16 peak; top-k rows/s & sparse-attn GB/s vs HBM roofline"
WORKLOAD = "hot-path step: vision attn (8547 tok, 16h, d80) + varlen causal GQA prefill " \
           "(8 seqs <= 32768 tok, 32/8h, d128) + top-k (323x2590, k 2048) + sparse MLA attn " \
           "(323 q x 128h, 576/512, 2048 paged idx)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS = {"vision": "attn_fwd_kernel<80>", "varlen": "attn_fwd_kernel<128>",
           "topk": "topk_select_kernel", "sparse": "sparse_attn_kernel"}
# this library's kernel launches per call of each part (the sparse call: the sort launch,
# then the attention launch)
LAUNCHES = {"vision": 1, "varlen": 1, "topk": 1, "sparse": 2}
KERNEL_SOURCES = {"vision": "attn_fwd.cu", "varlen": "attn_fwd.cu", "topk": "topk.cu",
                  "sparse": "sparse_attn.cu", "vision_qkv_rope": "qkv_rope.cu",
                  "varlen_fp8": "attn_fwd.cu"}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(part: str) -> str:
    h = hashlib.sha256()
    for fn in (KERNEL_SOURCES[part], "ptx.cuh"):
        with open(os.path.join(ROOT, "tiled_top_sparse_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(part: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(part)
    if not e or e.get("source_hash") != source_hash(part):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # The raw samples go to $TTS_CLOCKS_DIR when set (kept for inspection), else to a
        # temporary directory; the JSON line carries their summary either way.
        out_dir = os.environ.get("TTS_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a host float over all ranks (the step time that bounds the job)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workload
class Step:
    """Device-resident inputs/outputs of one hot-path step and the four calls."""

    def __init__(self, dev, small=False, shard=None):
        """shard = (rank, world): keep only this rank's units of the step (dense attention
        by (sequence, KV-head group), top-k by rows, sparse attention by queries), packed
        once here, outside any timed region. None: the whole step."""
        import tiled_top_sparse_gb300 as tts
        from tiled_top_sparse_gb300 import shard as S
        self.tts = tts
        self.dev = dev
        self.sharded = shard is not None
        self.vis = W.vision()
        # small: a profiling-sized varlen batch (still larger than L2 in total)
        self.var = W.varlen(lengths=[4096, 3000, 2000, 1000]) if small else W.varlen()
        self.tk = W.topk_inputs()
        self.sp = W.sparse_inputs()
        # the whole step's work (every rank's units together)
        self.flops_total = {"vision": self.vis.flops(), "varlen": self.var.flops(),
                            "sparse": self.sp.flops()}
        g = lambda t: t.to(dev)  # noqa: E731
        self.d_vis = [g(self.vis.q), g(self.vis.k), g(self.vis.v), g(self.vis.cu_seqlens_q),
                      g(self.vis.cu_seqlens_k)]
        self.d_var = [g(self.var.q), g(self.var.k), g(self.var.v), g(self.var.cu_seqlens_q),
                      g(self.var.cu_seqlens_k)]
        self.d_tk = [g(self.tk.logits), g(self.tk.row_starts), g(self.tk.row_lens)]
        self.d_sp = [g(self.sp.q), g(self.sp.kv_cache), g(self.sp.page_table), g(self.sp.idx)]
        self.mq = {"vision": (self.vis.max_seqlen_q, self.vis.max_seqlen_k),
                   "varlen": (self.var.max_seqlen_q, self.var.max_seqlen_k)}
        self.flops = dict(self.flops_total)
        self.topk_bytes = self.tk.bytes()
        self.gathered = self.sp.gathered_bytes()
        self.n_rows = self.tk.logits.shape[0]
        self.plan = None
        if shard is not None:
            rank, world = shard
            self.plan = {}
            for name, inp, d in (("vision", self.vis, self.d_vis), ("varlen", self.var,
                                                                   self.d_var)):
                hq, hkv = inp.q.shape[1], inp.k.shape[1]
                owned, load = S.plan_dense(inp.lengths_q, inp.lengths_k, hq, hkv, inp.causal,
                                           world)
                sh = S.pack_dense(*d, owned[rank], hq, hkv)
                d[:] = [sh.q, sh.k, sh.v, sh.cu_q, sh.cu_k]
                self.mq[name] = (sh.max_q, sh.max_k)
                self.flops[name] = self.flops_total[name] * load[rank] / max(1, sum(load))
                self.plan[name] = {"units": len(owned[rank]), "heads_per_call": sh.hq,
                                   "load_max_over_mean": max(load) * world / max(1, sum(load))}
            r0, r1 = S.split_range(self.n_rows, world, rank)
            self.d_tk = [t[r0:r1].contiguous() for t in self.d_tk]
            self.topk_bytes = self.tk.bytes() * (r1 - r0) / max(1, self.n_rows)
            self.n_rows = r1 - r0
            n0, n1 = S.split_range(self.sp.q.shape[0], world, rank)
            nq = self.sp.q.shape[0]
            self.d_sp[0] = self.d_sp[0][n0:n1].contiguous()
            self.d_sp[3] = self.d_sp[3][n0:n1].contiguous()
            self.flops["sparse"] = self.flops_total["sparse"] * (n1 - n0) / nq
            self.gathered = self.sp.gathered_bytes() * (n1 - n0) / nq
            self.plan["topk"] = {"rows": [r0, r1]}
            self.plan["sparse"] = {"queries": [n0, n1]}
        f32 = dict(dtype=torch.float32, device=dev)
        self.o_vis = torch.empty(self.d_vis[0].shape, **f32)
        self.l_vis = torch.empty(self.d_vis[0].shape[:2], **f32)
        self.o_var = torch.empty(self.d_var[0].shape, **f32)
        self.l_var = torch.empty(self.d_var[0].shape[:2], **f32)
        self.o_idx = torch.empty((self.d_tk[0].shape[0], self.tk.k), dtype=torch.int32,
                                 device=dev)
        nq_here = self.d_sp[0].shape[0]
        self.o_sp = torch.empty((nq_here, self.sp.q.shape[1], self.sp.dv), **f32)
        self.l_sp = torch.empty((nq_here, self.sp.q.shape[1]), **f32)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        # attention workspaces (each call's work-item counter): one per call, since the
        # step may run the two calls at the same time on different streams
        def attn_ws(d):
            n = tts.attn_workspace_bytes(d[0].shape[0], d[1].shape[0], d[0].shape[1],
                                         d[1].shape[1], d[0].shape[2], torch.bfloat16)
            return torch.empty(n, dtype=torch.uint8, device=dev)
        self.ws_vis, self.ws_var = attn_ws(self.d_vis), attn_ws(self.d_var)
        # sparse workspace: partial results of the split last wave
        self.ws_sp = torch.empty(max(16, tts.sparse_workspace_bytes(nq_here)),
                                 dtype=torch.uint8, device=dev)

    def inputs(self):
        return self.d_vis[:3] + self.d_var[:3] + self.d_tk[:1] + self.d_sp[:2] + self.d_sp[3:]

    def outputs(self):
        return [self.o_vis, self.l_vis, self.o_var, self.l_var, self.o_idx, self.o_sp, self.l_sp]

    def part(self, name):
        t = self.tts
        if name == "vision":
            q, k, v, cq, ck = self.d_vis
            t.attn_fwd_varlen(q, k, v, cq, ck, *self.mq["vision"], False, self.vis.scale,
                              out=self.o_vis, lse=self.l_vis, workspace=self.ws_vis,
                              status=self.status)
        elif name == "varlen":
            q, k, v, cq, ck = self.d_var
            t.attn_fwd_varlen(q, k, v, cq, ck, *self.mq["varlen"], True, self.var.scale,
                              out=self.o_var, lse=self.l_var, workspace=self.ws_var,
                              status=self.status)
        elif name == "topk":
            lg, rs, rl = self.d_tk
            t.topk_select(lg, rs, rl, self.tk.k, idx=self.o_idx, status=self.status)
        elif name == "sparse":
            q, kv, pt, ix = self.d_sp
            t.sparse_attn_paged(q, kv, pt, ix, self.sp.kv_len, self.sp.scale, dv=self.sp.dv,
                                out=self.o_sp, lse=self.l_sp, workspace=self.ws_sp,
                                status=self.status)

    PARTS = ("vision", "varlen", "topk", "sparse")

    def e2e_units(self, parts, varlen_chunks=3):
        """The step as copy/compute units for the end-to-end run: (name, inputs, outputs, run).

        The varlen batch is cut into `varlen_chunks` runs of whole consecutive sequences
        (a contiguous token range of q/k/v/out/lse each, with its own cu_seqlens), so its
        copies can overlap its compute; every other part is one unit. Inputs include the
        small index tensors (cu_seqlens, windows, page table); outputs are everything the
        calls write.
        """
        t = self.tts
        units = []
        # sparse first: small inputs, a large result, so the copy-out link starts early
        if "sparse" in parts:
            units.append(("sparse", list(self.d_sp), [self.o_sp, self.l_sp],
                          lambda: self.part("sparse")))
        if "varlen" in parts and self.sharded:
            units.append(("varlen", list(self.d_var), [self.o_var, self.l_var],
                          lambda: self.part("varlen")))
        elif "varlen" in parts:
            q, k, v, cq, ck = self.d_var
            cu = self.var.cu_seqlens_q.tolist()
            assert cu == self.var.cu_seqlens_k.tolist()
            n_seq = len(cu) - 1
            total = cu[-1]
            bounds, start = [], 0
            for c in range(1, varlen_chunks + 1):  # cut at the sequence end nearest c/n
                target = total * c / varlen_chunks
                end = min(range(start + 1, n_seq + 1), key=lambda e: abs(cu[e] - target)) \
                    if c < varlen_chunks else n_seq
                if end > start:
                    bounds.append((start, end))
                    start = end
            for (a, b) in bounds:
                t0, t1 = cu[a], cu[b]
                cuc = torch.tensor([x - t0 for x in cu[a:b + 1]], dtype=torch.int32,
                                   device=self.dev)
                mq = max(cu[i + 1] - cu[i] for i in range(a, b))
                ins = [q[t0:t1], k[t0:t1], v[t0:t1], cuc]
                outs = [self.o_var[t0:t1], self.l_var[t0:t1]]

                def run(t0=t0, t1=t1, cuc=cuc, mq=mq):
                    t.attn_fwd_varlen(q[t0:t1], k[t0:t1], v[t0:t1], cuc, cuc, mq, mq, True,
                                      self.var.scale, out=self.o_var[t0:t1],
                                      lse=self.l_var[t0:t1], workspace=self.ws_var,
                                      status=self.status)
                units.append((f"varlen[{a}:{b}]", ins, outs, run))
        if "vision" in parts:
            units.append(("vision", list(self.d_vis), [self.o_vis, self.l_vis],
                          lambda: self.part("vision")))
        if "topk" in parts:
            units.append(("topk", list(self.d_tk), [self.o_idx], lambda: self.part("topk")))
        return units


def topk_protocol(step, dev, peaks):
    """Top-k beyond the step: a ~6 MB launch is shorter than launch latency, so (1) a CUDA
    graph of 256 launches rotating over 64 input/output buffer sets (384 MB, > 2x L2, so
    every launch reads from HBM), graph time / launches; (2) one call over 16 x the rows
    (the same rows repeated; its indices are checked against the single-batch result)."""
    t = step.tts
    lg, rs, rl = step.d_tk
    k = step.tk.k
    rows = lg.shape[0]
    sets = [(lg.clone(), torch.empty((rows, k), dtype=torch.int32, device=dev))
            for _ in range(64)]
    n_launch = 256
    s = torch.cuda.Stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for x, o in sets[:4]:
            t.topk_select(x, rs, rl, k, idx=o, status=step.status)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n_launch):
                x, o = sets[i % len(sets)]
                t.topk_select(x, rs, rl, k, idx=o, status=step.status)
        g.replay()
        e0.record(s)
        g.replay()
        e1.record(s)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n_launch
    for _, o in sets:
        assert torch.equal(o, sets[0][1]), "top-k: rotating buffer sets disagree"
    reps = 16
    big = (lg.repeat(reps, 1), rs.repeat(reps), rl.repeat(reps))
    out_big = torch.empty((rows * reps, k), dtype=torch.int32, device=dev)
    with torch.cuda.stream(s):
        for _ in range(3):
            t.topk_select(*big, k, idx=out_big, status=step.status)
        e0.record(s)
        for _ in range(10):
            t.topk_select(*big, k, idx=out_big, status=step.status)
        e1.record(s)
    e1.synchronize()
    us_big = e0.elapsed_time(e1) * 1e3 / 10
    assert torch.equal(out_big, sets[0][1].repeat(reps, 1)), "top-k: scaled call disagrees"
    gbs = step.topk_bytes / (us * 1e-6) / 1e9
    gbs_big = reps * step.topk_bytes / (us_big * 1e-6) / 1e9
    del sets, big, out_big
    return {"graph_us_per_launch": us, "graph_rows_per_s": rows / (us * 1e-6),
            "graph_gbs": gbs, "graph_frac_hbm": gbs / peaks["hbm_gbs"],
            "graph_protocol": f"CUDA graph of {n_launch} launches over 64 rotating buffer sets",
            "scaled_rows": rows * reps, "scaled_us": us_big,
            "scaled_rows_per_s": rows * reps / (us_big * 1e-6), "scaled_gbs": gbs_big,
            "scaled_frac_hbm": gbs_big / peaks["hbm_gbs"]}


def topk_long_protocol(step, dev, peaks):
    """Long-row top-k (rows split over many CTAs), outside the step: the last 64 query
    rows of a 262144-token context, k = 2048. A CUDA graph of 16 calls rotating over 4
    input sets (256 MB, > L2, so every call reads its rows from HBM); graph time / calls.
    The indices of every set are checked against the first set's."""
    t = step.tts
    inp = W.topk_long_inputs()
    rows, cols = inp.logits.shape
    k = inp.k
    lg = inp.logits.to(dev)
    rs, rl = inp.row_starts.to(dev), inp.row_lens.to(dev)
    sets = [(lg.clone() if i else lg, torch.empty((rows, k), dtype=torch.int32, device=dev))
            for i in range(4)]
    ws = torch.empty(t.topk_long_workspace_bytes(rows, cols, k), dtype=torch.uint8, device=dev)
    n_call = 16
    s = torch.cuda.Stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for x, o in sets:
            t.topk_select_long(x, rs, rl, k, idx=o, workspace=ws, status=step.status)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(n_call):
                x, o = sets[i % len(sets)]
                t.topk_select_long(x, rs, rl, k, idx=o, workspace=ws, status=step.status)
        g.replay()
        e0.record(s)
        g.replay()
        e1.record(s)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n_call
    for _, o in sets:
        assert torch.equal(o, sets[0][1]), "long top-k: input sets disagree"
    nbytes = int(inp.row_lens.sum().item()) * 4 + rows * k * 4 + rows * 8
    gbs = nbytes / (us * 1e-6) / 1e9
    del sets, ws, lg
    return {"workload": f"{rows} rows x {cols} (last queries of a {cols}-token context), k {k}",
            "us_per_call": us, "launches_per_call": 3, "bytes": nbytes, "gbs": gbs,
            "frac_hbm": gbs / peaks["hbm_gbs"],
            "protocol": f"CUDA graph of {n_call} calls over 4 rotating input sets"}


def decode_protocol(step, dev, peaks, nreq=64):
    """Decode-shaped sparse attention outside the step: `nreq` requests (64; a small
    batch of 8 shows the key split filling the SMs), each with a 32768-token context (the
    paged cache's max_seq_len on p3) in its own shuffled pages of 64, one query, 2048
    indices; then each request's next KV row is written through its page table. The KV
    pool (2.4 GB for 64 requests) and the queries come from a seeded device generator
    (values do not affect the timing); page tables and index lists as in
    workloads.sparse_decode_inputs. Index sets rotate so that a round of them gathers
    about 300 MB (> L2); 20 calls timed with CUDA events."""
    t = step.tts
    ctx, ps, topk, dqk, dv = 32768, 64, 2048, 576, 512
    g = torch.Generator(device="cpu").manual_seed(W.SEEDS["decode"])
    per = ctx // ps + 1
    pool = nreq * per
    tables = torch.randperm(pool, generator=g).to(torch.int32).view(nreq, per).to(dev)
    lens = torch.full((nreq,), ctx, dtype=torch.int32, device=dev)
    n_sets = max(2, -(-(300 << 20) // (nreq * topk * dqk * 2)))
    idx_sets = [torch.stack([torch.randperm(ctx, generator=g)[:topk] for _ in range(nreq)])
                .to(torch.int32).to(dev) for _ in range(n_sets)]
    gd = torch.Generator(device=dev).manual_seed(W.SEEDS["decode"])
    kv = torch.randn(pool, ps, dqk, generator=gd, device=dev).to(torch.bfloat16)
    q = torch.randn(nreq, 128, dqk, generator=gd, device=dev).to(torch.bfloat16)
    kv_new = torch.randn(nreq, dqk, generator=gd, device=dev).to(torch.bfloat16)
    out = torch.empty((nreq, 128, dv), dtype=torch.float32, device=dev)
    lse = torch.empty((nreq, 128), dtype=torch.float32, device=dev)
    ws = torch.empty(max(t.sparse_workspace_bytes(nreq), 16), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(dqk)
    call = lambda i: t.sparse_attn_decode(q, kv, tables, lens, idx_sets[i % n_sets], scale,
                                          dv=dv, out=out, lse=lse, workspace=ws,
                                          status=step.status)
    s = torch.cuda.Stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def graph_us(fn, n):
        with torch.cuda.stream(s):
            for i in range(4):
                fn(i)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=s):
                for i in range(n):
                    fn(i)
            gr.replay()
            e0.record(s)
            gr.replay()
            e1.record(s)
        e1.synchronize()
        return e0.elapsed_time(e1) * 1e3 / n

    us = graph_us(call, 20)
    us_w = graph_us(lambda i: t.paged_kv_write(kv, tables, kv_new, lens, status=step.status), 20)
    gathered = nreq * topk * dqk * 2
    flops = 2.0 * 128 * nreq * topk * (dqk + dv)
    gbs = gathered / (us * 1e-6) / 1e9
    del kv, q, ws, idx_sets
    return {"workload": f"{nreq} requests x {ctx}-token contexts (pages of {ps}), "
                        f"128 heads, {topk} indices", "us_per_call": us,
            "gathered_bytes": gathered, "gathered_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
            "tflops": flops / (us * 1e-6) / 1e12, "kv_write_us": us_w,
            "protocol": f"CUDA graph of 20 calls over {n_sets} rotating index sets "
                        f"({n_sets * gathered / 1e6:.0f} MB gathered per round)"}


def qkv_rope_protocol(step, dev, peaks, flush):
    """Vision QKV projection + RoPE outside the step (the projection in front of the
    vision attention): 8547 tokens, hidden 1280, 16 heads of 80, positions 0..8546,
    cos/sin table of 32768 positions (built once, outside the timing). Each of 20
    calls is timed alone with CUDA events on its stream after a 256 MB L2 flush; the
    median is reported. The q / k / v of every call are checked against the first."""
    t = step.tts
    inp = W.vision_qkv_inputs()
    x, w = inp.x.to(dev), inp.w.to(dev)
    b, pos = inp.bias.to(dev), inp.positions.to(dev)
    cs = t.rope_cache(inp.max_pos, inp.d, inp.base, device=dev)
    n, hidden = inp.x.shape
    H, d = inp.heads, inp.d
    outs = [torch.empty((n, H, d), dtype=torch.bfloat16, device=dev) for _ in range(3)]
    ref = None
    s = torch.cuda.Stream(dev)
    times = []
    with torch.cuda.stream(s):
        for it in range(24):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            t.qkv_rope(x, w, b, pos, cs, H, q=outs[0], k=outs[1], v=outs[2], status=step.status)
            e1.record(s)
            e1.synchronize()
            if it >= 4:
                times.append(e0.elapsed_time(e1) * 1e3)
            if ref is None:
                ref = [o.clone() for o in outs]
    for o, r in zip(outs, ref):
        assert torch.equal(o, r), "qkv_rope: calls disagree"
    us = float(np.median(times))
    flops = inp.flops()
    tf = flops / (us * 1e-6) / 1e12
    nbytes = (n * hidden + inp.w.numel()) * 2 + 3 * n * H * d * 2 + b.numel() * 4 + n * 4
    del x, w, outs, ref, cs
    return {"workload": f"{n} tokens x hidden {hidden} -> q/k/v {H} heads x {d} "
                        f"(RoPE on q, k; table of {inp.max_pos} positions)",
            "kernel": "qkv_rope_kernel<80>", "us_per_call": us, "flops": flops,
            "tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"],
            "peak_source": "bf16_tflops (a call timed alone)",
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                         "traffic": profiled_traffic("vision_qkv_rope")},
            "bytes": nbytes, "gbs": nbytes / (us * 1e-6) / 1e9,
            "protocol": "median of 20 single calls, CUDA events, L2 flushed before each"}


def fp8_prefill_protocol(step, dev, peaks, flush):
    """The varlen prefill workload (8 sequences, 32 / 8 heads, d 128, causal) through the
    FP8 path, outside the step: the e4m3 quantization of q and k, then attention with e4m3
    q / k in Q K^T. Each of 20 rounds flushes L2 (256 MB) before the quantization and
    again before the attention, both timed with CUDA events on their stream; medians are
    reported. The output of every round is checked against the first."""
    t = step.tts
    q, k, v, cq, ck = step.d_var
    var = step.var
    out = torch.empty(var.q.shape, dtype=torch.float32, device=dev)
    lse = torch.empty(var.q.shape[:2], dtype=torch.float32, device=dev)
    q8, qs, k8, ks = t.quantize_fp8_prefill(q, k)
    s = torch.cuda.Stream(dev)
    tq, ta, ref = [], [], None
    with torch.cuda.stream(s):
        for it in range(24):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            flush.zero_()
            ev[0].record(s)
            t.quantize_fp8_prefill(q, k, q8=q8, q_scale=qs, k8=k8, k_scale=ks)
            ev[1].record(s)
            flush.zero_()
            ev[2].record(s)
            t.attn_fwd_varlen_fp8(q8, qs, k8, ks, v, cq, ck, var.max_seqlen_q,
                                  var.max_seqlen_k, True, var.scale, out=out, lse=lse,
                                  workspace=step.ws_var, status=step.status)
            ev[3].record(s)
            ev[3].synchronize()
            if it >= 4:
                tq.append(ev[0].elapsed_time(ev[1]) * 1e3)
                ta.append(ev[2].elapsed_time(ev[3]) * 1e3)
            if ref is None:
                ref = out.clone()
    assert torch.equal(out, ref), "fp8 prefill: rounds disagree"
    us_q, us_a = float(np.median(tq)), float(np.median(ta))
    flops = var.flops()
    tf = flops / (us_a * 1e-6) / 1e12
    qbytes = (q.numel() + k.numel()) * 2 * 2 + (q.numel() + k.numel()) + qs.numel() * 4
    del out, lse, q8, k8, ref
    return {"workload": "varlen causal GQA prefill (the step's batch), e4m3 q / k in Q K^T, "
                        "bf16 P V", "kernels": ["quant_rows_kernel", "head_amax_kernel",
                                                "head_scale_kernel", "attn_fwd_kernel<128, true>"],
            "us_quantize": us_q, "us_attention": us_a, "flops": flops, "tflops": tf,
            "frac_bf16_peak": tf / peaks["bf16_tflops"],
            "quantize_gbs": qbytes / (us_q * 1e-6) / 1e9,
            "peak_source": "bf16_tflops (half of the MMA work, P V, stays bf16)",
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
                         "traffic": profiled_traffic("varlen_fp8")},
            "protocol": "median of 20 rounds, CUDA events, L2 flushed before each call"}


# ----------------------------------------------------------------------------- CPU oracle
def oracle_sample(n_rows: int = 192, n_queries: int = 8):
    """Time the float64 oracle on bounded samples of each part.

    Returns {part: (work, seconds, description)}; work is FLOPs for the attention
    parts and rows for top-k.
    """
    import oracle
    oracle.build()
    vis, var, tk, sp = _inputs_cpu()
    g = np.random.default_rng(7)
    res = {}
    n = max(1, int(n_rows))
    tok = g.integers(0, 8547, n).astype(np.int32)
    head = g.integers(0, 16, n).astype(np.int32)
    t0 = time.perf_counter()
    oracle.attn_varlen(*vis["qkv"], vis["cq"], vis["ck"], False, vis["scale"], rows=(tok, head))
    res["vision"] = (n * 8547 * 80 * 4.0, time.perf_counter() - t0, f"{n} sampled rows")
    cq = var["cq"]
    T = int(cq[-1])
    tok = g.integers(0, T, n).astype(np.int32)
    head = g.integers(0, 32, n).astype(np.int32)
    b = np.searchsorted(cq, tok, side="right") - 1
    vis_keys = (tok - cq[b] + 1).astype(np.float64)  # causal, Lq == Lk
    t0 = time.perf_counter()
    oracle.attn_varlen(*var["qkv"], cq, var["ck"], True, var["scale"], rows=(tok, head))
    res["varlen"] = (float(vis_keys.sum()) * 128 * 4.0, time.perf_counter() - t0,
                     f"{n} sampled rows")
    t0 = time.perf_counter()
    oracle.topk(tk.logits.numpy(), tk.row_starts.numpy(), tk.row_lens.numpy(), tk.k)
    res["topk"] = (float(tk.logits.shape[0]), time.perf_counter() - t0, "all 323 rows")
    nq = max(1, int(n_queries))
    rows = g.choice(sp.q.shape[0], nq, replace=False)
    t0 = time.perf_counter()
    oracle.sparse_paged(sp.q.float().numpy()[rows], sp.kv_cache.float().numpy(),
                        sp.page_table.numpy(), sp.idx.numpy()[rows], sp.kv_len, sp.dv, sp.scale)
    valid = int((sp.idx[rows] >= 0).sum())
    res["sparse"] = (2.0 * 128 * valid * (576 + 512), time.perf_counter() - t0,
                     f"{nq} sampled queries")
    return res


_CPU_INPUTS = None


def _inputs_cpu():
    global _CPU_INPUTS
    if _CPU_INPUTS is None:
        vis, var, tk, sp = W.vision(), W.varlen(), W.topk_inputs(), W.sparse_inputs()
        pack = lambda d: {"qkv": [t.float().numpy() for t in (d.q, d.k, d.v)],  # noqa: E731
                          "cq": d.cu_seqlens_q.numpy(), "ck": d.cu_seqlens_k.numpy(),
                          "scale": d.scale}
        _CPU_INPUTS = (pack(vis), pack(var), tk, sp)
    return _CPU_INPUTS


def sized_sample(target_s: float):
    """Pick sample sizes so one oracle sample takes about target_s seconds."""
    probe = oracle_sample(16, 1)
    per_row = (probe["vision"][1] + probe["varlen"][1]) / 16
    per_q = probe["sparse"][1]
    fixed = probe["topk"][1]
    budget = max(0.05, target_s - fixed)
    # split the budget: half on dense rows, half on sparse queries
    n_rows = int(min(4096, max(1, 0.5 * budget / max(per_row, 1e-6))))
    n_q = int(min(323, max(1, 0.5 * budget / max(per_q, 1e-6))))
    return n_rows, n_q


def cpu_cores_used():
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def cpu_baseline_entry(res):
    attn_flops = res["vision"][0] + res["varlen"][0] + res["sparse"][0]
    attn_time = res["vision"][1] + res["varlen"][1] + res["sparse"][1]
    return {"value": attn_flops / attn_time / 1e12, "unit": "TFLOP/s", "cores": cpu_cores_used(),
            "kind": "oracle",
            "sample": "float64 oracle on bounded samples: vision %s, varlen %s, sparse %s; "
                      "top-k %s (%.1f rows/s)" % (res["vision"][2], res["varlen"][2],
                                                  res["sparse"][2], res["topk"][2],
                                                  res["topk"][0] / res["topk"][1])}


# ----------------------------------------------------------------------------- arms
def run_reference(args, rank, world):
    if rank != 0:
        return
    # Each step is a bounded sample so that warm-up + timed steps end within ~2 minutes.
    per_step = max(0.1, min(10.0, 100.0 / max(1, args.steps + args.warmup)))
    n_rows, n_q = sized_sample(per_step)
    steps = []
    res = None
    for _ in range(args.warmup):
        oracle_sample(n_rows, n_q)
    for _ in range(args.steps):
        res = oracle_sample(n_rows, n_q)
        steps.append(res)
    flops = sum(r["vision"][0] + r["varlen"][0] + r["sparse"][0] for r in steps)
    secs = sum(r["vision"][1] + r["varlen"][1] + r["sparse"][1] + r["topk"][1] for r in steps)
    value = flops / secs / 1e12
    cb = cpu_baseline_entry(res)
    cb["value"] = value
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": {"workload": WORKLOAD, "l2": "n/a (CPU)"},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_gpu(args, rank, world, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import tiled_top_sparse_gb300 as tts
    tts.lib()
    step = Step(dev, small=args.small, shard=(rank, world) if args.shard else None)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2
    parts = tuple(p for p in Step.PARTS if p in args.parts.split(","))

    gather = None
    if args.shard and args.gather and world > 1:
        # The one collective of a sharded step: every rank's results to every rank (raw
        # bytes, padded to the largest share), after its calls, inside the step's events.
        import torch.distributed as dist
        outs = [o for o in step.outputs()]
        nbytes = sum(o.numel() * o.element_size() for o in outs)
        mx = torch.tensor([nbytes], dtype=torch.int64, device=dev)
        dist.all_reduce(mx, op=dist.ReduceOp.MAX)
        send = torch.zeros(int(mx.item()), dtype=torch.uint8, device=dev)
        recv = torch.empty(world * send.numel(), dtype=torch.uint8, device=dev)

        def gather():
            off = 0
            for o in outs:
                b = o.numel() * o.element_size()
                send[off:off + b].copy_(o.reshape(-1).view(torch.uint8))
                off += b
            dist.all_gather_into_tensor(recv, send)

    def one_step(ev=None):
        """The parts one after another on one stream (events between them time each)."""
        for i, p in enumerate(parts):
            if ev is not None:
                ev[i].record(stream)
            step.part(p)
        if gather is not None:
            gather()
        if ev is not None:
            ev[len(parts)].record(stream)

    # The step's parts are independent (no part reads another's results), so the step
    # issues each on a stream of its own, the vision call first: the CTAs of the next
    # call take the SMs that a call's last, partial wave leaves idle.
    order = [p for p in ("vision", "varlen", "sparse", "topk") if p in parts]
    part_streams = {p: torch.cuda.Stream(dev) for p in order}
    ev_fork = torch.cuda.Event()
    ev_join = {p: torch.cuda.Event() for p in order}

    def concurrent_step(e0=None, e1=None):
        if e0 is not None:
            e0.record(stream)
        ev_fork.record(stream)
        for p in order:
            ps = part_streams[p]
            ps.wait_event(ev_fork)
            with torch.cuda.stream(ps):
                step.part(p)
            ev_join[p].record(ps)
        for p in order:
            stream.wait_event(ev_join[p])
        if gather is not None:
            gather()
        if e1 is not None:
            e1.record(stream)

    timed_step = one_step if args.serial else concurrent_step
    for _ in range(max(3, args.warmup)):
        one_step()
        concurrent_step()
    torch.cuda.synchronize()
    tts.check_status(step.status, "bench warm-up")

    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    with sampler:
        time.sleep(0.25)  # let the sampler start
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            flush.zero_()  # L2 flush between timed steps (outside the step's events)
            if args.serial:
                ev_step[k][0].record(stream)
                one_step()
                ev_step[k][1].record(stream)
            else:
                concurrent_step(*ev_step[k])
        torch.cuda.synchronize()
        t_wall1 = time.perf_counter()
        barrier(world)
    tts.check_status(step.status, "bench timed region")
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    # Per-part figures: the same steps with the parts one after another on one stream.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(parts) + 1)]
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for k in range(args.steps):
        flush.zero_()
        one_step(evs[k])
    torch.cuda.synchronize()
    tts.check_status(step.status, "bench per-part pass")
    per_part = {p: [] for p in parts}
    serial_ms = []
    for k in range(args.steps):
        e = evs[k]
        for i, p in enumerate(parts):
            per_part[p].append(e[i].elapsed_time(e[i + 1]))
        serial_ms.append(e[0].elapsed_time(e[len(parts)]))
    del timed_step
    ms_step_local = float(np.mean(step_ms))
    ms_step = max_over_ranks(ms_step_local, world)
    attn_flops = sum(step.flops[p] for p in parts if p in step.flops)
    # replicas: every rank runs the whole step; sharded: the ranks share one step
    job_flops = (sum(step.flops_total[p] for p in parts if p in step.flops_total)
                 if args.shard else world * attn_flops)
    value = job_flops / (ms_step * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    timed_s = t_wall1 - t_wall0
    tensor_peak = peaks["bf16_tflops_sustained"] if timed_s > 1.0 else peaks["bf16_tflops"]
    tensor_peak_name = "bf16_tflops_sustained" if timed_s > 1.0 else "bf16_tflops"
    comp = {}
    for p in parts:
        ms = float(np.mean(per_part[p]))
        c = {"ms": ms, "kernel": KERNELS[p], "launches_per_step": LAUNCHES[p]}
        if p in ("vision", "varlen"):
            tf = step.flops[p] / (ms * 1e-3) / 1e12
            c.update({"tflops": tf, "frac_bf16_peak": tf / tensor_peak})
        elif p == "topk":
            gbs = step.topk_bytes / (ms * 1e-3) / 1e9
            c.update({"rows_per_s": step.n_rows / (ms * 1e-3), "gbs": gbs,
                      "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": step.topk_bytes})
        else:
            gbs = step.gathered / (ms * 1e-3) / 1e9
            tf = step.flops[p] / (ms * 1e-3) / 1e12
            c.update({"gathered_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
                      "gathered_bytes": step.gathered, "tflops": tf,
                      "frac_bf16_peak": tf / tensor_peak})
        comp[p] = c
    extra = not args.shard  # the single-GPU protocols below measure whole workloads
    if "topk" in parts and rank == 0 and extra:
        comp["topk"].update(topk_protocol(step, dev, peaks))
        comp["topk_long"] = topk_long_protocol(step, dev, peaks)
    if "varlen" in parts and rank == 0 and extra:
        comp["varlen_fp8"] = fp8_prefill_protocol(step, dev, peaks, flush)
        tts.check_status(step.status, "bench fp8 prefill protocol")
    if "vision" in parts and rank == 0 and extra:
        comp["vision_qkv_rope"] = qkv_rope_protocol(step, dev, peaks, flush)
        tts.check_status(step.status, "bench qkv_rope protocol")
    if "sparse" in parts and rank == 0 and extra:
        comp["sparse_decode"] = decode_protocol(step, dev, peaks)
        comp["sparse_decode_small"] = decode_protocol(step, dev, peaks, nreq=8)
        tts.check_status(step.status, "bench decode protocol")
        tts.check_status(step.status, "bench top-k protocol")
    dom = max(parts, key=lambda p: comp[p]["ms"])
    dc = comp[dom]
    if dom in ("vision", "varlen"):
        roof = {"bound": "tensor", "achieved": dc["tflops"], "peak": tensor_peak,
                "unit": "TFLOP/s", "frac": dc["tflops"] / tensor_peak}
    elif dom == "topk":
        roof = {"bound": "hbm", "achieved": dc["gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": dc["frac_hbm"]}
    else:
        roof = {"bound": "tensor", "achieved": dc["tflops"], "peak": tensor_peak,
                "unit": "TFLOP/s", "frac": dc["tflops"] / tensor_peak}
    roof["kernel"] = dc["kernel"]
    roof["traffic"] = profiled_traffic(dom)
    roof["peak_source"] = f"{peak_src} ({'hbm_gbs' if roof['unit'] == 'GB/s' else tensor_peak_name})"

    # ---- end to end through the public API: pinned host inputs in, results out ----
    # Three streams: copies in, the calls, copies out. Each unit's calls wait for its
    # own inputs only and its copy-out waits for its calls, so the host link moves the
    # next unit's inputs and the previous unit's results while the GPU computes.
    e2e = None
    if rank == 0 or world > 1:
        units = step.e2e_units(parts)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        h_in = [[x.cpu().pin_memory() for x in u[1]] for u in units]
        h_out = [[torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in u[2]] for u in units]
        n_e2e = max(1, min(args.steps, 10))
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev_flush = torch.cuda.Event()
        ev_in = [torch.cuda.Event() for _ in units]
        ev_run = [torch.cuda.Event() for _ in units]
        times = []
        for _ in range(n_e2e + 1):  # the first pass warms the three-stream schedule
            flush.zero_()
            ev_flush.record(stream)
            s_in.wait_event(ev_flush)
            e0.record(s_in)
            for i, (name, ins, outs, run) in enumerate(units):
                with torch.cuda.stream(s_in):
                    for d, h in zip(ins, h_in[i]):
                        d.copy_(h, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                run()
                ev_run[i].record(stream)
                s_out.wait_event(ev_run[i])
                with torch.cuda.stream(s_out):
                    for h, d in zip(h_out[i], outs):
                        h.copy_(d, non_blocking=True)
            s_out.wait_event(ev_run[-1])
            e1.record(s_out)
            e1.synchronize()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        ms_e2e = max_over_ranks(float(np.median(times[1:])), world)
        e2e = {"value": job_flops / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": int(sum(x.numel() * x.element_size()
                                             for u in units for x in u[1])),
               "d2h_bytes_per_step": int(sum(x.numel() * x.element_size()
                                             for u in units for x in u[2])),
               "stat": f"median of {n_e2e} steps",
               "pipeline": "copy-in / compute / copy-out streams; units " +
                           ", ".join(u[0] for u in units)}
        tts.check_status(step.status, "bench e2e")

    if rank != 0:
        return
    cpu_base = None
    if world == 1 and not args.no_cpu_baseline:
        cpu_base = cpu_baseline_entry(oracle_sample(*sized_sample(15.0)))
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "strong" if args.shard else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "parallelism": (f"one step sharded over {world} GPUs: dense attention by "
                                   "(sequence, KV-head group), top-k by rows, sparse attention "
                                   "by queries" + (", results all-gathered" if gather else ""))
                   if args.shard else (f"replicas x{world}" if world > 1 else "single GPU"),
                   "shard_plan_rank0": step.plan, "lengths_varlen": step.var.lengths_q,
                   "schedule": ("the parts one after another on one stream" if args.serial
                                else "each part on a stream of its own (vision, varlen, sparse, "
                                     "top-k issued in that order; the parts are independent), "
                                     "so a part's last partial wave shares the GPU with the "
                                     "next part's first CTAs; per-part figures from a pass with "
                                     "the parts one after another"),
                   "ms_per_step_parts_in_sequence": float(np.mean(serial_ms)),
                   "l2": "flushed between steps (256 MB write outside the step's events); "
                         "step inputs also exceed L2",
                   "ms_wall_timed_region": (t_wall1 - t_wall0) * 1e3},
        "components": comp, "roofline": roof, "cpu_baseline": cpu_base, "e2e": e2e,
        "gpu_launches": sum(LAUNCHES[p] for p in parts) * args.steps, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--parts", default="vision,varlen,topk,sparse",
                    help="subset of the step to run (profiling); default: the whole hot path")
    ap.add_argument("--shard", action="store_true",
                    help="split one step's units over the ranks (strong scaling) instead of "
                         "running one whole step per rank (weak scaling, the default)")
    ap.add_argument("--gather", action="store_true",
                    help="with --shard: all-gather every rank's results inside the step")
    ap.add_argument("--serial", action="store_true",
                    help="time the step with its parts one after another on one stream")
    ap.add_argument("--small", action="store_true",
                    help="profiling-sized varlen batch (4 sequences, 10096 tokens)")
    args = ap.parse_args()
    rank, world, local = dist_init(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
