#!/usr/bin/env python3
"""Decode-attention benchmark (one JSON line on rank 0).

Headline workload: the Qwen3-8B-shaped layer (1 sequence, 16384 contiguous cells, 32
query / 8 KV heads, head_dim 128, f16 K/V, split 256).  One step = one decode token's
attention over all 36 layers: 36 kvattn_decode calls on 36 distinct layer buffers
(2.25 GiB of K/V, larger than L2, so the rotation defeats L2 reuse without a flush).

  value       effective KV GB/s over the timed steps (K + V bytes of every valid cell,
              read once per op), device-timed with CUDA events, inputs resident in HBM.
  roofline    the split-decode kernel alone (kvattn_decode_partials): its average launch
              duration over back-to-back launches replayed from a CUDA graph, CUDA events
              on its stream, against MEASURED_PEAKS.json hbm_gbs.
  e2e         the same metric through the public API from pinned host buffers: q copied
              in, 36 decode calls, out/lse copied back, every step, host-timed with a
              synchronize per step; the step's calls and copies are recorded once as a
              CUDA graph and replayed (e2e_eager: the same with every call launched from
              Python).
  us_per_op_interleaved  the layer's cost when other kernels run between the attention
              calls (a stand-in projection GEMV before each call, so no attention launch
              overlaps the previous one): step time with attention minus the stand-ins' own.
  workloads   the other decode-attention workloads (tiny, multi-slot plan, Q8_0 long
              context, window + host tail) timed the same way; each carries its own
              cpu_baseline (the oracle on all host cores and on one thread).  The tiny
              workload also reports device time per call from a replayed CUDA graph.
  cpu_baseline  the fp64 oracle on the host cores over a bounded sample of the workload.

--impl reference times the oracle (the plain CPU implementation) on the same metric.
Under torchrun each rank runs an independent replica (no collective on the data path).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/op and effective KV GB/s vs 8 TB/s HBM (PCIe for host tail)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


# ------------------------------------------------------------------ helpers

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(torch, ms, world, device):
    """The slowest rank's time (ms): every replica's work counts only once all are done."""
    if world > 1:
        t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    return ms


def whole_job_gbs(bytes_per_rank_step, world, ms_per_step):
    """Whole-job throughput: the bytes every rank processed per step over the slowest rank's
    step time."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "kv_cache_decode_02_gb300", "csrc")
    for name in ("decode.cu", "kvattn_internal.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(profile_name: str):
    """dram bytes per launch recorded by an ncu summary under profiles/, if it was taken
    on the current kernel source (otherwise None)."""
    path = os.path.join(ROOT, "profiles", profile_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != kernel_source_hash():
        return None
    return int(t.group(1))


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = os.path.join("/tmp", f"kvattn_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
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
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm

class Qwen3Layers:
    """36 distinct layer buffers of the Qwen3-8B-shaped decode workload."""

    def __init__(self, K, torch, layers):
        from kv_cache_decode_02_gb300 import inputs
        w = inputs.QWEN3_8B_LAYER
        self.w = w
        self.layers = layers
        D, Hk, H, N = w.head_dim, w.n_head_kv, w.n_head, w.n_cells
        self.q_host = torch.empty((layers, 1, H, D), dtype=torch.float16).pin_memory()
        self.k, self.v = [], []
        self.kv_host0 = None
        for l in range(layers):
            if l == 0:
                # layer 0 comes from the shared seeded generator so the oracle can check it
                q0 = inputs.make_q(w, layer=0)
                k0, v0 = inputs.make_kv_f16(w, layer=0)
                self.kv_host0 = (q0, k0, v0)
                self.q_host[0].copy_(torch.from_numpy(q0))
                self.k.append(torch.from_numpy(k0).cuda())
                self.v.append(torch.from_numpy(v0).cuda())
            else:
                self.q_host[l].copy_(inputs.normal_f16_torch((1000 + w.number, l), (1, H, D), "cpu"))
                self.k.append(inputs.normal_f16_torch((2000 + w.number, l), (N, Hk, D), "cuda"))
                self.v.append(inputs.normal_f16_torch((3000 + w.number, l), (N, Hk, D), "cuda"))
        self.q = self.q_host.cuda()
        self.lens = torch.tensor([N], dtype=torch.int32, device="cuda")
        self.out = torch.empty((layers, 1, H, D), dtype=torch.float32, device="cuda")
        self.lse = torch.empty((layers, 1, H), dtype=torch.float32, device="cuda")
        self.out_host = torch.empty_like(self.out, device="cpu").pin_memory()
        self.lse_host = torch.empty_like(self.lse, device="cpu").pin_memory()
        self.ws = K.decode_workspace(1, H, D, N, w.split)
        n_split = -(-N // w.split)
        self.part_o = torch.empty((1, n_split, H, D), dtype=torch.float32, device="cuda")
        self.part_lse = torch.empty((1, n_split, H), dtype=torch.float32, device="cuda")
        self.bytes_per_op = N * Hk * D * 2 * 2
        self.scale = 1.0 / math.sqrt(D)

    def call(self, K, l, stream):
        w = self.w
        K.kvattn_decode(self.q[l], self.k[l], self.v[l], None, None, K.KVATTN_KV_F16, w.n_cells, None, 0,
                        self.lens, 1, w.n_cells, w.n_head, w.n_head_kv, w.head_dim, w.split, self.scale,
                        self.out[l], self.lse[l], self.ws, self.ws.numel(), stream)

    def call_partials(self, K, l, stream):
        w = self.w
        K.kvattn_decode_partials(self.q[l], self.k[l], self.v[l], None, None, K.KVATTN_KV_F16, w.n_cells,
                                 None, 0, self.lens, 1, w.n_cells, w.n_head, w.n_head_kv, w.head_dim,
                                 w.split, self.scale, self.part_o, self.part_lse, self.ws,
                                 self.ws.numel(), stream)

    def step(self, K, stream):
        for l in range(self.layers):
            self.call(K, l, stream)


def time_events(torch, stream, fn, iters):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(iters):
        fn()
    end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / iters  # ms


def h2d_bandwidth(torch):
    """Pinned host -> device copy bandwidth (GB/s): one 1 GiB copy and 1 MiB copies."""
    n = 1 << 30
    host = torch.empty(n, dtype=torch.uint8).pin_memory()
    devb = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    big = []
    for _ in range(5):
        big.append(time_events(torch, s, lambda: devb.copy_(host, non_blocking=True), 1))
    mib = 1 << 20
    chunks = [(host[i * mib:(i + 1) * mib], devb[i * mib:(i + 1) * mib]) for i in range(1024)]

    def many():
        for h, d in chunks:
            d.copy_(h, non_blocking=True)
    small = [time_events(torch, s, many, 1) for _ in range(3)]
    del host, devb
    return n / (min(big) * 1e-3) / 1e9, n / (min(small) * 1e-3) / 1e9


def quantized_kv_torch(torch, w):
    """Device K/V planes of a Q8_0, Q8_0-key / Q4_0-value or Q4_0 workload, drawn with a seeded torch
    generator in the value ranges of the seeded numpy generators (int8 in [-127, 127], Q8_0
    scales U(0.001, 0.02); 4-bit pairs as bytes in [0, 255], Q4_0 scales U(0.001, 0.3))."""
    N, Hk, D = w.n_cells, w.n_head_kv, w.head_dim
    g = torch.Generator(device="cuda")
    g.manual_seed(2000 + w.number)
    if w.kv_type == "q4_0":
        kq = torch.randint(0, 256, (N, Hk, D // 2), dtype=torch.uint8, device="cuda", generator=g)
        kd = (torch.rand((N, Hk, D // 32), device="cuda", generator=g) * 0.299 + 0.001).half()
    else:
        kq = torch.randint(-127, 128, (N, Hk, D), dtype=torch.int8, device="cuda", generator=g)
        kd = (torch.rand((N, Hk, D // 32), device="cuda", generator=g) * 0.019 + 0.001).half()
    if w.kv_type in ("q8_0_q4_0", "q4_0"):
        vq = torch.randint(0, 256, (N, Hk, D // 2), dtype=torch.uint8, device="cuda", generator=g)
        vd = (torch.rand((N, Hk, D // 32), device="cuda", generator=g) * 0.299 + 0.001).half()
    else:
        vq = torch.randint(-127, 128, (N, Hk, D), dtype=torch.int8, device="cuda", generator=g)
        vd = (torch.rand((N, Hk, D // 32), device="cuda", generator=g) * 0.019 + 0.001).half()
    return kq, vq, kd, vd


def bench_workloads(K, torch, stream, peak):
    """Secondary measurements of the other decode-attention workloads (device-timed)."""
    from kv_cache_decode_02_gb300 import inputs
    res = {}
    iters = 20

    def add(name, nbytes, ms, extra=None):
        d = {"us_per_op": round(ms * 1e3, 2), "kv_gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
             "frac_of_measured_hbm": round(nbytes / (ms * 1e-3) / 1e9 / peak, 3),
             "frac_of_8tbs": round(nbytes / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 3), "kv_bytes": int(nbytes)}
        if extra:
            d.update(extra)
        res[name] = d

    def timed(fn, n=iters):
        """Mean device time (ms) of n back-to-back calls on `stream`, after one warm-up call.

        Every gated input is larger than the 129 MB L2, so nothing is flushed between calls
        (a flush by writing a buffer would leave dirty lines whose write-back the next call
        pays for)."""
        fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / n

    # tiny (L2-resident, launch-latency-bound: reported, not gated)
    w = inputs.TINY
    q = torch.from_numpy(inputs.make_q(w)).cuda()
    k, v = (torch.from_numpy(x).cuda() for x in inputs.make_kv_f16(w))
    lens = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    ws = K.decode_workspace(1, w.n_head, w.head_dim, w.n_cells, w.split)
    out = torch.empty((1, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, w.n_head), dtype=torch.float32, device="cuda")
    fn = lambda: K.kvattn_decode(q, k, v, None, None, 0, w.n_cells, None, 0, lens, 1, w.n_cells, w.n_head,
                                 w.n_head_kv, w.head_dim, w.split, 1 / math.sqrt(w.head_dim), out, lse, ws,
                                 ws.numel(), stream)
    fn()
    ms_eager = timed(fn)
    # the same calls recorded as one CUDA graph of 64 back-to-back calls and replayed: device
    # time per call without the host's enqueue (the eager figure above is bound by it)
    n_rec = 64
    g_tiny = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn_side = lambda: K.kvattn_decode(q, k, v, None, None, 0, w.n_cells, None, 0, lens, 1, w.n_cells, w.n_head,
                                          w.n_head_kv, w.head_dim, w.split, 1 / math.sqrt(w.head_dim), out, lse, ws,
                                          ws.numel(), side)
        fn_side()
    torch.cuda.synchronize()
    with torch.cuda.graph(g_tiny):
        cur = torch.cuda.current_stream()
        for _ in range(n_rec):
            K.kvattn_decode(q, k, v, None, None, 0, w.n_cells, None, 0, lens, 1, w.n_cells, w.n_head, w.n_head_kv,
                            w.head_dim, w.split, 1 / math.sqrt(w.head_dim), out, lse, ws, ws.numel(), cur)
    torch.cuda.synchronize()
    ms_graph = timed(lambda: g_tiny.replay(), 10) / n_rec
    del g_tiny
    add(w.name, w.n_cells * w.n_head_kv * w.head_dim * 4, ms_eager,
        {"gated": False, "how": "eager ctypes calls, back to back (host enqueue bound)",
         "us_per_op_graph": round(ms_graph * 1e3, 3),
         "graph_how": f"{n_rec} calls recorded in one CUDA graph, replayed; device time per call"})

    # causal multi-query decode: the Qwen3-8B-shaped layer verifying 4 and 8 draft tokens (16
    # and 32 query rows per KV head read every K/V byte once); 8 rotating layer buffers
    # exceed L2
    w = inputs.QWEN3_8B_LAYER
    n_buf = 8
    kvs = [(inputs.normal_f16_torch((2000 + w.number, l), (w.n_cells, w.n_head_kv, w.head_dim), "cuda"),
            inputs.normal_f16_torch((3000 + w.number, l), (w.n_cells, w.n_head_kv, w.head_dim), "cuda"))
           for l in range(n_buf)]
    lens = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    for n_q in (4, 8, 16):  # 16, 32 and 64 query rows per KV head (64: the tcgen05 kernel)
        qm = torch.randn((1, n_q, w.n_head, w.head_dim), device="cuda").half()
        wsm = torch.zeros(K.kvattn_decode_multi_workspace_bytes(1, n_q, w.n_head, w.head_dim, w.n_cells, 0),
                          dtype=torch.uint8, device="cuda")
        om = torch.empty((1, n_q, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
        lm = torch.empty((1, n_q, w.n_head), dtype=torch.float32, device="cuda")
        it = [0]

        def mq():
            kb, vb = kvs[it[0] % n_buf]
            it[0] += 1
            K.kvattn_decode_multi(qm, kb, vb, None, None, 0, w.n_cells, None, 0, lens, 1, w.n_cells, n_q, w.n_head,
                                  w.n_head_kv, w.head_dim, 0, 1 / math.sqrt(w.head_dim), om, lm, wsm,
                                  wsm.numel(), stream)
        add(f"qwen3_8b_layer_verify_nq{n_q}", w.n_cells * w.n_head_kv * w.head_dim * 4, timed(mq, 40),
            {"n_q": n_q, "query_rows_per_kv_head": n_q * w.n_head // w.n_head_kv, "split": "automatic"})
    del kvs

    # multi-slot GQA-6 through the compact plan (descriptors + decode + merge)
    w = inputs.MULTISLOT_PLAN
    lay = inputs.make_unified_layout(w)
    plan, plens = K.build_cell_plan(lay.encoded_cells, w.n_cells)
    kk = inputs.normal_f16_torch((2000 + w.number, 0), (w.n_cells, w.n_head_kv, w.head_dim), "cuda")
    vv = inputs.normal_f16_torch((3000 + w.number, 0), (w.n_cells, w.n_head_kv, w.head_dim), "cuda")
    q = torch.from_numpy(inputs.make_q(w)).cuda()
    plan_d = torch.from_numpy(plan).cuda()
    lens_d = torch.from_numpy(plens).cuda()
    ws = K.decode_workspace(w.n_seq, w.n_head, w.head_dim, plan.shape[1], w.split)
    out = torch.empty((w.n_seq, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
    lse = torch.empty((w.n_seq, w.n_head), dtype=torch.float32, device="cuda")
    fn = lambda: K.kvattn_decode(q, kk, vv, None, None, 0, w.n_cells, plan_d, plan.shape[1], lens_d, w.n_seq,
                                 plan.shape[1], w.n_head, w.n_head_kv, w.head_dim, w.split,
                                 1 / math.sqrt(w.head_dim), out, lse, ws, ws.numel(), stream)
    fn()
    valid = int((plan >= 0).sum())
    add(w.name, valid * w.n_head_kv * w.head_dim * 4, timed(fn), {"valid_cells": valid,
                                                                 "plan_entries": int(plens.sum())})
    # the same slots verifying 8 draft tokens each: 48 query rows per KV head (the tcgen05
    # kernel, every row of a KV head in one unit); split 512 (147 us against 157 us at 256)
    n_q, vsplit = 8, 512
    qm = inputs.normal_f16_torch((1000 + w.number, 8), (w.n_seq, n_q, w.n_head, w.head_dim), "cuda")
    wsm = torch.zeros(K.kvattn_decode_multi_workspace_bytes(w.n_seq, n_q, w.n_head, w.head_dim, plan.shape[1],
                                                            vsplit), dtype=torch.uint8, device="cuda")
    om = torch.empty((w.n_seq, n_q, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
    lm = torch.empty((w.n_seq, n_q, w.n_head), dtype=torch.float32, device="cuda")
    fm = lambda: K.kvattn_decode_multi(qm, kk, vv, None, None, 0, w.n_cells, plan_d, plan.shape[1], lens_d,
                                       w.n_seq, plan.shape[1], n_q, w.n_head, w.n_head_kv, w.head_dim, vsplit,
                                       1 / math.sqrt(w.head_dim), om, lm, wsm, wsm.numel(), stream)
    fm()
    add(w.name + "_verify_nq8", valid * w.n_head_kv * w.head_dim * 4, timed(fm),
        {"n_q": n_q, "query_rows_per_kv_head": n_q * w.n_head // w.n_head_kv, "split": vsplit})
    del kk, vv

    # a serving batch: 64 sequences x 4096 cells in one call, the automatic split
    w = inputs.BATCH64
    S, N = w.n_seq, w.n_cells
    kk = inputs.normal_f16_torch((2000 + w.number, 0), (S, N, w.n_head_kv, w.head_dim), "cuda")
    vv = inputs.normal_f16_torch((3000 + w.number, 0), (S, N, w.n_head_kv, w.head_dim), "cuda")
    q = torch.from_numpy(inputs.make_q(w)).cuda()
    lens = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    sp = K.kvattn_select_split(0, S, N, w.n_head_kv, w.head_dim)
    ws = K.decode_workspace(S, w.n_head, w.head_dim, N, sp)
    out = torch.empty((S, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
    lse = torch.empty((S, w.n_head), dtype=torch.float32, device="cuda")
    fn = lambda: K.kvattn_decode(q, kk, vv, None, None, 0, N, None, 0, lens, S, N, w.n_head, w.n_head_kv,
                                 w.head_dim, 0, 1 / math.sqrt(w.head_dim), out, lse, ws, ws.numel(), stream)
    fn()
    add(w.name, S * N * w.n_head_kv * w.head_dim * 4, timed(fn), {"split": sp, "n_seq": S})
    del kk, vv

    # f16 head_dim 256 long context, the automatic split
    w = inputs.F16_D256_LONG
    kk = inputs.normal_f16_torch((2000 + w.number, 0), (w.n_cells, w.n_head_kv, w.head_dim), "cuda")
    vv = inputs.normal_f16_torch((3000 + w.number, 0), (w.n_cells, w.n_head_kv, w.head_dim), "cuda")
    q = torch.from_numpy(inputs.make_q(w)).cuda()
    lens = torch.tensor(w.seq_lens, dtype=torch.int32, device="cuda")
    sp = K.kvattn_select_split(0, 1, w.n_cells, w.n_head_kv, w.head_dim)
    ws = K.decode_workspace(1, w.n_head, w.head_dim, w.n_cells, sp)
    out = torch.empty((1, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, w.n_head), dtype=torch.float32, device="cuda")
    fn = lambda: K.kvattn_decode(q, kk, vv, None, None, 0, w.n_cells, None, 0, lens, 1, w.n_cells, w.n_head,
                                 w.n_head_kv, w.head_dim, 0, 1 / math.sqrt(w.head_dim), out, lse, ws, ws.numel(),
                                 stream)
    fn()
    add(w.name, w.n_cells * w.n_head_kv * w.head_dim * 4, timed(fn), {"split": sp})
    # the same cache verifying 4 draft tokens (8 query rows per KV head), the same split
    n_q = 4
    qm = torch.randn((1, n_q, w.n_head, w.head_dim), device="cuda").half()
    wsm = torch.zeros(K.kvattn_decode_multi_workspace_bytes(1, n_q, w.n_head, w.head_dim, w.n_cells, sp),
                      dtype=torch.uint8, device="cuda")
    om = torch.empty((1, n_q, w.n_head, w.head_dim), dtype=torch.float32, device="cuda")
    lm = torch.empty((1, n_q, w.n_head), dtype=torch.float32, device="cuda")
    fm = lambda: K.kvattn_decode_multi(qm, kk, vv, None, None, 0, w.n_cells, None, 0, lens, 1, w.n_cells, n_q,
                                       w.n_head, w.n_head_kv, w.head_dim, sp, 1 / math.sqrt(w.head_dim), om, lm,
                                       wsm, wsm.numel(), stream)
    fm()
    add(w.name + "_verify_nq4", w.n_cells * w.n_head_kv * w.head_dim * 4, timed(fm),
        {"n_q": n_q, "query_rows_per_kv_head": n_q * w.n_head // w.n_head_kv, "split": sp})
    del kk, vv

    # Q8_0 long context, head_dim 128 and 256; and Q8_0 keys with Q4_0 values
    for w in (inputs.Q8_LONG_D128, inputs.Q8_LONG_D256, inputs.Q8Q4_LONG_D128, inputs.Q8Q4_LONG_D256,
              inputs.Q4_LONG_D128, inputs.Q4_LONG_D256):
        N, Hk, D = w.n_cells, w.n_head_kv, w.head_dim
        kq, vq, kd, vd = quantized_kv_torch(torch, w)
        kv_type = {"q8_0": 1, "q8_0_q4_0": 2, "q4_0": 3}[w.kv_type]
        q = torch.from_numpy(inputs.make_q(w)).cuda()
        lens = torch.tensor([N], dtype=torch.int32, device="cuda")
        ws = K.decode_workspace(1, w.n_head, D, N, w.split)
        out = torch.empty((1, w.n_head, D), dtype=torch.float32, device="cuda")
        lse = torch.empty((1, w.n_head), dtype=torch.float32, device="cuda")
        fn = lambda: K.kvattn_decode(q, kq, vq, kd, vd, kv_type, N, None, 0, lens, 1, N, w.n_head, Hk, D,
                                     w.split, 1 / math.sqrt(D), out, lse, ws, ws.numel(), stream)
        fn()
        # per (cell, head): K and V rows of D int8 (or D/2 bytes of 4-bit values) + D/32 f16 scales
        kb, vb = (D // 2 if kv_type == 3 else D), (D if kv_type == 1 else D // 2)
        kv_bytes = N * Hk * ((kb + D // 16) + (vb + D // 16))
        add(w.name, kv_bytes, timed(fn))
        if w is inputs.Q8_LONG_D128 or w is inputs.Q8_LONG_D256:
            # the same cache verifying 4 draft tokens (16 query rows per KV head)
            n_q = 4
            qm = torch.randn((1, n_q, w.n_head, D), device="cuda").half()
            wsm = torch.zeros(K.kvattn_decode_multi_workspace_bytes(1, n_q, w.n_head, D, N, w.split),
                              dtype=torch.uint8, device="cuda")
            om = torch.empty((1, n_q, w.n_head, D), dtype=torch.float32, device="cuda")
            lm = torch.empty((1, n_q, w.n_head), dtype=torch.float32, device="cuda")
            fm = lambda: K.kvattn_decode_multi(qm, kq, vq, kd, vd, kv_type, N, None, 0, lens, 1, N, n_q, w.n_head,
                                               Hk, D, w.split, 1 / math.sqrt(D), om, lm, wsm, wsm.numel(), stream)
            fm()
            add(w.name + "_verify_nq4", kv_bytes, timed(fm), {"n_q": n_q, "query_rows_per_kv_head": 16})
        del kq, vq, kd, vd

    # window + pinned-host tail
    w, q, k_win, v_win, k_tail, v_tail = window_tail_inputs(torch, inputs)
    N, Hk, D, H = w.n_cells, w.n_head_kv, w.head_dim, w.n_head
    n_tail = N - w.n_window
    wt = K.WindowTail()
    ws = wt.workspace(H, Hk, D, w.n_window, n_tail, w.split, w.tile_cells, w.tail_split)
    out = torch.empty((H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((H,), dtype=torch.float32, device="cuda")
    copy_stream = torch.cuda.Stream()
    fn = lambda: wt(q, k_win, v_win, k_tail, v_tail, split=w.split, tile_cells=w.tile_cells,
                    tail_split=w.tail_split, out=out, lse=lse, ws=ws, compute_stream=stream,
                    copy_stream=copy_stream)
    fn()
    torch.cuda.synchronize()
    ms_wt = timed(fn, 5)
    host_t0 = time.perf_counter()
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    host_ms = (time.perf_counter() - host_t0) * 1e3 / 3
    tail_bytes = n_tail * Hk * D * 4
    win_bytes = w.n_window * Hk * D * 4
    h2d_big, h2d_1mib = h2d_bandwidth(torch)
    tail_gbs = tail_bytes / (ms_wt * 1e-3) / 1e9
    res[w.name] = {"ms_per_op": round(ms_wt, 3), "tail_bytes": tail_bytes, "window_bytes": win_bytes,
                   "tail_gbs": round(tail_gbs, 1), "h2d_gbs_1gib_copy": round(h2d_big, 1),
                   "h2d_gbs_1mib_copies": round(h2d_1mib, 1),
                   "frac_of_measured_h2d": round(tail_gbs / h2d_big, 3),
                   "host_ms_per_call": round(host_ms, 3),
                   "model_ms": round(tail_bytes / (h2d_big * 1e9) * 1e3, 3)}
    wt.close()
    # the same window + tail, the tail read in place from pinned host memory (no staging)
    fn = lambda: K.window_tail_direct(q, k_win, v_win, k_tail, v_tail, split=w.split, tail_split=w.tail_split,
                                      out=out, lse=lse, ws=ws_direct, stream=stream)
    ws_direct = torch.zeros(K.kvattn_window_tail_direct_workspace_bytes(H, Hk, D, w.n_window, n_tail, w.split,
                                                                        w.tail_split), dtype=torch.uint8,
                            device="cuda")
    fn()
    torch.cuda.synchronize()
    ms_d = timed(fn, 5)
    gbs_d = tail_bytes / (ms_d * 1e-3) / 1e9
    res[w.name + "_direct"] = {"ms_per_op": round(ms_d, 3), "tail_bytes": tail_bytes, "tail_gbs": round(gbs_d, 1),
                              "frac_of_measured_h2d": round(gbs_d / h2d_big, 3),
                              "how": "tail rows read in place from pinned host memory by the decode kernel"}
    del k_win, v_win, k_tail, v_tail, ws, ws_direct
    for w in (inputs.STACK_TAIL_295MIB, inputs.STACK_TAIL_1815MIB):
        res[w.name] = bench_layer_stack(K, torch, w, h2d_big)
    return res


def bench_layer_stack(K, torch, w, h2d_gbs):
    """One decode token over a stack of layers that each attend a resident window and stream
    a pinned host tail, in each way the library offers, against the pages' model
    t = resident compute + tail bytes / host-link bandwidth."""
    from kv_cache_decode_02_gb300 import inputs
    L, H, Hk, D = w.layers, w.n_head, w.n_head_kv, w.head_dim
    n_win, n_tail = w.n_window, w.n_cells - w.n_window
    cs, xs = torch.cuda.Stream(), torch.cuda.Stream()
    kw = [inputs.normal_f16_torch((2000 + w.number, l), (n_win, Hk, D), "cuda") for l in range(L)]
    vw = [inputs.normal_f16_torch((3000 + w.number, l), (n_win, Hk, D), "cuda") for l in range(L)]
    kt, vt = [], []
    for l in range(L):
        kt.append(inputs.normal_f16_torch((2000 + w.number, L + l), (n_tail, Hk, D), "cuda").cpu().pin_memory())
        vt.append(inputs.normal_f16_torch((3000 + w.number, L + l), (n_tail, Hk, D), "cuda").cpu().pin_memory())
    q = torch.cat([torch.from_numpy(inputs.make_q(w, layer=l)) for l in range(L)]).cuda()
    out = torch.empty((L, H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((L, H), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()

    def timed(fn, n=3):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cs)
        for _ in range(n):
            fn()
        b.record(cs)
        b.synchronize()
        return a.elapsed_time(b) / n

    def staged(wt, ws, tile, tails=True):
        for l in range(L):
            wt(q[l], kw[l], vw[l], kt[l] if tails else None, vt[l] if tails else None, split=w.split,
               tile_cells=tile, tail_split=w.tail_split, out=out[l], lse=lse[l], ws=ws, compute_stream=cs,
               copy_stream=xs)

    tail_bytes = L * n_tail * Hk * D * 4
    ms = {}
    wt = K.WindowTail()
    ws = wt.workspace(H, Hk, D, n_win, n_tail, w.split, 512, w.tail_split)
    ms["resident_only"] = timed(lambda: staged(wt, ws, 512, tails=False))
    ms["staged_1mib_tiles_graphs"] = timed(lambda: staged(wt, ws, 512))
    wt.close()
    wt = K.WindowTail(prefetch=True)
    ws = wt.workspace(H, Hk, D, n_win, n_tail, w.split, w.tile_cells, w.tail_split)
    ms["prefetch_layer_tiles"] = timed(lambda: staged(wt, ws, w.tile_cells))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        staged(wt, ws, w.tile_cells)

    def replay():
        with torch.cuda.stream(cs):
            g.replay()
    ms["prefetch_layer_tiles_captured_step"] = timed(replay)
    del g
    wt.close()
    wsd = torch.zeros(K.kvattn_window_tail_direct_workspace_bytes(H, Hk, D, n_win, n_tail, w.split, w.tail_split),
                      dtype=torch.uint8, device="cuda")

    def direct():
        for l in range(L):
            K.window_tail_direct(q[l], kw[l], vw[l], kt[l], vt[l], split=w.split, tail_split=w.tail_split,
                                 out=out[l], lse=lse[l], ws=wsd, stream=cs)
    ms["direct"] = timed(direct)
    link_ms = tail_bytes / (h2d_gbs * 1e9) * 1e3
    d = {"layers": L, "n_window": n_win, "n_tail_per_layer": n_tail, "tail_bytes_per_token": tail_bytes,
         "link_ms": round(link_ms, 3), "model_ms": round(ms["resident_only"] + link_ms, 3)}
    for k_, v_ in ms.items():
        d[k_ + "_ms"] = round(v_, 3)
        if k_ != "resident_only":
            d[k_ + "_frac_of_link"] = round(link_ms / v_, 3)
    return d


def cpu_baseline_sample(budget_s=12.0):
    """The fp64 oracle (as it stands) on layer-0 inputs of the headline workload, repeated for
    about budget_s seconds of host time."""
    import oracle
    from kv_cache_decode_02_gb300 import inputs
    w = inputs.QWEN3_8B_LAYER
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w)
    threads = oracle.default_threads()
    nbytes = w.n_cells * w.n_head_kv * w.head_dim * 4
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.decode_f16(q, k, v, list(w.seq_lens), n_threads=threads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    # the same oracle on one core, for a short sample
    reps1, t1 = 0, time.perf_counter()
    while True:
        oracle.decode_f16(q, k, v, list(w.seq_lens), n_threads=1)
        reps1 += 1
        el1 = time.perf_counter() - t1
        if el1 >= min(3.0, budget_s / 4):
            break
    return {"value": round(nbytes * reps / el / 1e9, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"fp64 C oracle (OpenMP) on layer 0 of 36, {reps} repetition(s) in {el:.1f} s",
            "single_core": {"value": round(nbytes * reps1 / el1 / 1e9, 3), "unit": "GB/s",
                            "sample": f"{reps1} repetition(s) in {el1:.1f} s on one thread"}}


def interleaved_layer_cost(K, torch, data, reps=20):
    """The headline layer's cost inside a decode step, where other kernels run between the
    attention calls.  A stand-in for the rest of a layer -- one token through a 4096 x 12288
    bf16 projection (100 MB of weights; four rotating matrices, so L2 holds none of them) --
    runs before each of the kvattn_decode calls, so no attention launch overlaps the previous
    one (the stand-in neither lets dependents start early nor waits for them).  Both step
    forms -- stand-ins alone, stand-ins with attention -- are captured as CUDA graphs and
    replayed; the attention's cost per layer is their difference over the layers."""
    L = data.layers
    x = torch.randn((1, 4096), device="cuda", dtype=torch.bfloat16)
    Ws = [torch.randn((4096, 12288), device="cuda", dtype=torch.bfloat16) for _ in range(4)]
    y = torch.empty((1, 12288), device="cuda", dtype=torch.bfloat16)

    def standins(st):
        for l in range(L):
            torch.mm(x, Ws[l % 4], out=y)

    def with_attention(st):
        for l in range(L):
            torch.mm(x, Ws[l % 4], out=y)
            data.call(K, l, st)

    graphs = {}
    for name, fn in (("standins", standins), ("interleaved", with_attention)):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        torch.cuda.synchronize()
        graphs[name] = g
    cur = torch.cuda.current_stream()
    best = {name: float("inf") for name in graphs}
    for _ in range(3):                       # alternate the two forms, keep each one's best
        for name, g in graphs.items():
            for _ in range(3):
                g.replay()
            best[name] = min(best[name], time_events(torch, cur, g.replay, reps))
    del graphs, Ws
    us = (best["interleaved"] - best["standins"]) * 1e3 / L
    return {"us_per_op_interleaved": round(us, 3),
            "kv_gbs_interleaved": round(data.bytes_per_op / (us * 1e-6) / 1e9, 1),
            "step_ms_standins": round(best["standins"], 4), "step_ms_with_attention": round(best["interleaved"], 4),
            "how": (f"{L} x (stand-in bf16 GEMV 1x4096 @ 4096x12288, then kvattn_decode), CUDA graph, minus "
                    f"{L} stand-ins alone; per layer")}


def oracle_workload_baselines(budget_s=1.0):
    """The fp64 oracle (as it stands) on each workload of the decode-attention configurations,
    on this host's cores: all the cores of the process's affinity set over the whole op
    (repeated for about budget_s seconds, at least once), and one thread over an eighth of
    the cells of the larger workloads (the oracle's cost is linear in cells), scaled to the
    whole op.  Inputs come from the seeded numpy generators; the window + tail op is sampled
    on 65536 of its cells on all cores as well."""
    import oracle
    from oracle import plan_oracle as po
    from kv_cache_decode_02_gb300 import inputs
    threads = oracle.default_threads()
    res = {}

    def measure(name, fn, nbytes, sample, frac_all=1.0, frac_one=1.0):
        """fn(threads, frac): one oracle call over that fraction of the op's cells."""
        reps, t0 = 0, time.perf_counter()
        while True:
            fn(threads, frac_all)
            reps += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        ms_all = (time.perf_counter() - t0) * 1e3 / reps / frac_all
        t1 = time.perf_counter()
        fn(1, frac_one)
        ms_one = (time.perf_counter() - t1) * 1e3 / frac_one
        res[name] = {"ms_per_op": round(ms_all, 3), "kv_gbs": round(nbytes / (ms_all * 1e-3) / 1e9, 3),
                     "cores": threads, "kind": "oracle",
                     "sample": (f"{sample}; {reps} call(s) on {threads} threads" +
                                (f" over {frac_all:g} of the cells" if frac_all < 1 else "") +
                                (f"; one thread over {frac_one:g} of the cells, scaled" if frac_one < 1 else "")),
                     "single_core": {"ms_per_op": round(ms_one, 3),
                                     "kv_gbs": round(nbytes / (ms_one * 1e-3) / 1e9, 3)}}

    def lens_frac(lens, frac):
        return [max(1, int(round(L * frac))) for L in lens]

    for w in (inputs.TINY, inputs.QWEN3_8B_LAYER, inputs.F16_D256_LONG):
        q = inputs.make_q(w)
        k, v = inputs.make_kv_f16(w)
        measure(w.name, lambda t, f: oracle.decode_f16(q, k, v, lens_frac(w.seq_lens, f), n_threads=t),
                w.n_cells * w.n_head_kv * w.head_dim * 4, "fp64 C oracle", frac_one=1.0 if w is inputs.TINY else 0.125)
    w = inputs.BATCH64
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w)
    # one thread: 8 of the 64 sequences
    measure(w.name, lambda t, f: oracle.decode_f16(q[:max(1, int(w.n_seq * f))], k[:max(1, int(w.n_seq * f))],
                                                   v[:max(1, int(w.n_seq * f))], list(w.seq_lens)[:max(1, int(w.n_seq * f))],
                                                   n_threads=t),
            w.n_seq * w.n_cells * w.n_head_kv * w.head_dim * 4, "fp64 C oracle", frac_one=0.125)
    del k, v

    w = inputs.MULTISLOT_PLAN
    lay = inputs.make_unified_layout(w)
    plan, plens = po.build_cell_plan(lay.encoded_cells, w.n_cells)
    q = inputs.make_q(w)
    k = inputs.normal_f16(np.random.default_rng([2000 + w.number, 0]), (w.n_cells, w.n_head_kv, w.head_dim))
    v = inputs.normal_f16(np.random.default_rng([3000 + w.number, 0]), (w.n_cells, w.n_head_kv, w.head_dim))
    inputs.nan_fill_unselected(k, v, np.concatenate(lay.selected))
    valid = int((plan >= 0).sum())
    measure(w.name, lambda t, f: oracle.decode_f16(q, k, v, lens_frac(plens, f), plan=plan, n_threads=t),
            valid * w.n_head_kv * w.head_dim * 4, "fp64 C oracle through the plan", frac_one=0.125)
    del k, v

    for w, make, fn in ((inputs.Q8_LONG_D128, inputs.make_kv_q8, oracle.decode_q8_0),
                        (inputs.Q8_LONG_D256, inputs.make_kv_q8, oracle.decode_q8_0),
                        (inputs.Q8Q4_LONG_D128, inputs.make_kv_q8q4, oracle.decode_q8_0_q4_0),
                        (inputs.Q8Q4_LONG_D256, inputs.make_kv_q8q4, oracle.decode_q8_0_q4_0),
                        (inputs.Q4_LONG_D128, inputs.make_kv_q4, oracle.decode_q4_0),
                        (inputs.Q4_LONG_D256, inputs.make_kv_q4, oracle.decode_q4_0)):
        D = w.head_dim
        q = inputs.make_q(w)
        (kq, kd), (vq, vd) = make(w)
        nbytes = w.n_cells * w.n_head_kv * ((kq.shape[-1] + D // 16) + (vq.shape[-1] + D // 16))
        measure(w.name, lambda t, f: fn(q, kq, kd, vq, vd, lens_frac(w.seq_lens, f), n_threads=t), nbytes,
                "fp64 C oracle", frac_one=0.125)
        del kq, kd, vq, vd

    w = inputs.WINDOW_TAIL
    n_s = 65536
    q = inputs.make_q(w)
    k, v = inputs.make_kv_f16(w, n_cells=n_s)
    measure(w.name, lambda t, f: oracle.decode_f16(q, k, v, [max(1, int(w.n_cells * f))], n_threads=t),
            w.n_cells * w.n_head_kv * w.head_dim * 4, "fp64 C oracle on the sequence fully resident",
            frac_all=n_s / w.n_cells, frac_one=n_s / w.n_cells / 8)
    return res


def run_ours(args):
    import torch
    from kv_cache_decode_02_gb300 import kvattn as K

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peak, peak_kind = measured_peaks()
    stream = torch.cuda.current_stream()
    data = Qwen3Layers(K, torch, args.layers)

    # parity spot check of layer 0 against the oracle (rank 0)
    parity = None
    if rank == 0 and not args.no_parity:
        import oracle
        data.call(K, 0, stream)
        torch.cuda.synchronize()
        q0, k0, v0 = data.kv_host0
        wo, wl = oracle.decode_f16(q0, k0, v0, list(data.w.seq_lens))
        diff = data.out[0].cpu().numpy().astype(np.float64) - wo
        parity = {"max_abs_o": float(np.max(np.abs(diff))),
                  "max_abs_lse": float(np.max(np.abs(data.lse[0].cpu().numpy() - wl))),
                  "rmse_o": float(np.sqrt(np.mean(diff ** 2))),
                  "tolerance": {"max_abs_o": 2e-3, "max_abs_lse": 1e-4, "rmse_o": 3e-4},
                  "layer": 0}

    # capture one step (all layers) into a CUDA graph
    graph = None
    if not args.eager:
        data.step(K, stream)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            data.step(K, side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            data.step(K, torch.cuda.current_stream())
        torch.cuda.synchronize()

    def step():
        if graph is not None:
            graph.replay()
        else:
            data.step(K, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    # keep the GPU under load for ~1 s so that the clock samples see it (not timed)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        for _ in range(50):
            step()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(torch, ev0.elapsed_time(ev1) / args.steps, world, "cuda")
    step_bytes = data.bytes_per_op * args.layers
    value = whole_job_gbs(step_bytes, world, ms)

    # the dominant kernel alone: its average launch duration over back-to-back launches
    # (one per layer buffer, replayed from a CUDA graph so host launch cost cannot gap
    # them), events on the launching stream at both ends
    for l in range(args.layers):
        data.call_partials(K, l, stream)
    torch.cuda.synchronize()
    kgraph = None
    if not args.eager:
        kgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kgraph):
            for l in range(args.layers):
                data.call_partials(K, l, torch.cuda.current_stream())
        torch.cuda.synchronize()

    def kernel_pass():
        if kgraph is not None:
            kgraph.replay()
        else:
            for l in range(args.layers):
                data.call_partials(K, l, stream)
    kernel_pass()
    reps = max(1, args.kernel_reps)
    n_launch = reps * args.layers
    ka, kb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ka.record(stream)
    for _ in range(reps):
        kernel_pass()
    kb.record(stream)
    torch.cuda.synchronize()
    kern_ms = ka.elapsed_time(kb) / n_launch
    del kgraph
    achieved = data.bytes_per_op / (kern_ms * 1e-3) / 1e9
    traffic = profiled_traffic("split_decode_f16_qwen3_8b_layer.md")

    # the layer with other kernels between the attention calls (no cross-call overlap)
    inter = None
    if not args.no_interleaved and not args.eager:
        inter = interleaved_layer_cost(K, torch, data)

    # end to end through the API with host buffers
    e2e = e2e_eager = None
    if not args.no_e2e:
        def e2e_step(st):
            data.q.copy_(data.q_host, non_blocking=True)
            data.step(K, st)
            data.out_host.copy_(data.out, non_blocking=True)
            data.lse_host.copy_(data.lse, non_blocking=True)

        def host_timed(fn):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(args.steps):
                fn()
                stream.synchronize()
            return (time.perf_counter() - t0) / args.steps

        # eager: every call launched from Python
        el_eager = host_timed(lambda: e2e_step(stream))
        # graph: the same public-API calls and copies recorded once and replayed per step
        el_graph = None
        if not args.eager:
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                e2e_step(torch.cuda.current_stream())
            torch.cuda.synchronize()
            el_graph = host_timed(g_e2e.replay)
            del g_e2e
        el = el_graph if el_graph is not None else el_eager
        io = {"h2d_bytes_per_step": int(data.q_host.numel() * 2),
              "d2h_bytes_per_step": int(data.out.numel() * 4 + data.lse.numel() * 4)}
        e2e = {"value": round(step_bytes / el / 1e9, 1), "unit": "GB/s", "ms_per_step": round(el * 1e3, 4), **io,
               "how": ("pinned q in, 36 kvattn_decode calls, out/lse out, recorded once as a CUDA graph and "
                       "replayed; host-timed per step with a synchronize" if el_graph is not None else
                       "pinned q in, 36 eager kvattn_decode calls, out/lse out, host-timed per step")}
        e2e_eager = {"value": round(step_bytes / el_eager / 1e9, 1), "unit": "GB/s",
                     "ms_per_step": round(el_eager * 1e3, 4), **io,
                     "how": "pinned q in, 36 eager kvattn_decode calls from Python, out/lse out, host-timed per step"}

    workloads = None
    if rank == 0 and not args.no_workloads:
        del graph
        workloads = bench_workloads(K, torch, stream, peak)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sample(args.cpu_budget)
        if workloads is not None and not args.no_workload_cpu:
            for name, d in oracle_workload_baselines().items():
                if name in workloads:
                    workloads[name]["cpu_baseline"] = d
                elif name == "qwen3_8b_layer_n16384":
                    cpu["per_layer_oracle"] = d

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"qwen3_8b_layer_n16384 x{args.layers} layers", "n_seq": 1,
                       "n_cells": data.w.n_cells, "n_head": data.w.n_head, "n_head_kv": data.w.n_head_kv,
                       "head_dim": data.w.head_dim, "split": data.w.split, "kv": "f16",
                       "l2": "36 distinct layer buffers (2.25 GiB) rotate; larger than the 129 MB L2, no flush",
                       "launch": "eager" if args.eager else f"CUDA graph of {args.layers} x kvattn_decode",
                       "parallelism": f"replicas x{world}"},
            "us_per_op": round(ms * 1e3 / args.layers, 3),
            "us_per_op_interleaved": inter["us_per_op_interleaved"] if inter else None,
            "interleaved": inter,
            "us_per_token_36_layers": round(ms * 1e3 * 36 / args.layers, 2),
            "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 3),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 3), "traffic": traffic, "peak_kind": peak_kind,
                         "kernel": "split_decode_f16_d128", "kernel_us": round(kern_ms * 1e3, 3),
                         "algorithmic_bytes_per_launch": data.bytes_per_op},
            "gpu_launches": args.steps * args.layers * 2,
            "clocks": clocks, "parity": parity, "e2e": e2e, "e2e_eager": e2e_eager, "cpu_baseline": cpu,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    """The plain fp64 CPU oracle on the headline workload: each step is one layer of the
    36 (a bounded sample), reported in the same unit."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from kv_cache_decode_02_gb300 import inputs
    w = inputs.QWEN3_8B_LAYER
    threads = oracle.default_threads()
    nbytes = w.n_cells * w.n_head_kv * w.head_dim * 4
    data = [(inputs.make_q(w, layer=l), *inputs.make_kv_f16(w, layer=l)) for l in range(2)]
    for i in range(args.warmup):
        q, k, v = data[i % 2]
        oracle.decode_f16(q, k, v, list(w.seq_lens), n_threads=threads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        q, k, v = data[i % 2]
        oracle.decode_f16(q, k, v, list(w.seq_lens), n_threads=threads)
    el = time.perf_counter() - t0
    value = nbytes * args.steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "qwen3_8b_layer_n16384 (one layer per step)", "n_seq": 1,
                       "n_cells": w.n_cells, "n_head": w.n_head, "n_head_kv": w.n_head_kv,
                       "head_dim": w.head_dim, "split": w.split, "kv": "f16"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"one of 36 layers per step, {args.steps} steps"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def window_tail_inputs(torch, inputs, n_tail=None):
    """The window + tail workload: the resident window on the device, the older tail in
    pinned host memory (filled through the device in 64K-cell pieces), and q.  n_tail: a
    shorter tail (profiling the host link on a small case); the window is unchanged."""
    import dataclasses
    w = inputs.WINDOW_TAIL
    if n_tail is not None:
        w = dataclasses.replace(w, name=f"window_tail_n{w.n_window + n_tail}", n_cells=w.n_window + n_tail,
                                seq_lens=(w.n_window + n_tail,))
    N, Hk, D = w.n_cells, w.n_head_kv, w.head_dim
    n_tail = N - w.n_window
    k_win = inputs.normal_f16_torch((2000 + w.number, 1), (w.n_window, Hk, D), "cuda")
    v_win = inputs.normal_f16_torch((3000 + w.number, 1), (w.n_window, Hk, D), "cuda")
    k_tail = torch.empty((n_tail, Hk, D), dtype=torch.float16).pin_memory()
    v_tail = torch.empty((n_tail, Hk, D), dtype=torch.float16).pin_memory()
    chunk = 65536
    for lo in range(0, n_tail, chunk):
        hi = min(n_tail, lo + chunk)
        k_tail[lo:hi].copy_(inputs.normal_f16_torch((2000 + w.number, 2, lo), (hi - lo, Hk, D), "cuda"))
        v_tail[lo:hi].copy_(inputs.normal_f16_torch((3000 + w.number, 2, lo), (hi - lo, Hk, D), "cuda"))
    q = torch.from_numpy(inputs.make_q(w)[0]).cuda()
    return w, q, k_win, v_win, k_tail, v_tail


def profile_verify(args):
    """--kernel-reps calls of causal multi-query decode on the Qwen3-8B-shaped layer (16384
    cells, 32/8 heads, split 256) verifying 4, 8 or 16 draft tokens, for profilers."""
    import torch
    from kv_cache_decode_02_gb300 import inputs
    from kv_cache_decode_02_gb300 import kvattn as K
    w = inputs.QWEN3_8B_LAYER
    n_q = int(args.profile_workload.rsplit("nq", 1)[1])
    N, H, Hk, D = w.n_cells, w.n_head, w.n_head_kv, w.head_dim
    k = inputs.normal_f16_torch((2000 + w.number, 0), (N, Hk, D), "cuda")
    v = inputs.normal_f16_torch((3000 + w.number, 0), (N, Hk, D), "cuda")
    q = inputs.normal_f16_torch((1000 + w.number, 9), (1, n_q, H, D), "cuda")
    lens = torch.tensor([N], dtype=torch.int32, device="cuda")
    ws = torch.zeros(K.kvattn_decode_multi_workspace_bytes(1, n_q, H, D, N, w.split), dtype=torch.uint8,
                     device="cuda")
    for _ in range(args.kernel_reps):
        K.decode_multi(q, k, v, lens, split=w.split, ws=ws)
    torch.cuda.synchronize()
    print(f"{args.profile_workload}: {args.kernel_reps} calls done")


def profile_plan(args):
    """--kernel-reps kvattn_decode calls of the multi-slot plan workload (4 GQA-6 sequences
    through a compact plan with ~10 % holes, split 256), for profilers."""
    import torch
    from kv_cache_decode_02_gb300 import inputs
    from kv_cache_decode_02_gb300 import kvattn as K
    w = inputs.MULTISLOT_PLAN
    lay = inputs.make_unified_layout(w)
    plan, plens = K.build_cell_plan(lay.encoded_cells, w.n_cells)
    k = inputs.normal_f16_torch((2000 + w.number, 0), (w.n_cells, w.n_head_kv, w.head_dim), "cuda")
    v = inputs.normal_f16_torch((3000 + w.number, 0), (w.n_cells, w.n_head_kv, w.head_dim), "cuda")
    q = torch.from_numpy(inputs.make_q(w)).cuda()
    plan_d = torch.from_numpy(plan).cuda()
    lens_d = torch.from_numpy(plens).cuda()
    for _ in range(args.kernel_reps):
        K.decode(q, k, v, lens_d, split=w.split, cell_plan=plan_d, n_cells=w.n_cells)
    torch.cuda.synchronize()
    print(f"{args.profile_workload}: {args.kernel_reps} calls done ({int((plan >= 0).sum())} valid cells)")


def profile_interleaved(args):
    """--kernel-reps decode steps of the headline layers with the stand-in projection before
    each kvattn_decode call (launched eagerly), for an ncu launch list."""
    import torch
    from kv_cache_decode_02_gb300 import kvattn as K
    data = Qwen3Layers(K, torch, args.layers)
    x = torch.randn((1, 4096), device="cuda", dtype=torch.bfloat16)
    Ws = [torch.randn((4096, 12288), device="cuda", dtype=torch.bfloat16) for _ in range(4)]
    y = torch.empty((1, 12288), device="cuda", dtype=torch.bfloat16)
    st = torch.cuda.current_stream()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()          # a profiler started with --profile-from-start off sees only the steps
    for _ in range(args.kernel_reps):
        for l in range(args.layers):
            torch.mm(x, Ws[l % 4], out=y)
            data.call(K, l, st)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    print(f"qwen3_8b_interleaved: {args.kernel_reps} steps done")


def profile_window_tail(args):
    """--kernel-reps calls of the window + tail op (staged 1 MiB tiles through the copy
    kernel, or the tail read in place), for profilers (no timing, no JSON line).  The
    window_tail_n81920 names keep the 16384-cell window with a 65536-cell tail (268 MB of
    pinned host memory), small enough for multi-pass counter captures."""
    import torch
    from kv_cache_decode_02_gb300 import inputs
    from kv_cache_decode_02_gb300 import kvattn as K
    small = args.profile_workload.startswith("window_tail_n81920")
    w, q, k_win, v_win, k_tail, v_tail = window_tail_inputs(torch, inputs, 65536 if small else None)
    Hk, D, H = w.n_head_kv, w.head_dim, w.n_head
    n_tail = w.n_cells - w.n_window
    out = torch.empty((H, D), dtype=torch.float32, device="cuda")
    lse = torch.empty((H,), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    if args.profile_workload.endswith("_direct"):
        ws = torch.zeros(K.kvattn_window_tail_direct_workspace_bytes(H, Hk, D, w.n_window, n_tail, w.split,
                                                                     w.tail_split), dtype=torch.uint8, device="cuda")
        for _ in range(args.kernel_reps):
            K.window_tail_direct(q, k_win, v_win, k_tail, v_tail, split=w.split, tail_split=w.tail_split,
                                 out=out, lse=lse, ws=ws, stream=stream)
    else:
        wt = K.WindowTail()
        ws = wt.workspace(H, Hk, D, w.n_window, n_tail, w.split, w.tile_cells, w.tail_split)
        copy_stream = torch.cuda.Stream()
        for _ in range(args.kernel_reps):
            wt(q, k_win, v_win, k_tail, v_tail, split=w.split, tile_cells=w.tile_cells, tail_split=w.tail_split,
               out=out, lse=lse, ws=ws, compute_stream=stream, copy_stream=copy_stream)
        torch.cuda.synchronize()
        wt.close()
    torch.cuda.synchronize()
    print(f"{args.profile_workload}: {args.kernel_reps} calls done")


def PROFILE_WORKLOADS(inputs):
    return (inputs.Q8_LONG_D128, inputs.Q8_LONG_D256, inputs.Q8Q4_LONG_D128, inputs.Q8Q4_LONG_D256,
            inputs.Q4_LONG_D128, inputs.Q4_LONG_D256)


def profile_workload(args):
    """A few launches of one decode-attention workload's kvattn_decode_partials, for
    profilers (no timing, no JSON line).  Inputs are built on the device with torch RNG in
    the workload's shapes and value ranges."""
    import torch
    from kv_cache_decode_02_gb300 import inputs
    from kv_cache_decode_02_gb300 import kvattn as K
    w = {x.name: x for x in PROFILE_WORKLOADS(inputs)}[args.profile_workload]
    N, H, Hk, D = w.n_cells, w.n_head, w.n_head_kv, w.head_dim
    kq, vq, kd, vd = quantized_kv_torch(torch, w)
    kv_type = {"q8_0": K.KVATTN_KV_Q8_0, "q8_0_q4_0": K.KVATTN_KV_Q8_0_Q4_0, "q4_0": K.KVATTN_KV_Q4_0}[w.kv_type]
    q = torch.from_numpy(inputs.make_q(w)).cuda()
    lens = torch.tensor([N], dtype=torch.int32, device="cuda")
    n_split = -(-N // w.split)
    part_o = torch.empty((1, n_split, H, D), dtype=torch.float32, device="cuda")
    part_lse = torch.empty((1, n_split, H), dtype=torch.float32, device="cuda")
    ws = K.decode_workspace(1, H, D, N, w.split)
    for _ in range(args.kernel_reps):
        K.kvattn_decode_partials(q, kq, vq, kd, vd, kv_type, N, None, 0, lens, 1, N, H, Hk, D, w.split,
                                 1 / math.sqrt(D), part_o, part_lse, ws, ws.numel())
    torch.cuda.synchronize()
    print(f"{args.profile_workload}: {args.kernel_reps} launches done")


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=36)
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before timing")
    ap.add_argument("--kernel-reps", type=int, default=20)
    ap.add_argument("--eager", action="store_true", help="launch each call instead of a CUDA graph")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-workload-cpu", action="store_true", help="skip the oracle on each secondary workload")
    ap.add_argument("--no-interleaved", action="store_true")
    ap.add_argument("--profile-workload", choices=["qwen3_8b_interleaved", "q8_0_n131072_d128", "q8_0_n131072_d256", "q8_0_q4_0_n131072_d128",
                                                   "q8_0_q4_0_n131072_d256", "q4_0_n131072_d128",
                                                   "q4_0_n131072_d256", "window_tail_n524288",
                                                   "window_tail_n524288_direct", "window_tail_n81920",
                                                   "window_tail_n81920_direct", "qwen3_8b_layer_verify_nq4",
                                                   "qwen3_8b_layer_verify_nq8", "qwen3_8b_layer_verify_nq16",
                                                   "multislot_gqa6_plan"],
                    help="only launch this workload's split decode (window + tail: the whole op) "
                         "--kernel-reps times (for ncu)")
    args = ap.parse_args()
    if args.profile_workload:
        if args.profile_workload == "qwen3_8b_interleaved":
            profile_interleaved(args)
        elif args.profile_workload.startswith("window_tail"):
            profile_window_tail(args)
        elif args.profile_workload.startswith("qwen3_8b_layer_verify"):
            profile_verify(args)
        elif args.profile_workload == "multislot_gqa6_plan":
            profile_plan(args)
        else:
            profile_workload(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
