#!/usr/bin/env python3
"""Throughput of the Hierarchical Sparse Indexer decode hot path on GB300.

One step = one pass of the whole path over the resident workload:
  per Full layer: quantise q (NVFP4), score every visible key (tcgen05 FP4),
                  exact top-512;
  then (decoder workloads): the candidate pool from the fused block maxima
                  (blocks of 8, keep 2048, newest pinned, boolean bit table),
                  and per Reindex layer: quantise q, score only the pooled
                  keys (whole 576-byte blocks gathered), exact top-512.
The headline runs on NVFP4 records (72 B per key). After the timed steps the
JSON line also carries:
  mxfp4          the step on MXFP4 records (68 B per key, the pages' own format);
  reindex        one Reindex layer timed alone, and the pages' dense masked form;
  mainkv_gather  gather(main_kv, topk) of every layer's top-512 from the FP4 main KV;
  serve          decode steps over growing caches (append, step, gathers per token).
The default workload is 64 decode queries at 1,048,576 visible keys each with
4 Reindex layers. K caches are generated from the seeded recipe, quantised on
the GPU and stay resident (4.83 GB > L2, so no L2 flush is needed).

Output: one JSON line (rank 0). `value` is (query, key) pairs scored per
second over the whole job; `e2e` repeats the measurement with each step's
inputs (bf16 q, w) copied from pinned host memory and its results (top-512
indices and values of every layer) copied back inside the timed region.
`--impl reference` times the CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import inputs  # noqa: E402

METRIC = "indexer (query,key) pairs scored/s + top-512/s at 1M ctx; % FP4-TC/HBM roofline"
UNIT = "pairs/s"
K_TOP = 512
PROFILE_SUMMARY = {"nvfp4": os.path.join(ROOT, "profiles", "score_full_decode_b64_n1m.md"),
                   "mxfp4": os.path.join(ROOT, "profiles", "score_full_mxfp4_decode_b64_n1m.md")}
KERNEL_SOURCES = ["score.cuh", "ptx.cuh", "common.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["hsi", "reference"], default="hsi")
    ap.add_argument("--workload", type=int, default=2, help="0..3 (see inputs.workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--format", choices=["nvfp4", "mxfp4"], default="nvfp4",
                    help="record format of the headline step")
    ap.add_argument("--no-mxfp4", action="store_true", help="skip the extra step on MXFP4 records")
    ap.add_argument("--no-mainkv", action="store_true", help="skip the main-KV gather measurement")
    ap.add_argument("--no-serve", action="store_true", help="skip the serving-step measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the calibration, the other workloads and the chunked-prefill workload")
    ap.add_argument("--profile", action="store_true", help="cudaProfilerStart/Stop around the timed steps")
    ap.add_argument("--queries", type=int, default=0, help="use only the first N queries (profiling captures)")
    ap.add_argument("--case", choices=["prefill_score", "prefill_layer", "rowsel", "gather", "reindex", "reindex_gather", "pool"], default=None,
                    help="run only one kernel's case, --steps times, and exit (profiling captures): the chunked-"
                         "prefill scoring phase, the whole prefill layer, the prefill selection phase, or the "
                         "main-KV gather of five layers' top-512 lists")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers --

def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "long_context_decode_lightning_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(fmt: str = "nvfp4"):
    """dram bytes per launch of the scoring kernel (records of format fmt) from
    the committed ncu summary, if it was taken on the current kernel source."""
    try:
        txt = open(PROFILE_SUMMARY[fmt]).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="hsi_clocks_", suffix=".csv")
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------- device workload --

class DeviceWorkload:
    """The workload resident on one GPU, and one step of the path over it."""

    HEADROOM = 256  # rows of room per cache for appended decode tokens

    def __init__(self, wl: inputs.Workload, dev, log, fmt: int = 0):
        import torch

        import long_context_decode_lightning_gb300 as hsi
        self.torch, self.hsi, self.wl, self.dev = torch, hsi, wl, dev
        # record format of q and K: NVFP4 (576-byte records, tensor scales) or
        # MXFP4 (544-byte records, no tensor scales: g_q and g_k stay None)
        self.fmt = fmt
        self.mx = fmt == hsi.FMT_MXFP4
        REC = self.rec = hsi.rec_bytes(fmt)
        B = wl.B
        self.B = B
        self.maxv = max(wl.n_visible)
        signs = wl.signs()
        seqs = sorted(set(wl.query_seq))
        # --- K caches: one record buffer per Full layer, sequences back to back
        self.k_rec, self.g_k = [], []
        rec_off = {}
        off = 0
        for s in seqs:
            rec_off[s] = off
            off += hsi.n_records(wl.seq_len[s] + self.HEADROOM)
        t0 = time.time()
        stage = [torch.empty(max(wl.seq_len) * 128, dtype=torch.int16).pin_memory() for _ in range(2)]
        stage_dev = [torch.empty(max(wl.seq_len) * 128, dtype=torch.int16, device=dev) for _ in range(2)]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        qws = hsi.workspace(hsi.WS_QUANTIZE, 1, 0, device=dev)
        i = 0
        for layer in range(wl.full_layers):
            krec = torch.zeros(off * REC, dtype=torch.uint8, device=dev)
            gseq = torch.empty(len(seqs), dtype=torch.float32, device=dev)
            for si, s in enumerate(seqs):
                n = wl.seq_len[s]
                j = i % 2
                done[j].synchronize()
                host = stage[j][: n * 128].numpy().view(np.uint16)
                inputs.normal_bf16(wl.seed, inputs.tensor_id(inputs.KIND_K, layer, s), n * 128, out=host)
                stage_dev[j][: n * 128].copy_(stage[j][: n * 128], non_blocking=True)
                dst = krec[rec_off[s] * REC:(rec_off[s] + hsi.n_records(n)) * REC]
                if self.mx:
                    hsi.quantize_mxfp4(stage_dev[j][: n * 128].view(n, 128), 1, n, signs, dst)
                else:
                    hsi.quantize_nvfp4(stage_dev[j][: n * 128].view(n, 128), 1, n, signs, gseq[si:si + 1], dst,
                                       ws=qws)
                done[j].record()
                i += 1
            self.k_rec.append(krec)
            self.g_k.append(None if self.mx else
                            torch.stack([gseq[seqs.index(s)] for s in wl.query_seq]).contiguous())
        torch.cuda.synchronize()
        del stage, stage_dev
        log(f"K caches generated and quantised ({'MXFP4' if self.mx else 'NVFP4'}) in {time.time() - t0:.1f} s "
            f"({off * REC * wl.full_layers / 1e9:.2f} GB)")
        self.k_off = torch.tensor([rec_off[s] for s in wl.query_seq], dtype=torch.int64, device=dev)
        self.n_vis = torch.tensor(wl.n_visible, dtype=torch.int32, device=dev)
        # rows each query's caches hold (appends past the visible rows go up to here)
        self.capacity = torch.tensor([wl.seq_len[s] + self.HEADROOM for s in wl.query_seq], dtype=torch.int32,
                                     device=dev)
        self.maxv_cap = self.maxv + self.HEADROOM
        # --- per-step inputs: bf16 q and fp32 w of every layer, one contiguous buffer
        self.layers = wl.full_layers + (wl.reindex_layers if wl.build_pool else 0)
        L = self.layers
        q_host = np.stack([np.concatenate([wl.q_bf16(l, b) for b in range(B)]) for l in range(L)])  # [L][B*32][128]
        w_host = np.stack([np.stack([wl.w(l, b) for b in range(B)]) for l in range(L)])  # [L][B][32]
        self.q_bytes = q_host.nbytes
        self.in_host = torch.empty(q_host.nbytes + w_host.nbytes, dtype=torch.uint8).pin_memory()
        self.in_host[: q_host.nbytes].numpy()[:] = q_host.reshape(-1).view(np.uint8)
        self.in_host[q_host.nbytes:].numpy()[:] = w_host.reshape(-1).view(np.uint8)
        self.in_dev = self.in_host.to(dev)
        self.q = self.in_dev[: q_host.nbytes].view(torch.int16).view(L, B * 32, 128)
        self.w = self.in_dev[q_host.nbytes:].view(torch.float32).view(L, B, 32)
        # --- outputs and scratch
        self.q_rec = torch.empty(L, B * 4 * REC, dtype=torch.uint8, device=dev)
        self.g_q = [None] * L if self.mx else torch.empty(L, B, dtype=torch.float32, device=dev)
        self.scores = torch.empty(B, self.maxv_cap, dtype=torch.float32, device=dev)
        self.bmax = torch.empty(B, hsi.n_records(self.maxv), dtype=torch.float32, device=dev)
        self.out_dev = torch.empty(L * B * K_TOP * 8, dtype=torch.uint8, device=dev)
        # two host result buffers: step i reads its results back into buffer i % 2
        # while the host still holds step i - 1's
        self.out_host2 = [torch.empty_like(self.out_dev, device="cpu").pin_memory() for _ in range(2)]
        self.out_host = self.out_host2[0]
        self.idx = self.out_dev[: L * B * K_TOP * 4].view(torch.int32).view(L, B, K_TOP)
        self.val = self.out_dev[L * B * K_TOP * 4:].view(torch.float32).view(L, B, K_TOP)
        self.ws_q = hsi.workspace(hsi.WS_QUANTIZE, B, 0, device=dev)
        self.ws_topk = hsi.workspace(hsi.WS_TOPK, B, self.maxv, K_TOP, device=dev)
        self.ws_full = hsi.workspace(hsi.WS_FULL_LAYER, B, self.maxv_cap, K_TOP, device=dev)
        if wl.build_pool:
            self.ids = torch.empty(B, wl.n_keep, dtype=torch.int32, device=dev)
            self.nk = torch.empty(B, dtype=torch.int32, device=dev)
            self.npool = torch.empty(B, dtype=torch.int32, device=dev)
            self.bits = torch.empty(B, (self.maxv_cap + 31) // 32, dtype=torch.int32, device=dev)
            self.ws_pool = hsi.workspace(hsi.WS_POOL, B, self.maxv, 8, device=dev)
            self.pool_scores = torch.empty(B, wl.n_keep * 8, dtype=torch.float32, device=dev)
            self.ws_rtopk = hsi.workspace(hsi.WS_REINDEX_LAYER, B, wl.n_keep * 8, K_TOP, device=dev)
            self.pool_rec = torch.empty(B, wl.n_keep * REC, dtype=torch.uint8, device=dev)
        self.ev_score = []
        # the Full layer that builds the pool writes no score row: its top-512 is
        # taken from the pool's blocks, scored again (the same scores, the same top-512)
        self.pooled_topk = wl.build_pool
        self.pool_sum = None
        self.wl_signs = signs
        self.graphs = []

    def quant_q(self, l):
        """Quantise layer l's queries (all B) into q_rec[l]."""
        if self.mx:
            self.hsi.quantize_mxfp4(self.q[l], self.B, 32, self.wl_signs, self.q_rec[l])
        else:
            self.hsi.quantize_nvfp4(self.q[l], self.B, 32, self.wl_signs, self.g_q[l], self.q_rec[l], ws=self.ws_q)

    def step(self):
        """One step as individual launches (the same calls the graphs hold)."""
        for _, fn in self.segments():
            fn()

    # -- the step as CUDA graphs: [q quantisation] [scoring] [selection and the
    # rest], per Full layer, so that the scoring kernel can be timed between replays
    def segments(self, maxv=None):
        """The step's calls; maxv: the host bound on the visible lengths (the
        caches' capacity for a step over growing caches)."""
        hsi, wl, B = self.hsi, self.wl, self.B
        maxv = self.maxv if maxv is None else maxv
        segs = []

        def rest():
            # the Reindex layers stream the compacted pool, each query quantised
            # right before its layer
            for r in range(wl.reindex_layers):
                l = wl.full_layers + r
                self.quant_q(l)
                hsi.reindex_layer(self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[0], self.g_k[0], self.k_off,
                                  self.n_vis, self.ids, self.nk, self.npool, B, self.pool_scores, K_TOP,
                                  self.idx[l], self.val[l], n_keep=wl.n_keep, ws=self.ws_rtopk,
                                  pool_rec=self.pool_rec, pool_rec_ready=True, fmt=self.fmt)

        for l in range(wl.full_layers):
            segs.append(("pre", lambda l=l: self.quant_q(l)))
            # the Full layer (scores, top-512, pool) as the fused call, issued in
            # phases so that the scoring kernel can be timed alone
            pool = wl.build_pool and l == wl.full_layers - 1

            def fl(ph, l=l, pool=pool):
                hsi.full_layer(
                    self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[l], self.g_k[l], self.k_off, self.n_vis, B,
                    maxv, None if (pool and self.pooled_topk) else self.scores, K_TOP, self.idx[l], self.val[l],
                    block_ids=self.ids if pool else None, n_kept=self.nk if pool else None,
                    n_pool=self.npool if pool else None, pool_bits=self.bits if pool else None,
                    n_keep=wl.n_keep, ws=self.ws_full, phases=ph, fmt=self.fmt)
            segs.append(("score", lambda fl=fl: fl(hsi.PHASE_SCORE)))
            if pool:
                def post(fl=fl, l=l):
                    # model order on one stream: the pool; the Full layer's top-512
                    # from it (the pool's blocks gathered and scored again with the
                    # Full query: the full row's scores and top-512), which leaves
                    # the gathered records compacted for the Reindex layers; then
                    # those layers, whose queries a model computes only after the
                    # Full layer's attention over that top-512
                    fl(hsi.PHASE_POOL)
                    hsi.reindex_layer(self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[l], self.g_k[l], self.k_off,
                                      self.n_vis, self.ids, self.nk, self.npool, B, self.pool_scores, K_TOP,
                                      self.idx[l], self.val[l], n_keep=wl.n_keep, ws=self.ws_rtopk,
                                      pool_rec=self.pool_rec if wl.reindex_layers else None,
                                      pool_rec_ready=False, fmt=self.fmt)
                    rest()
                segs.append(("post", post))
            else:
                segs.append(("post", lambda fl=fl: fl(hsi.PHASE_SELECT)))
        merged = []
        for kind, fn in segs:  # fuse neighbouring non-scoring segments into one graph
            if merged and kind != "score" and merged[-1][0] != "score":
                prev = merged[-1][1]
                merged[-1] = (merged[-1][0], lambda a=prev, b=fn: (a(), b()))
            else:
                merged.append((kind, fn))
        return merged

    def reindex_timings(self, reps=20):
        """One Reindex layer, timed alone on the resident pool: the whole layer
        through the compacted pool (scan with the fused key histogram, then the
        selection), a plain top-k of the pooled scores (no histogram), the
        compaction, and the gathering scorer. Each figure is one CUDA graph of
        `reps` back-to-back calls (as the step runs them: graphs, programmatic
        dependent launch), timed with events around its replay, so that the
        host's per-call launch cost, which exceeds these layers' device time,
        is not what is measured."""
        torch, hsi, wl, B = self.torch, self.hsi, self.wl, self.B
        l = wl.full_layers

        def t(fn):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(reps):
                    fn()
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            return 1000.0 * e0.elapsed_time(e1) / reps

        layer = t(lambda: hsi.reindex_layer(self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[0], self.g_k[0],
                                            self.k_off, self.n_vis, self.ids, self.nk, self.npool, B,
                                            self.pool_scores, K_TOP, self.idx[l], self.val[l], n_keep=wl.n_keep,
                                            ws=self.ws_rtopk, pool_rec=self.pool_rec, fmt=self.fmt))
        topk = t(lambda: hsi.topk(self.pool_scores, self.npool, B, wl.n_keep * 8, K_TOP, self.idx[l], self.val[l],
                                  block_ids=self.ids, ws=self.ws_rtopk))
        compact = t(lambda: hsi.pool_gather(self.k_rec[0], self.k_off, self.n_vis, self.ids, self.nk, B,
                                            self.pool_rec, n_keep=wl.n_keep, fmt=self.fmt))
        gather = t(lambda: hsi.score_pool(self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[0], self.g_k[0],
                                          self.k_off, self.n_vis, self.ids, self.nk, wl.n_keep, B,
                                          self.pool_scores, fmt=self.fmt))
        # the scan of the compacted pool alone (query b's n_pool[b] keys at record
        # b n_keep, left there by the compaction above): the scoring of the
        # Reindex layers that stream the pool
        pool_off = torch.arange(B, dtype=torch.int64, device=self.dev) * wl.n_keep
        stream = t(lambda: hsi.score_full(self.q_rec[l], self.g_q[l], self.w[l], self.pool_rec, self.g_k[0],
                                          pool_off, self.npool, B, wl.n_keep * 8, self.pool_scores, fmt=self.fmt))
        first = t(lambda: hsi.reindex_layer(self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[0], self.g_k[0],
                                            self.k_off, self.n_vis, self.ids, self.nk, self.npool, B,
                                            self.pool_scores, K_TOP, self.idx[l], self.val[l], n_keep=wl.n_keep,
                                            ws=self.ws_rtopk, pool_rec=self.pool_rec, pool_rec_ready=False,
                                            fmt=self.fmt))
        # the pages' masked form of the same layer, kept for comparison: every
        # visible position scored with the Reindex query, the pool's bit table
        # applied as -inf, then the top-512
        def dense():
            hsi.score_full(self.q_rec[l], self.g_q[l], self.w[l], self.k_rec[0], self.g_k[0], self.k_off,
                           self.n_vis, B, self.maxv, self.scores, fmt=self.fmt)
            hsi.mask_scores(self.scores, self.n_vis, self.bits, B, self.maxv)
            hsi.topk(self.scores, self.n_vis, B, self.maxv, K_TOP, self.idx[l], self.val[l], ws=self.ws_topk)
        dense_us = t(dense)
        # the pool phase alone on the block maxima and their histogram the step's
        # Full scan left in the workspace: threshold bin, candidates, the pool
        pool_us = t(lambda: hsi.full_layer(self.q_rec[0], self.g_q[0], self.w[0], self.k_rec[0], self.g_k[0],
                                           self.k_off, self.n_vis, B, self.maxv,
                                           None if self.pooled_topk else self.scores, K_TOP, self.idx[0],
                                           self.val[0], block_ids=self.ids, n_kept=self.nk, n_pool=self.npool,
                                           pool_bits=self.bits, n_keep=wl.n_keep, ws=self.ws_full,
                                           phases=hsi.PHASE_POOL, fmt=self.fmt))
        pooled_bytes = int(self.nk.clamp(max=wl.n_keep).sum().item()) * self.rec
        return {"layer_us": layer, "first_layer_us": first, "plain_topk_us": topk, "compact_us": compact,
                "pool_phase_us": pool_us,
                "gather_score_us": gather, "stream_score_us": stream, "dense_masked_layer_us": dense_us,
                "dense_over_pooled": dense_us / layer, "pooled_bytes_per_layer": pooled_bytes}

    def capture(self):
        torch = self.torch
        self.step()  # also sets every kernel's attributes before capture
        torch.cuda.synchronize()
        self.graphs = []
        for kind, fn in self.segments():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            self.graphs.append((kind, g))
        # the end-to-end step as one graph: inputs in from pinned host memory, the
        # whole path, results out to pinned host memory (one launch per step); one
        # graph per host result buffer
        self.graph_e2e = []
        for buf in self.out_host2:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.in_dev.copy_(self.in_host, non_blocking=True)
                self.step()
                buf.copy_(self.out_dev, non_blocking=True)
            self.graph_e2e.append(g)
        self.ev_e2e = [torch.cuda.Event(), torch.cuda.Event()]
        torch.cuda.synchronize()

    def replay(self, time_score=False):
        torch = self.torch
        for kind, g in self.graphs:
            if time_score and kind == "score":
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                self.ev_score.append((e0, e1))
            else:
                g.replay()

    def step_e2e(self, i=0):
        """End-to-end step i: its graph (inputs in, the path, results out to host
        buffer i % 2), then the host waits until step i - 1's results are in host
        memory, so that one step is always queued behind the running one and the
        GPU does not idle while the host launches."""
        self.graph_e2e[i % 2].replay()
        self.ev_e2e[i % 2].record()
        if i > 0:
            self.ev_e2e[(i - 1) % 2].synchronize()

    def pairs_per_step(self):
        full = self.wl.full_layers * int(sum(self.wl.n_visible))
        pooled = 0
        if self.wl.build_pool:
            if self.pool_sum is None:
                self.torch.cuda.synchronize()
                self.pool_sum = int(self.npool.sum().item())
            pooled = self.wl.reindex_layers * self.pool_sum
        return full + pooled, full, pooled

    def score_bytes_per_launch(self):
        """Algorithmic bytes of one Full-layer scoring launch: 72 B (NVFP4) or 68 B
        (MXFP4) per visible key read, 4 B per block maximum written, 4 B per
        score written unless the top-512 comes from the pool, q/w/scales read."""
        n = int(sum(self.wl.n_visible))
        nb = sum((v + 7) // 8 for v in self.wl.n_visible)
        key_bytes = self.rec // 8
        scales = 0 if self.mx else 8
        score_row = 0 if (self.wl.build_pool and self.pooled_topk) else n * 4
        return (n * key_bytes + score_row + (nb * 4 if self.wl.build_pool else 0)
                + self.B * (4 * self.rec + 32 * 4 + scales))


class MainKV:
    """The FP4 main-KV caches of a workload, resident on one GPU: the caches of
    all sequences back to back, seq_len entries of 288 bytes each (19.3 GB for
    64 x 1M). Entry e of the buffer holds pattern entry e mod P: the first
    P = 131072 generated main-KV entries of the workload's first sequence,
    quantised on the GPU once and replicated (a gather's cost depends on where
    the selected entries sit, not on their values)."""
    PATTERN = 131072

    def __init__(self, wl: inputs.Workload, dev, log, headroom: int = 0):
        import torch

        import long_context_decode_lightning_gb300 as hsi
        seqs = sorted(set(wl.query_seq))
        start, off = {}, 0
        for s in seqs:
            start[s] = off
            off += wl.seq_len[s] + headroom
        self.entries = off
        E = hsi.KV_ENTRY_BYTES
        t0 = time.time()
        self.kv = torch.empty(off * E, dtype=torch.uint8, device=dev)
        self.P = P = min(self.PATTERN, off)
        self.pattern_seq = seqs[0]
        x = torch.from_numpy(wl.kv_bf16(seqs[0], rows=P).view(np.int16)).to(dev)
        hsi.quantize_mainkv(x, self.kv[: P * E])
        reps = off // P
        if reps > 1:
            self.kv[: reps * P * E].view(reps, P * E)[1:].copy_(self.kv[: P * E].expand(reps - 1, -1))
        if off > reps * P:
            self.kv[reps * P * E:].copy_(self.kv[: (off - reps * P) * E])
        torch.cuda.synchronize()
        self.off = torch.tensor([start[s] for s in wl.query_seq], dtype=torch.int64, device=dev)
        log(f"main KV: {off} entries, {off * E / 1e9:.2f} GB, filled in {time.time() - t0:.1f} s")

    def pattern_index(self, b_off: int, i: int) -> int:
        """The pattern entry that entry i of the cache starting at entry b_off holds."""
        return (b_off + i) % self.P


# ----------------------------------------------------------- CPU oracle --

def serving_steps(W: DeviceWorkload, M: MainKV, wl: inputs.Workload, dev, args, timed, log):
    """Decode steps over growing caches: each step appends one token per query
    (its indexer K row into every Full layer's cache, with the cache's fixed
    tensor scale, and its main-KV entry), then runs the whole path and gathers
    every layer's top-512 from the main KV; one CUDA graph per step, replayed
    while the caches grow by one row per step. Returns the JSON object."""
    import torch

    import long_context_decode_lightning_gb300 as hsi
    B, T = W.B, max(args.warmup, 1) + args.steps + 1
    kx = np.empty((T, B, 128), np.uint16)
    vx = np.empty((T, B, hsi.KV_DIM), np.uint16)
    for b in range(B):  # the sequences' own next rows
        s, n = wl.query_seq[b], wl.n_visible[b]
        kx[:, b] = wl.k_bf16(0, s, first_row=n, rows=T)
        vx[:, b] = wl.kv_bf16(s, first_row=n, rows=T)
    new_k = torch.from_numpy(kx.view(np.int16)).to(dev)
    new_v = torch.from_numpy(vx.view(np.int16)).to(dev)
    k_stage = torch.empty(B, 128, dtype=torch.int16, device=dev)
    v_stage = torch.empty(B, hsi.KV_DIM, dtype=torch.int16, device=dev)
    rows = torch.empty(W.layers, B, K_TOP, hsi.KV_DIM, dtype=torch.int16, device=dev)
    n_start = int(W.n_vis.max().item())

    assert wl.full_layers == 1, "decoder workloads: one Full layer's K cache per sequence"

    def step():
        hsi.append_token(k_stage, W.wl_signs, W.g_k[0], W.k_rec[0], W.k_off, W.n_vis, W.capacity, B, kv_x=v_stage,
                         kv=M.kv, kv_off=M.off, fmt=W.fmt)
        for _, fn in W.segments(maxv=W.maxv_cap):
            fn()
        hsi.gather_mainkv_layers(M.kv, M.off, W.n_vis, W.idx, K_TOP, B, rows)  # every layer's top-512, one launch

    k_stage.copy_(new_k[0])
    v_stage.copy_(new_v[0])
    step()  # the first token outside the graph (sets every launch attribute)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    state = {"i": 1}

    def one():
        i = state["i"]
        k_stage.copy_(new_k[i])
        v_stage.copy_(new_v[i])
        graph.replay()
        state["i"] = i + 1
    for _ in range(max(args.warmup, 1)):
        one()
    torch.cuda.synchronize()
    ms = timed(one, args.steps)
    n_end = int(W.n_vis.max().item())
    log(f"serving: {args.steps} steps, context {n_start} -> {n_end}")
    return {"ms_per_step": ms / args.steps, "tokens_per_s": B * args.steps / (ms / 1e3), "queries": B,
            "context_start": n_start, "context_end": n_end,
            "note": "per step: append one token per query (indexer K row with the cache's fixed tensor scale, "
                    "main-KV entry), the whole indexer path over the grown caches (max_visible = capacity), "
                    "and the gathers of every layer's top-512 from the main KV; one CUDA graph, inputs staged "
                    "by two device copies"}


def oracle_sample_setup(wl: inputs.Workload, nq: int, fmt: str = "nvfp4"):
    """Oracle inputs for the first nq queries (quantised by the oracle itself, in
    the record format fmt: "nvfp4" or "mxfp4")."""
    import oracle
    signs = wl.signs()
    L = wl.full_layers + (wl.reindex_layers if wl.build_pool else 0)

    def quant(x):
        return (oracle.quantize_mx(x, signs), 1.0) if fmt == "mxfp4" else oracle.quantize(x, signs)

    def prep(b):
        s = wl.query_seq[b]
        ks = [quant(wl.k_bf16(l, s)) for l in range(wl.full_layers)]
        qs = [quant(wl.q_bf16(l, b)) + (wl.w(l, b),) for l in range(L)]
        return ks, qs

    return oracle.map_queries(prep, list(range(nq)), threads=nq)


def oracle_query_step(wl: inputs.Workload, b: int, ks, qs, fmt: str = "nvfp4"):
    """The whole path for one query on the oracle; returns pairs scored."""
    import oracle
    n = wl.n_visible[b]
    pairs = 0
    scores = None
    for l in range(wl.full_layers):
        qrec, gq, w = qs[l]
        krec, gk = ks[l]
        scores, _ = oracle.score_full(qrec, gq, w, krec, gk, n, fmt=fmt)
        oracle.topk(scores, n, K_TOP)
        pairs += n
    if wl.build_pool:
        ids, nk, npool, _ = oracle.pool(scores, n, wl.block_size, wl.n_keep, want_mask=True)
        krec, gk = ks[0]
        for r in range(wl.reindex_layers):
            qrec, gq, w = qs[wl.full_layers + r]
            ps, _ = oracle.score_pool(qrec, gq, w, krec, gk, n, ids, nk, wl.n_keep, wl.block_size, fmt=fmt)
            oracle.topk_pool(ps, npool, ids, K_TOP, wl.block_size)
            pairs += npool
    return pairs


def oracle_timed(wl, prepared, nq, fmt: str = "nvfp4"):
    import oracle
    t0 = time.perf_counter()
    pairs = oracle.map_queries(lambda b: oracle_query_step(wl, b, *prepared[b], fmt=fmt), list(range(nq)),
                               threads=nq)
    return sum(pairs), time.perf_counter() - t0


def cpu_sample_size(wl: inputs.Workload):
    """All host cores, one query per thread (at most the workload's queries)."""
    return max(1, min(os.cpu_count() or 1, wl.B))


# ------------------------------------------------------------ calibration --

def calibrate(dev, log, n_sm: int):
    """The rooflines of this GPU measured with the path's own instructions: a
    read-only stream of 4 GB (16-byte loads from every SM, and bulk copies of
    18 KB through a shared-memory ring), and back-to-back block-scaled FP4
    MMAs (M = 128, K = 64, N = 32 .. 256) on every SM. Best of 5 launches each."""
    import torch

    import long_context_decode_lightning_gb300 as hsi
    buf = torch.ones(4 << 30, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int64, device=dev)

    def best(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return min(ts)

    out = {"hbm_read_gbs": {}, "fp4_mma_tflops": {}}
    ms = best(lambda: hsi.calib_read(buf, 0, sink=sink))
    out["hbm_read_gbs"]["ldg16"] = buf.numel() / (ms / 1e3) / 1e9
    ms = best(lambda: hsi.calib_read(buf, 1, chunk=18432, stages=8, sink=sink))
    out["hbm_read_gbs"]["bulk18k"] = buf.numel() / (ms / 1e3) / 1e9
    del buf
    for n in (32, 64, 128, 256):
        iters = 16000 * 256 // n if n < 256 else 24000
        ms = best(lambda: hsi.calib_mma(n, iters, sink=sink, device=dev))
        out["fp4_mma_tflops"][str(n)] = 2.0 * 128 * n * 64 * iters * n_sm / (ms / 1e3) / 1e12
    assert hsi.device_error() == 0, "device error during calibration"
    log(f"calibration: read {out['hbm_read_gbs']}, FP4 MMA {out['fp4_mma_tflops']}")
    out["note"] = ("read-only HBM bandwidth (4 GB, 16-byte loads / 18 KB bulk copies) and dense block-scaled FP4 "
                   "tensor throughput (tcgen05.mma kind::mxf4nvf4, M=128, K=64, shared-memory operands), measured "
                   "in this run by hsi_calib_read / hsi_calib_mma; best of 5")
    return out


def flush_l2(dev, _buf={}):
    """Write 256 MB (twice the L2) so that the next step reads its inputs from HBM."""
    import torch
    if "b" not in _buf:
        _buf["b"] = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    _buf["b"].zero_()


def time_steps_flushed(fn, K: int, dev) -> list:
    """K replays of fn, each timed alone with events after an L2 flush (ms each)."""
    import torch
    out = []
    for _ in range(K):
        flush_l2(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def decode_config(idx: int, dev, args, log, peaks):
    """One of the other decode / encoder workloads, as the headline step runs
    (CUDA graphs), each step timed alone after an L2 flush (their caches can fit
    in L2). Roofline: the scans' key bytes (72 per visible key per Full layer,
    576 per pooled block per Reindex layer) over the step time."""
    import torch

    import long_context_decode_lightning_gb300 as hsi
    wl = inputs.workload(idx)
    W = DeviceWorkload(wl, dev, log)
    W.capture()
    for _ in range(max(args.warmup, 1)):
        W.replay()
    torch.cuda.synchronize()
    assert hsi.device_error() == 0, f"device error in workload {wl.name}"
    ts = time_steps_flushed(W.replay, args.steps, dev)
    ms = float(np.median(ts))
    pairs, full, pooled = W.pairs_per_step()
    key_bytes = wl.full_layers * sum(wl.n_visible) * 72
    if wl.build_pool:
        key_bytes += wl.reindex_layers * int(W.nk.clamp(max=wl.n_keep).sum().item()) * W.rec
    peak = float(peaks["hbm_gbs"])
    gbs = key_bytes / (ms / 1e3) / 1e9
    res = {"workload": wl.name, "notes": wl.notes, "ms_per_step": ms, "pairs_per_s": pairs / (ms / 1e3),
           "top512_selections_per_s": W.B * W.layers / (ms / 1e3), "pairs_per_step": pairs,
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                        "bytes_per_step": key_bytes, "peak_kind": "measured copy bandwidth",
                        "ideal_ms": key_bytes / (peak * 1e9) * 1e3},
           "timing": "median of per-step CUDA-event times, L2 flushed (256 MB written) before each step"}
    if idx == 0:
        res["note"] = ("latency-bound: 2.4 MB of keys is well under one microsecond of HBM time, so the step is "
                       "the launch and dependency chain of its kernels, not bandwidth")
    del W
    torch.cuda.empty_cache()
    return res


class PrefillWorkload:
    """Chunked prefill: 8192 consecutive queries on one 131,072-key cache (query
    t sees 122,881 + t keys). One step: quantise the 8192 queries' q, then
    hsi_prefill_layer: four queries per tensor-core tile, scores and block maxima
    written, then each query's top-512 and pool from the block maxima and the
    candidate blocks' scores."""

    def __init__(self, wl: inputs.Workload, dev, log, queries: int = 0):
        import torch

        import long_context_decode_lightning_gb300 as hsi
        if queries:  # the first `queries` queries only (a multiple of 4), for profiling captures
            wl.query_seq = wl.query_seq[:queries]
            wl.n_visible = wl.n_visible[:queries]
        self.torch, self.hsi, self.wl = torch, hsi, wl
        signs = wl.signs()
        self.signs = signs
        n = wl.seq_len[0]
        B = self.B = wl.B
        self.n = n
        t0 = time.time()
        kb = torch.from_numpy(wl.k_bf16(0, 0).view(np.int16)).to(dev)
        self.k_rec = torch.empty(hsi.n_records(n) * hsi.REC_BYTES, dtype=torch.uint8, device=dev)
        g1 = torch.empty(1, device=dev)
        hsi.quantize_nvfp4(kb, 1, n, signs, g1, self.k_rec)
        del kb
        self.g_k = g1.repeat(B)
        self.k_off = torch.zeros(B, dtype=torch.int64, device=dev)
        q_host = np.concatenate([wl.q_bf16(0, t) for t in range(B)])
        self.q = torch.from_numpy(q_host.view(np.int16)).to(dev)
        self.w = torch.from_numpy(np.stack([wl.w(0, t) for t in range(B)])).to(dev)
        self.q_rec = torch.empty(B * 4 * hsi.REC_BYTES, dtype=torch.uint8, device=dev)
        self.g_q = torch.empty(B, device=dev)
        self.ws_q = hsi.workspace(hsi.WS_QUANTIZE, B, 0, device=dev)
        self.nv = torch.tensor(wl.n_visible, dtype=torch.int32, device=dev)
        self.scores = torch.empty(B, n, device=dev)
        self.idx = torch.empty(B, K_TOP, dtype=torch.int32, device=dev)
        self.val = torch.empty(B, K_TOP, device=dev)
        self.ids = torch.empty(B, wl.n_keep, dtype=torch.int32, device=dev)
        self.nk = torch.empty(B, dtype=torch.int32, device=dev)
        self.npool = torch.empty(B, dtype=torch.int32, device=dev)
        self.bits = torch.empty(B, (n + 31) // 32, dtype=torch.int32, device=dev)
        self.ws = hsi.workspace(hsi.WS_PREFILL_LAYER, B, n, K_TOP, device=dev)
        log(f"prefill workload ready in {time.time() - t0:.1f} s")

    def quant(self):
        self.hsi.quantize_nvfp4(self.q, self.B, 32, self.signs, self.g_q, self.q_rec, ws=self.ws_q)

    def layer(self, phases):
        self.hsi.prefill_layer(self.q_rec, self.g_q, self.w, self.k_rec, self.g_k, self.k_off, self.nv, self.B,
                               self.n, self.scores, K_TOP, self.idx, self.val, group=4, block_ids=self.ids,
                               n_kept=self.nk, n_pool=self.npool, pool_bits=self.bits, n_keep=self.wl.n_keep,
                               ws=self.ws, phases=phases)


def run_case(args, dev, log):
    """One kernel's case for a profiling capture: set up, run it --steps times, check the device status."""
    import torch

    import long_context_decode_lightning_gb300 as hsi
    if args.case in ("prefill_score", "prefill_layer", "rowsel"):
        P = PrefillWorkload(inputs.workload(4), dev, log, queries=args.queries)
        P.quant()
        if args.case == "rowsel":
            P.layer(hsi.PHASE_SCORE)
        for _ in range(args.steps):
            if args.case == "prefill_score":
                P.layer(hsi.PHASE_SCORE)
            elif args.case == "rowsel":
                P.layer(hsi.PHASE_SELECT)
            else:
                P.quant()
                P.layer(hsi.PHASE_ALL)
    elif args.case in ("reindex", "reindex_gather", "pool"):
        # the decode step's Reindex layer (streaming the compacted pool, or gathering
        # it), or the pool selection, on the resident state one step left behind
        wl = inputs.workload(2)
        if args.queries:
            wl.query_seq = wl.query_seq[: args.queries]
            wl.n_visible = wl.n_visible[: args.queries]
        W = DeviceWorkload(wl, dev, log)
        W.step()
        l = wl.full_layers
        for _ in range(args.steps):
            if args.case == "pool":
                hsi.full_layer(W.q_rec[0], W.g_q[0], W.w[0], W.k_rec[0], W.g_k[0], W.k_off, W.n_vis, W.B, W.maxv,
                               None if W.pooled_topk else W.scores, K_TOP, W.idx[0], W.val[0], block_ids=W.ids, n_kept=W.nk, n_pool=W.npool,
                               pool_bits=W.bits, n_keep=wl.n_keep, ws=W.ws_full, phases=hsi.PHASE_POOL)
            else:
                hsi.reindex_layer(W.q_rec[l], W.g_q[l], W.w[l], W.k_rec[0], W.g_k[0], W.k_off, W.n_vis, W.ids,
                                  W.nk, W.npool, W.B, W.pool_scores, K_TOP, W.idx[l], W.val[l], n_keep=wl.n_keep,
                                  ws=W.ws_rtopk, pool_rec=W.pool_rec, pool_rec_ready=args.case == "reindex")
    else:  # the five layers' gathers of a decode step, random selections, one launch each
        wl = inputs.workload(2)
        if args.queries:
            wl.query_seq = wl.query_seq[: args.queries]
            wl.n_visible = wl.n_visible[: args.queries]
        M = MainKV(wl, dev, log)
        B, L = wl.B, 5
        g = torch.Generator(device="cpu").manual_seed(1)
        idx = torch.randint(0, min(wl.n_visible), (L, B, K_TOP), generator=g, dtype=torch.int32).to(dev)
        nv = torch.tensor(wl.n_visible, dtype=torch.int32, device=dev)
        out = torch.empty(L, B, K_TOP, hsi.KV_DIM, dtype=torch.int16, device=dev)
        for _ in range(args.steps):
            hsi.gather_mainkv_layers(M.kv, M.off, nv, idx, K_TOP, B, out)
    torch.cuda.synchronize()
    assert hsi.device_error() == 0, f"device error in case {args.case}"
    log(f"case {args.case}: {args.steps} runs ok")


def prefill_config(dev, args, log, peaks, calib, clk_mhz, n_sm):
    """The chunked-prefill workload (compute-bound), timed as graphs of its
    three segments with the scoring segment timed on its own, against the
    larger of its three bounds: dense FP4 tensor time at the calibrated rate of
    the kernel's MMA shape (N = 128), the epilogue's issue time (per (query,
    key) pair 32 ReLU maxima and 16 packed fp32 fmas, 4 warp instructions per
    cycle per SM at the sampled SM clock) and the HBM time of its bytes."""
    import torch

    import long_context_decode_lightning_gb300 as hsi
    wl = inputs.workload(4)
    P = PrefillWorkload(wl, dev, log)
    segs = [("pre", P.quant), ("score", lambda: P.layer(hsi.PHASE_SCORE)),
            ("post", lambda: P.layer(hsi.PHASE_SELECT))]
    for _, fn in segs:
        fn()
    torch.cuda.synchronize()
    assert hsi.device_error() == 0, "device error in the prefill workload"
    graphs = []
    for kind, fn in segs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        graphs.append((kind, g))
    ev = []

    def replay():
        for kind, g in graphs:
            if kind == "score":
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                g.replay()
                e1.record()
                ev.append((e0, e1))
            else:
                g.replay()
    for _ in range(max(args.warmup, 1)):
        replay()
    torch.cuda.synchronize()
    ev.clear()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        replay()
    e1.record()
    torch.cuda.synchronize()
    assert hsi.device_error() == 0, "device error in the prefill steps"
    ms = e0.elapsed_time(e1) / args.steps
    score_ms = float(np.mean([a.elapsed_time(b) for a, b in ev]))
    pairs = int(sum(wl.n_visible))
    flop = pairs * 32 * 128 * 2
    t_tensor = flop / (calib["fp4_mma_tflops"]["128"] * 1e12) * 1e3
    t_alu = pairs * 48 / 32 / (4 * n_sm * clk_mhz * 1e6) * 1e3
    nb = sum((v + 7) // 8 for v in wl.n_visible)
    hbm_bytes = (hsi.n_records(P.n) * hsi.REC_BYTES + P.B * (4 * hsi.REC_BYTES + 32 * 4 + 32 * 128 * 2)
                 + pairs * 4 + nb * 4 * 2 + P.B * (513 * 8 * 4 + (P.n + 31) // 32 * 4 + K_TOP * 8 + wl.n_keep * 4))
    t_hbm = hbm_bytes / (float(peaks["hbm_gbs"]) * 1e9) * 1e3
    bounds = {"tensor": t_tensor, "alu": t_alu, "hbm": t_hbm}
    bind = max(bounds, key=bounds.get)
    res = {"workload": wl.name, "notes": wl.notes, "ms_per_step": ms, "pairs_per_s": pairs / (ms / 1e3),
           "top512_selections_per_s": P.B / (ms / 1e3), "pool_builds_per_s": P.B / (ms / 1e3),
           "pairs_per_step": pairs, "score_ms": score_ms, "select_and_quant_ms": ms - score_ms,
           "fp4_pflops_achieved": flop / (score_ms / 1e3) / 1e15,
           "roofline": {"bound": bind, "achieved": pairs / (ms / 1e3), "peak": pairs / (bounds[bind] / 1e3),
                        "unit": "pairs/s", "frac": bounds[bind] / ms, "bounds_ms": bounds,
                        "score_kernel_frac": bounds[bind] / score_ms,
                        "tensor_peak_tflops": calib["fp4_mma_tflops"]["128"], "sm_clock_mhz": clk_mhz,
                        "hbm_bytes_per_step": hbm_bytes,
                        "note": "frac = the binding bound's time over the whole layer's time (q quantisation, "
                                "scoring, selection); score_kernel_frac over the scoring kernel alone"}}
    del P, graphs
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------- multi-rank --

def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: every rank of the job processed its own units,
    so the job's throughput is all units over this time."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: float, world: int, steps: int, ms: float) -> float:
    """Whole-job throughput: the units of all ranks over the slowest rank's time."""
    return units_per_rank * world * steps / (ms / 1e3)


# ------------------------------------------------------------------- main --

def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    log = (lambda m: print(f"[bench] {m}", file=sys.stderr, flush=True)) if rank == 0 else (lambda m: None)
    wl = inputs.workload(args.workload)
    if args.queries:
        wl.query_seq = wl.query_seq[: args.queries]
        wl.n_visible = wl.n_visible[: args.queries]
        wl.name += f"_first{args.queries}"
    config = {"workload": wl.name, "queries": wl.B, "context": max(wl.n_visible), "full_layers": wl.full_layers,
              "reindex_layers": wl.reindex_layers if wl.build_pool else 0, "k": K_TOP,
              "block": wl.block_size if wl.build_pool else None, "keep": wl.n_keep if wl.build_pool else None,
              "format": args.format, "l2": "no flush: resident inputs exceed L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        nq = cpu_sample_size(wl)
        log(f"oracle sample: {nq} queries of {wl.name}")
        prepared = oracle_sample_setup(wl, nq, args.format)
        for _ in range(args.warmup):
            oracle_timed(wl, prepared, nq, args.format)
        tot_pairs, tot_t = 0, 0.0
        for _ in range(args.steps):
            p, t = oracle_timed(wl, prepared, nq, args.format)
            tot_pairs += p
            tot_t += t
        v = tot_pairs / tot_t
        sample = f"{nq} of {wl.B} queries per step, full path per query, one thread per query"
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": 1,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_t / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": config,
                          "cpu_baseline": {"value": v, "unit": UNIT, "cores": nq, "kind": "oracle", "sample": sample},
                          "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return

    import torch
    import long_context_decode_lightning_gb300 as hsi
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hsi.build() if rank == 0 else None
    if world > 1:
        dist.barrier()
    hsi.device_check()
    if args.case:
        run_case(args, dev, log)
        return
    fmt = hsi.FMT_MXFP4 if args.format == "mxfp4" else hsi.FMT_NVFP4
    W = DeviceWorkload(wl, dev, log, fmt=fmt)
    l0 = hsi.kernel_launches()
    W.step()
    torch.cuda.synchronize()
    launches_per_step = hsi.kernel_launches() - l0
    W.capture()
    for _ in range(args.warmup):
        W.replay()
    torch.cuda.synchronize()
    assert hsi.device_error() == 0, "device error during warm-up"
    pairs, pairs_full, pairs_pool = W.pairs_per_step()

    def timed(fn, K, sync_each=False):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            fn()
            if sync_each:
                torch.cuda.current_stream().synchronize()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        return max_over_ranks(ms, dev) if world > 1 else ms

    with ClockSampler(local) as clk:
        if args.profile:
            torch.cuda.profiler.start()
        ms = timed(lambda: W.replay(time_score=True), args.steps)
        if args.profile:
            torch.cuda.profiler.stop()
    launches = launches_per_step * args.steps  # graph replays of the captured launches
    assert hsi.device_error() == 0, "device error during the timed steps"
    score_ms = float(np.mean([a.elapsed_time(b) for a, b in W.ev_score]))
    # end to end: host inputs in, host results out, every step
    for i in range(2):
        W.step_e2e(i)
    torch.cuda.synchronize()
    it = iter(range(args.steps))
    ms_e2e = timed(lambda: W.step_e2e(next(it)), args.steps)  # the end event follows the last step's copy out
    assert hsi.device_error() == 0, "device error during the end-to-end steps"
    reindex = W.reindex_timings() if wl.build_pool else None
    assert hsi.device_error() == 0, "device error during the Reindex timings"

    value = job_value(pairs, world, args.steps, ms)
    value_e2e = job_value(pairs, world, args.steps, ms_e2e)
    sel = job_value(W.B * W.layers, world, args.steps, ms)
    peaks, peak_kind = measured_peaks()
    bytes_launch = W.score_bytes_per_launch()
    achieved = bytes_launch / (score_ms / 1e3) / 1e9
    traffic = recorded_traffic(args.format)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp4 (e2m1 x e2m1, e8m0 block scales, fp32 accumulate)" if W.mx else
                 "nvfp4 (e2m1 x e2m1, e4m3 block scales, fp32 accumulate)",
        "data": "synthetic", "config": config,
        "top512_selections_per_s": sel,
        "pairs_per_step": {"full": pairs_full, "pooled": pairs_pool},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                     "frac": achieved / float(peaks["hbm_gbs"]), "traffic": traffic,
                     "kernel": f"hsi_score_full (score_kernel<1,false> {args.format.upper()})",
                     "bytes_per_launch": bytes_launch, "ms_per_launch": score_ms,
                     "peak_kind": f"{peak_kind} copy bandwidth"},
        "e2e": {"value": value_e2e, "unit": UNIT, "h2d_bytes_per_step": int(W.in_host.numel()),
                "d2h_bytes_per_step": int(W.out_host.numel()), "ms_per_step": ms_e2e / args.steps},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if reindex is not None:
        peak = float(peaks["hbm_gbs"])
        gbs = lambda us: reindex["pooled_bytes_per_layer"] / (us * 1e-6) / 1e9
        line["pool_builds_per_s"] = job_value(W.B, world, args.steps, ms)
        line["reindex"] = dict(reindex, **{
            "layer_gbs": gbs(reindex["layer_us"]), "layer_frac": gbs(reindex["layer_us"]) / peak,
            "gather_score_gbs": gbs(reindex["gather_score_us"]),
            "gather_score_frac": gbs(reindex["gather_score_us"]) / peak,
            "stream_score_gbs": gbs(reindex["stream_score_us"]),
            "stream_score_frac": gbs(reindex["stream_score_us"]) / peak,
            "note": "one layer timed alone on the resident pool, each figure a CUDA graph of 20 calls; fractions "
                    "of the measured copy bandwidth for the pooled bytes (the layer figure includes its zeroing "
                    "and selection; stream_score is the Reindex layers' scoring, which reads the compacted pool; "
                    "gather_score the one gather per step)"})
    serve = not args.no_serve and wl.build_pool and wl.full_layers == 1
    M = MainKV(wl, dev, log, headroom=DeviceWorkload.HEADROOM) if (not args.no_mainkv or serve) else None
    if not args.no_mainkv:
        # gather(main_kv, topk) of every layer's top-512 of the last step, into bf16
        kv_out = torch.empty(W.layers, W.B, K_TOP, hsi.KV_DIM, dtype=torch.int16, device=dev)

        def gathers():  # every layer's top-512 in one launch
            hsi.gather_mainkv_layers(M.kv, M.off, W.n_vis, W.idx, K_TOP, W.B, kv_out)
        gathers()  # sets the launch attributes before capture
        torch.cuda.synchronize()
        g_graph = torch.cuda.CUDAGraph()  # the step's gathers as one graph, as the step itself runs
        with torch.cuda.graph(g_graph):
            gathers()
        for _ in range(max(args.warmup, 1)):
            g_graph.replay()
        torch.cuda.synchronize()
        assert hsi.device_error() == 0, "device error in the main-KV gather"
        ms_g = timed(g_graph.replay, args.steps)
        valid = int((W.idx >= 0).sum().item())
        bytes_g = valid * hsi.KV_ENTRY_BYTES + W.layers * W.B * K_TOP * (hsi.KV_DIM * 2 + 4)
        gbs_g = bytes_g / (ms_g / args.steps / 1e3) / 1e9
        line["mainkv_gather"] = {
            "us_per_step": 1000 * ms_g / args.steps, "gathers_per_step": W.layers,
            "entries_per_step": W.layers * W.B * K_TOP, "bytes_per_step": bytes_g,
            "roofline": {"bound": "hbm", "achieved": gbs_g, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs_g / float(peaks["hbm_gbs"]), "traffic": None,
                         "kernel": "hsi_gather_mainkv_layers (mainkv_gather_kernel), all layers in one launch"},
            "note": "the top-512 of each of the step's layers gathered from 288-byte FP4 main-KV entries "
                    f"({M.entries * hsi.KV_ENTRY_BYTES / 1e9:.1f} GB resident) and decoded to bf16 rows; "
                    "bytes = 288 read + 1024 written + 4 of index per selected entry"}
        del g_graph, kv_out
    if not args.no_mxfp4 and not W.mx:
        # the same step on MXFP4 records (its own K caches and queries)
        Wm = DeviceWorkload(wl, dev, log, fmt=hsi.FMT_MXFP4)
        Wm.capture()
        for _ in range(args.warmup):
            Wm.replay()
        torch.cuda.synchronize()
        assert hsi.device_error() == 0, "device error during the MXFP4 warm-up"
        ms_mx = timed(lambda: Wm.replay(time_score=True), args.steps)
        assert hsi.device_error() == 0, "device error during the MXFP4 steps"
        score_mx = float(np.mean([a.elapsed_time(b) for a, b in Wm.ev_score]))
        bytes_mx = Wm.score_bytes_per_launch()
        gbs_mx = bytes_mx / (score_mx / 1e3) / 1e9
        line["mxfp4"] = {
            "value": job_value(Wm.pairs_per_step()[0], world, args.steps, ms_mx), "unit": UNIT,
            "ms_per_step": ms_mx / args.steps, "key_bytes": Wm.rec // 8,
            "roofline": {"bound": "hbm", "achieved": gbs_mx, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs_mx / float(peaks["hbm_gbs"]), "traffic": recorded_traffic("mxfp4"),
                         "kernel": "hsi_score_full (score_kernel<1,false> MXFP4)", "bytes_per_launch": bytes_mx,
                         "ms_per_launch": score_mx},
            "note": "the same step and workload on MXFP4 records (32-element groups, E8M0 scales); the "
                    "pool and selections follow from its own scores"}
        del Wm
    if serve:
        line["serve"] = serving_steps(W, M, wl, dev, args, timed, log)
        assert hsi.device_error() == 0, "device error during the serving steps"
    del M
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    if not args.no_configs:
        del W
        torch.cuda.empty_cache()
        calib = calibrate(dev, log, n_sm)
        line["peaks"] = calib
        clk = line["clocks"].get("sm_mhz") or 2070.0
        line["configs"] = {}
        for idx in (0, 1, 3):
            line["configs"][str(idx)] = decode_config(idx, dev, args, log, peaks)
        with ClockSampler(local) as pclk:
            line["prefill"] = prefill_config(dev, args, log, peaks, calib, clk, n_sm)
        line["prefill"]["clocks"] = pclk.summary()
    if rank == 0 and not args.no_cpu_baseline:
        nq = cpu_sample_size(wl)
        log(f"cpu baseline: oracle on {nq} queries, one per host core, then one query on one core")
        prepared = oracle_sample_setup(wl, nq, args.format)
        p, t = oracle_timed(wl, prepared, nq, args.format)
        p1, t1 = oracle_timed(wl, prepared, 1, args.format)
        line["cpu_baseline"] = {"value": p / t, "unit": UNIT, "cores": nq, "host_cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{nq} of {wl.B} queries, whole path per query, one thread per query "
                                          f"on {nq} cores, {t:.1f} s wall",
                                "one_core": {"value": p1 / t1, "unit": UNIT, "cores": 1,
                                             "sample": f"1 query, whole path, one thread, {t1:.1f} s wall"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
