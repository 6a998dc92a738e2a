"""Shared set-up for the GPU parity tests: seeded inputs pushed through both the
CUDA path (via the C ABI) and the oracle."""
from __future__ import annotations

import numpy as np
import torch

import inputs
import oracle

import long_context_decode_lightning_gb300 as hsi

DEV = "cuda"


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)


def gpu_quantize_mx(x_bf16: np.ndarray, n_tensors: int, rpt: int, signs):
    x = dev_bf16(x_bf16.reshape(n_tensors * rpt, 128))
    rec = torch.full((n_tensors * hsi.n_records(rpt) * hsi.MX_REC_BYTES,), 0xA5, dtype=torch.uint8, device=DEV)
    hsi.quantize_mxfp4(x, n_tensors, rpt, signs, rec)
    return rec


def gpu_quantize(x_bf16: np.ndarray, n_tensors: int, rpt: int, signs, mode=0, g=None, fmt=hsi.FMT_NVFP4):
    if fmt == hsi.FMT_MXFP4:  # no tensor scale: g is a placeholder of ones
        return gpu_quantize_mx(x_bf16, n_tensors, rpt, signs), torch.ones(n_tensors, device=DEV)
    x = dev_bf16(x_bf16.reshape(n_tensors * rpt, 128))
    rec = torch.empty(n_tensors * hsi.n_records(rpt) * hsi.REC_BYTES, dtype=torch.uint8, device=DEV)
    gt = torch.empty(n_tensors, dtype=torch.float32, device=DEV) if g is None else \
        torch.tensor(g, dtype=torch.float32, device=DEV)
    hsi.quantize_nvfp4(x, n_tensors, rpt, signs, gt, rec, mode=mode)
    return rec, gt


class Caches:
    """K caches of several sequences in one buffer of block records."""

    def __init__(self, wl: inputs.Workload, layer: int, seqs, lengths, fmt=hsi.FMT_NVFP4):
        self.fmt = fmt
        self.signs = wl.signs()
        self.lengths = list(lengths)
        self.rec_off = []
        self.host_rec, self.host_g = [], []
        parts, gs = [], []
        off = 0
        for s, n in zip(seqs, lengths):
            kb = wl.k_bf16(layer, s, rows=n)
            rec, g = gpu_quantize(kb, 1, n, self.signs, fmt=fmt)
            parts.append(rec)
            gs.append(g)
            self.rec_off.append(off)
            off += hsi.n_records(n)
            self.host_rec.append(kb)
        self.k_rec = torch.cat(parts)
        self.g = torch.cat(gs)

    def oracle_rec(self, i):
        if self.fmt == hsi.FMT_MXFP4:
            return oracle.quantize_mx(self.host_rec[i], self.signs), 1.0
        rec, g = oracle.quantize(self.host_rec[i], self.signs)
        return rec, g


def gpu_queries(wl: inputs.Workload, layer: int, queries, fmt=hsi.FMT_NVFP4):
    qb = np.concatenate([wl.q_bf16(layer, b) for b in queries])
    rec, g = gpu_quantize(qb, len(queries), 32, wl.signs(), fmt=fmt)
    w = torch.from_numpy(np.stack([wl.w(layer, b) for b in queries])).to(DEV)
    return rec, g, w


def oracle_query(wl, layer, b, fmt=hsi.FMT_NVFP4):
    if fmt == hsi.FMT_MXFP4:
        return oracle.quantize_mx(wl.q_bf16(layer, b), wl.signs()), 1.0, wl.w(layer, b)
    rec, g = oracle.quantize(wl.q_bf16(layer, b), wl.signs())
    return rec, g, wl.w(layer, b)


def i32(v):
    return torch.tensor(v, dtype=torch.int32, device=DEV)


def i64(v):
    return torch.tensor(v, dtype=torch.int64, device=DEV)


def assert_sets_match_except_near_ties(got, want, value, tol, kth):
    """End-to-end selections from two score computations that each lie within
    a per-item tolerance of the exact value: the sets may differ only in items
    whose oracle value lies near the k-th value. If item x is in one set but
    not the other, some item y of the symmetric difference was ranked the other
    way round, and |v_x - kth| <= |v_x - v_y| <= tol(x) + tol(y); so every item
    x of the difference must satisfy |v_x - kth| <= tol(x) + max_y tol(y).
    value(x), tol(x): the oracle's value and tolerance of item x."""
    diff = set(int(x) for x in got) ^ set(int(x) for x in want)
    if not diff:
        return
    slack = max(tol(x) for x in diff)
    for x in diff:
        assert abs(value(x) - kth) <= tol(x) + slack, (x, value(x), kth, tol(x), slack)
