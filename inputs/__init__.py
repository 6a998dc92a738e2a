"""Seeded synthetic inputs for the Hierarchical Sparse Indexer workloads.

This module draws random numbers and describes the five workloads; it holds
none of the indexer's arithmetic. The oracle and the CUDA path both take their
inputs from here, so both see identical bf16 values.

Recipe (the same for every workload):
  * q and k: N(0, 1) drawn with splitmix64 + Box-Muller, rounded to bf16.
  * w: N(0, 1/32) in fp32.
  * context lengths (mixed-length decode batch): uniform integers in [lo, hi].
  * the random signs of the Hadamard rotation: 128 values of +-1, one vector per
    workload, shared by q and k so that rotated dot products are preserved.
Each tensor is its own stream keyed by (seed, tensor id); see ``tensor_id``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_SO = os.path.join(_HERE, "libhsigen.so")
_lib = None

H = 32  # indexer heads
D = 128  # head dimension

KIND_Q, KIND_K, KIND_W, KIND_LEN, KIND_SIGNS, KIND_KV = 1, 2, 3, 4, 5, 6
DKV = 512  # main-KV entry width


def build(force: bool = False) -> str:
    """Compile the generator into a shared library beside its source."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, i64, dbl, vp, i32 = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_double,
                                  ctypes.c_void_p, ctypes.c_int)
        L.gen_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
        L.gen_normal_f32.argtypes = [u64, u64, u64, u64, dbl, vp, i32]
        L.gen_uniform_int.argtypes = [u64, u64, u64, i64, i64, vp]
        L.gen_signs.argtypes = [u64, u64, u64, vp]
        L.gen_words.argtypes = [u64, u64, u64, u64, vp]
        L.gen_mix64.argtypes = [u64]
        L.gen_mix64.restype = u64
        for f in (L.gen_normal_bf16, L.gen_normal_f32, L.gen_uniform_int, L.gen_signs, L.gen_words):
            f.restype = None
        _lib = L
    return _lib


def tensor_id(kind: int, layer: int = 0, index: int = 0) -> int:
    """Stream id of one tensor: kind in bits 40+, layer in bits 32-39, index below."""
    return (kind << 40) | (layer << 32) | index


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, tid: int, n: int, sigma: float = 1.0, first: int = 0,
                out: np.ndarray | None = None) -> np.ndarray:
    """n bf16 values (as uint16 bit patterns) of a N(0, sigma^2) stream."""
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    assert out.dtype == np.uint16 and out.size == n and out.flags.c_contiguous
    lib().gen_normal_bf16(seed, tid, first, n, sigma, out.ctypes.data, _threads())
    return out


def normal_f32(seed: int, tid: int, n: int, sigma: float = 1.0, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().gen_normal_f32(seed, tid, first, n, sigma, out.ctypes.data, _threads())
    return out


def uniform_int(seed: int, tid: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    lib().gen_uniform_int(seed, tid, n, lo, hi, out.ctypes.data)
    return out


def signs(seed: int, n: int = D) -> np.ndarray:
    out = np.empty(n, dtype=np.int8)
    lib().gen_signs(seed, tensor_id(KIND_SIGNS), n, out.ctypes.data)
    return out


def words(seed: int, tid: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    lib().gen_words(seed, tid, first, n, out.ctypes.data)
    return out


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# The five workloads.
# ---------------------------------------------------------------------------


@dataclass
class Workload:
    """One seeded workload.

    ``seq_len[s]`` is the number of keys in K cache ``s``; ``query_seq[b]`` the
    cache query b reads and ``n_visible[b]`` how many of its leading keys it sees.
    A "Full" layer scores every visible key; a "Reindex" layer scores only the
    candidate pool built by the Full layer before it.
    """
    name: str
    seed: int
    seq_len: list[int]
    query_seq: list[int]
    n_visible: list[int]
    full_layers: int = 1          # Full layers, each with its own K caches
    reindex_layers: int = 0       # pooled Reindex layers after the (last) Full layer
    build_pool: bool = True
    k: int = 512
    block_size: int = 8
    n_keep: int = 2048
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.query_seq)

    def k_bf16(self, layer: int, seq: int, first_row: int = 0, rows: int | None = None) -> np.ndarray:
        """bf16 bits [rows][128] of K cache ``seq`` of Full layer ``layer``."""
        n = self.seq_len[seq]
        rows = n - first_row if rows is None else rows
        a = normal_bf16(self.seed, tensor_id(KIND_K, layer, seq), rows * D, 1.0, first_row * D)
        return a.reshape(rows, D)

    def kv_bf16(self, seq: int, first_row: int = 0, rows: int | None = None) -> np.ndarray:
        """bf16 bits [rows][512] of the main-KV cache of sequence ``seq`` (N(0, 1):
        entries after an RMSNorm with unit weights have unit RMS)."""
        n = self.seq_len[seq]
        rows = n - first_row if rows is None else rows
        a = normal_bf16(self.seed, tensor_id(KIND_KV, 0, seq), rows * DKV, 1.0, first_row * DKV)
        return a.reshape(rows, DKV)

    def q_bf16(self, layer: int, query: int) -> np.ndarray:
        """bf16 bits [32][128] of the indexer query of ``query`` at ``layer``.

        Layers 0 .. full_layers-1 are Full layers; full_layers + r is Reindex r.
        """
        return normal_bf16(self.seed, tensor_id(KIND_Q, layer, query), H * D).reshape(H, D)

    def w(self, layer: int, query: int) -> np.ndarray:
        return normal_f32(self.seed, tensor_id(KIND_W, layer, query), H, (1.0 / 32.0) ** 0.5)

    def signs(self) -> np.ndarray:
        return signs(self.seed)


def workload(idx: int) -> Workload:
    """The five workloads (index 0..4), sizes exactly as they are specified."""
    if idx == 0:
        return Workload("decode_b1_n32k", 0, [32768], [0], [32768], 1, 1, True,
                        notes="single decode query, one Full layer over 32768 keys, pool, one Reindex layer")
    if idx == 1:
        lens = uniform_int(1, tensor_id(KIND_LEN), 16, 4096, 131072).tolist()
        return Workload("decode_b16_mixed", 1, lens, list(range(16)), list(lens), 1, 4, True,
                        notes="16 decode queries, context lengths uniform in [4096, 131072], Full + pool + 4 Reindex")
    if idx == 2:
        n = 1 << 20
        return Workload("decode_b64_n1m", 2, [n] * 64, list(range(64)), [n] * 64, 1, 4, True,
                        notes="64 decode queries at 1,048,576 visible keys each, Full + pool + 4 Reindex")
    if idx == 3:
        n = 1 << 19
        return Workload("encoder_b64_3x512k", 3, [n] * 64, list(range(64)), [n] * 64, 3, 0, False,
                        notes="64 queries, 3 independent Full layers of 524,288 keys each, top-512, no pool")
    if idx == 4:
        n = 131072
        nq = 8192
        return Workload("prefill_8192_on_131k", 4, [n], [0] * nq, [122881 + t for t in range(nq)], 1, 0, True,
                        notes="8192 chunked-prefill queries on one 131,072-key cache, query t sees keys [0, 122880+t]")
    raise ValueError(idx)


def scaled_workload(idx: int, shrink: int) -> Workload:
    """A smaller copy of workload ``idx`` (lengths divided by ``shrink``) for quick tests."""
    w = workload(idx)
    f = lambda n: max(1, n // shrink)
    w.seq_len = [f(n) for n in w.seq_len]
    w.n_visible = [min(f(n), w.seq_len[s]) for n, s in zip(w.n_visible, w.query_seq)]
    w.name += f"_div{shrink}"
    return w
