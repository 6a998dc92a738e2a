"""ORACLE -- test infrastructure, not the product.

ctypes binding of ``oracle.c``: a plain single-threaded CPU restatement of the
Hierarchical Sparse Indexer decode path (NVFP4 and MXFP4 codecs, rotation,
quantisation, fp64 scoring, full-sort top-k, the candidate pool, pooled
Reindex scoring).
Only the tests, the smoke check and the bench's CPU-baseline leg use it; the
CUDA path never imports it.

Every function here works on one query (or one tensor) at a time. ``map_queries``
runs a function over many queries on a thread pool; ctypes releases the GIL
during each C call, so the threads run on separate cores.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

REC_BYTES = 576
MX_REC_BYTES = 544
FMTS = {"nvfp4": 0, "mxfp4": 1}
ROWS_PER_REC = 8
H = 32
D = 128


def build(force: bool = False) -> str:
    """Compile the oracle (no FMA contraction, IEEE fp32/fp64, no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        vp, i64, i32, f32, u8 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint8
        L.hsio_e2m1_value.argtypes = [u8]
        L.hsio_e2m1_value.restype = ctypes.c_double
        L.hsio_e4m3_value.argtypes = [u8]
        L.hsio_e4m3_value.restype = ctypes.c_double
        L.hsio_e4m3_encode.argtypes = [f32]
        L.hsio_e4m3_encode.restype = u8
        L.hsio_e2m1_encode.argtypes = [f32]
        L.hsio_e2m1_encode.restype = u8
        L.hsio_fwht128.argtypes = [vp]
        L.hsio_fwht128.restype = None
        L.hsio_quantize.argtypes = [vp, i64, vp, i32, vp, vp]
        L.hsio_quantize.restype = i32
        L.hsio_decode_row.argtypes = [vp, i64, f32, vp]
        L.hsio_decode_row.restype = None
        L.hsio_e8m0_value.argtypes = [u8]
        L.hsio_e8m0_value.restype = ctypes.c_double
        L.hsio_mx_scale_exp.argtypes = [f32]
        L.hsio_mx_scale_exp.restype = i32
        L.hsio_quantize_mx.argtypes = [vp, i64, vp, vp]
        L.hsio_quantize_mx.restype = i32
        L.hsio_decode_row_mx.argtypes = [vp, i64, vp]
        L.hsio_decode_row_mx.restype = None
        L.hsio_score_full_fmt.argtypes = [i32, vp, f32, vp, vp, f32, i64, vp]
        L.hsio_score_full_fmt.restype = i64
        L.hsio_score_rows_fmt.argtypes = [i32, vp, f32, vp, vp, f32, vp, i64, vp, vp]
        L.hsio_score_rows_fmt.restype = i64
        L.hsio_score_pool_fmt.argtypes = [i32, vp, f32, vp, vp, f32, i64, vp, ctypes.c_int32, ctypes.c_int32,
                                          i32, vp]
        L.hsio_score_pool_fmt.restype = i64
        L.hsio_mainkv_quantize.argtypes = [vp, i64, vp]
        L.hsio_mainkv_quantize.restype = i32
        L.hsio_mainkv_decode.argtypes = [vp, i64, vp]
        L.hsio_mainkv_decode.restype = None
        L.hsio_mainkv_gather.argtypes = [vp, i64, vp, i32, vp]
        L.hsio_mainkv_gather.restype = i32
        L.hsio_topk.argtypes = [vp, i64, i32, vp, vp]
        L.hsio_topk.restype = i64
        L.hsio_pool.argtypes = [vp, i64, i32, i32, vp, vp, vp, vp]
        L.hsio_pool.restype = i32
        L.hsio_topk_pool.argtypes = [vp, i64, vp, i32, i32, vp, vp]
        L.hsio_topk_pool.restype = i64
        L.hsio_topk_masked.argtypes = [vp, i64, vp, i32, vp, vp]
        L.hsio_topk_masked.restype = i64
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codecs ----

def e2m1_value(code: int) -> float:
    return lib().hsio_e2m1_value(code)


def e4m3_value(code: int) -> float:
    return lib().hsio_e4m3_value(code)


def e2m1_encode(x: float) -> int:
    return int(lib().hsio_e2m1_encode(float(x)))


def e4m3_encode(x: float) -> int:
    return int(lib().hsio_e4m3_encode(float(x)))


def e8m0_value(code: int) -> float:
    return lib().hsio_e8m0_value(code)


def mx_scale_exp(amax: float) -> int:
    """Exponent e of the MXFP4 group scale 2^e for a group whose largest magnitude is amax."""
    return int(lib().hsio_mx_scale_exp(float(amax)))


def fwht128(v: np.ndarray) -> np.ndarray:
    out = _c(v, np.float32).copy()
    assert out.size == D
    lib().hsio_fwht128(_p(out))
    return out


# -------------------------------------------------------------- quantise ----

def n_records(rows: int) -> int:
    return (rows + ROWS_PER_REC - 1) // ROWS_PER_REC


def quantize(x_bf16: np.ndarray, signs: np.ndarray, g: float | None = None):
    """Quantise one tensor (bf16 bits [rows][128]) -> (records uint8 [nrec*576], g).

    g None: computed from the tensor's amax (mode 0); else used as given (mode 1).
    """
    x = _c(x_bf16, np.uint16).reshape(-1, D)
    s = _c(signs, np.int8)
    rec = np.empty(n_records(x.shape[0]) * REC_BYTES, dtype=np.uint8)
    gg = np.array([0.0 if g is None else g], dtype=np.float32)
    rc = lib().hsio_quantize(_p(x), x.shape[0], _p(s), 0 if g is None else 1, _p(gg), _p(rec))
    if rc != 0:
        raise ValueError("oracle quantize: non-finite input or bad scale")
    return rec, float(gg[0])


def quantize_mx(x_bf16: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Quantise one tensor (bf16 bits [rows][128]) -> MXFP4 records uint8 [nrec*544] (no tensor scale)."""
    x = _c(x_bf16, np.uint16).reshape(-1, D)
    s = _c(signs, np.int8)
    rec = np.empty(n_records(x.shape[0]) * MX_REC_BYTES, dtype=np.uint8)
    if lib().hsio_quantize_mx(_p(x), x.shape[0], _p(s), _p(rec)) != 0:
        raise ValueError("oracle quantize_mx: non-finite input")
    return rec


def decode_row(records: np.ndarray, row: int, g: float = 1.0, fmt: str = "nvfp4") -> np.ndarray:
    out = np.empty(D, dtype=np.float64)
    if fmt == "mxfp4":
        lib().hsio_decode_row_mx(_p(records), row, _p(out))
    else:
        lib().hsio_decode_row(_p(records), row, g, _p(out))
    return out


def decode_rows(records: np.ndarray, rows: int, g: float = 1.0, fmt: str = "nvfp4") -> np.ndarray:
    return np.stack([decode_row(records, r, g, fmt) for r in range(rows)])


# --------------------------------------------------------------- main KV ----

KV_DIM, KV_BYTES = 512, 288


def mainkv_quantize(x_bf16: np.ndarray) -> np.ndarray:
    """bf16 bits [n][512] -> FP4 main-KV entries uint8 [n*288] (E2M1, E4M3 per 16, no global scale)."""
    x = _c(x_bf16, np.uint16).reshape(-1, KV_DIM)
    kv = np.empty(x.shape[0] * KV_BYTES, dtype=np.uint8)
    if lib().hsio_mainkv_quantize(_p(x), x.shape[0], _p(kv)) != 0:
        raise ValueError("oracle mainkv_quantize: non-finite input")
    return kv


def mainkv_decode(kv: np.ndarray, i: int) -> np.ndarray:
    out = np.empty(KV_DIM, dtype=np.float64)
    lib().hsio_mainkv_decode(_p(kv), i, _p(out))
    return out


def mainkv_gather(kv: np.ndarray, n_vis: int, idx: np.ndarray) -> np.ndarray:
    """gather(main_kv, topk) for one query -> bf16 bits [k][512] (zeros for idx < 0)."""
    idx = _c(idx, np.int32)
    out = np.empty((idx.size, KV_DIM), dtype=np.uint16)
    rc = lib().hsio_mainkv_gather(_p(kv), n_vis, _p(idx), idx.size, _p(out))
    if rc != 0:
        raise ValueError(f"oracle mainkv_gather: status {rc}")
    return out


# ----------------------------------------------------------------- score ----

def score_full(q_rec, g_q, w, k_rec, g_k, n_vis, fmt="nvfp4"):
    """fp32 scores of keys [0, n_vis) for one query; returns (scores, macs).
    fmt "mxfp4": MXFP4 records, g_q and g_k ignored (no tensor scale)."""
    out = np.empty(max(n_vis, 1), dtype=np.float32)
    w = _c(w, np.float32)
    f = FMTS[fmt]
    g_q, g_k = (1.0, 1.0) if f else (g_q, g_k)
    macs = lib().hsio_score_full_fmt(f, _p(q_rec), g_q, _p(w), _p(k_rec), g_k, n_vis, _p(out))
    return out[:n_vis], macs


def score_rows(q_rec, g_q, w, k_rec, g_k, rows, fmt="nvfp4"):
    """Scores and parity tolerances of the listed keys for one query."""
    rows = _c(rows, np.int64)
    out = np.empty(max(rows.size, 1), dtype=np.float32)
    tol = np.empty(max(rows.size, 1), dtype=np.float64)
    w = _c(w, np.float32)
    f = FMTS[fmt]
    g_q, g_k = (1.0, 1.0) if f else (g_q, g_k)
    lib().hsio_score_rows_fmt(f, _p(q_rec), g_q, _p(w), _p(k_rec), g_k, _p(rows), rows.size, _p(out), _p(tol))
    return out[:rows.size], tol[:rows.size]


# ----------------------------------------------------------------- top-k ----

def topk(scores: np.ndarray, n_valid: int, k: int):
    s = _c(scores, np.float32)
    idx = np.empty(k, dtype=np.int32)
    val = np.empty(k, dtype=np.float32)
    m = lib().hsio_topk(_p(s), n_valid, k, _p(idx), _p(val))
    if m < 0:
        raise ValueError("oracle topk: NaN score")
    return idx, val


# ------------------------------------------------------------------ pool ----

def pool(scores: np.ndarray, n_vis: int, block_size: int = 8, n_keep: int = 2048, want_mask=True):
    """-> (block_ids int32 [n_keep] ascending, -1 padded; n_kept; n_pool; mask uint8 [n_vis])"""
    s = _c(scores, np.float32)
    ids = np.empty(n_keep, dtype=np.int32)
    nk = np.zeros(1, dtype=np.int32)
    npool = np.zeros(1, dtype=np.int64)
    mask = np.empty(max(n_vis, 1), dtype=np.uint8) if want_mask else None
    rc = lib().hsio_pool(_p(s), n_vis, block_size, n_keep, _p(ids), _p(nk), _p(npool),
                         _p(mask) if want_mask else None)
    if rc != 0:
        raise ValueError("oracle pool: NaN score")
    return ids, int(nk[0]), int(npool[0]), (mask[:n_vis] if want_mask else None)


def score_pool(q_rec, g_q, w, k_rec, g_k, n_vis, block_ids, n_kept, n_keep=2048, block_size=8, fmt="nvfp4"):
    out = np.empty(n_keep * block_size, dtype=np.float32)
    w = _c(w, np.float32)
    ids = _c(block_ids, np.int32)
    f = FMTS[fmt]
    g_q, g_k = (1.0, 1.0) if f else (g_q, g_k)
    macs = lib().hsio_score_pool_fmt(f, _p(q_rec), g_q, _p(w), _p(k_rec), g_k, n_vis, _p(ids), n_kept, n_keep,
                                     block_size, _p(out))
    return out, macs


def topk_pool(pool_scores, n_pool, block_ids, k=512, block_size=8):
    s = _c(pool_scores, np.float32)
    ids = _c(block_ids, np.int32)
    idx = np.empty(k, dtype=np.int32)
    val = np.empty(k, dtype=np.float32)
    lib().hsio_topk_pool(_p(s), n_pool, _p(ids), block_size, k, _p(idx), _p(val))
    return idx, val


def topk_masked(scores_all, n_vis, mask, k=512):
    s = _c(scores_all, np.float32)
    m = _c(mask, np.uint8)
    idx = np.empty(k, dtype=np.int32)
    val = np.empty(k, dtype=np.float32)
    lib().hsio_topk_masked(_p(s), n_vis, _p(m), k, _p(idx), _p(val))
    return idx, val


# ------------------------------------------------------------- batching ----

def map_queries(fn, items, threads: int | None = None):
    """Run fn over items on `threads` OS threads (the C calls release the GIL)."""
    threads = threads or max(1, os.cpu_count() or 1)
    if threads == 1 or len(items) <= 1:
        return [fn(x) for x in items]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(fn, items))
