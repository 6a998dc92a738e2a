"""Python binding of libhsi, the GB300 hot path of the Hierarchical Sparse Indexer.

Argument marshalling only: every function passes device pointers of torch
tensors, sizes and the current CUDA stream to the C ABI declared in
``include/hsi.h`` and raises ``HsiError`` on a non-OK status. No step of the
path runs in Python or torch. The library must have been built (``build()``);
importing this module on a machine without it raises at the first call.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_SO = os.path.join(_PKG, "libhsi.so")
_lib = None

HEADS, DIM, REC_ROWS, REC_BYTES, MX_REC_BYTES = 32, 128, 8, 576, 544
PHASE_SCORE, PHASE_SELECT, PHASE_ALL, PHASE_TOPK, PHASE_POOL = 1, 2, 3, 4, 8
FMT_NVFP4, FMT_MXFP4 = 0, 1  # hsi_format: NVFP4 (576-byte records, tensor scales) or MXFP4 (544 bytes)

STATUS = {0: "HSI_OK", -1: "HSI_ERR_INVALID_ARG", -2: "HSI_ERR_UNSUPPORTED", -3: "HSI_ERR_CUDA",
          -4: "HSI_ERR_DEVICE_TIMEOUT", -5: "HSI_ERR_WORKSPACE", -6: "HSI_ERR_DEVICE_ARG", -7: "HSI_ERR_TOO_LARGE"}
WS_QUANTIZE, WS_SCORE, WS_TOPK, WS_POOL, WS_FULL_LAYER, WS_REINDEX_LAYER, WS_PREFILL_LAYER = 0, 1, 2, 3, 4, 5, 6

EXPORTS = ["hsi_quantize_nvfp4", "hsi_score_full", "hsi_topk", "hsi_candidate_pool", "hsi_score_pool",
           "hsi_workspace_size", "hsi_device_error", "hsi_device_check", "hsi_status_string",
           "hsi_kernel_launches", "hsi_calib_read", "hsi_calib_mma", "hsi_full_layer", "hsi_reindex_layer",
           "hsi_topk_noalloc", "hsi_debug_set", "hsi_pool_gather", "hsi_quantize_mxfp4", "hsi_quantize_mainkv",
           "hsi_gather_mainkv", "hsi_append_token", "hsi_mask_scores", "hsi_prefill_layer",
           "hsi_gather_mainkv_layers"]


class HsiError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)}")


def nvcc_command(out: str = _SO) -> list[str]:
    return ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
            "-Xcompiler", "-fPIC", "-shared", "-o", out, os.path.join(_CSRC, "hsi.cu")]


def build(force: bool = False) -> str:
    """Compile libhsi.so for sm_103a in the package directory."""
    srcs = [os.path.join(_CSRC, f) for f in os.listdir(_CSRC)] + [os.path.join(_ROOT, "include", "hsi.h")]
    newest = max(os.path.getmtime(s) for s in srcs)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(nvcc_command(tmp))
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_SO):
            raise RuntimeError(f"libhsi is not built ({_SO} missing); run __graft_entry__.build()")
        L = ctypes.CDLL(_SO)
        vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        L.hsi_quantize_nvfp4.argtypes = [vp, i64, i64, vp, ctypes.c_int, vp, vp, vp, sz, vp]
        L.hsi_quantize_mxfp4.argtypes = [vp, i64, i64, vp, vp, vp]
        L.hsi_quantize_mainkv.argtypes = [vp, i64, vp, vp]
        L.hsi_gather_mainkv.argtypes = [vp, vp, vp, vp, i64, i32, i32, vp, vp]
        L.hsi_gather_mainkv_layers.argtypes = [vp, vp, vp, vp, i64, i64, i32, i32, i32, vp, i64, vp]
        L.hsi_append_token.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, ctypes.c_int, vp]
        L.hsi_mask_scores.argtypes = [vp, i64, vp, vp, i64, i32, i64, vp]
        L.hsi_score_full.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, vp, i64, vp, i64, ctypes.c_int, vp,
                                     sz, vp]
        L.hsi_topk.argtypes = [vp, i64, vp, i32, i64, i32, vp, i64, i32, vp, vp, vp, sz, vp]
        L.hsi_candidate_pool.argtypes = [vp, i64, vp, i64, vp, i32, i64, i32, i32, vp, vp, vp, vp, i64, vp, sz, vp]
        L.hsi_score_pool.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, vp, i64, ctypes.c_int, vp, sz,
                                     vp]
        L.hsi_full_layer.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, vp, i64, i32, vp, vp, i32, vp, vp, vp,
                                     vp, i64, i32, ctypes.c_int, vp, sz, vp]
        L.hsi_prefill_layer.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, vp, i64, i32, vp, vp, i32, vp, vp,
                                        vp, vp, i64, i32, ctypes.c_int, vp, sz, vp]
        L.hsi_reindex_layer.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, i32, vp, i64, i32, vp,
                                        vp, ctypes.c_int, vp, sz, vp]
        L.hsi_pool_gather.argtypes = [vp, vp, vp, vp, vp, i32, i32, vp, ctypes.c_int, vp]
        L.hsi_topk_noalloc.argtypes = [vp, i64, vp, i32, i64, i32, vp, i64, i32, vp, vp, vp]
        L.hsi_debug_set.argtypes = [ctypes.c_int, ctypes.c_longlong]
        L.hsi_workspace_size.argtypes = [ctypes.c_int, i32, i64, i32]
        L.hsi_workspace_size.restype = sz
        L.hsi_device_error.argtypes = [vp]
        L.hsi_device_check.argtypes = []
        L.hsi_status_string.argtypes = [ctypes.c_int]
        L.hsi_status_string.restype = ctypes.c_char_p
        L.hsi_calib_read.argtypes = [vp, sz, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp]
        L.hsi_calib_mma.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp]
        L.hsi_kernel_launches.argtypes = []
        L.hsi_kernel_launches.restype = ctypes.c_uint64
        for name in ("hsi_quantize_nvfp4", "hsi_score_full", "hsi_topk", "hsi_candidate_pool", "hsi_score_pool",
                     "hsi_device_error", "hsi_device_check", "hsi_calib_read", "hsi_calib_mma", "hsi_full_layer",
                     "hsi_reindex_layer", "hsi_topk_noalloc", "hsi_debug_set", "hsi_pool_gather",
                     "hsi_quantize_mxfp4", "hsi_quantize_mainkv", "hsi_gather_mainkv", "hsi_append_token",
                     "hsi_mask_scores", "hsi_prefill_layer", "hsi_gather_mainkv_layers"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn: str, st: int):
    if st != 0:
        raise HsiError(fn, st)


def workspace_size(kind: int, B: int, max_n: int, k: int = 0) -> int:
    return int(lib().hsi_workspace_size(kind, B, max_n, k))


def workspace(kind: int, B: int, max_n: int, k: int = 0, device="cuda") -> torch.Tensor | None:
    """A caller-owned scratch buffer for one call (256-byte aligned by torch)."""
    n = workspace_size(kind, B, max_n, k)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().hsi_kernel_launches())


DEBUG_WAIT_LIMIT_NS, DEBUG_SKIP_FIRST_COPY = 1, 2


def debug_set(what: int, value: int):
    """Diagnostics: the kernels' wait limit, or the test switch that makes a wait run out."""
    _check("hsi_debug_set", lib().hsi_debug_set(what, value))


def device_check():
    _check("hsi_device_check", lib().hsi_device_check())


def device_error(stream=None) -> int:
    """Synchronise, then return and clear the sticky device status (0 = OK)."""
    return int(lib().hsi_device_error(_stream(stream)))


def calib_read(buf: torch.Tensor, method: int = 0, chunk: int = 9216, stages: int = 12, sink=None, stream=None):
    sink = torch.zeros(1, dtype=torch.int64, device=buf.device) if sink is None else sink
    _check("hsi_calib_read", lib().hsi_calib_read(_ptr(buf), buf.numel() * buf.element_size(), method, chunk,
                                                  stages, _ptr(sink), _stream(stream)))


def calib_mma(n: int, iters: int, sink=None, device="cuda", stream=None):
    sink = torch.zeros(1, dtype=torch.int64, device=device) if sink is None else sink
    _check("hsi_calib_mma", lib().hsi_calib_mma(n, iters, _ptr(sink), _stream(stream)))


def n_records(rows: int) -> int:
    return (rows + REC_ROWS - 1) // REC_ROWS


def quantize_nvfp4(x: torch.Tensor, n_tensors: int, rows_per_tensor: int, signs, g: torch.Tensor,
                   rec: torch.Tensor, mode: int = 0, ws: torch.Tensor | None = None, stream=None):
    """x: bf16 (or its int16 bits) [n_tensors*rows_per_tensor, 128] on the device."""
    s8 = (ctypes.c_int8 * 128)(*[int(v) for v in signs])
    if mode == 0 and ws is None:
        ws = workspace(WS_QUANTIZE, n_tensors, 0, device=x.device)
    _check("hsi_quantize_nvfp4", lib().hsi_quantize_nvfp4(
        _ptr(x), n_tensors, rows_per_tensor, s8, mode, _ptr(g), _ptr(rec), _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def quantize_mxfp4(x: torch.Tensor, n_tensors: int, rows_per_tensor: int, signs, rec: torch.Tensor, stream=None):
    """x: bf16 (or its int16 bits) [n_tensors*rows_per_tensor, 128] -> MXFP4 records (no tensor scale)."""
    s8 = (ctypes.c_int8 * 128)(*[int(v) for v in signs])
    _check("hsi_quantize_mxfp4", lib().hsi_quantize_mxfp4(
        _ptr(x), n_tensors, rows_per_tensor, s8, _ptr(rec), _stream(stream)))


KV_DIM, KV_ENTRY_BYTES = 512, 288


def quantize_mainkv(x: torch.Tensor, kv: torch.Tensor, stream=None):
    """x: bf16 (or its int16 bits) [n, 512] -> FP4 main-KV entries kv [n*288] bytes."""
    n = x.numel() // KV_DIM
    _check("hsi_quantize_mainkv", lib().hsi_quantize_mainkv(_ptr(x), n, _ptr(kv), _stream(stream)))


def gather_mainkv(kv, kv_off, n_visible, idx, k, B, out, ld_idx=None, stream=None):
    """gather(main_kv, topk): out [B, k, 512] bf16 bits = the entries idx selects, decoded (0 rows for -1)."""
    ld_idx = idx.shape[-1] if ld_idx is None else ld_idx
    _check("hsi_gather_mainkv", lib().hsi_gather_mainkv(
        _ptr(kv), _ptr(kv_off), _ptr(n_visible), _ptr(idx), ld_idx, k, B, _ptr(out), _stream(stream)))


def gather_mainkv_layers(kv, kv_off, n_visible, idx, k, B, out, stream=None):
    """gather(main_kv, topk) for L layers in one launch: idx [L, B, ld_idx] int32, out [L, B, k, 512] bf16 bits."""
    L, ld_idx = idx.shape[0], idx.shape[-1]
    _check("hsi_gather_mainkv_layers", lib().hsi_gather_mainkv_layers(
        _ptr(kv), _ptr(kv_off), _ptr(n_visible), _ptr(idx), ld_idx, idx.stride(0), L, k, B, _ptr(out),
        out.stride(0), _stream(stream)))


def append_token(k_x, signs, g_k, k_rec, k_rec_off, n_visible, capacity, B, kv_x=None, kv=None, kv_off=None,
                 fmt=FMT_NVFP4, stream=None):
    """One decode token into every query's caches (K row, optional main-KV entry); n_visible += 1 on the device."""
    s8 = (ctypes.c_int8 * 128)(*[int(v) for v in signs])
    _check("hsi_append_token", lib().hsi_append_token(
        _ptr(k_x), s8, _ptr(g_k), _ptr(k_rec), _ptr(k_rec_off), _ptr(kv_x), _ptr(kv), _ptr(kv_off),
        _ptr(n_visible), _ptr(capacity), B, fmt, _stream(stream)))


def mask_scores(scores, n_visible, pool_bits, B, max_visible, ld=None, ld_bits=None, stream=None):
    """The masked Reindex form: -inf at the visible positions outside each query's pool bit table."""
    ld = scores.shape[-1] if ld is None else ld
    ld_bits = pool_bits.shape[-1] if ld_bits is None else ld_bits
    _check("hsi_mask_scores", lib().hsi_mask_scores(_ptr(scores), ld, _ptr(n_visible), _ptr(pool_bits), ld_bits, B,
                                                    max_visible, _stream(stream)))


def rec_bytes(fmt: int = FMT_NVFP4) -> int:
    return MX_REC_BYTES if fmt == FMT_MXFP4 else REC_BYTES


def score_full(q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B, max_visible, scores, ld=None,
               block_max=None, ldb=0, group=1, fmt=FMT_NVFP4, stream=None):
    """scores None (block_max given): the block maxima only, no score row."""
    ld = (scores.shape[-1] if scores is not None else 0) if ld is None else ld
    if block_max is not None and not ldb:
        ldb = block_max.shape[-1]
    _check("hsi_score_full", lib().hsi_score_full(
        _ptr(q_rec), _ptr(g_q), _ptr(w), _ptr(k_rec), _ptr(g_k), _ptr(k_rec_off), _ptr(n_visible), B,
        max_visible, group, _ptr(scores), ld, _ptr(block_max), ldb, fmt, None, 0, _stream(stream)))


def topk(scores, n_valid, B, max_valid, k, out_idx, out_val, ld=None, block_ids=None, ld_blocks=0,
         block_size=8, ws=None, stream=None):
    ld = scores.shape[-1] if ld is None else ld
    if ws is None:
        ws = workspace(WS_TOPK, B, max_valid, k, device=scores.device)
    if block_ids is not None and not ld_blocks:
        ld_blocks = block_ids.shape[-1]
    _check("hsi_topk", lib().hsi_topk(
        _ptr(scores), ld, _ptr(n_valid), B, max_valid, k, _ptr(block_ids), ld_blocks, block_size,
        _ptr(out_idx), _ptr(out_val), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def topk_noalloc(scores, n_valid, B, max_valid, k, out_idx, out_val, ld=None, block_ids=None, ld_blocks=0,
                 block_size=8, stream=None):
    """hsi_topk for callers that cannot allocate: no workspace argument; the
    long-row passes use the library's fixed 8 MiB device scratch instead."""
    ld = scores.shape[-1] if ld is None else ld
    if block_ids is not None and not ld_blocks:
        ld_blocks = block_ids.shape[-1]
    _check("hsi_topk_noalloc", lib().hsi_topk_noalloc(
        _ptr(scores), ld, _ptr(n_valid), B, max_valid, k, _ptr(block_ids), ld_blocks, block_size,
        _ptr(out_idx), _ptr(out_val), _stream(stream)))


def candidate_pool(n_visible, B, max_visible, block_ids, n_kept, n_pool, scores=None, ld=0, block_max=None,
                   ldb=0, block_size=8, n_keep=2048, pool_bits=None, ld_bits=0, ws=None, stream=None):
    if scores is not None and not ld:
        ld = scores.shape[-1]
    if block_max is not None and not ldb:
        ldb = block_max.shape[-1]
    if pool_bits is not None and not ld_bits:
        ld_bits = pool_bits.shape[-1]
    if ws is None:
        dev = (scores if scores is not None else block_max).device
        ws = workspace(WS_POOL, B, max_visible, block_size, device=dev)
    _check("hsi_candidate_pool", lib().hsi_candidate_pool(
        _ptr(scores), ld, _ptr(block_max), ldb, _ptr(n_visible), B, max_visible, block_size, n_keep,
        _ptr(block_ids), _ptr(n_kept), _ptr(n_pool), _ptr(pool_bits), ld_bits, _ptr(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def score_pool(q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, block_ids, n_kept, n_keep, B, pool_scores,
               ld=None, fmt=FMT_NVFP4, stream=None):
    ld = pool_scores.shape[-1] if ld is None else ld
    _check("hsi_score_pool", lib().hsi_score_pool(
        _ptr(q_rec), _ptr(g_q), _ptr(w), _ptr(k_rec), _ptr(g_k), _ptr(k_rec_off), _ptr(n_visible),
        _ptr(block_ids), _ptr(n_kept), n_keep, B, _ptr(pool_scores), ld, fmt, None, 0, _stream(stream)))


def full_layer(q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B, max_visible, scores, k, top_idx, top_val,
               block_ids=None, n_kept=None, n_pool=None, pool_bits=None, n_keep=2048, ld=None, ld_bits=0, ws=None,
               phases=3, fmt=FMT_NVFP4, stream=None):
    """Full layer: scores, top-k and (block_ids given) the candidate pool.
    phases: 1 scoring only, 2 selection only (after 1, same workspace), 3 both;
    4 the top-k only, 8 the pool only (after 1; the two may run on two streams).
    scores None: no score row; the top-k is taken from the pool (phase 4 after 8)."""
    ld = (scores.shape[-1] if scores is not None else 0) if ld is None else ld
    if pool_bits is not None and not ld_bits:
        ld_bits = pool_bits.shape[-1]
    if ws is None:
        ws = workspace(WS_FULL_LAYER, B, max_visible, k, device=top_idx.device)
    _check("hsi_full_layer", lib().hsi_full_layer(
        _ptr(q_rec), _ptr(g_q), _ptr(w), _ptr(k_rec), _ptr(g_k), _ptr(k_rec_off), _ptr(n_visible), B, max_visible,
        _ptr(scores), ld, k, _ptr(top_idx), _ptr(top_val), n_keep, _ptr(block_ids), _ptr(n_kept), _ptr(n_pool),
        _ptr(pool_bits), ld_bits, phases, fmt, _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def prefill_layer(q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, B, max_visible, scores, k, top_idx, top_val,
                  group=4, block_ids=None, n_kept=None, n_pool=None, pool_bits=None, n_keep=2048, ld=None, ld_bits=0,
                  ws=None, phases=3, fmt=FMT_NVFP4, stream=None):
    """Chunked-prefill layer: scores (groups of `group` queries share a cache), then each
    query's top-k and (block_ids given) pool from the block maxima.
    phases: 1 scoring only, 2 selection only (after 1, same workspace), 3 both."""
    ld = scores.shape[-1] if ld is None else ld
    if pool_bits is not None and not ld_bits:
        ld_bits = pool_bits.shape[-1]
    if ws is None:
        ws = workspace(WS_PREFILL_LAYER, B, max_visible, k, device=scores.device)
    _check("hsi_prefill_layer", lib().hsi_prefill_layer(
        _ptr(q_rec), _ptr(g_q), _ptr(w), _ptr(k_rec), _ptr(g_k), _ptr(k_rec_off), _ptr(n_visible), B, max_visible,
        group, _ptr(scores), ld, k, _ptr(top_idx), _ptr(top_val), n_keep, _ptr(block_ids), _ptr(n_kept),
        _ptr(n_pool), _ptr(pool_bits), ld_bits, phases, fmt, _ptr(ws), 0 if ws is None else ws.numel(),
        _stream(stream)))


def pool_gather(k_rec, k_rec_off, n_visible, block_ids, n_kept, B, pool_rec, n_keep=2048, fmt=FMT_NVFP4,
                stream=None):
    """Compact each query's pooled K records into pool_rec [B][n_keep][record bytes] (block-list order)."""
    _check("hsi_pool_gather", lib().hsi_pool_gather(
        _ptr(k_rec), _ptr(k_rec_off), _ptr(n_visible), _ptr(block_ids), _ptr(n_kept), n_keep, B, _ptr(pool_rec),
        fmt, _stream(stream)))


def reindex_layer(q_rec, g_q, w, k_rec, g_k, k_rec_off, n_visible, block_ids, n_kept, n_pool, B, pool_scores, k,
                  top_idx, top_val, n_keep=2048, ld=None, ws=None, pool_rec=None, pool_rec_ready=True, fmt=FMT_NVFP4,
                  stream=None):
    """Reindex layer: pooled scores and the top-k inside the pool (global positions).
    pool_rec None: gathered from k_rec. pool_rec with pool_rec_ready: the compacted pool
    (pool_gather, or an earlier layer) is streamed; without: gathered from k_rec and the
    compacted pool left in pool_rec."""
    ld = pool_scores.shape[-1] if ld is None else ld
    if ws is None:
        ws = workspace(WS_REINDEX_LAYER, B, 8 * n_keep, k, device=pool_scores.device)
    _check("hsi_reindex_layer", lib().hsi_reindex_layer(
        _ptr(q_rec), _ptr(g_q), _ptr(w), _ptr(k_rec), _ptr(g_k), _ptr(k_rec_off), _ptr(pool_rec),
        1 if pool_rec_ready else 0, _ptr(n_visible),
        _ptr(block_ids),
        _ptr(n_kept), _ptr(n_pool), n_keep, B, _ptr(pool_scores), ld, k, _ptr(top_idx), _ptr(top_val), fmt,
        _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))
