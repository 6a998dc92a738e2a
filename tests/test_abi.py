"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every
function include/hsi.h declares, and rejects bad host-side arguments before it
touches the device."""
import ctypes
import os
import re
import shutil

import pytest

import long_context_decode_lightning_gb300 as hsi
from conftest import ROOT

needs_nvcc = pytest.mark.skipif(shutil.which("nvcc") is None, reason="nvcc not on PATH")


def _declared():
    src = open(os.path.join(ROOT, "include", "hsi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hsi_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    hsi.build()
    return hsi.lib()


@needs_nvcc
def test_exports_every_declared_function(L):
    names = _declared()
    assert set(names) == set(hsi.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


@needs_nvcc
def test_status_strings(L):
    for code in hsi.STATUS:
        s = L.hsi_status_string(code)
        assert s and s != b"unknown status"
    assert L.hsi_status_string(12345) == b"unknown status"


@needs_nvcc
def test_workspace_sizes(L):
    assert hsi.workspace_size(hsi.WS_SCORE, 64, 1 << 20) == 0
    assert hsi.workspace_size(hsi.WS_QUANTIZE, 3, 0) >= 12
    assert hsi.workspace_size(hsi.WS_TOPK, 4, 16384, 512) == 0  # fits in shared memory
    big = hsi.workspace_size(hsi.WS_TOPK, 4, 1 << 20, 512)
    assert big >= 4 * 4096 * 4 + 4 * 16384 * 8
    pool8 = hsi.workspace_size(hsi.WS_POOL, 2, 1 << 20, 8)
    assert pool8 >= 2 * (1 << 17) * 4


@needs_nvcc
def test_host_validation_rejects_bad_arguments(L):
    fake = 1 << 20  # never dereferenced: validation fails first
    s8 = (ctypes.c_int8 * 128)(*([1] * 128))
    bad_signs = (ctypes.c_int8 * 128)(*([2] * 128))
    # quantize: null x, bad sizes, bad mode, bad signs, unaligned record buffer
    assert L.hsi_quantize_nvfp4(None, 1, 1, s8, 0, fake, fake, fake, 256, None) == -1
    assert L.hsi_quantize_nvfp4(fake, 0, 1, s8, 0, fake, fake, fake, 256, None) == -1
    assert L.hsi_quantize_nvfp4(fake, 1, 1, s8, 2, fake, fake, fake, 256, None) == -1
    assert L.hsi_quantize_nvfp4(fake, 1, 1, bad_signs, 0, fake, fake, fake, 256, None) == -1
    assert L.hsi_quantize_nvfp4(fake, 1, 1, s8, 0, fake, fake + 8, fake, 256, None) == -1
    assert L.hsi_quantize_nvfp4(fake, 1, 1, s8, 0, fake, fake, None, 0, None) == -5
    # score_full: group 3 unsupported, ld too small, B not a multiple of the group
    args = [fake] * 7
    assert L.hsi_score_full(*args, 1, 100, 3, fake, 100, None, 0, 0, None, 0, None) == -2
    assert L.hsi_score_full(*args, 1, 100, 1, fake, 99, None, 0, 0, None, 0, None) == -1
    assert L.hsi_score_full(*args, 6, 100, 4, fake, 100, None, 0, 0, None, 0, None) == -1
    assert L.hsi_score_full(*args, 1, 100, 1, fake, 100, fake, 12, 0, None, 0, None) == -1
    # record format: unknown format; NVFP4 needs its tensor scales (MXFP4 has none)
    assert L.hsi_score_full(*args, 1, 100, 1, fake, 100, None, 0, 2, None, 0, None) == -1
    assert L.hsi_score_full(fake, None, *[fake] * 5, 1, 100, 1, fake, 100, None, 0, 0, None, 0, None) == -1
    assert L.hsi_pool_gather(fake, fake, fake, fake, fake, 2048, 1, fake + 4096, 3, None) == -1
    # main KV: null input, unaligned entries, k out of range, ld_idx < k
    assert L.hsi_quantize_mainkv(None, 4, fake, None) == -1
    assert L.hsi_quantize_mainkv(fake, 4, fake + 8, None) == -1
    assert L.hsi_quantize_mainkv(fake, 0, fake, None) == -1
    assert L.hsi_gather_mainkv(fake, fake, fake, fake, 512, 0, 4, fake, None) == -1
    assert L.hsi_gather_mainkv(fake, fake, fake, fake, 512, 5000, 4, fake, None) == -1
    assert L.hsi_gather_mainkv(fake, fake, fake, fake, 511, 512, 4, fake, None) == -1
    assert L.hsi_gather_mainkv(fake + 4, fake, fake, fake, 512, 512, 4, fake, None) == -1
    # append_token: NVFP4 needs the tensor scales; main KV needs its buffer and offsets; unaligned rows
    assert L.hsi_append_token(fake, s8, None, fake, fake, None, None, None, fake, fake, 4, 0, None) == -1
    assert L.hsi_append_token(fake, s8, fake, fake, fake, fake, None, None, fake, fake, 4, 0, None) == -1
    assert L.hsi_append_token(fake + 8, s8, fake, fake, fake, None, None, None, fake, fake, 4, 0, None) == -1
    assert L.hsi_append_token(fake, bad_signs, fake, fake, fake, None, None, None, fake, fake, 4, 0, None) == -1
    assert L.hsi_append_token(fake, s8, fake, fake, fake, None, None, None, fake, fake, 0, 0, None) == -1
    # mask_scores: ld or the bit table's stride too short for max_visible
    assert L.hsi_mask_scores(fake, 99, fake, fake, 4, 1, 100, None) == -1
    assert L.hsi_mask_scores(fake, 100, fake, fake, 3, 1, 100, None) == -1
    # quantize_mxfp4: null x, bad signs, unaligned records
    assert L.hsi_quantize_mxfp4(None, 1, 1, s8, fake, None) == -1
    assert L.hsi_quantize_mxfp4(fake, 1, 1, bad_signs, fake, None) == -1
    assert L.hsi_quantize_mxfp4(fake, 1, 1, s8, fake + 8, None) == -1
    # topk: k out of range, workspace missing for a long row
    assert L.hsi_topk(fake, 10, fake, 1, 10, 0, None, 0, 8, fake, fake, None, 0, None) == -1
    assert L.hsi_topk(fake, 10, fake, 1, 10, 4096, None, 0, 8, fake, fake, None, 0, None) == -1
    assert L.hsi_topk(fake, 1 << 20, fake, 1, 1 << 20, 512, None, 0, 8, fake, fake, None, 0, None) == -5
    # pool: block size, keep, block maxima only for block 8
    assert L.hsi_candidate_pool(fake, 100, None, 0, fake, 1, 100, 0, 16, fake, fake, fake, None, 0, fake, 1 << 20,
                                None) == -1
    assert L.hsi_candidate_pool(fake, 100, None, 0, fake, 1, 100, 8, 5000, fake, fake, fake, None, 0, fake,
                                1 << 20, None) == -1
    assert L.hsi_candidate_pool(None, 0, fake, 100, fake, 1, 100, 4, 16, fake, fake, fake, None, 0, fake, 1 << 20,
                                None) == -1
    # score_pool: ld shorter than 8 * n_keep
    assert L.hsi_score_pool(*args, fake, fake, 2048, 1, fake, 2048 * 8 - 1, 0, None, 0, None) == -1
    # score_full: neither a score row nor block maxima
    assert L.hsi_score_full(*args, 1, 100, 1, None, 0, None, 0, 0, None, 0, None) == -1
    # full_layer without scores: needs the pool, n_keep - 1 >= k; n_keep <= 2048, a multiple of 32
    ws_big = 1 << 40
    def fl(scores, k, n_keep, ids):
        return L.hsi_full_layer(*args, 1, 1 << 20, scores, 0, k, fake, fake, n_keep, ids, fake, fake, None, 0, 3, 0,
                                fake, ws_big, None)
    assert fl(None, 512, 2048, None) == -1
    assert fl(None, 512, 512, fake) == -1
    assert fl(None, 512, 4096, fake) == -2
    assert fl(None, 512, 2047, fake) == -2
