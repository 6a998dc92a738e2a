"""Failure detection on the GPU without a fault: a wait that nothing will ever
satisfy (the producer is told to skip its first copy) must run out after the
wait limit, the kernel must report HSI_ERR_DEVICE_TIMEOUT through the sticky
error word, and the context must stay usable for correct work afterwards."""
import time

import numpy as np
import pytest
import torch

import inputs
import oracle
from cases import DEV, Caches, gpu_queries, i32, i64, oracle_query

import long_context_decode_lightning_gb300 as hsi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hsi.build()
    hsi.device_check()
    yield
    hsi.debug_set(hsi.DEBUG_SKIP_FIRST_COPY, 0)
    hsi.debug_set(hsi.DEBUG_WAIT_LIMIT_NS, 1_000_000_000)


def test_wait_that_never_completes_times_out_and_context_survives():
    wl = inputs.workload(0)
    n = 5000
    caches = Caches(wl, 0, [0], [n])
    q_rec, g_q, w = gpu_queries(wl, 0, [0])
    scores = torch.zeros(1, n, device=DEV)
    assert hsi.device_error() == 0
    hsi.debug_set(hsi.DEBUG_WAIT_LIMIT_NS, 20_000_000)  # 20 ms
    hsi.debug_set(hsi.DEBUG_SKIP_FIRST_COPY, 1)
    t0 = time.time()
    hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, i64([0]), i32([n]), 1, n, scores)
    st = hsi.device_error()
    dt = time.time() - t0
    assert st == -4, hsi.STATUS.get(st, st)  # HSI_ERR_DEVICE_TIMEOUT
    assert dt < 5.0
    assert hsi.device_error() == 0  # the word was cleared
    # normal operation again, correct results on the same context
    hsi.debug_set(hsi.DEBUG_SKIP_FIRST_COPY, 0)
    hsi.debug_set(hsi.DEBUG_WAIT_LIMIT_NS, 1_000_000_000)
    hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, i64([0]), i32([n]), 1, n, scores)
    assert hsi.device_error() == 0
    krec, gk = caches.oracle_rec(0)
    qrec, gq, wo = oracle_query(wl, 0, 0)
    ref, tol = oracle.score_rows(qrec, gq, wo, krec, gk, np.arange(n))
    assert np.all(np.abs(scores.cpu().numpy()[0] - ref) <= tol)


def test_length_past_the_host_bound_is_clamped_and_reported():
    """A device-side length larger than the bound the caller gave on the host
    (which sized the rows) is a malformed argument: the selection kernels clamp
    it to the bound, so no pass reads past a row, and report it through the
    sticky word; the results are those of the clamped length."""
    B, n = 3, 20000
    g = torch.Generator(device="cpu").manual_seed(11)
    s = (torch.randn(B, n, generator=g) * 3).to(DEV)
    k = 512
    bad = i32([n, n + 5, 2 * n])  # rows 1 and 2 claim more than max_valid = n items
    ok = i32([n, n, n])
    gi = torch.empty(B, k, dtype=torch.int32, device=DEV)
    gv = torch.empty(B, k, device=DEV)
    assert hsi.device_error() == 0
    hsi.topk(s, bad, B, n, k, gi, gv)
    assert hsi.device_error() == -6  # HSI_ERR_DEVICE_ARG
    ri = torch.empty_like(gi)
    rv = torch.empty_like(gv)
    hsi.topk(s, ok, B, n, k, ri, rv)
    assert hsi.device_error() == 0
    assert torch.equal(gi, ri) and torch.equal(gv, rv)
