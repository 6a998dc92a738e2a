"""The pages' masked Reindex form on the GPU, kept for comparison: score every
visible position with the Reindex query, set the positions outside the pool's
bit table to -inf, take the top-512. It must give exactly the pooled Reindex
layer's top-512 (the scores of a position are the same fp32 number on both
paths), and exactly the oracle's masked form on the same scores."""
import numpy as np
import pytest
import torch

import inputs
import oracle
from cases import DEV, Caches, gpu_queries, i32, i64

import long_context_decode_lightning_gb300 as hsi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hsi.build()
    hsi.device_check()
    yield
    assert hsi.device_error() == 0


def test_mask_scores_bit_exact():
    rng = np.random.default_rng(21)
    lengths = [1, 31, 33, 1000, 70001]
    B, n = len(lengths), max(lengths)
    sc = rng.standard_normal((B, n + 7)).astype(np.float32)
    words = (n + 31) // 32
    bits = rng.integers(0, 2 ** 32, (B, words + 1), dtype=np.uint64).astype(np.uint32)
    bits[2, :] = 0xFFFFFFFF
    s = torch.from_numpy(sc).to(DEV)
    hsi.mask_scores(s, i32(lengths), torch.from_numpy(bits.view(np.int32)).to(DEV), B, n)
    assert hsi.device_error() == 0
    want = sc.copy()
    for b, nb in enumerate(lengths):
        pos = np.arange(nb)
        keep = (bits[b, pos // 32] >> (pos % 32)) & 1
        want[b, :nb][keep == 0] = -np.inf
    assert np.array_equal(s.cpu().numpy(), want)


@pytest.mark.parametrize("lengths", [[3, 20000, 131073]])
def test_dense_masked_reindex_equals_pooled_layer(lengths):
    wl = inputs.workload(1)
    B, maxv = len(lengths), max(lengths)
    caches = Caches(wl, 0, range(B), lengths)
    q0, g0, w0 = gpu_queries(wl, 0, range(B))
    nv, off = i32(lengths), i64(caches.rec_off)
    s_f = torch.empty(B, maxv, device=DEV)
    i_f = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    v_f = torch.empty(B, 512, device=DEV)
    ids = torch.empty(B, 2048, dtype=torch.int32, device=DEV)
    nk, npool = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    bits = torch.zeros(B, (maxv + 31) // 32, dtype=torch.int32, device=DEV)
    hsi.full_layer(q0, g0, w0, caches.k_rec, caches.g, off, nv, B, maxv, s_f, 512, i_f, v_f, block_ids=ids, n_kept=nk,
                   n_pool=npool, pool_bits=bits)
    q1, g1, w1 = gpu_queries(wl, 1, range(B))
    # pooled: the Reindex layer as deployed
    ps = torch.empty(B, 2048 * 8, device=DEV)
    ri_p = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_p = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids, nk, npool, B, ps, 512, ri_p, rv_p)
    # dense: every position scored, masked, top-512
    s_d = torch.empty(B, maxv, device=DEV)
    hsi.score_full(q1, g1, w1, caches.k_rec, caches.g, off, nv, B, maxv, s_d)
    s_unmasked = s_d.clone()
    hsi.mask_scores(s_d, nv, bits, B, maxv)
    ri_d = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_d = torch.empty(B, 512, device=DEV)
    hsi.topk(s_d, nv, B, maxv, 512, ri_d, rv_d)
    assert hsi.device_error() == 0
    assert torch.equal(ri_d, ri_p) and torch.equal(rv_d, rv_p)
    su, bt = s_unmasked.cpu().numpy(), bits.cpu().numpy().view(np.uint32)
    for b, n in enumerate(lengths):
        pos = np.arange(n)
        mask = ((bt[b, pos // 32] >> (pos % 32)) & 1).astype(np.uint8)
        oi, ov = oracle.topk_masked(su[b], n, mask)
        assert np.array_equal(ri_d.cpu().numpy()[b], oi) and np.array_equal(rv_d.cpu().numpy()[b], ov), b
