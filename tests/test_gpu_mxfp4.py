"""The MXFP4 indexer format on the GPU (through the C ABI) against the oracle.

MXFP4 is the format the pages give for the indexer q and K: 32-element groups
with a power-of-two (E8M0) scale, 544-byte records, no tensor scale. Bars as
for NVFP4: quantisation bit-exact; scores within
|d| <= 1e-4 * sum_j |w_j| * sum_d |qhat_jd khat_d| / 128 per pair; every
consumer of the records (block maxima, selections, pool gather, pooled scans,
prefill groups) bit-identical to the separate calls on the same scores.
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import inputs
import oracle
from cases import DEV, Caches, gpu_queries, gpu_quantize_mx, i32, i64, oracle_query

import long_context_decode_lightning_gb300 as hsi

pytestmark = pytest.mark.gpu
MX = hsi.FMT_MXFP4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    hsi.build()
    hsi.device_check()
    yield
    assert hsi.device_error() == 0


# ---------------------------------------------------------------- quantise --

@pytest.mark.parametrize("rows,tensors", [(1, 1), (7, 3), (32, 64), (1000, 2), (4099, 1)])
def test_quantize_mx_bit_exact(rows, tensors):
    s = inputs.workload(0).signs()
    x = inputs.normal_bf16(21, 78, tensors * rows * 128).reshape(tensors * rows, 128)
    rec = gpu_quantize_mx(x, tensors, rows, s)
    assert hsi.device_error() == 0
    nrec = hsi.n_records(rows)
    got = rec.cpu().numpy().reshape(tensors, nrec * 544)
    for t in range(tensors):
        ref = oracle.quantize_mx(x[t * rows:(t + 1) * rows], s)
        assert np.array_equal(got[t], ref), f"tensor {t}: {np.flatnonzero(got[t] != ref)[:10]}"


def test_quantize_mx_extremes():
    """Group scales from 2^-127 to 2^100: zero rows, bf16 subnormals, huge rows,
    exact powers of two (the scale rule's boundary m = 1.5) and mixed signs."""
    s = np.where(np.arange(128) % 5 == 0, -1, 1).astype(np.int8)
    rng = np.random.default_rng(9)
    f = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-80, 80, (64, 1)))).astype(np.float32)
    f[3] = 0.0
    f[4] = 1e-40  # bf16 subnormal
    f[5, :] = 0.0
    f[5, 0] = 6.0  # rotated: +-6 everywhere, scale 2^0 exactly at the boundary
    f[6, :] = 0.0
    f[6, 0] = 1.5 * 2.0 ** 90
    f[7] = np.where(np.arange(128) < 64, 1e30, -1e-30)
    x = (f.view(np.uint32) >> 16).astype(np.uint16)
    rec = gpu_quantize_mx(x, 1, 64, s)
    assert hsi.device_error() == 0
    assert np.array_equal(rec.cpu().numpy(), oracle.quantize_mx(x, s))


def test_quantize_mx_non_finite_input_is_reported():
    s = np.ones(128, dtype=np.int8)
    x = np.zeros((8, 128), dtype=np.uint16)
    x[2, 7] = 0x7F80  # +inf in bf16
    gpu_quantize_mx(x, 1, 8, s)
    assert hsi.device_error() == -6  # HSI_ERR_DEVICE_ARG


# ------------------------------------------------------------------- score --

def _mx_scores(wl, lengths, layer=0):
    B, maxv = len(lengths), max(lengths)
    caches = Caches(wl, layer, range(B), lengths, fmt=MX)
    q_rec, _, w = gpu_queries(wl, layer, range(B), fmt=MX)
    scores = torch.full((B, maxv), float("nan"), device=DEV)
    bmax = torch.full((B, hsi.n_records(maxv)), float("nan"), device=DEV)
    # no tensor scales in MXFP4: the g pointers are not read
    hsi.score_full(q_rec, None, w, caches.k_rec, None, i64(caches.rec_off), i32(lengths), B, maxv, scores,
                   block_max=bmax, fmt=MX)
    assert hsi.device_error() == 0
    return caches, q_rec, w, scores, bmax


@pytest.mark.parametrize("lengths", [[1], [129], [5000], [300, 1, 4097, 2048, 131]])
def test_score_full_mx_within_tolerance(lengths):
    wl = inputs.workload(1)
    caches, _, _, scores, bmax = _mx_scores(wl, lengths)
    sg, bm = scores.cpu().numpy(), bmax.cpu().numpy()
    for b, n in enumerate(lengths):
        krec, _ = caches.oracle_rec(b)
        qrec, _, w = oracle_query(wl, 0, b, fmt=MX)
        ref, tol = oracle.score_rows(qrec, 1.0, w, krec, 1.0, np.arange(n), fmt="mxfp4")
        d = np.abs(sg[b, :n].astype(np.float64) - ref)
        assert np.all(d <= tol), f"query {b}: worst {np.max(d / tol):.3g} x tol"
        assert np.all(np.isnan(sg[b, n:])), "wrote past n_visible"
        nb = hsi.n_records(n)
        exp = np.array([sg[b, 8 * j:min(n, 8 * j + 8)].max() for j in range(nb)], dtype=np.float32)
        assert np.array_equal(bm[b, :nb], exp)


def test_score_mx_single_head_is_relu_of_decoded_gemv():
    wl = inputs.workload(0)
    n = 777
    caches = Caches(wl, 0, [0], [n], fmt=MX)
    q_rec, _, _ = gpu_queries(wl, 0, [0], fmt=MX)
    krec, _ = caches.oracle_rec(0)
    qrec_o, _, _ = oracle_query(wl, 0, 0, fmt=MX)
    qd = oracle.decode_rows(qrec_o, 32, fmt="mxfp4")
    kd = oracle.decode_rows(krec, n, fmt="mxfp4")
    for j in (0, 17, 31):
        w = torch.zeros(1, 32, device=DEV)
        w[0, j] = 1.0
        scores = torch.empty(1, n, device=DEV)
        hsi.score_full(q_rec, None, w, caches.k_rec, None, i64([0]), i32([n]), 1, n, scores, fmt=MX)
        ref = np.maximum(kd @ qd[j], 0.0) / 128.0
        tol = 1e-4 * (np.abs(kd) @ np.abs(qd[j])) / 128.0
        assert np.all(np.abs(scores.cpu().numpy()[0] - ref) <= tol)


def test_score_mx_groups_of_very_different_scale():
    """Each row's four groups sit 2^4 apart, so every K step's two scales and
    the two steps' scales differ: a scale read from the wrong byte or group
    is off by at least 16x."""
    rng = np.random.default_rng(41)
    Hm = scipy.linalg.hadamard(128).astype(np.float64)
    s = np.ones(128, dtype=np.int8)
    mag = 2.0 ** (4 * (np.arange(128) // 32) - 6)

    def bf16_rows(n, perm):
        y = rng.standard_normal((n, 128)) * mag[perm]
        x = (y @ Hm / 128).astype(np.float32)
        return (x.view(np.uint32) >> 16).astype(np.uint16)

    n = 1000
    kb = bf16_rows(n, np.arange(128))
    qb = bf16_rows(32, np.arange(128)[::-1])
    krec = gpu_quantize_mx(kb, 1, n, s)
    qrec = gpu_quantize_mx(qb, 1, 32, s)
    w = torch.from_numpy(rng.standard_normal((1, 32)).astype(np.float32)).to(DEV)
    scores = torch.empty(1, n, device=DEV)
    hsi.score_full(qrec, None, w, krec, None, i64([0]), i32([n]), 1, n, scores, fmt=MX)
    assert hsi.device_error() == 0
    ref, tol = oracle.score_rows(oracle.quantize_mx(qb, s), 1.0, w.cpu().numpy()[0], oracle.quantize_mx(kb, s), 1.0,
                                 np.arange(n), fmt="mxfp4")
    assert np.all(np.abs(scores.cpu().numpy()[0] - ref) <= tol)


@pytest.mark.parametrize("n_cache,n_vis", [(3000, [2990, 2991, 2992, 3000, 5, 6, 7, 8])])
def test_score_full_mx_group4_shared_cache(n_cache, n_vis):
    wl = inputs.workload(4)
    B = len(n_vis)
    caches = Caches(wl, 0, [0], [n_cache], fmt=MX)
    q_rec, _, w = gpu_queries(wl, 0, range(B), fmt=MX)
    scores = torch.full((B, n_cache), float("nan"), device=DEV)
    hsi.score_full(q_rec, None, w, caches.k_rec, None, i64([0] * B), i32(n_vis), B, n_cache, scores, group=4,
                   fmt=MX)
    assert hsi.device_error() == 0
    sg = scores.cpu().numpy()
    krec, _ = caches.oracle_rec(0)
    for b, n in enumerate(n_vis):
        qrec, _, wo = oracle_query(wl, 0, b, fmt=MX)
        ref, tol = oracle.score_rows(qrec, 1.0, wo, krec, 1.0, np.arange(n), fmt="mxfp4")
        assert np.all(np.abs(sg[b, :n] - ref) <= tol), b
        assert np.isnan(sg[b, n:]).all()


# ------------------------------------------------------- pool and layers --

@pytest.mark.parametrize("lengths", [[3, 20000, 200003]])
def test_full_and_reindex_layer_mx_match_separate_calls(lengths):
    wl = inputs.workload(1)
    B, maxv = len(lengths), max(lengths)
    caches, q_rec, w, s_sep, bm = _mx_scores(wl, lengths)
    nv, off = i32(lengths), i64(caches.rec_off)
    i_sep = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    v_sep = torch.empty(B, 512, device=DEV)
    hsi.topk(s_sep, nv, B, maxv, 512, i_sep, v_sep)
    ids_sep = torch.empty(B, 2048, dtype=torch.int32, device=DEV)
    nk_sep, np_sep = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    hsi.candidate_pool(nv, B, maxv, ids_sep, nk_sep, np_sep, block_max=bm)

    s_f = torch.full((B, maxv), float("nan"), device=DEV)
    i_f = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    v_f = torch.empty(B, 512, device=DEV)
    ids_f = torch.empty(B, 2048, dtype=torch.int32, device=DEV)
    nk_f, np_f = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    hsi.full_layer(q_rec, None, w, caches.k_rec, None, off, nv, B, maxv, s_f, 512, i_f, v_f, block_ids=ids_f,
                   n_kept=nk_f, n_pool=np_f, fmt=MX)
    assert hsi.device_error() == 0
    for b, n in enumerate(lengths):
        assert torch.equal(s_f[b, :n], s_sep[b, :n])
    assert torch.equal(i_f, i_sep) and torch.equal(v_f, v_sep)
    assert torch.equal(nk_f, nk_sep) and torch.equal(np_f, np_sep)
    sg = s_f.cpu().numpy()
    for b, n in enumerate(lengths):
        ri, _ = oracle.topk(sg[b], n, 512)
        assert np.array_equal(i_f.cpu().numpy()[b], ri)
        oi, onk, _, _ = oracle.pool(sg[b], n, want_mask=False)
        assert int(nk_f[b]) == onk and np.array_equal(ids_f.cpu().numpy()[b][:onk], oi[:onk])

    # Reindex layer: gathered pooled scan vs the oracle's pooled scores
    q1, _, w1 = gpu_queries(wl, 1, range(B), fmt=MX)
    ps_sep = torch.empty(B, 2048 * 8, device=DEV)
    hsi.score_pool(q1, None, w1, caches.k_rec, None, off, nv, ids_f, nk_f, 2048, B, ps_sep, fmt=MX)
    assert hsi.device_error() == 0
    pss = ps_sep.cpu().numpy()
    for b, n in enumerate(lengths):
        krec, _ = caches.oracle_rec(b)
        qrec, _, wo = oracle_query(wl, 1, b, fmt=MX)
        k = int(nk_f[b])
        slots = np.arange(8 * k)
        pos = ids_f.cpu().numpy()[b][slots // 8].astype(np.int64) * 8 + slots % 8
        vis = pos < n
        ref, tol = oracle.score_rows(qrec, 1.0, wo, krec, 1.0, pos[vis], fmt="mxfp4")
        assert np.all(np.abs(pss[b, slots[vis]] - ref) <= tol), b
        assert np.isneginf(pss[b, slots[~vis]]).all()
    ri_sep = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_sep = torch.empty(B, 512, device=DEV)
    hsi.topk(ps_sep, np_f, B, 2048 * 8, 512, ri_sep, rv_sep, block_ids=ids_f)

    ps_r = torch.empty(B, 2048 * 8, device=DEV)
    ri_r = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_r = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, None, w1, caches.k_rec, None, off, nv, ids_f, nk_f, np_f, B, ps_r, 512, ri_r, rv_r,
                      fmt=MX)
    assert hsi.device_error() == 0
    assert torch.equal(ri_r, ri_sep) and torch.equal(rv_r, rv_sep)

    # the compacted pool of 544-byte records, then the streamed and the
    # gathering-and-storing forms of the layer
    pool_rec = torch.full((B, 2048 * 544), 0xA5, dtype=torch.uint8, device=DEV)
    hsi.pool_gather(caches.k_rec, off, nv, ids_f, nk_f, B, pool_rec, fmt=MX)
    assert hsi.device_error() == 0
    kr = caches.k_rec.cpu().numpy().reshape(-1, 544)
    pr = pool_rec.cpu().numpy().reshape(B, 2048, 544)
    for b in range(B):
        k = int(nk_f[b])
        assert np.array_equal(pr[b, :k], kr[caches.rec_off[b] + ids_f[b, :k].cpu().numpy()])
        assert np.all(pr[b, k:] == 0xA5)
    ps_c = torch.full((B, 2048 * 8), float("nan"), device=DEV)
    ri_c = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_c = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, None, w1, caches.k_rec, None, off, nv, ids_f, nk_f, np_f, B, ps_c, 512, ri_c, rv_c,
                      pool_rec=pool_rec, fmt=MX)
    assert hsi.device_error() == 0
    for b in range(B):
        k8 = 8 * int(nk_f[b])
        assert torch.equal(ps_c[b, :k8], ps_sep[b, :k8])
    assert torch.equal(ri_c, ri_sep) and torch.equal(rv_c, rv_sep)
    pool_rec2 = torch.full((B, 2048 * 544), 0x5A, dtype=torch.uint8, device=DEV)
    ps_g = torch.empty(B, 2048 * 8, device=DEV)
    ri_g = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_g = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, None, w1, caches.k_rec, None, off, nv, ids_f, nk_f, np_f, B, ps_g, 512, ri_g, rv_g,
                      pool_rec=pool_rec2, pool_rec_ready=False, fmt=MX)
    assert hsi.device_error() == 0
    pr2 = pool_rec2.cpu().numpy().reshape(B, 2048, 544)
    for b in range(B):
        k = int(nk_f[b])
        assert np.array_equal(pr2[b, :k], pr[b, :k])
        assert np.all(pr2[b, k:] == 0x5A)
    assert torch.equal(ri_g, ri_sep) and torch.equal(rv_g, rv_sep)
