"""Parity of the CUDA path (through the C ABI) with the oracle, stage by stage.

Bars: quantisation bit-exact; scores within
|d| <= 1e-4 * sum_j |w_j| * sum_d |qhat_jd khat_d| (scales applied) per pair;
top-k, pool and Reindex top-k bit-exact when fed the same fp32 scores.
"""
import numpy as np
import pytest
import torch

import inputs
import oracle
from cases import DEV, Caches, assert_sets_match_except_near_ties, gpu_queries, gpu_quantize, i32, i64, oracle_query

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


# ---------------------------------------------------------------- quantise --

@pytest.mark.parametrize("rows,tensors", [(1, 1), (7, 3), (32, 5), (1000, 2), (4099, 1)])
def test_quantize_bit_exact(rows, tensors):
    wl = inputs.workload(0)
    s = wl.signs()
    x = inputs.normal_bf16(11, 77, tensors * rows * 128).reshape(tensors * rows, 128)
    rec, g = gpu_quantize(x, tensors, rows, s)
    nrec = hsi.n_records(rows)
    got = rec.cpu().numpy().reshape(tensors, nrec * 576)
    gg = g.cpu().numpy()
    for t in range(tensors):
        ref, gr = oracle.quantize(x[t * rows:(t + 1) * rows], s)
        assert np.float32(gr) == gg[t]
        assert np.array_equal(got[t], ref), f"tensor {t}: {np.flatnonzero(got[t] != ref)[:10]}"


def test_quantize_mode1_and_extremes():
    s = np.where(np.arange(128) % 3 == 0, -1, 1).astype(np.int8)
    rng = np.random.default_rng(3)
    f = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    f[5] = 0.0
    f[6, :] = 1e-30
    x = (f.view(np.uint32) >> 16).astype(np.uint16)
    rec, g = gpu_quantize(x, 1, 64, s)
    ref, gr = oracle.quantize(x, s)
    assert np.array_equal(rec.cpu().numpy(), ref)
    rec1, _ = gpu_quantize(x, 1, 64, s, mode=1, g=[gr * 0.5])
    ref1, _ = oracle.quantize(x, s, g=np.float32(gr * 0.5))
    assert np.array_equal(rec1.cpu().numpy(), ref1)


# ------------------------------------------------------------------- score --

def _score_case(wl, lengths, layer=0):
    B = len(lengths)
    caches = Caches(wl, layer, range(B), lengths)
    q_rec, g_q, w = gpu_queries(wl, layer, range(B))
    maxv = max(lengths)
    scores = torch.full((B, maxv), float("nan"), device=DEV)
    bmax = torch.full((B, hsi.n_records(maxv)), float("nan"), device=DEV)
    hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, i64(caches.rec_off), i32(lengths), B, maxv, scores,
                   block_max=bmax)
    assert hsi.device_error() == 0
    return caches, scores.cpu().numpy(), bmax.cpu().numpy()


@pytest.mark.parametrize("lengths", [[1], [7], [128], [129], [5000], [300, 1, 4097, 2048, 131]])
def test_score_full_within_tolerance(lengths):
    wl = inputs.workload(1)
    caches, sg, bm = _score_case(wl, lengths)
    for b, n in enumerate(lengths):
        krec, gk = caches.oracle_rec(b)
        qrec, gq, w = oracle_query(wl, 0, b)
        ref, tol = oracle.score_rows(qrec, gq, w, krec, gk, np.arange(n))
        d = np.abs(sg[b, :n].astype(np.float64) - ref)
        assert np.all(d <= tol), f"query {b}: worst {np.max(d / tol):.3g} x tol"
        assert np.all(np.isnan(sg[b, n:])), "wrote past n_visible"
        nb = hsi.n_records(n)
        exp = np.array([sg[b, 8 * j:min(n, 8 * j + 8)].max() for j in range(nb)], dtype=np.float32)
        assert np.array_equal(bm[b, :nb], exp)


def test_score_full_pairs_scored_mac_identity():
    # special case: one head weighted 1, others 0 -> ReLU of one decoded dot product
    wl = inputs.workload(0)
    n = 777
    caches = Caches(wl, 0, [0], [n])
    q_rec, g_q, _ = gpu_queries(wl, 0, [0])
    krec, gk = caches.oracle_rec(0)
    qrec_o, gq_o, _ = oracle_query(wl, 0, 0)
    qd = oracle.decode_rows(qrec_o, 32, gq_o)
    kd = oracle.decode_rows(krec, n, gk)
    for j in (0, 17, 31):
        w = torch.zeros(1, 32, device=DEV)
        w[0, j] = 1.0
        scores = torch.empty(1, n, device=DEV)
        hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, i64([0]), i32([n]), 1, n, scores)
        ref = np.maximum(kd @ qd[j], 0.0) / 128.0
        tol = 1e-4 * (np.abs(kd) @ np.abs(qd[j])) / 128.0
        assert np.all(np.abs(scores.cpu().numpy()[0] - ref) <= tol)


# ------------------------------------------------------------------- top-k --

def _gpu_topk(scores_np, n_valid, k, block_ids=None, block_size=8):
    B, ld = scores_np.shape
    s = torch.from_numpy(np.ascontiguousarray(scores_np)).to(DEV)
    idx = torch.empty(B, k, dtype=torch.int32, device=DEV)
    val = torch.empty(B, k, dtype=torch.float32, device=DEV)
    bid = None if block_ids is None else torch.from_numpy(block_ids).to(DEV)
    hsi.topk(s, i32(n_valid), B, max(n_valid), k, idx, val, block_ids=bid, block_size=block_size)
    assert hsi.device_error() == 0
    return idx.cpu().numpy(), val.cpu().numpy()


@pytest.mark.parametrize("n,k", [(1, 512), (100, 512), (511, 512), (512, 512), (513, 512), (16384, 512),
                                 (16385, 512), (100000, 512), (300000, 2048), (5000, 1)])
def test_topk_bit_exact(n, k):
    rng = np.random.default_rng(n + k)
    sc = rng.standard_normal((3, n)).astype(np.float32) * 4
    sc[1, ::7] = sc[1, min(3, n - 1)]  # many exact ties
    sc[2, : n // 2] = -0.0
    sc[2, n // 2:] = 0.0
    gi, gv = _gpu_topk(sc, [n, n, n], k)
    for b in range(3):
        ri, rv = oracle.topk(sc[b], n, k)
        assert np.array_equal(gi[b], ri), f"row {b}"
        assert np.array_equal(gv[b][ri >= 0], rv[ri >= 0])


def test_topk_outliers_and_infinities():
    """Rows whose k-th key lies far below the largest ones (the selection's
    first window, which ends at the largest finite key, misses it), rows whose
    k best are all tied at the top, and rows holding +inf / -inf."""
    rng = np.random.default_rng(11)
    n = 40000
    sc = rng.standard_normal((5, n)).astype(np.float32)
    sc[0, rng.choice(n, 7, replace=False)] = np.float32(1e30)  # outliers, k-th key below the window
    sc[1, rng.choice(n, 300, replace=False)] = np.float32(3e5)
    sc[2, :600] = sc[2].max()  # the k best tied at the top
    sc[3, rng.choice(n, 20, replace=False)] = np.inf
    sc[3, rng.choice(n, 20, replace=False)] = -np.inf
    sc[4, rng.choice(n, 600, replace=False)] = np.inf  # more +inf than k
    for rows in (sc, sc[:, :9000]):  # long rows (histogram path) and rows that fit shared memory
        m = rows.shape[1]
        gi, gv = _gpu_topk(np.ascontiguousarray(rows), [m] * 5, 512)
        for b in range(5):
            ri, rv = oracle.topk(rows[b], m, 512)
            assert np.array_equal(gi[b], ri), f"row {b}, n {m}"
            assert np.array_equal(gv[b], rv)


def test_topk_ragged_rows_and_all_equal():
    # all-equal rows exercise every survivor path: shared memory, survivors in
    # L2 (40000 > 16384), survivor overflow with a re-read of the row (100000)
    n = [1, 20000, 40000, 3, 100000]
    ld = max(n)
    sc = np.full((len(n), ld), 2.5, dtype=np.float32)
    gi, _ = _gpu_topk(sc, n, 512)
    for b in range(len(n)):
        ri, _ = oracle.topk(sc[b], n[b], 512)
        assert np.array_equal(gi[b], ri)


def test_topk_with_block_map():
    rng = np.random.default_rng(5)
    ids = np.sort(rng.choice(100000, 2048, replace=False)).astype(np.int32)[None, :]
    ps = rng.standard_normal((1, 2048 * 8)).astype(np.float32)
    npool = 2048 * 8 - 5
    gi, gv = _gpu_topk(ps, [npool], 512, block_ids=ids)
    ri, rv = oracle.topk_pool(ps[0], npool, ids[0])
    assert np.array_equal(gi[0], ri) and np.array_equal(gv[0], rv)


# -------------------------------------------------------------------- pool --

def _gpu_pool(scores_np, n_vis, bs=8, keep=2048, use_bmax=False):
    B, ld = scores_np.shape
    s = torch.from_numpy(np.ascontiguousarray(scores_np)).to(DEV)
    ids = torch.empty(B, keep, dtype=torch.int32, device=DEV)
    nk = torch.empty(B, dtype=torch.int32, device=DEV)
    npool = torch.empty(B, dtype=torch.int32, device=DEV)
    bits = torch.empty(B, (ld + 31) // 32, dtype=torch.int32, device=DEV)
    if use_bmax:
        nb = (ld + bs - 1) // bs
        bm = np.full((B, nb), -np.inf, dtype=np.float32)
        for b in range(B):
            for j in range((n_vis[b] + bs - 1) // bs):
                bm[b, j] = scores_np[b, j * bs:min(n_vis[b], j * bs + bs)].max()
        hsi.candidate_pool(i32(n_vis), B, max(n_vis), ids, nk, npool, block_max=torch.from_numpy(bm).to(DEV),
                           block_size=bs, n_keep=keep, pool_bits=bits)
    else:
        hsi.candidate_pool(i32(n_vis), B, max(n_vis), ids, nk, npool, scores=s, block_size=bs, n_keep=keep,
                           pool_bits=bits)
    assert hsi.device_error() == 0
    return ids.cpu().numpy(), nk.cpu().numpy(), npool.cpu().numpy(), bits.cpu().numpy().view(np.uint32)


def _bits_to_mask(bits_row, n):
    return ((bits_row[np.arange(n) // 32] >> (np.arange(n) % 32)) & 1).astype(np.uint8)


@pytest.mark.parametrize("n_vis", [[1], [9], [16384], [16385], [20001, 131072, 50], [1048576]])
@pytest.mark.parametrize("use_bmax", [False, True])
def test_pool_bit_exact(n_vis, use_bmax):
    rng = np.random.default_rng(sum(n_vis))
    ld = max(n_vis)
    sc = rng.standard_normal((len(n_vis), ld)).astype(np.float32)
    if len(n_vis) > 1:
        sc[1, ::3] = 1.0  # ties between block maxima
    gi, gk, gp, gb = _gpu_pool(sc, n_vis, use_bmax=use_bmax)
    for b, n in enumerate(n_vis):
        ri, rk, rp, rm = oracle.pool(sc[b], n)
        assert gk[b] == rk and gp[b] == rp
        assert np.array_equal(gi[b][:rk], ri[:rk]) and (gi[b][rk:] == -1).all()
        assert np.array_equal(_bits_to_mask(gb[b], n), rm)


def test_pool_past_the_bitmap_range():
    """More blocks than the in-order bitmap of the final selection covers
    (262144): the kept ids are put in order by a sort instead."""
    n = 2_100_000
    rng = np.random.default_rng(21)
    sc = rng.standard_normal((1, n)).astype(np.float32)
    gi, gk, gp, gb = _gpu_pool(sc, [n])
    ri, rk, rp, rm = oracle.pool(sc[0], n)
    assert gk[0] == rk and gp[0] == rp
    assert np.array_equal(gi[0][:rk], ri[:rk])
    assert np.array_equal(_bits_to_mask(gb[0], n), rm)


@pytest.mark.parametrize("case", ["few_values", "neg_inf_blocks", "pos_inf", "one_value", "keep_1"])
def test_pool_crafted_rows_past_the_shared_memory_size(case):
    """Rows of more than 16384 blocks take the candidate list and the pool's
    final kernel (second-level bins, the tied bin ranked) or, for heavy ties and
    more +inf keys than places, the general block select: crafted rows for
    every route, against the oracle."""
    rng = np.random.default_rng(len(case))
    n_vis = [300001, 140003, 131072]
    ld = max(n_vis)
    sc = rng.standard_normal((len(n_vis), ld)).astype(np.float32)
    keep = 2048
    if case == "few_values":
        sc = np.round(sc * 4) / 4
    elif case == "neg_inf_blocks":
        sc[:, 8 * 1000:8 * 60000] = -np.inf  # whole blocks dropped
    elif case == "pos_inf":
        sc[0, rng.integers(0, n_vis[0], 3000)] = np.inf  # more +inf blocks than places
        sc[1, rng.integers(0, n_vis[1], 100)] = np.inf
    elif case == "one_value":
        sc[:] = 0.5
    else:
        keep = 1
    gi, gk, gp, gb = _gpu_pool(sc, n_vis, keep=keep)
    for b, n in enumerate(n_vis):
        ri, rk, rp, rm = oracle.pool(sc[b], n, 8, keep)
        assert gk[b] == rk and gp[b] == rp, (case, b)
        assert np.array_equal(gi[b][:rk], ri[:rk]) and (gi[b][rk:] == -1).all(), (case, b)
        assert np.array_equal(_bits_to_mask(gb[b], n), rm), (case, b)


@pytest.mark.parametrize("bs,keep", [(4, 6), (1, 5), (3, 100), (8, 1)])
def test_pool_small_block_and_keep(bs, keep):
    rng = np.random.default_rng(bs * 100 + keep)
    n_vis = [61, 1, 200, 997]
    sc = rng.choice([-1.0, 0.0, 0.5, 2.0], (4, 997)).astype(np.float32)
    gi, gk, gp, gb = _gpu_pool(sc, n_vis, bs=bs, keep=keep)
    for b, n in enumerate(n_vis):
        ri, rk, rp, rm = oracle.pool(sc[b], n, bs, keep)
        assert gk[b] == rk and gp[b] == rp
        assert np.array_equal(gi[b][:rk], ri[:rk])
        assert np.array_equal(_bits_to_mask(gb[b], n), rm)


# ------------------------------------------------------------ pooled score --

@pytest.mark.parametrize("lengths", [[20000], [3, 16384, 16391, 70001]])
def test_score_pool_within_tolerance_and_reindex_topk(lengths):
    wl = inputs.workload(1)
    B = len(lengths)
    caches, sg, _ = _score_case(wl, lengths, layer=0)
    gi, gk, gp, _ = _gpu_pool(sg, lengths)
    q_rec, g_q, w = gpu_queries(wl, 1, range(B))
    ps = torch.full((B, 2048 * 8), float("nan"), device=DEV)
    hsi.score_pool(q_rec, g_q, w, caches.k_rec, caches.g, i64(caches.rec_off), i32(lengths),
                   torch.from_numpy(gi).to(DEV), i32(gk.tolist()), 2048, B, ps)
    assert hsi.device_error() == 0
    psg = ps.cpu().numpy()
    for b, n in enumerate(lengths):
        krec, gkk = caches.oracle_rec(b)
        qrec, gq, wq = oracle_query(wl, 1, b)
        ref, _ = oracle.score_pool(qrec, gq, wq, krec, gkk, n, gi[b], gk[b])
        m = int(gp[b])
        pos = np.array([gi[b][i // 8] * 8 + i % 8 for i in range(m)])
        _, tol = oracle.score_rows(qrec, gq, wq, krec, gkk, pos)
        assert np.all(np.abs(psg[b, :m] - ref[:m]) <= tol)
        assert np.isneginf(psg[b, m:8 * gk[b]]).all()
        assert np.isnan(psg[b, 8 * gk[b]:]).all()
    # Reindex top-512 on the GPU's pooled scores, bit-exact, global positions
    ri_g, _ = _gpu_topk(psg, gp.tolist(), 512, block_ids=gi)
    for b in range(B):
        ri, _ = oracle.topk_pool(psg[b], int(gp[b]), gi[b])
        assert np.array_equal(ri_g[b], ri)


# ---------------------------------------------------------------- end to end --

def test_end_to_end_topk_and_pool_match_except_near_ties():
    """Oracle's own path vs the GPU path: top-512 sets agree except positions
    whose oracle score is within tolerance of the k-th score, and pools agree
    except blocks whose oracle block maximum is within tolerance of the
    2048th block value (a block maximum's tolerance is the largest of its
    positions')."""
    wl = inputs.workload(0)
    n = 32768
    caches, sg, _ = _score_case(wl, [n])
    gidx, _ = _gpu_topk(sg, [n], 512)
    krec, gk = caches.oracle_rec(0)
    qrec, gq, w = oracle_query(wl, 0, 0)
    so, _ = oracle.score_full(qrec, gq, w, krec, gk, n)
    _, tol = oracle.score_rows(qrec, gq, w, krec, gk, np.arange(n))
    oidx, oval = oracle.topk(so, n, 512)
    assert_sets_match_except_near_ties(gidx[0], oidx, lambda p: so[p], lambda p: tol[p], oval[-1])
    # pools: the GPU's pool of its own scores vs the oracle's pool of its scores
    nv = i32([n])
    gids = torch.empty(1, 2048, dtype=torch.int32, device=DEV)
    gnk, gnp = torch.empty(1, dtype=torch.int32, device=DEV), torch.empty(1, dtype=torch.int32, device=DEV)
    hsi.candidate_pool(nv, 1, n, gids, gnk, gnp, scores=torch.from_numpy(sg).to(DEV))
    oids, onk, _, _ = oracle.pool(so, n)
    nblk = (n + 7) // 8
    bmax_o = so[: nblk * 8].reshape(nblk, 8).max(1)
    btol = tol[: nblk * 8].reshape(nblk, 8).max(1)
    ranked = np.lexsort((np.arange(nblk), -bmax_o))
    ranked = ranked[ranked != nblk - 1]  # the pinned newest block ranks first on both sides
    kth_block = bmax_o[ranked[2048 - 2]]
    assert int(gnk[0]) == onk == 2048
    assert nblk - 1 in set(gids[0].tolist()) and nblk - 1 in set(oids[:onk].tolist())
    assert_sets_match_except_near_ties(gids[0].cpu().numpy(), oids[:onk], lambda j: bmax_o[j], lambda j: btol[j],
                                       kth_block)


# ------------------------------------------------------- composite layers --

@pytest.mark.parametrize("lengths", [[3, 20000, 200003], [16384, 131073]])
def test_full_and_reindex_layer_match_separate_calls(lengths):
    """hsi_full_layer (histograms fused into the scoring kernel) and
    hsi_reindex_layer give exactly what the separate calls give."""
    wl = inputs.workload(1)
    B, maxv = len(lengths), max(lengths)
    caches = Caches(wl, 0, range(B), lengths)
    q_rec, g_q, w = gpu_queries(wl, 0, range(B))
    nv, off = i32(lengths), i64(caches.rec_off)
    s_sep = torch.empty(B, maxv, device=DEV)
    bm = torch.empty(B, hsi.n_records(maxv), device=DEV)
    hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_sep, block_max=bm)
    i_sep = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    v_sep = torch.empty(B, 512, device=DEV)
    hsi.topk(s_sep, nv, B, maxv, 512, i_sep, v_sep)
    ids_sep = torch.empty(B, 2048, dtype=torch.int32, device=DEV)
    nk_sep, np_sep = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    bits_sep = torch.zeros(B, (maxv + 31) // 32, dtype=torch.int32, device=DEV)
    hsi.candidate_pool(nv, B, maxv, ids_sep, nk_sep, np_sep, scores=s_sep, pool_bits=bits_sep)

    s_f = torch.empty(B, maxv, device=DEV)
    i_f = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    v_f = torch.empty(B, 512, device=DEV)
    ids_f = torch.empty(B, 2048, dtype=torch.int32, device=DEV)
    nk_f, np_f = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    bits_f = torch.zeros(B, (maxv + 31) // 32, dtype=torch.int32, device=DEV)
    hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_f, 512, i_f, v_f, block_ids=ids_f,
                   n_kept=nk_f, n_pool=np_f, pool_bits=bits_f)
    assert hsi.device_error() == 0
    for b, n in enumerate(lengths):
        assert torch.equal(s_f[b, :n], s_sep[b, :n])
    assert torch.equal(i_f, i_sep) and torch.equal(v_f, v_sep)
    assert torch.equal(nk_f, nk_sep) and torch.equal(np_f, np_sep)
    for b in range(B):
        k = int(nk_sep[b])
        assert torch.equal(ids_f[b, :k], ids_sep[b, :k])
        words = (lengths[b] + 31) // 32
        assert torch.equal(bits_f[b, :words], bits_sep[b, :words])
    # oracle on the GPU scores: the fused path is still the exact selection
    sg = s_f.cpu().numpy()
    for b, n in enumerate(lengths):
        ri, _ = oracle.topk(sg[b], n, 512)
        assert np.array_equal(i_f.cpu().numpy()[b], ri)
        oi, onk, onp, _ = oracle.pool(sg[b], n)
        assert int(nk_f[b]) == onk and np.array_equal(ids_f.cpu().numpy()[b][:onk], oi[:onk])

    # the selection phase run again (twice) over the same scores and workspace
    # starts from the same state and gives the same top-k and pool
    ws = hsi.workspace(hsi.WS_FULL_LAYER, B, maxv, 512, device=DEV)
    i_r, v_r, ids_r = torch.empty_like(i_f), torch.empty_like(v_f), torch.empty_like(ids_f)
    nk_r, np_r, bits_r = torch.empty_like(nk_f), torch.empty_like(np_f), torch.zeros_like(bits_f)
    s_r = torch.empty_like(s_f)
    for phases in (1, 2, 2):
        hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_r, 512, i_r, v_r, block_ids=ids_r,
                       n_kept=nk_r, n_pool=np_r, pool_bits=bits_r, ws=ws, phases=phases)
    assert hsi.device_error() == 0
    assert torch.equal(i_r, i_f) and torch.equal(v_r, v_f)
    assert torch.equal(nk_r, nk_f) and torch.equal(np_r, np_f) and torch.equal(bits_r, bits_f)
    for b in range(B):
        assert torch.equal(ids_r[b, :int(nk_f[b])], ids_f[b, :int(nk_f[b])])
    # the two selections as separate phases, the pool first: separate parts of
    # the workspace, so their order (or running them on two streams) is free
    i_r.fill_(7), v_r.fill_(7), ids_r.fill_(7), nk_r.fill_(7), np_r.fill_(7), bits_r.zero_()
    for phases in (hsi.PHASE_SCORE, hsi.PHASE_POOL, hsi.PHASE_TOPK):
        hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_r, 512, i_r, v_r, block_ids=ids_r,
                       n_kept=nk_r, n_pool=np_r, pool_bits=bits_r, ws=ws, phases=phases)
    assert hsi.device_error() == 0
    assert torch.equal(i_r, i_f) and torch.equal(v_r, v_f)
    assert torch.equal(nk_r, nk_f) and torch.equal(np_r, np_f) and torch.equal(bits_r, bits_f)
    for b in range(B):
        assert torch.equal(ids_r[b, :int(nk_f[b])], ids_f[b, :int(nk_f[b])])

    q1, g1, w1 = gpu_queries(wl, 1, range(B))
    ps_sep = torch.empty(B, 2048 * 8, device=DEV)
    hsi.score_pool(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids_f, nk_f, 2048, B, ps_sep)
    ri_sep = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_sep = torch.empty(B, 512, device=DEV)
    hsi.topk(ps_sep, np_f, B, 2048 * 8, 512, ri_sep, rv_sep, block_ids=ids_f)
    ps_r = torch.empty(B, 2048 * 8, device=DEV)
    ri_r = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_r = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids_f, nk_f, np_f, B, ps_r, 512, ri_r, rv_r)
    assert hsi.device_error() == 0
    assert torch.equal(ri_r, ri_sep) and torch.equal(rv_r, rv_sep)

    # the compacted pool: records bit-exact copies, and the streamed Reindex
    # layer gives the gathered one's scores and selection
    pool_rec = torch.full((B, 2048 * 576), 0xA5, dtype=torch.uint8, device=DEV)
    hsi.pool_gather(caches.k_rec, off, nv, ids_f, nk_f, B, pool_rec)
    assert hsi.device_error() == 0
    kr = caches.k_rec.cpu().numpy().reshape(-1, 576)
    pr = pool_rec.cpu().numpy().reshape(B, 2048, 576)
    for b in range(B):
        k = int(nk_f[b])
        want = kr[caches.rec_off[b] + ids_f[b, :k].cpu().numpy()]
        assert np.array_equal(pr[b, :k], want)
        assert np.all(pr[b, k:] == 0xA5)  # slots past n_kept untouched
    ps_c = torch.full((B, 2048 * 8), float("nan"), device=DEV)
    ri_c = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_c = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids_f, nk_f, np_f, B, ps_c, 512, ri_c, rv_c,
                      pool_rec=pool_rec)
    assert hsi.device_error() == 0
    for b in range(B):
        k8 = 8 * int(nk_f[b])
        assert torch.equal(ps_c[b, :k8], ps_sep[b, :k8])
        assert torch.isnan(ps_c[b, k8:]).all()  # slots past the pool untouched
    assert torch.equal(ri_c, ri_sep) and torch.equal(rv_c, rv_sep)

    # a gathering layer that leaves the compacted pool behind: the same records
    # as the compaction call, and the same scores and selection
    pool_rec2 = torch.full((B, 2048 * 576), 0x5A, dtype=torch.uint8, device=DEV)
    ps_g = torch.full((B, 2048 * 8), float("nan"), device=DEV)
    ri_g = torch.empty(B, 512, dtype=torch.int32, device=DEV)
    rv_g = torch.empty(B, 512, device=DEV)
    hsi.reindex_layer(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids_f, nk_f, np_f, B, ps_g, 512, ri_g, rv_g,
                      pool_rec=pool_rec2, pool_rec_ready=False)
    assert hsi.device_error() == 0
    pr2 = pool_rec2.cpu().numpy().reshape(B, 2048, 576)
    for b in range(B):
        k = int(nk_f[b])
        assert np.array_equal(pr2[b, :k], pr[b, :k])
        assert np.all(pr2[b, k:] == 0x5A)
        assert torch.equal(ps_g[b, :8 * k], ps_sep[b, :8 * k])
    assert torch.equal(ri_g, ri_sep) and torch.equal(rv_g, rv_sep)


@pytest.mark.parametrize("k,n_keep", [(512, 544), (64, 96), (1, 32)])
def test_full_layer_without_scores_small_pools(k, n_keep):
    """The top-k from the pool when the pool is barely larger than k blocks
    (n_keep - 1 >= k): still the top-k of the whole row."""
    wl = inputs.workload(1)
    lengths = [20000, 140000, 4000]
    B, maxv = len(lengths), max(lengths)
    caches = Caches(wl, 0, range(B), lengths)
    q_rec, g_q, w = gpu_queries(wl, 0, range(B))
    nv, off = i32(lengths), i64(caches.rec_off)
    s_ref = torch.empty(B, maxv, device=DEV)
    ri, rv = torch.empty(B, k, dtype=torch.int32, device=DEV), torch.empty(B, k, device=DEV)
    ids = torch.empty(B, n_keep, dtype=torch.int32, device=DEV)
    nk, npl = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_ref, k, ri, rv, block_ids=ids,
                   n_kept=nk, n_pool=npl, n_keep=n_keep)
    gi, gv = torch.full((B, k), 7, dtype=torch.int32, device=DEV), torch.full((B, k), 7.0, device=DEV)
    ids2 = torch.empty_like(ids)
    nk2, np2 = torch.empty_like(nk), torch.empty_like(npl)
    hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, None, k, gi, gv, block_ids=ids2,
                   n_kept=nk2, n_pool=np2, n_keep=n_keep)
    assert hsi.device_error() == 0
    assert torch.equal(gi, ri) and torch.equal(gv, rv)
    assert torch.equal(nk2, nk) and torch.equal(np2, npl)
    sg = s_ref.cpu().numpy()
    for b, n in enumerate(lengths):
        oi, _ = oracle.topk(sg[b], n, k)
        assert np.array_equal(gi.cpu().numpy()[b], oi), b


@pytest.mark.parametrize("lengths", [[3, 20000, 200003], [16384, 131073, 9000]])
def test_full_layer_without_scores(lengths):
    """With scores = NULL the Full layer writes no score row and takes its
    top-k from the pool's re-scored blocks: the same top-k, pool and table as
    with the score row, in one call and as separate phases."""
    wl = inputs.workload(1)
    B, maxv = len(lengths), max(lengths)
    caches = Caches(wl, 0, range(B), lengths)
    q_rec, g_q, w = gpu_queries(wl, 0, range(B))
    nv, off = i32(lengths), i64(caches.rec_off)

    def outs():
        return (torch.full((B, 512), 7, dtype=torch.int32, device=DEV), torch.full((B, 512), 7.0, device=DEV),
                torch.full((B, 2048), 7, dtype=torch.int32, device=DEV), torch.full((B,), 7, dtype=torch.int32,
                device=DEV), torch.full((B,), 7, dtype=torch.int32, device=DEV),
                torch.zeros(B, (maxv + 31) // 32, dtype=torch.int32, device=DEV))

    s_ref = torch.empty(B, maxv, device=DEV)
    ref = outs()
    hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_ref, 512, ref[0], ref[1],
                   block_ids=ref[2], n_kept=ref[3], n_pool=ref[4], pool_bits=ref[5])
    ws = hsi.workspace(hsi.WS_FULL_LAYER, B, maxv, 512, device=DEV)
    for split in (False, True):
        got = outs()
        kw = dict(block_ids=got[2], n_kept=got[3], n_pool=got[4], pool_bits=got[5], ws=ws)
        if split:
            for ph in (hsi.PHASE_SCORE, hsi.PHASE_POOL, hsi.PHASE_TOPK):
                hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, None, 512, got[0], got[1],
                               phases=ph, **kw)
        else:
            hsi.full_layer(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, None, 512, got[0], got[1], **kw)
        assert hsi.device_error() == 0
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), split
        assert torch.equal(got[3], ref[3]) and torch.equal(got[4], ref[4]), split
        for b, n in enumerate(lengths):
            kb = int(ref[3][b])
            assert torch.equal(got[2][b, :kb], ref[2][b, :kb]), (split, b)
            assert torch.equal(got[5][b, :(n + 31) // 32], ref[5][b, :(n + 31) // 32]), (split, b)
    # the oracle's top-k on the score row
    sg = s_ref.cpu().numpy()
    for b, n in enumerate(lengths):
        oi, _ = oracle.topk(sg[b], n, 512)
        assert np.array_equal(ref[0].cpu().numpy()[b], oi)
    # block maxima without a score row
    bm_ref = torch.empty(B, hsi.n_records(maxv), device=DEV)
    hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, s_ref, block_max=bm_ref)
    bm = torch.full_like(bm_ref, float("nan"))
    hsi.score_full(q_rec, g_q, w, caches.k_rec, caches.g, off, nv, B, maxv, None, block_max=bm)
    assert hsi.device_error() == 0
    for b, n in enumerate(lengths):
        nb = (n + 7) // 8
        assert torch.equal(bm[b, :nb], bm_ref[b, :nb])


def test_step_in_model_order():
    """The decode step's composition: the Full layer's top-512 taken from the
    pool by the gathering Reindex call (which leaves the pool compacted) is the
    Full layer's own pooled top-512, and a Reindex layer that streams that
    compacted pool gives what it gives when it gathers the records."""
    wl = inputs.workload(1)
    lengths = [3, 20000, 200003]
    B, maxv, n_keep, k = len(lengths), max(lengths), 2048, 512
    caches = Caches(wl, 0, range(B), lengths)
    nv, off = i32(lengths), i64(caches.rec_off)
    q0, g0, w0 = gpu_queries(wl, 0, range(B))  # the Full layer's query
    q1, g1, w1 = gpu_queries(wl, 1, range(B))  # a Reindex layer's query
    ids = torch.empty(B, n_keep, dtype=torch.int32, device=DEV)
    nk, npl = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)

    def outs():
        return torch.full((B, k), 7, dtype=torch.int32, device=DEV), torch.full((B, k), 7.0, device=DEV)

    ri, rv = outs()
    hsi.full_layer(q0, g0, w0, caches.k_rec, caches.g, off, nv, B, maxv, None, k, ri, rv, block_ids=ids,
                   n_kept=nk, n_pool=npl, n_keep=n_keep)
    pool_rec = torch.zeros(B, n_keep * 576, dtype=torch.uint8, device=DEV)
    ps = torch.empty(B, n_keep * 8, device=DEV)
    ws = hsi.workspace(hsi.WS_REINDEX_LAYER, B, n_keep * 8, k, device=DEV)
    fi, fv = outs()
    hsi.reindex_layer(q0, g0, w0, caches.k_rec, caches.g, off, nv, ids, nk, npl, B, ps, k, fi, fv, n_keep=n_keep,
                      ws=ws, pool_rec=pool_rec, pool_rec_ready=False)
    assert hsi.device_error() == 0
    assert torch.equal(fi, ri) and torch.equal(fv, rv)
    si, sv = outs()
    hsi.reindex_layer(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids, nk, npl, B, ps, k, si, sv, n_keep=n_keep,
                      ws=ws, pool_rec=pool_rec, pool_rec_ready=True)
    gi, gv = outs()
    hsi.reindex_layer(q1, g1, w1, caches.k_rec, caches.g, off, nv, ids, nk, npl, B, ps, k, gi, gv, n_keep=n_keep,
                      ws=ws)
    assert hsi.device_error() == 0
    assert torch.equal(si, gi) and torch.equal(sv, gv)


def _caches_from_rows(wl, rows_per_cache):
    """K caches built from given bf16 rows (one array [n][128] per cache)."""
    parts, gs, offs, off = [], [], [], 0
    for kb in rows_per_cache:
        rec, g = gpu_quantize(kb, 1, kb.shape[0], wl.signs())
        parts.append(rec)
        gs.append(g)
        offs.append(off)
        off += hsi.n_records(kb.shape[0])
    return torch.cat(parts), torch.cat(gs), offs


@pytest.mark.parametrize("case", ["repeated_keys", "one_key", "three_keys", "unaligned_rows"])
def test_reindex_layer_selection_paths(case):
    """The Reindex layer's selection takes the k-th key's bin from the
    histogram its scoring kernel fills, then orders few kept items by their
    bins' ranks, many (heavy ties) by radix passes, and reads rows that are
    not 16-byte aligned with plain loads. Every route gives what the general
    top-k (hsi_topk) gives on the same pooled scores, and the oracle's top-k."""
    wl = inputs.workload(1)
    lengths = [140000, 20000, 16390]  # the first row's 17,500 blocks take the Full layer's bounded pool route
    B = len(lengths)
    rng = np.random.default_rng(11)
    base = [wl.k_bf16(0, b, rows=n) for b, n in enumerate(lengths)]
    if case == "repeated_keys":  # exact score ties spread over the whole range
        rows = [kb[rng.integers(0, 3000, kb.shape[0])] for kb in base]
    elif case == "one_key":  # every score of a query equal
        rows = [np.repeat(kb[:1], kb.shape[0], axis=0) for kb in base]
    elif case == "three_keys":
        rows = [kb[rng.integers(0, 3, kb.shape[0])] for kb in base]
    else:
        rows = base
    k_rec, gk, offs = _caches_from_rows(wl, rows)
    q_rec, g_q, w = gpu_queries(wl, 0, range(B))
    nv, off = i32(lengths), i64(offs)
    maxv = max(lengths)
    s_f = torch.empty(B, maxv, device=DEV)
    i_f, v_f = torch.empty(B, 512, dtype=torch.int32, device=DEV), torch.empty(B, 512, device=DEV)
    ids = torch.empty(B, 2048, dtype=torch.int32, device=DEV)
    nk, npl = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    bits = torch.full((B, (maxv + 31) // 32), 7, dtype=torch.int32, device=DEV)
    hsi.full_layer(q_rec, g_q, w, k_rec, gk, off, nv, B, maxv, s_f, 512, i_f, v_f, block_ids=ids, n_kept=nk,
                   n_pool=npl, pool_bits=bits)
    assert hsi.device_error() == 0
    # the Full layer's pool equals the stand-alone pool selection on its scores
    ids_sep = torch.full((B, 2048), 7, dtype=torch.int32, device=DEV)
    nk_sep, np_sep = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    bits_sep = torch.zeros(B, (maxv + 31) // 32, dtype=torch.int32, device=DEV)
    hsi.candidate_pool(nv, B, maxv, ids_sep, nk_sep, np_sep, scores=s_f, pool_bits=bits_sep)
    assert torch.equal(nk, nk_sep) and torch.equal(npl, np_sep), case
    for b, n in enumerate(lengths):
        kb = int(nk_sep[b])
        assert torch.equal(ids[b, :kb], ids_sep[b, :kb]) and bool((ids[b, kb:] == -1).all()), (case, b)
        words = (n + 31) // 32
        assert torch.equal(bits[b, :words], bits_sep[b, :words]), (case, b)
    oi, onk, onp, _ = oracle.pool(s_f[0].cpu().numpy(), lengths[0])
    assert int(nk[0]) == onk and int(npl[0]) == onp and np.array_equal(ids[0].cpu().numpy()[:onk], oi[:onk])
    q1, g1, w1 = gpu_queries(wl, 1, range(B))
    ld = 2048 * 8 + (1 if case == "unaligned_rows" else 0)
    ps_sep = torch.empty(B, ld, device=DEV)[:, :2048 * 8]
    hsi.score_pool(q1, g1, w1, k_rec, gk, off, nv, ids, nk, 2048, B, ps_sep, ld=ld)
    ri_sep, rv_sep = torch.empty(B, 512, dtype=torch.int32, device=DEV), torch.empty(B, 512, device=DEV)
    hsi.topk(ps_sep, npl, B, 2048 * 8, 512, ri_sep, rv_sep, block_ids=ids, ld=ld)
    pool_rec = torch.empty(B, 2048 * 576, dtype=torch.uint8, device=DEV)
    for ready in (False, True):  # gathering (leaves the compacted pool), then streaming it
        ps = torch.empty(B, ld, device=DEV)[:, :2048 * 8]
        ri, rv = torch.full((B, 512), 7, dtype=torch.int32, device=DEV), torch.full((B, 512), 7.0, device=DEV)
        hsi.reindex_layer(q1, g1, w1, k_rec, gk, off, nv, ids, nk, npl, B, ps, 512, ri, rv, ld=ld,
                          pool_rec=pool_rec, pool_rec_ready=ready)
        assert hsi.device_error() == 0
        assert torch.equal(ri, ri_sep) and torch.equal(rv, rv_sep), (case, ready)
    sg, idn, nkh, nph = ps_sep.cpu().numpy(), ids.cpu().numpy(), nk.cpu().numpy(), npl.cpu().numpy()
    for b in range(B):
        oi, ov = oracle.topk_pool(sg[b], int(nph[b]), idn[b], 512)
        assert np.array_equal(ri_sep.cpu().numpy()[b], oi), (case, b)


# ------------------------------------------------------- grouped (prefill) --

@pytest.mark.parametrize("n_cache,n_vis", [(3000, [2990, 2991, 2992, 3000, 5, 6, 7, 8]),
                                           (20000, [19000 + 37 * i for i in range(12)])])
def test_score_full_group4_shared_cache(n_cache, n_vis):
    """Chunked prefill: groups of 4 consecutive queries share one cache and are
    scored in one N = 128 tensor-core tile; each query keeps its own causal limit."""
    wl = inputs.workload(4)
    B = len(n_vis)
    caches = Caches(wl, 0, [0], [n_cache])
    q_rec, g_q, w = gpu_queries(wl, 0, range(B))
    gk = caches.g.repeat(B)
    off = i64([0] * B)
    scores = torch.full((B, n_cache), float("nan"), device=DEV)
    hsi.score_full(q_rec, g_q, w, caches.k_rec, gk, off, i32(n_vis), B, n_cache, scores, group=4)
    assert hsi.device_error() == 0
    sg = scores.cpu().numpy()
    krec, gko = caches.oracle_rec(0)
    for b, n in enumerate(n_vis):
        qrec, gq, wo = oracle_query(wl, 0, b)
        ref, tol = oracle.score_rows(qrec, gq, wo, krec, gko, np.arange(n))
        assert np.all(np.abs(sg[b, :n] - ref) <= tol), b
        assert np.isnan(sg[b, n:]).all()
