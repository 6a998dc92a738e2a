"""Parity of the chunked-prefill layer (hsi_prefill_layer): scores of groups of
queries sharing one cache, then every query's top-k and candidate pool taken
from the block maxima and the candidate blocks' scores only.

Bars: scores bit-identical to hsi_score_full with the same grouping; top-k,
pool ids, counts and the boolean table bit-exact against the oracle's top-k
and pool on the same fp32 scores (and so equal to hsi_topk and
hsi_candidate_pool on them). The selection phase is also driven on crafted
scores (heavy ties, -inf, short rows, rows whose tied blocks overflow the
staging buffer) written straight into the workspace."""
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


def _outputs(B, maxv, k, n_keep):
    return dict(
        top_idx=torch.full((B, k), 7, dtype=torch.int32, device=DEV),
        top_val=torch.full((B, k), 7.0, device=DEV),
        block_ids=torch.full((B, n_keep), 7, dtype=torch.int32, device=DEV),
        n_kept=torch.full((B,), 7, dtype=torch.int32, device=DEV),
        n_pool=torch.full((B,), 7, dtype=torch.int32, device=DEV),
        pool_bits=torch.full((B, (maxv + 31) // 32), 7, dtype=torch.int32, device=DEV))


def _check_against_oracle(scores, lengths, out, k, n_keep):
    sg = scores.cpu().numpy()
    ti, tv = out["top_idx"].cpu().numpy(), out["top_val"].cpu().numpy()
    ids, nk, npl = out["block_ids"].cpu().numpy(), out["n_kept"].cpu().numpy(), out["n_pool"].cpu().numpy()
    bits = out["pool_bits"].cpu().numpy().view(np.uint32)
    for b, n in enumerate(lengths):
        oi, ov = oracle.topk(sg[b], n, k)
        assert np.array_equal(ti[b], oi), f"query {b} (n={n}): top-k"
        assert np.array_equal(tv[b].view(np.uint32), ov.view(np.uint32)) or np.array_equal(tv[b], ov)
        pi, pk, pn, mask = oracle.pool(sg[b], n, 8, n_keep)
        assert nk[b] == pk and npl[b] == pn, f"query {b} (n={n}): counts {nk[b]},{npl[b]} vs {pk},{pn}"
        assert np.array_equal(ids[b], pi), f"query {b} (n={n}): pool ids"
        if n:
            gm = ((bits[b][np.arange(n) // 32] >> (np.arange(n) % 32)) & 1).astype(np.uint8)
            assert np.array_equal(gm, mask), f"query {b} (n={n}): boolean table"


@pytest.mark.parametrize("n_cache,n_vis", [
    (20000, [20000, 19999, 16384, 16385]),
    (131072, [122881, 122882, 122883, 122884, 131072, 131071, 40000, 9]),
    (3000, [1, 2, 8, 9]),
])
def test_prefill_layer_scores_topk_pool(n_cache, n_vis):
    wl = inputs.workload(4)
    B, k, n_keep = len(n_vis), 512, 2048
    caches = Caches(wl, 0, [0], [n_cache])
    gk = caches.g.repeat(B)
    q_rec, g_q, w = gpu_queries(wl, 0, range(B))
    off = i64([0] * B)
    nv = i32(n_vis)
    ref = torch.full((B, n_cache), float("nan"), device=DEV)
    hsi.score_full(q_rec, g_q, w, caches.k_rec, gk, off, nv, B, n_cache, ref, group=4)
    scores = torch.full((B, n_cache), float("nan"), device=DEV)
    out = _outputs(B, n_cache, k, n_keep)
    hsi.prefill_layer(q_rec, g_q, w, caches.k_rec, gk, off, nv, B, n_cache, scores, k, group=4, n_keep=n_keep, **out)
    assert hsi.device_error() == 0
    for b, n in enumerate(n_vis):
        assert torch.equal(scores[b, :n], ref[b, :n])
    _check_against_oracle(scores, n_vis, out, k, n_keep)


def _select_on(scores, lengths, k=512, n_keep=2048):
    """The selection phase alone on given scores: the block maxima are written
    into the workspace where the scoring phase leaves them."""
    B, maxv = scores.shape
    nb = (maxv + 7) // 8
    ldb = (nb + 3) // 4 * 4  # rows of block maxima padded to 16 bytes
    ws = hsi.workspace(hsi.WS_PREFILL_LAYER, B, maxv, k, device=DEV)
    pad = torch.full((B, nb * 8), float("-inf"), device=DEV)
    for b, n in enumerate(lengths):
        pad[b, :n] = scores[b, :n]
    ws[: B * ldb * 4].view(torch.float32).view(B, ldb)[:, :nb] = pad.view(B, nb, 8).amax(2)
    out = _outputs(B, maxv, k, n_keep)
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    hsi.prefill_layer(dummy, torch.ones(B, device=DEV), torch.zeros(B, 32, device=DEV), dummy,
                      torch.ones(B, device=DEV), i64([0] * B), i32(lengths), B, maxv, scores, k, group=1,
                      n_keep=n_keep, ws=ws, phases=hsi.PHASE_SELECT, **out)
    assert hsi.device_error() == 0
    return out


def test_prefill_select_crafted_ties_and_edges():
    g = torch.Generator(device="cpu").manual_seed(5)
    maxv = 140000
    lengths = [140000, 16384, 16383, 2049 * 8, 2048 * 8 + 1, 513 * 8, 100, 1, 0, 131072]
    B = len(lengths)
    s = torch.randn(B, maxv, generator=g)
    s[0] = torch.round(s[0] * 2) / 2          # few distinct values: ties everywhere
    s[1, ::3] = float("-inf")                  # -inf scores
    s[2] = 0.0                                  # one value: every block tied
    s[2, 5] = -0.0
    s[3, 8 * 100:8 * 600] = float("-inf")      # whole blocks at -inf
    s[9] = torch.randint(0, 3, (maxv,), generator=g).float()  # tied maxima beyond the staging buffer
    out = _select_on(s.to(DEV), lengths)
    _check_against_oracle(s, lengths, out, 512, 2048)


@pytest.mark.parametrize("k,n_keep", [(1, 1), (100, 64), (2048, 2048), (512, 4096)])
def test_prefill_select_k_and_keep(k, n_keep):
    g = torch.Generator(device="cpu").manual_seed(k + n_keep)
    maxv = 70000
    lengths = [70000, 33333, 8, 5000]
    s = torch.randn(len(lengths), maxv, generator=g) * 3
    out = _select_on(s.to(DEV), lengths, k, n_keep)
    _check_against_oracle(s, lengths, out, k, n_keep)
