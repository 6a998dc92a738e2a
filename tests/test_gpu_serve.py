"""Incremental decode on the GPU (through the C ABI): tokens appended one at a
time to K and main-KV caches equal the caches quantised at once by the oracle
(NVFP4 with the cache's fixed tensor scale, MXFP4, main KV), and a serving step
captured once as a CUDA graph and replayed over the growing caches gives what
separate calls give at the final lengths."""
import numpy as np
import pytest
import torch

import inputs
import oracle
from cases import DEV, dev_bf16, gpu_quantize, i32, i64

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


class Growing:
    """Caches of several sequences with room to grow: the first n0[b] rows
    quantised at once (NVFP4 mode 0 gives each cache its tensor scale), the
    next tokens appended one per call."""

    def __init__(self, wl, n0, room, fmt):
        self.wl, self.n0, self.fmt = wl, list(n0), fmt
        self.B = B = len(n0)
        self.cap = [n + room for n in n0]
        self.signs = wl.signs()
        R = hsi.rec_bytes(fmt)
        self.R = R
        self.k_off = np.concatenate([[0], np.cumsum([hsi.n_records(c) for c in self.cap])[:-1]]).astype(np.int64)
        self.kv_off = np.concatenate([[0], np.cumsum(self.cap)[:-1]]).astype(np.int64)
        self.k_rec = torch.zeros(int(self.k_off[-1] + hsi.n_records(self.cap[-1])) * R, dtype=torch.uint8, device=DEV)
        self.kv = torch.zeros(int(self.kv_off[-1] + self.cap[-1]) * 288, dtype=torch.uint8, device=DEV)
        self.g = torch.ones(B, dtype=torch.float32, device=DEV)
        for b, n in enumerate(n0):
            kb = wl.k_bf16(0, b, rows=n)
            rec, g = gpu_quantize(kb, 1, n, self.signs, fmt=fmt)
            o = int(self.k_off[b]) * R
            self.k_rec[o:o + rec.numel()] = rec
            self.g[b] = g[0]
            x = dev_bf16(wl.kv_bf16(b, rows=n))
            hsi.quantize_mainkv(x, self.kv[int(self.kv_off[b]) * 288:(int(self.kv_off[b]) + n) * 288])
        self.n_vis = i32(self.n0)
        self.capacity = i32(self.cap)
        self.k_off_d, self.kv_off_d = i64(self.k_off.tolist()), i64(self.kv_off.tolist())
        self.k_stage = torch.empty(B, 128, dtype=torch.int16, device=DEV)
        self.kv_stage = torch.empty(B, 512, dtype=torch.int16, device=DEV)

    def token_rows(self, step):
        """bf16 rows of the token appended at `step` (the sequences' own next rows)."""
        k = np.stack([self.wl.k_bf16(0, b, first_row=self.n0[b] + step, rows=1)[0] for b in range(self.B)])
        kv = np.stack([self.wl.kv_bf16(b, first_row=self.n0[b] + step, rows=1)[0] for b in range(self.B)])
        return k, kv

    def stage(self, step):
        k, kv = self.token_rows(step)
        self.k_stage.copy_(dev_bf16(k))
        self.kv_stage.copy_(dev_bf16(kv))

    def append(self):
        hsi.append_token(self.k_stage, self.signs, None if self.fmt == hsi.FMT_MXFP4 else self.g, self.k_rec,
                         self.k_off_d, self.n_vis, self.capacity, self.B, kv_x=self.kv_stage, kv=self.kv,
                         kv_off=self.kv_off_d, fmt=self.fmt)

    def check_against_oracle(self, steps):
        k_all = self.k_rec.cpu().numpy()
        kv_all = self.kv.cpu().numpy()
        for b in range(self.B):
            n = self.n0[b] + steps
            kb = self.wl.k_bf16(0, b, rows=n)
            if self.fmt == hsi.FMT_MXFP4:
                ref = oracle.quantize_mx(kb, self.signs)
            else:
                ref, _ = oracle.quantize(kb, self.signs, g=float(self.g[b].item()))
            o = int(self.k_off[b]) * self.R
            assert np.array_equal(k_all[o:o + ref.size], ref), f"K cache {b}"
            refkv = oracle.mainkv_quantize(self.wl.kv_bf16(b, rows=n))
            o = int(self.kv_off[b]) * 288
            assert np.array_equal(kv_all[o:o + refkv.size], refkv), f"main KV {b}"


@pytest.mark.parametrize("fmt", [hsi.FMT_NVFP4, hsi.FMT_MXFP4])
def test_appended_tokens_equal_the_cache_quantised_at_once(fmt):
    wl = inputs.workload(1)
    G = Growing(wl, [5, 8, 1000, 4099], room=16, fmt=fmt)
    for step in range(12):  # crosses record boundaries in every cache
        G.stage(step)
        G.append()
    assert hsi.device_error() == 0
    assert G.n_vis.cpu().tolist() == [n + 12 for n in G.n0]
    G.check_against_oracle(12)


def test_append_past_capacity_is_reported_and_writes_nothing():
    wl = inputs.workload(1)
    G = Growing(wl, [7, 30], room=1, fmt=hsi.FMT_NVFP4)
    G.stage(0)
    G.append()
    assert hsi.device_error() == 0
    before_k, before_kv = G.k_rec.clone(), G.kv.clone()
    G.stage(1)
    G.append()  # both caches are full now
    assert hsi.device_error() == -6
    assert G.n_vis.cpu().tolist() == [8, 31]
    assert torch.equal(G.k_rec, before_k) and torch.equal(G.kv, before_kv)


def test_serving_step_graph_over_growing_caches():
    """append -> quantise q -> Full layer (scores, top-512, pool) -> 2 Reindex
    layers -> gather(main_kv, topk), captured once and replayed 9 times; then
    the same calls made separately at the final lengths give the same results."""
    wl = inputs.workload(1)
    n0 = [20000, 16380, 40001]
    G = Growing(wl, n0, room=16, fmt=hsi.FMT_NVFP4)
    B, cap = G.B, max(G.cap)
    signs = G.signs
    q = [dev_bf16(np.concatenate([wl.q_bf16(l, b) for b in range(B)])) for l in range(3)]
    w = [torch.from_numpy(np.stack([wl.w(l, b) for b in range(B)])).to(DEV) for l in range(3)]

    def outputs():
        return dict(q_rec=[torch.empty(B * 4 * 576, dtype=torch.uint8, device=DEV) for _ in range(3)],
                    g_q=[torch.empty(B, device=DEV) for _ in range(3)],
                    scores=torch.empty(B, cap, device=DEV),
                    idx=[torch.empty(B, 512, dtype=torch.int32, device=DEV) for _ in range(3)],
                    val=[torch.empty(B, 512, device=DEV) for _ in range(3)],
                    ids=torch.empty(B, 2048, dtype=torch.int32, device=DEV),
                    nk=torch.empty(B, dtype=torch.int32, device=DEV),
                    npool=torch.empty(B, dtype=torch.int32, device=DEV),
                    ps=torch.empty(B, 2048 * 8, device=DEV),
                    rows=torch.empty(3, B, 512, 512, dtype=torch.int16, device=DEV),
                    ws_full=hsi.workspace(hsi.WS_FULL_LAYER, B, cap, 512, device=DEV),
                    ws_r=hsi.workspace(hsi.WS_REINDEX_LAYER, B, 2048 * 8, 512, device=DEV),
                    pool_rec=torch.empty(B, 2048 * 576, dtype=torch.uint8, device=DEV))

    def step(o, n_vis, with_append):
        if with_append:
            G.append()
        for l in range(3):
            hsi.quantize_nvfp4(q[l], B, 32, signs, o["g_q"][l], o["q_rec"][l])
        hsi.full_layer(o["q_rec"][0], o["g_q"][0], w[0], G.k_rec, G.g, G.k_off_d, n_vis, B, cap, o["scores"], 512,
                       o["idx"][0], o["val"][0], block_ids=o["ids"], n_kept=o["nk"], n_pool=o["npool"],
                       ws=o["ws_full"])
        for r in (1, 2):
            hsi.reindex_layer(o["q_rec"][r], o["g_q"][r], w[r], G.k_rec, G.g, G.k_off_d, n_vis, o["ids"], o["nk"],
                              o["npool"], B, o["ps"], 512, o["idx"][r], o["val"][r], ws=o["ws_r"],
                              pool_rec=o["pool_rec"], pool_rec_ready=r > 1)
        for l in range(3):
            hsi.gather_mainkv(G.kv, G.kv_off_d, n_vis, o["idx"][l], 512, B, o["rows"][l])

    og = outputs()
    G.stage(0)
    step(og, G.n_vis, True)  # the first token, outside the graph (sets launch attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(og, G.n_vis, True)
    # capture records the launches without running them: the lengths are still n0 + 1
    for t in range(1, 10):
        G.stage(t)
        graph.replay()
    torch.cuda.synchronize()
    assert hsi.device_error() == 0
    assert G.n_vis.cpu().tolist() == [n + 10 for n in n0]
    G.check_against_oracle(10)
    os_ = outputs()
    step(os_, G.n_vis, False)  # the same step at the final lengths, separate calls, no append
    torch.cuda.synchronize()
    assert hsi.device_error() == 0
    for l in range(3):
        assert torch.equal(og["idx"][l], os_["idx"][l]) and torch.equal(og["val"][l], os_["val"][l]), l
        assert torch.equal(og["rows"][l], os_["rows"][l]), l
    assert torch.equal(og["ids"], os_["ids"]) and torch.equal(og["nk"], os_["nk"])
    assert torch.equal(og["npool"], os_["npool"])
    for b, n in enumerate(n0):
        assert torch.equal(og["scores"][b, :n + 10], os_["scores"][b, :n + 10])
    # the newest position is in every pool (its block is pinned)
    ids = og["ids"].cpu().numpy()
    for b, n in enumerate(n0):
        assert (n + 10 - 1) // 8 in ids[b, :int(og["nk"][b])]
