"""The FP4 main KV and gather(main_kv, topk) on the GPU (through the C ABI)
against the oracle: entries bit-exact, gathered bf16 rows bit-exact (every
decoded value is exact in bf16), padding rows zero, bad indices reported."""
import numpy as np
import pytest
import torch

import inputs
import oracle
from cases import DEV, dev_bf16, i32, i64

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


def _gpu_kv(x):
    kv = torch.full((x.shape[0] * 288,), 0xA5, dtype=torch.uint8, device=DEV)
    hsi.quantize_mainkv(dev_bf16(x), kv)
    return kv


@pytest.mark.parametrize("n", [1, 7, 1000, 4099])
def test_quantize_mainkv_bit_exact(n):
    x = inputs.normal_bf16(31, 81, n * 512).reshape(n, 512)
    kv = _gpu_kv(x)
    assert hsi.device_error() == 0
    assert np.array_equal(kv.cpu().numpy(), oracle.mainkv_quantize(x))


def test_quantize_mainkv_extremes():
    """Zero groups, bf16 subnormals (scales that round to 0 or to E4M3
    subnormals), groups past 2688 (scale saturates at 448, codes at 6), mixed signs."""
    rng = np.random.default_rng(5)
    f = (rng.standard_normal((64, 512)) * np.exp(rng.uniform(-30, 12, (64, 32))).repeat(16, 1)).astype(np.float32)
    f[1] = 0.0
    f[2] = 1e-40
    f[3, :256] = 5000.0
    f[3, 256:] = -1e-3
    f[4] = np.where(np.arange(512) % 2 == 0, 7.0, -7.0)
    x = (f.view(np.uint32) >> 16).astype(np.uint16)
    kv = _gpu_kv(x)
    assert hsi.device_error() == 0
    assert np.array_equal(kv.cpu().numpy(), oracle.mainkv_quantize(x))


def test_quantize_mainkv_non_finite_is_reported():
    x = np.zeros((3, 512), dtype=np.uint16)
    x[1, 100] = 0x7FC0  # NaN
    _gpu_kv(x)
    assert hsi.device_error() == -6


def test_gather_decodes_every_code_and_scale():
    """Entries holding every (code, scale) pair of valid E4M3 scales."""
    rows = []
    scales = [c for c in range(256) if c not in (0x7F, 0xFF)]
    for i in range(0, len(scales), 32):
        sc = np.array((scales[i:i + 32] * 2)[:32], dtype=np.uint8)
        e = np.zeros(288, dtype=np.uint8)
        codes = (np.arange(512) * 7 + i) % 16
        for c in range(512):
            e[c // 2] |= codes[c] << (4 * (c & 1))
        e[256:] = sc
        rows.append(e)
    kv_h = np.concatenate(rows)
    n = len(rows)
    kv = torch.from_numpy(kv_h).to(DEV)
    idx = np.arange(n, dtype=np.int32)[::-1].copy()
    out = torch.empty(1, n, 512, dtype=torch.int16, device=DEV)
    hsi.gather_mainkv(kv, i64([0]), i32([n]), torch.from_numpy(idx).view(1, n).to(DEV), n, 1, out)
    assert hsi.device_error() == 0
    got = out.cpu().numpy().view(np.uint16)[0]
    assert np.array_equal(got, oracle.mainkv_gather(kv_h, n, idx))


def test_gather_topk_of_several_caches():
    """Caches of 5, 300 and 20000 entries back to back; each query's row of a
    wider index buffer (ld 600) holds a top-512-style list: its own positions,
    -1 padding past a short cache."""
    lengths = [5, 300, 20000]
    xs = [inputs.normal_bf16(40 + j, 82, n * 512).reshape(n, 512) for j, n in enumerate(lengths)]
    kv_h = [oracle.mainkv_quantize(x) for x in xs]
    kv = torch.cat([_gpu_kv(x) for x in xs])
    off = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64)
    rng = np.random.default_rng(6)
    idx = np.full((3, 600), -7, dtype=np.int32)
    for b, n in enumerate(lengths):
        sel = rng.permutation(n)[:512].astype(np.int32)
        idx[b, :512] = -1
        idx[b, :sel.size] = sel
    out = torch.full((3, 512, 512), 0x5A5A, dtype=torch.int16, device=DEV)
    hsi.gather_mainkv(kv, i64(off.tolist()), i32(lengths), torch.from_numpy(idx).to(DEV), 512, 3, out, ld_idx=600)
    assert hsi.device_error() == 0
    got = out.cpu().numpy().view(np.uint16)
    for b, n in enumerate(lengths):
        assert np.array_equal(got[b], oracle.mainkv_gather(kv_h[b], n, idx[b, :512])), b


def test_gather_index_past_the_cache_is_reported_and_zeroed():
    x = inputs.normal_bf16(50, 83, 64 * 512).reshape(64, 512)
    kv_h = oracle.mainkv_quantize(x)
    kv = _gpu_kv(x)
    idx = np.array([[3, 64, 10, -1]], dtype=np.int32)
    out = torch.full((1, 4, 512), 0x5A5A, dtype=torch.int16, device=DEV)
    hsi.gather_mainkv(kv, i64([0]), i32([64]), torch.from_numpy(idx).to(DEV), 4, 1, out)
    assert hsi.device_error() == -6
    got = out.cpu().numpy().view(np.uint16)[0]
    ok = np.array([3, -1, 10, -1], dtype=np.int32)
    assert np.array_equal(got, oracle.mainkv_gather(kv_h, 64, ok))


@pytest.mark.parametrize("B,k", [(3, 7), (1, 1), (5, 513)])
def test_gather_ragged_list_lengths(B, k):
    """List lengths that leave a warp's last entries past the end (4 per warp)."""
    n = 1000
    x = inputs.normal_bf16(60 + k, 84, n * 512).reshape(n, 512)
    kv_h = oracle.mainkv_quantize(x)
    kv = _gpu_kv(x)
    rng = np.random.default_rng(k)
    idx = rng.integers(-1, n, (B, k + 2)).astype(np.int32)
    out = torch.full((B, k, 512), 0x5A5A, dtype=torch.int16, device=DEV)
    hsi.gather_mainkv(kv, i64([0] * B), i32([n] * B), torch.from_numpy(idx).to(DEV), k, B, out, ld_idx=k + 2)
    assert hsi.device_error() == 0
    got = out.cpu().numpy().view(np.uint16)
    for b in range(B):
        assert np.array_equal(got[b], oracle.mainkv_gather(kv_h, n, idx[b, :k])), b


@pytest.mark.parametrize("L,B,k", [(5, 3, 7), (2, 1, 1), (3, 4, 513)])
def test_gather_layers_in_one_launch(L, B, k):
    """Every layer's list in one launch (hsi_gather_mainkv_layers): each layer's
    rows equal the oracle's gather of that layer's list, ragged ends included."""
    n = 1000
    x = inputs.normal_bf16(70 + k, 85, n * 512).reshape(n, 512)
    kv_h = oracle.mainkv_quantize(x)
    kv = _gpu_kv(x)
    rng = np.random.default_rng(L * 100 + k)
    lengths = [n - 7 * b for b in range(B)]
    idx = np.stack([rng.integers(-1, lengths[b], (L, k)) for b in range(B)], 1).astype(np.int32)  # [L][B][k]
    out = torch.full((L, B, k, 512), 0x5A5A, dtype=torch.int16, device=DEV)
    hsi.gather_mainkv_layers(kv, i64([0] * B), i32(lengths), torch.from_numpy(idx).to(DEV), k, B, out)
    assert hsi.device_error() == 0
    got = out.cpu().numpy().view(np.uint16)
    for l in range(L):
        for b in range(B):
            assert np.array_equal(got[l, b], oracle.mainkv_gather(kv_h, lengths[b], idx[l, b])), (l, b)
