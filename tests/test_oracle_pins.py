"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values printed
on the pages (tests/golden), library routines (torch's fp8 cast, scipy's
Hadamard matrix, Python's sort), closed forms, invariants and brute force.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import inputs
import oracle
from conftest import golden_rows

D, H = 128, 32


# ------------------------------------------------------------------ codecs --

def test_e2m1_values_match_page_table():
    for code, mag in golden_rows("e2m1_values.txt"):
        c, m = int(code), float(mag)
        assert oracle.e2m1_value(c) == m
        assert oracle.e2m1_value(c | 8) == -m
    distinct = {oracle.e2m1_value(c) for c in range(16)}
    assert len(distinct) == 15  # +0 and -0 compare equal: 15 values


def test_e2m1_rounding_golden_midpoints():
    for x, code in golden_rows("e2m1_rounding.txt"):
        assert oracle.e2m1_encode(float(x)) == int(code), x
        assert oracle.e2m1_encode(-float(x)) == int(code) | 8, x


def test_e2m1_encode_is_nearest_and_monotone():
    xs = np.linspace(0, 8, 20001, dtype=np.float32)
    vals = np.array([oracle.e2m1_value(c) for c in range(8)])
    prev = 0
    for x in xs:
        c = oracle.e2m1_encode(float(x))
        assert c >= prev
        prev = c
        err = abs(float(x) - vals[c])
        assert err <= np.min(np.abs(float(x) - vals)) + 0.0


def test_e4m3_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], c
    assert oracle.e4m3_value(0x7E) == 448.0  # 448 * 6 = 2688 (page: 去掉全局 scale 之后范围仍然够用)


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        np.linspace(0, 448, 50001),
        np.exp(rng.uniform(np.log(1e-4), np.log(448), 50000)),
        # exact midpoints between neighbouring codes: ties go to the even code
        np.array([(oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)) / 2 for c in range(126)]),
    ]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert (mine == ref).all()
    # negative values keep their sign
    neg = torch.from_numpy(-xs[:2000]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine_neg = np.array([oracle.e4m3_encode(-float(x)) for x in xs[:2000]], dtype=np.uint8)
    nz = xs[:2000] != 0
    assert (mine_neg[nz] == neg[nz]).all()


def test_e4m3_saturates_at_448():
    for x in [448.0, 449.0, 464.0, 480.0, 1e6]:
        assert oracle.e4m3_encode(x) == 0x7E


# ---------------------------------------------------------------- rotation --

def test_fwht_is_sylvester_hadamard():
    cols = np.stack([oracle.fwht128(np.eye(D, dtype=np.float32)[i]) for i in range(D)], 1)
    assert (cols == scipy.linalg.hadamard(D)).all()
    assert (cols @ cols.T == D * np.eye(D)).all()


def test_fwht_twice_is_128x_on_small_integers():
    rng = np.random.default_rng(1)
    x = rng.integers(-50, 50, D).astype(np.float32)
    assert (oracle.fwht128(oracle.fwht128(x)) == D * x).all()


def test_rotation_preserves_dot_products():
    rng = np.random.default_rng(2)
    q = rng.standard_normal(D)
    k = rng.standard_normal(D)
    s = rng.choice([-1.0, 1.0], D)
    Hm = scipy.linalg.hadamard(D).astype(np.float64)
    assert abs((Hm @ (s * q)) @ (Hm @ (s * k)) / D - q @ k) < 1e-9


# ---------------------------------------------------------------- quantise --

def _rand_tensor(seed, rows):
    return inputs.normal_bf16(seed, 99, rows * D).reshape(rows, D)


def test_quantize_tensor_scale_and_range():
    x = _rand_tensor(3, 40)
    s = inputs.signs(3)
    rec, g = oracle.quantize(x, s)
    Hm = scipy.linalg.hadamard(D).astype(np.float64)
    y = (inputs.bf16_to_f32(x).astype(np.float64) * s) @ Hm.T
    amax = np.abs(y).max()
    assert g == pytest.approx(amax / 2688.0, rel=1e-6)
    dec = oracle.decode_rows(rec, 40, g)
    # largest representable magnitude is 6 * 448 * g = amax_T
    assert np.abs(dec).max() <= 6 * 448 * g * (1 + 1e-6)
    assert np.abs(dec).max() >= amax * (1 - 0.07)


def test_quantize_error_within_half_step():
    x = _rand_tensor(4, 64)
    s = inputs.signs(4)
    rec, g = oracle.quantize(x, s)
    Hm = scipy.linalg.hadamard(D).astype(np.float64)
    y = (inputs.bf16_to_f32(x).astype(np.float64) * s) @ Hm.T
    dec = oracle.decode_rows(rec, 64, g)
    for r in range(64):
        for grp in range(8):
            sl = slice(16 * grp, 16 * grp + 16)
            yb, db = y[r, sl], dec[r, sl]
            amax_b = np.abs(yb).max()
            nz = np.abs(db[db != 0])
            sc = nz.min() / 0.5 if nz.size else 0.0  # not the scale itself; only a bound below
            # decoded block max within one E4M3 step (12.5%) of the true block max
            assert np.abs(db).max() <= amax_b * 1.13 + 1e-12
            assert np.abs(db).max() >= amax_b / 1.13 - 1e-12
            # every element within half the widest E2M1 gap (1.0 between 4 and 6) of
            # the block scale, which is at most amax_b / 6 * 1.0625
            assert np.all(np.abs(yb - db) <= amax_b / 6 * 1.0625 * 1.0 + 1e-9)
            del sc


def test_quantize_codes_and_scales_are_brute_force_nearest():
    """Every NVFP4 scale byte is torch's E4M3 cast (round to nearest even,
    saturating at 448) of amax_b / (6 g) in fp32, and every code is the nearest
    E2M1 magnitude (ties to the even code, saturating at 6) of y / (E4M3(sb) g)
    with the sign of y; g = amax_T / 2688 in fp32."""
    rows = 24
    x = _rand_tensor(13, rows)
    x[5] = 0  # an all-zero row: every block scale 0, every code 0
    s = inputs.signs(13)
    rec, g = oracle.quantize(x, s)
    xf = inputs.bf16_to_f32(x)
    y = np.stack([oracle.fwht128((xf[r] * s).astype(np.float32)) for r in range(rows)])
    assert np.float32(g) == np.float32(np.abs(y).max()) / np.float32(2688)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    six_g = np.float32(6) * np.float32(g)
    for r in range(rows):
        d = oracle.decode_row(rec, r, g)
        for grp in range(8):
            yb = y[r, 16 * grp:16 * grp + 16]
            ratio = min(np.float32(np.abs(yb).max()) / six_g, np.float32(448))
            sb = torch.tensor([ratio], dtype=torch.float32).to(torch.float8_e4m3fn)
            assert rec[(r // 8) * 576 + 512 + (r % 8) * 8 + grp] == sb.view(torch.uint8).item()
            sbv = float(sb.to(torch.float64).item())
            sc = np.float32(np.float32(sbv) * np.float32(g))
            for t in range(16):
                if sc == 0:
                    c = 0
                else:
                    a = float(np.abs(yb[t]) / sc)  # fp32 division, as the recipe states
                    dist = np.abs(mags - a)
                    best = np.flatnonzero(dist == dist.min())
                    c = best[0] if best.size == 1 else best[best % 2 == 0][0]
                want = math.copysign(mags[c] * sbv * g, float(yb[t]))
                assert d[16 * grp + t] == want or (mags[c] == 0 and d[16 * grp + t] == 0)
    assert np.all(oracle.decode_row(rec, 5, g) == 0)


def test_quantize_mode1_reuses_scale_and_is_deterministic():
    x = _rand_tensor(5, 17)
    s = inputs.signs(5)
    rec0, g0 = oracle.quantize(x, s)
    rec1, g1 = oracle.quantize(x, s, g=g0)
    assert g1 == g0 and (rec0 == rec1).all()
    assert rec0.size == 3 * 576
    # padding rows of the last record are zero
    dec = oracle.decode_row(rec0, 17, g0)
    assert (dec == 0).all()


def test_quantize_zero_tensor():
    x = np.zeros((8, D), dtype=np.uint16)
    rec, g = oracle.quantize(x, np.ones(D, dtype=np.int8))
    assert g == 1.0 and (rec == 0).all()


# ----------------------------------------------------------------- MXFP4 --

def test_fp4_format_sizes_match_page_table():
    for fmt, group, sbits, bpe, per_key in golden_rows("fp4_formats.txt"):
        group, sbits, bpe, per_key = int(group), int(sbits), float(bpe), int(per_key)
        assert 4 + sbits / group == bpe
        x = np.zeros((8, D), dtype=np.uint16)
        rec = oracle.quantize_mx(x, np.ones(D, dtype=np.int8)) if fmt == "mxfp4" else \
            oracle.quantize(x, np.ones(D, dtype=np.int8))[0]
        assert rec.size == 8 * per_key, fmt


def test_e8m0_decode_matches_library_all_codes():
    codes = list(range(256))
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.tensor(codes, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).tolist()
    else:  # the OCP MX definition: 2^(b - 127), 0xFF NaN
        ref = [math.ldexp(1.0, c - 127) if c != 255 else math.nan for c in codes]
    for c in codes:
        v = oracle.e8m0_value(c)
        assert (math.isnan(v) and math.isnan(ref[c])) or v == ref[c], c


def test_mx_scale_is_the_smallest_power_of_two_covering_amax_over_6():
    # closed forms: 6 * 2^e >= amax > 6 * 2^(e-1)
    assert oracle.mx_scale_exp(6.0) == 0
    assert oracle.mx_scale_exp(3.0) == -1
    assert oracle.mx_scale_exp(1.5) == -2
    assert oracle.mx_scale_exp(float(np.nextafter(np.float32(1.5), np.float32(2)))) == -1
    assert oracle.mx_scale_exp(0.0) == -127
    assert oracle.mx_scale_exp(1e-45) == -127
    assert oracle.mx_scale_exp(float(np.finfo(np.float32).max)) == 126
    rng = np.random.default_rng(31)
    for a in np.exp(rng.uniform(-80, 80, 3000)).astype(np.float32):
        e = oracle.mx_scale_exp(float(a))
        assert math.ldexp(6.0, e) >= float(a)
        assert e == -127 or math.ldexp(6.0, e - 1) < float(a)


def _bf16(x):
    b = (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert (inputs.bf16_to_f32(b) == np.asarray(x, dtype=np.float32)).all()
    return b


def test_quantize_mx_layout_one_hot_rows():
    # y = H x is one-hot (6 at element e) when x = 6 H[e] / 128 (+-0.046875, exact in bf16),
    # so element e must decode to 6 with scale 2^0 and every other group to 0 with scale byte 0
    Hm = scipy.linalg.hadamard(D).astype(np.float64)
    cases = [(0, 0), (1, 1), (2, 31), (3, 32), (4, 77), (5, 126), (6, 127), (7, 64), (8, 5)]
    x = np.zeros((len(cases), D))
    for r, e in cases:
        x[r] = 6.0 * Hm[e] / D
    rec = oracle.quantize_mx(_bf16(x), np.ones(D, dtype=np.int8))
    assert rec.size == 2 * 544
    want = np.zeros(2 * 544, dtype=np.uint8)
    for r, e in cases:
        base = (r // 8) * 544
        rr = r % 8
        byte = base + (e // 32) * 128 + rr * 16 + (e % 32) // 2
        want[byte] |= 7 << (4 * (e & 1))
        want[base + 512 + rr * 4 + e // 32] = 127
    assert (rec == want).all()
    for r, e in cases:
        d = oracle.decode_row(rec, r, fmt="mxfp4")
        assert d[e] == 6.0 and np.count_nonzero(d) == 1


def test_quantize_mx_constant_rows_closed_form():
    # x = c e_0 with signs +1 gives y = c in all 128 elements (first Sylvester column)
    cs = [6.0, -5.0, 1.0, 0.75, -40.0, 0.0]
    x = np.zeros((len(cs), D))
    x[:, 0] = cs
    rec = oracle.quantize_mx(_bf16(x), np.ones(D, dtype=np.int8))
    # c = 6: scale 1, code 6.0; -5: scale 1, 5 ties between 4 and 6 -> even code (4);
    # 1: scale 1/4, code 4.0; 0.75: scale 1/8, 6.0; -40: scale 8, 5 -> 4 (tie to even); 0: zeros
    want = [(127, 6.0), (127, -4.0), (125, 4.0), (124, 6.0), (130, -4.0), (0, 0.0)]
    for r, (sb, cv) in enumerate(want):
        d = oracle.decode_row(rec, r, fmt="mxfp4")
        assert (rec[512 + r * 4: 512 + r * 4 + 4] == sb).all(), r
        assert (d == cv * math.ldexp(1.0, sb - 127)).all(), r


def test_quantize_mx_codes_are_brute_force_nearest():
    x = _rand_tensor(12, 24)
    s = inputs.signs(12)
    rec = oracle.quantize_mx(x, s)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    xf = inputs.bf16_to_f32(x)
    for r in range(24):
        y = oracle.fwht128((xf[r] * s).astype(np.float32)).astype(np.float64)
        d = oracle.decode_row(rec, r, fmt="mxfp4")
        for grp in range(4):
            yg = y[32 * grp: 32 * grp + 32]
            amax = np.abs(yg).max()
            sc = math.ldexp(1.0, int(rec[(r // 8) * 544 + 512 + (r % 8) * 4 + grp]) - 127)
            assert 6 * sc >= amax and (amax == 0 or 3 * sc < amax)
            for t in range(32):
                a = abs(yg[t]) / sc
                dist = np.abs(mags - a)
                best = np.flatnonzero(dist == dist.min())
                c = best[0] if best.size == 1 else best[best % 2 == 0][0]  # tie: even code
                assert d[32 * grp + t] == math.copysign(mags[c] * sc, yg[t]) or (mags[c] == 0 and d[32 * grp + t] == 0)


def test_quantize_mx_padding_rows_are_zero():
    rec = oracle.quantize_mx(_rand_tensor(13, 17), inputs.signs(13))
    assert rec.size == 3 * 544
    last = rec[2 * 544:].reshape(-1)
    for rr in range(1, 8):  # row 16 is real; rows 17..23 are padding
        for e in range(D):
            assert last[(e // 32) * 128 + rr * 16 + (e % 32) // 2] == 0
        assert (last[512 + rr * 4: 512 + rr * 4 + 4] == 0).all()


def test_score_mx_equals_unrotated_formula_when_quantisation_is_exact():
    s, qb, qx, kb, kx = _sparse_exact_case(16)
    qrec = oracle.quantize_mx(qb, s)
    krec = oracle.quantize_mx(kb, s)
    w = np.random.default_rng(17).standard_normal(H).astype(np.float32)
    scores, macs = oracle.score_full(qrec, 1.0, w, krec, 1.0, 50, fmt="mxfp4")
    ref = np.maximum(kx @ qx.T, 0.0) @ w.astype(np.float64)
    assert np.allclose(scores, ref, rtol=2e-6, atol=1e-9)
    assert macs == 50 * 4096
    rows = np.array([0, 9, 49])
    part, tol = oracle.score_rows(qrec, 1.0, w, krec, 1.0, rows, fmt="mxfp4")
    assert (part == scores[rows]).all() and (tol > 0).all()


def test_score_mx_tracks_unquantised_formula_and_pool_slots():
    wl = inputs.workload(0)
    s = wl.signs()
    qb, kb = wl.q_bf16(0, 0), wl.k_bf16(0, 0, rows=2000)
    qrec, krec = oracle.quantize_mx(qb, s), oracle.quantize_mx(kb, s)
    w = wl.w(0, 0)
    sc, _ = oracle.score_full(qrec, 1.0, w, krec, 1.0, 2000, fmt="mxfp4")
    ref = np.maximum(inputs.bf16_to_f32(kb).astype(np.float64) @ inputs.bf16_to_f32(qb).astype(np.float64).T,
                     0.0) @ w.astype(np.float64)
    assert np.corrcoef(sc, ref)[0, 1] > 0.95
    # the scale is carried: same magnitude as the unquantised score (no stray 2^k)
    assert 0.5 < np.abs(sc).mean() / np.abs(ref).mean() < 2.0
    ids = np.array([3, 0, 249, 17] + [-1] * 4, dtype=np.int32)
    ps, _ = oracle.score_pool(qrec, 1.0, w, krec, 1.0, 1997, ids, 4, n_keep=8, fmt="mxfp4")
    for j, b in enumerate(ids[:4]):
        for r in range(8):
            pos = b * 8 + r
            assert ps[8 * j + r] == (sc[pos] if pos < 1997 else -np.inf)
    assert np.isneginf(ps[32:]).all()


# ----------------------------------------------------------------- main KV --

def _kv_entry(codes, scales):
    """One 288-byte main-KV entry from 512 codes and 32 scale bytes (the layout definition)."""
    e = np.zeros(288, dtype=np.uint8)
    for c in range(512):
        e[c // 2] |= (int(codes[c]) & 15) << (4 * (c & 1))
    e[256:] = scales
    return e


def test_mainkv_entry_size_matches_page():
    ((dims, group, payload, scales, total),) = golden_rows("mainkv_format.txt")
    dims, group, payload, scales, total = map(int, (dims, group, payload, scales, total))
    assert dims * 4 // 8 == payload and dims // group == scales and payload + scales == total
    kv = oracle.mainkv_quantize(np.zeros((3, dims), dtype=np.uint16))
    assert kv.size == 3 * total


def test_mainkv_decode_every_code_and_scale_against_library():
    e2m1 = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6] * 2) * np.repeat([1, -1], 8)
    sc = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for sbase in range(0, 256, 32):
        scales = np.arange(sbase, sbase + 32, dtype=np.uint8)
        codes = np.arange(512) % 16
        e = _kv_entry(codes, scales)
        d = oracle.mainkv_decode(e, 0)
        ref = e2m1[codes] * sc[scales[np.arange(512) // 16]]
        fin = ~np.isnan(ref)
        assert np.array_equal(d[fin], ref[fin])
        if fin.all():  # exact in bf16: torch's bf16 cast returns the same value
            g = oracle.mainkv_gather(e, 1, np.array([0]))[0]
            tb = torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(g, tb)


def test_mainkv_quantize_closed_forms():
    # group g of entry 0 is constant v_g: scale E4M3_RN(|v|/6), every code the same
    vals = [6.0, 7.0, 0.0, -3.0, 448.0 * 6, 1e-3, 5.0, -0.75]
    x = np.zeros((1, 512), dtype=np.float32)
    for g, v in enumerate(vals):
        x[0, 16 * g:16 * g + 16] = v
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    kv = oracle.mainkv_quantize(xb)
    d = oracle.mainkv_decode(kv, 0)
    xf = inputs.bf16_to_f32(xb)[0]
    # 6 -> scale 1, code 6; 7 -> 7/6 rounds to scale 1.125, 7/1.125 saturates to 6 -> 6.75;
    # 0 -> scale 0, zeros; -3 -> scale 0.5, -6 -> -3; 2688 -> scale 448, 6 -> 2688;
    # 5 -> scale 0.8125 (5/6 = 0.8333 rounds down), 5/0.8125 = 6.15 -> 6 -> 4.875;
    # -0.75 -> scale 0.125, -6 -> -0.75
    want = {0: 6.0, 1: 6.75, 2: 0.0, 3: -3.0, 4: 2688.0, 6: 4.875, 7: -0.75}
    for g, v in want.items():
        assert (d[16 * g:16 * g + 16] == v).all(), (g, d[16 * g])
    # 1e-3 (bf16 0.000999..): a subnormal E4M3 scale; check against the definition
    a = float(np.abs(xf[80:96]).max())
    sb = torch.tensor([np.float32(a) / np.float32(6)]).to(torch.float8_e4m3fn).view(torch.uint8).item()
    assert kv[256 + 5] == sb


def test_mainkv_codes_are_brute_force_nearest():
    x = inputs.normal_bf16(14, 79, 20 * 512).reshape(20, 512)
    kv = oracle.mainkv_quantize(x)
    xf = inputs.bf16_to_f32(x)
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for i in range(20):
        d = oracle.mainkv_decode(kv, i)
        for g in range(32):
            xg = xf[i, 16 * g:16 * g + 16]
            amax = np.float32(np.abs(xg).max())
            sb = torch.tensor([amax / np.float32(6)]).to(torch.float8_e4m3fn)
            assert kv[i * 288 + 256 + g] == sb.view(torch.uint8).item()
            sc = float(sb.to(torch.float64).item())
            for t in range(16):
                a = float(np.float32(abs(xg[t])) / np.float32(sc))
                dist = np.abs(mags - a)
                best = np.flatnonzero(dist == dist.min())
                c = best[0] if best.size == 1 else best[best % 2 == 0][0]
                assert abs(d[16 * g + t]) == mags[c] * sc


def test_mainkv_gather_order_padding_and_range():
    x = inputs.normal_bf16(15, 80, 40 * 512).reshape(40, 512)
    kv = oracle.mainkv_quantize(x)
    idx = np.array([7, 0, 39, -1, 7, -1], dtype=np.int32)
    g = oracle.mainkv_gather(kv, 40, idx)
    for t, i in enumerate(idx):
        if i < 0:
            assert (g[t] == 0).all()
        else:
            want = oracle.mainkv_decode(kv, int(i)).astype(np.float32).view(np.uint32) >> 16
            assert np.array_equal(g[t], want.astype(np.uint16))
    with pytest.raises(ValueError):
        oracle.mainkv_gather(kv, 39, idx)  # 39 is past the 39 visible entries


# ------------------------------------------------------------------- score --

def _sparse_exact_case(seed):
    """q, k whose rotated rows have at most two non-zeros from the E2M1 set, so
    that NVFP4 holds them exactly (up to the fp32 tensor scale)."""
    rng = np.random.default_rng(seed)
    Hm = scipy.linalg.hadamard(D).astype(np.float64)
    s = np.ones(D, dtype=np.int8)

    def rows(n):
        ys = np.zeros((n, D))
        for r in range(n):
            # both non-zeros in one 16-element group, whose block scale then
            # decodes to g * 448, so every E2M1 value is held exactly
            grp = rng.integers(0, D // 16)
            i, j = grp * 16 + rng.choice(16, 2, replace=False)
            ys[r, i] = 6.0 * rng.choice([-1, 1])
            ys[r, j] = rng.choice([0.5, 1, 1.5, 2, 3, 4, 6]) * rng.choice([-1, 1])
        xs = ys @ Hm / D  # H^-1 = H / 128; entries are (+-a +- b)/128: exact in bf16
        b = (xs.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert (inputs.bf16_to_f32(b) == xs).all()
        return b, xs

    qb, qx = rows(H)
    kb, kx = rows(50)
    return s, qb, qx, kb, kx


def test_score_equals_unrotated_formula_when_quantisation_is_exact():
    s, qb, qx, kb, kx = _sparse_exact_case(6)
    qrec, gq = oracle.quantize(qb, s)
    krec, gk = oracle.quantize(kb, s)
    w = np.random.default_rng(7).standard_normal(H).astype(np.float32)
    scores, macs = oracle.score_full(qrec, gq, w, krec, gk, 50)
    # page formula on the original (unrotated) vectors, in double
    ref = np.maximum(kx @ qx.T, 0.0) @ w.astype(np.float64)
    assert np.allclose(scores, ref, rtol=2e-6, atol=1e-9)
    assert macs == 50 * 4096


def test_score_single_head_is_relu_of_decoded_gemv():
    wl = inputs.workload(0)
    s = wl.signs()
    qrec, gq = oracle.quantize(wl.q_bf16(0, 0), s)
    krec, gk = oracle.quantize(wl.k_bf16(0, 0, rows=300), s)
    qd = oracle.decode_rows(qrec, H, gq)
    kd = oracle.decode_rows(krec, 300, gk)
    for j in (0, 13, 31):
        w = np.zeros(H, dtype=np.float32)
        w[j] = 1.0
        sc, _ = oracle.score_full(qrec, gq, w, krec, gk, 300)
        ref = np.maximum(kd @ qd[j], 0.0) / 128.0
        assert np.allclose(sc, ref.astype(np.float32), rtol=1e-6, atol=0)


def test_score_tracks_unquantised_formula():
    wl = inputs.workload(0)
    s = wl.signs()
    qb, kb = wl.q_bf16(0, 0), wl.k_bf16(0, 0, rows=2000)
    qrec, gq = oracle.quantize(qb, s)
    krec, gk = oracle.quantize(kb, s)
    w = wl.w(0, 0)
    sc, _ = oracle.score_full(qrec, gq, w, krec, gk, 2000)
    ref = np.maximum(inputs.bf16_to_f32(kb).astype(np.float64) @ inputs.bf16_to_f32(qb).astype(np.float64).T,
                     0.0) @ w.astype(np.float64)
    assert np.corrcoef(sc, ref)[0, 1] > 0.97
    # a transposed or sign-flipped operand destroys the correlation
    bad = np.maximum(-(inputs.bf16_to_f32(kb).astype(np.float64) @ inputs.bf16_to_f32(qb).astype(np.float64).T),
                     0.0) @ w.astype(np.float64)
    assert np.corrcoef(sc, bad)[0, 1] < 0.5


def test_score_rows_matches_full_and_tolerance_positive():
    wl = inputs.workload(0)
    s = wl.signs()
    qrec, gq = oracle.quantize(wl.q_bf16(0, 0), s)
    krec, gk = oracle.quantize(wl.k_bf16(0, 0, rows=500), s)
    w = wl.w(0, 0)
    full, _ = oracle.score_full(qrec, gq, w, krec, gk, 500)
    rows = np.array([0, 7, 8, 123, 499])
    part, tol = oracle.score_rows(qrec, gq, w, krec, gk, rows)
    assert (part == full[rows]).all()
    assert (tol > 0).all()
    # the bound exceeds the largest possible fp32 rounding of the score itself
    assert (tol > np.abs(part) * 2e-7).all()


def test_mac_counts_reproduce_page_totals():
    per_key = 4096
    for name, keys, printed, sig in golden_rows("mac_counts.txt"):
        keys, printed, sig = int(keys), float(printed), int(sig)
        got = keys * per_key
        if sig == 0:
            assert got == printed, name
        else:  # the page rounds to `sig` significant figures
            assert float(f"{got:.{sig - 1}e}") == printed, (name, got, printed)
    # per key, counted by the oracle itself on a pooled Reindex layer
    wl = inputs.workload(0)
    s = wl.signs()
    qrec, gq = oracle.quantize(wl.q_bf16(0, 0), s)
    krec, gk = oracle.quantize(wl.k_bf16(0, 0, rows=16384), s)
    ids = np.arange(2048, dtype=np.int32)
    _, macs = oracle.score_pool(qrec, gq, wl.w(0, 0), krec, gk, 16384, ids, 2048)
    assert macs == 16384 * 4096  # ~6.7e7 per pooled layer


# ------------------------------------------------------------------- top-k --

def test_topk_brute_force_small():
    rng = np.random.default_rng(8)
    for n in range(0, 9):
        for trial in range(30):
            vals = rng.choice([-1.5, -0.0, 0.0, 0.25, 1.0, 2.0], n).astype(np.float32)
            for k in (1, 3, 8):
                idx, val = oracle.topk(vals, n, k)
                ref = sorted(range(n), key=lambda i: (-float(vals[i]), i))[:k]
                m = len(ref)
                assert list(idx[:m]) == ref
                assert (idx[m:] == -1).all() and np.isneginf(val[m:]).all()
                assert (val[:m] == vals[ref]).all()


def test_topk_all_equal_gives_lowest_indices():
    vals = np.full(5000, 3.25, dtype=np.float32)
    idx, _ = oracle.topk(vals, 5000, 512)
    assert (idx == np.arange(512)).all()


def test_topk_signed_zero_ties_by_index():
    vals = np.array([-0.0, 0.0, -0.0, -1.0], dtype=np.float32)
    idx, _ = oracle.topk(vals, 4, 3)
    assert list(idx) == [0, 1, 2]


# -------------------------------------------------------------------- pool --

def _check_pool_definition(scores, n_vis, bs, keep, ids, nk, npool, mask):
    nblk = -(-n_vis // bs)
    bval = np.full(nblk, -np.inf)
    for b in range(nblk):
        bval[b] = scores[b * bs:min(n_vis, b * bs + bs)].max()
    if n_vis:
        bval[(n_vis - 1) // bs] = np.inf
    K = set(ids[:nk].tolist())
    assert list(ids[:nk]) == sorted(K)
    assert nk == min(keep, nblk)
    if n_vis:
        assert (n_vis - 1) // bs in K
    for b in K:
        for c in set(range(nblk)) - K:
            assert (bval[b], -b) > (bval[c], -c)
    exp_mask = np.array([1 if (sidx // bs) in K else 0 for sidx in range(n_vis)], dtype=np.uint8)
    assert (mask == exp_mask).all()
    assert npool == exp_mask.sum()


def test_pool_brute_force_tiny():
    rng = np.random.default_rng(9)
    for bs in (1, 2, 3, 4):
        for keep in range(1, 9):
            for n_vis in (1, 2, 5, 9, 17, 33, 64):
                scores = rng.choice([-2.0, -1.0, 0.0, 0.5, 1.0, 3.0], n_vis).astype(np.float32)
                ids, nk, npool, mask = oracle.pool(scores, n_vis, bs, keep)
                _check_pool_definition(scores, n_vis, bs, keep, ids, nk, npool, mask)


def test_pool_page_figure_block4_keep6():
    rng = np.random.default_rng(10)
    scores = rng.standard_normal(60).astype(np.float32)
    ids, nk, npool, mask = oracle.pool(scores, 58, 4, 6)
    assert nk == 6 and npool <= 24
    _check_pool_definition(scores, 58, 4, 6, ids, nk, npool, mask)


def test_pool_short_context_keeps_everything():
    rng = np.random.default_rng(11)
    for n_vis in (1, 100, 16383, 16384):
        scores = rng.standard_normal(n_vis).astype(np.float32)
        ids, nk, npool, mask = oracle.pool(scores, n_vis)
        assert npool == n_vis and mask.all()
        assert nk == -(-n_vis // 8)


def test_pool_bound_pin_and_nesting():
    rng = np.random.default_rng(12)
    n_vis = 50001
    scores = rng.standard_normal(n_vis).astype(np.float32)
    ids, nk, npool, mask = oracle.pool(scores, n_vis)
    assert nk == 2048 and npool <= 16384
    assert (n_vis - 1) // 8 == ids[nk - 1]
    assert npool == 2047 * 8 + 1  # the pinned block holds only one visible position
    top, _ = oracle.topk(scores, n_vis, 512)
    assert mask[top].all()  # top-512 inside the pool inside the visible range


def test_pool_drops_minus_inf_blocks():
    scores = np.array([-np.inf] * 8 + [1.0] * 8 + [-np.inf] * 8 + [2.0], dtype=np.float32)
    ids, nk, npool, mask = oracle.pool(scores, 25, 8, 4)
    assert list(ids[:nk]) == [1, 3] and npool == 9


# ----------------------------------------------------------------- reindex --

def test_pooled_reindex_equals_page_masked_form():
    wl = inputs.workload(0)
    s = wl.signs()
    n_vis = 20003
    krec, gk = oracle.quantize(wl.k_bf16(0, 0, rows=n_vis), s)
    q0, g0 = oracle.quantize(wl.q_bf16(0, 0), s)
    q1, g1 = oracle.quantize(wl.q_bf16(1, 0), s)
    full0, _ = oracle.score_full(q0, g0, wl.w(0, 0), krec, gk, n_vis)
    ids, nk, npool, mask = oracle.pool(full0, n_vis)
    assert nk == 2048
    ps, _ = oracle.score_pool(q1, g1, wl.w(1, 0), krec, gk, n_vis, ids, nk)
    assert np.isneginf(ps[npool:]).all() and np.isfinite(ps[:npool]).all()
    idx, val = oracle.topk_pool(ps, npool, ids)
    full1, _ = oracle.score_full(q1, g1, wl.w(1, 0), krec, gk, n_vis)
    midx, mval = oracle.topk_masked(full1, n_vis, mask)
    assert (idx == midx).all() and (val == mval).all()
    assert mask[idx].all()


# --------------------------------------------------------------- generator --

def test_splitmix64_published_vector():
    G = 0x9E3779B97F4A7C15
    want = [int(r[0]) for r in golden_rows("splitmix64.txt")]
    got = [inputs.lib().gen_mix64((1234567 + G * (i + 1)) % (1 << 64)) for i in range(5)]
    assert got == want


def test_generator_normal_moments_and_determinism():
    a = inputs.bf16_to_f32(inputs.normal_bf16(0, 5, 400000)).astype(np.float64)
    assert abs(a.mean()) < 0.01 and abs(a.var() - 1) < 0.01
    assert abs(((a - a.mean()) ** 4).mean() / a.var() ** 2 - 3) < 0.05
    b = inputs.normal_bf16(0, 5, 1000, first=1000)
    assert (inputs.normal_bf16(0, 5, 2000)[1000:] == b).all()
    w = inputs.normal_f32(0, 6, 200000, sigma=(1 / 32) ** 0.5)
    assert abs(w.var() - 1 / 32) < 1e-3


def test_workload_recipes():
    w1 = inputs.workload(1)
    assert w1.B == 16 and all(4096 <= n <= 131072 for n in w1.seq_len)
    w4 = inputs.workload(4)
    assert w4.B == 8192 and w4.n_visible[0] == 122881 and w4.n_visible[-1] == 131072
    w2 = inputs.workload(2)
    assert w2.B == 64 and w2.seq_len[0] == 1 << 20 and w2.reindex_layers == 4
