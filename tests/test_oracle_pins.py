"""Pins of the CPU oracle against facts that do not come from the oracle itself:
library conversions (torch, ml_dtypes), closed forms, rational-arithmetic
brute force, and invariants. No GPU needed."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4_moe_oracle as O
from nvfp4_w4a4_moe_permute_gb300 import inputs as IN

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
FMT = json.load(open(os.path.join(GOLDEN, "nvfp4_format.json")))

ml_dtypes = pytest.importorskip("ml_dtypes")


def _sweep_f32(n=400000, seed=1, hi=8.0):
    rng = np.random.default_rng(seed)
    a = rng.uniform(-hi, hi, n).astype(np.float32)
    # dense grid of exact quarter and eighth points (ties and near-ties)
    g = (np.arange(-64 * 8, 64 * 8 + 1) / 64.0).astype(np.float32)
    nxt = np.nextafter(g, np.float32(np.inf))
    prv = np.nextafter(g, np.float32(-np.inf))
    return np.concatenate([a, g, nxt, prv]).astype(np.float32)


# ---------------------------------------------------------------- BF16

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    a = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        rng.standard_normal(1000).astype(np.float32) * 1e-39,
                        np.array([0.0, -0.0, 1.0, 3.0e38, -3.0e38, 1 + 2 ** -8, 1 + 3 * 2 ** -8],
                                 dtype=np.float32)])
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16(a), ref)
    assert np.array_equal(O.bf16_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_f64_to_bf16_single_rounding():
    # 1 + 2^-8 + 2^-30: above the BF16 midpoint; a float32 detour would land on the
    # midpoint and round to even (1.0). One rounding must give 1 + 2^-7.
    v = np.array([1 + 2 ** -8 + 2 ** -30, -(1 + 2 ** -8 + 2 ** -30), 1 + 2 ** -8])
    out = O.bf16_to_f32(O.f64_to_bf16(v))
    assert out.tolist() == [1 + 2 ** -7, -(1 + 2 ** -7), 1.0]
    # agrees with the float32 path wherever the value is a float32
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(50000) * 100).astype(np.float32)
    assert np.array_equal(O.f64_to_bf16(a.astype(np.float64)), O.f32_to_bf16(a))


def test_f64_to_bf16_brute_force_rational():
    rng = np.random.default_rng(5)
    vals = rng.standard_normal(300) * np.exp2(rng.integers(-20, 20, 300))
    got = O.bf16_to_f32(O.f64_to_bf16(vals)).astype(np.float64)
    for v, g in zip(vals, got):
        fv = Fraction(float(v))
        e = math.floor(math.log2(abs(v)))
        q = Fraction(2) ** (e - 7)
        lo = (fv / q).__floor__()
        cands = [lo * q, (lo + 1) * q]
        d = [abs(fv - c) for c in cands]
        if d[0] < d[1]:
            best = cands[0]
        elif d[1] < d[0]:
            best = cands[1]
        else:
            best = cands[0] if lo % 2 == 0 else cands[1]
        assert Fraction(float(g)) == best


# ---------------------------------------------------------------- E2M1

def test_e2m1_all_16_codes_decode_to_grid():
    ref = np.arange(16, dtype=np.uint8).view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    got = O.e2m1_decode(np.arange(16))
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    assert np.array_equal(got, ref)
    assert sorted(set(np.abs(got).tolist())) == FMT["e2m1_magnitudes"]


@pytest.mark.parametrize("case", FMT["e2m1_ties"] + FMT["e2m1_saturation"] + FMT["e2m1_negative_underflow"])
def test_e2m1_golden_cases(case):
    v, code = case
    assert int(O.e2m1_rn(np.array([v], dtype=np.float32))[0]) == code


def test_e2m1_rounding_brute_force_and_ml_dtypes():
    a = _sweep_f32()
    got = O.e2m1_rn(a)
    # brute force: nearest grid magnitude by exhaustive distance, ties to even code
    mags = np.array(FMT["e2m1_magnitudes"])
    d = np.abs(np.abs(a.astype(np.float64))[:, None] - mags[None, :])
    best = d.min(axis=1)
    cand = d == best[:, None]
    even_pick = np.where(cand[:, ::2].any(axis=1),
                         np.argmax(cand & (np.arange(8) % 2 == 0), axis=1),
                         np.argmax(cand, axis=1))
    bf = even_pick | (np.signbit(a).astype(np.int64) << 3)
    assert np.array_equal(got, bf.astype(np.uint8))
    ref = a.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- E4M3

def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float32)
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert float(O.e4m3_decode(np.array([FMT["e4m3_max_code"]]))[0]) == FMT["e4m3_max"]


def test_e4m3_rounding_matches_libraries():
    rng = np.random.default_rng(2)
    vals = O.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    s = np.concatenate([
        np.exp2(rng.uniform(-14, 10, 300000)),
        mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9), vals,
        [0.0, 447.9, 448.0, 460.0, 464.0, 464.1, 1e6, 3e38],
    ]).astype(np.float32)
    got = O.e4m3_rn_satfinite(s)
    clamped = np.minimum(s, np.float32(448.0))
    ref = clamped.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    assert np.array_equal(got, ref)
    ref_t = torch.from_numpy(clamped).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref_t)


def test_block_scale_is_nearest_e4m3_of_amax_over_6():
    """scale = amax/6 * g before E4M3 rounding: the stored scale is the finite E4M3
    value nearest to that fp32 product (exhaustive search over all codes)."""
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-10, 10, (64, 1)))).astype(np.float32)
    codes, sf, g = O.quantize_per_row(x)
    amax_b = np.abs(x.reshape(64, 16, 16)).max(axis=2)
    s = ((amax_b / np.float32(6)) * g[:, None]).astype(np.float32).astype(np.float64)
    allv = O.e4m3_decode(np.arange(127, dtype=np.uint8)).astype(np.float64)
    d = np.abs(s[..., None] - allv)
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # ties go to the even code
    pick = np.where(cand.sum(-1) > 1, np.argmax(cand & (np.arange(127) % 2 == 0), axis=-1), np.argmax(cand, -1))
    assert np.array_equal(sf, pick.astype(np.uint8))


# ---------------------------------------------------------------- quantization

def test_exact_round_trip_on_scaled_grid():
    rng = np.random.default_rng(11)
    mags = np.array(FMT["e2m1_magnitudes"])
    for j in range(-20, 21, 5):
        R, C = 8, 128
        v = rng.choice(mags, size=(R, C)) * rng.choice([-1.0, 1.0], size=(R, C))
        v.reshape(R, C // 16, 16)[:, :, 3] = 6.0 * rng.choice([-1.0, 1.0], size=(R, C // 16))
        x = (v * 2.0 ** j).astype(np.float32)
        codes, sf, g = O.quantize_per_row(x)
        assert np.all(sf == FMT["e4m3_max_code"])
        assert np.array_equal(O.dequantize(codes, sf, g), x.astype(np.float64))


def test_dequant_error_bound():
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((256, 512)) * np.exp2(rng.integers(-8, 8, (256, 1)))).astype(np.float32)
    x[:, 7] *= 50  # outlier channel: many blocks far below the row max
    codes, sf, g = O.quantize_per_row(x)
    xh = O.dequantize(codes, sf, g)
    sfv = np.repeat(O.e4m3_decode(sf).astype(np.float64), 16, axis=1)
    enc = g.astype(np.float64)[:, None] / sfv
    v = np.abs(x.astype(np.float64) * enc)
    delta = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
    amax_b = np.repeat(np.abs(x).reshape(256, 32, 16).max(axis=2), 16, axis=1).astype(np.float64)
    s = amax_b / 6 * g.astype(np.float64)[:, None]
    normal = s >= 2.0 ** -6
    err = np.abs(x - xh)
    bound = (sfv / g[:, None]) * delta + 2.0 ** -20 * np.abs(x)
    assert np.all(err[normal] <= bound[normal])
    assert np.all(err[~normal] <= amax_b[~normal] * (1 + 2.0 ** -20))
    assert normal.mean() > 0.5


def test_row_max_gets_code_six_and_scale_448():
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((500, 64)) * np.exp2(rng.uniform(-30, 30, (500, 1)))).astype(np.float32)
    codes, sf, g = O.quantize_per_row(x)
    q = O.unpack_codes(codes)
    i = np.argmax(np.abs(x), axis=1)
    r = np.arange(500)
    assert np.all((q[r, i] & 7) == 7)
    assert np.all(sf[r, i // 16] == FMT["e4m3_max_code"])


def test_zero_and_denormal_rows():
    x = np.zeros((2, 32), dtype=np.float32)
    x[1, :4] = np.float32(1e-40)  # BF16-representable subnormal scale
    x[1, 5] = np.float32(-3e-40)
    codes, sf, g = O.quantize_per_row(x)
    assert np.all(codes[0] == 0) and np.all(sf[0] == 0) and g[0] == 1.0
    assert np.isfinite(g[1]) and g[1] == np.finfo(np.float32).max
    xh = O.dequantize(codes, sf, g)
    assert np.all(np.isfinite(xh))
    assert np.all(np.abs(xh[1] - x[1]) <= np.abs(x[1]).max())


def test_per_token_scaling_is_batch_invariant():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal((300, 256)) * np.exp2(rng.integers(-6, 6, (300, 1)))).astype(np.float32)
    c0, s0, g0 = O.quantize_per_row(x)
    p = rng.permutation(300)
    c1, s1, g1 = O.quantize_per_row(x[p])
    assert np.array_equal(c1, c0[p]) and np.array_equal(s1, s0[p]) and np.array_equal(g1, g0[p])
    # the same token embedded in a different batch
    other = (rng.standard_normal((50, 256)) * 1000).astype(np.float32)
    c2, s2, g2 = O.quantize_per_row(np.concatenate([other, x[:10]]))
    assert np.array_equal(c2[50:], c0[:10]) and np.array_equal(s2[50:], s0[:10])


def test_negative_control_tensor_wide_scale_depends_on_batch():
    """The invariance test above can fail: the tensor-wide policy changes a token's
    codes when a large-valued neighbour joins the batch."""
    rng = np.random.default_rng(15)
    x = rng.standard_normal((10, 256)).astype(np.float32)
    c0, s0, _ = O.quantize_tensor_wide_activations(x)
    other = (rng.standard_normal((5, 256)) * 1000).astype(np.float32)
    c1, s1, _ = O.quantize_tensor_wide_activations(np.concatenate([other, x]))
    assert not (np.array_equal(c1[5:], c0) and np.array_equal(s1[5:], s0))


# ---------------------------------------------------------------- SF layout

def test_sf_swizzle_matches_reshape_definition():
    rng = np.random.default_rng(16)
    for R, C16 in [(1, 4), (100, 8), (128, 4), (300, 128), (257, 48), (64, 3)]:
        sf = rng.integers(0, 127, (R, C16)).astype(np.uint8)
        Rp, Kc = O.roundup(R, 128), O.roundup(C16, 4)
        pad = np.zeros((Rp, Kc), dtype=np.uint8)
        pad[:R, :C16] = sf
        ref = pad.reshape(Rp // 128, 4, 32, Kc // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
        assert np.array_equal(O.swizzle_sf(sf), ref)
        assert np.array_equal(O.unswizzle_sf(ref, R, C16), sf)
    r, c = np.meshgrid(np.arange(256), np.arange(12), indexing="ij")
    offs = O.sf_swizzle_offset(r, c, 12).ravel()
    assert np.array_equal(np.sort(offs), np.arange(256 * 12))


# ---------------------------------------------------------------- permutation

def test_permute_brute_force():
    rng = np.random.default_rng(17)
    for trial in range(40):
        T, k, E = int(rng.integers(1, 40)), int(rng.integers(1, 5)), int(rng.integers(1, 9))
        ids = rng.integers(-1, E + 1, (T, k)).astype(np.int32)
        if trial % 3 == 0:
            ids = rng.integers(0, E, (T, k)).astype(np.int32)
        p = O.moe_permute(ids, E)
        pairs = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k) if 0 <= ids[t, j] < E)
        assert [t for _, t, _ in pairs] == p["perm_src"].tolist()
        assert [j for _, _, j in pairs] == p["perm_slot"].tolist()
        counts = [sum(1 for e2, _, _ in pairs if e2 == e) for e in range(E)]
        assert p["expert_offsets"].tolist() == [0] + list(np.cumsum(counts))
        assert p["sf_row_offsets"].tolist() == [0] + list(np.cumsum([(c + 127) // 128 * 128 for c in counts]))
        assert p["n_bad"] == T * k - len(pairs)
        for r, (e, t, j) in enumerate(pairs):
            assert p["dest_row"][t, j] == r
        bad = (ids < 0) | (ids >= E)
        assert np.all(p["dest_row"][bad] == -1)


def test_permute_quant_rows_are_token_quantizations():
    d = IN.make_moe_inputs("tiny")
    E = d["cfg"]["E"]
    pq = O.moe_permute_quant(d["x"], d["topk_ids"], d["topk_w"], E)
    xf = O.bf16_to_f32(d["x"])
    for r in [0, 5, 17, len(pq["perm_src"]) - 1]:
        c, s, g = O.quantize_per_row(xf[pq["perm_src"][r]][None])
        assert np.array_equal(pq["codes"][r], c[0]) and np.array_equal(pq["sf"][r], s[0])
        assert pq["row_g"][r] == g[0]
        assert pq["perm_w"][r] == d["topk_w"][pq["perm_src"][r], pq["perm_slot"][r]]
    # every expert region unswizzles back to its rows; padding bytes are zero
    kc = O.roundup(d["cfg"]["H"] // 16, 4)
    for e in range(E):
        a, b = pq["expert_offsets"][e], pq["expert_offsets"][e + 1]
        base = pq["sf_row_offsets"][e] * kc
        n = (pq["sf_row_offsets"][e + 1] - pq["sf_row_offsets"][e]) * kc
        reg = pq["sf_swizzled"][base:base + n]
        assert np.array_equal(O.unswizzle_sf(reg, b - a, d["cfg"]["H"] // 16), pq["sf"][a:b])
        mask = np.ones(n, dtype=bool)
        r, c = np.meshgrid(np.arange(b - a), np.arange(d["cfg"]["H"] // 16), indexing="ij")
        mask[O.sf_swizzle_offset(r, c, kc)] = False
        assert np.all(reg[mask] == 0)


# ---------------------------------------------------------------- grouped GEMM

def _exact_rational(a_codes, a_sf, a_g, b_codes, b_sf, b_g, off, m, n):
    e = int(np.searchsorted(off, m, side="right") - 1)
    K = a_codes.shape[1] * 2
    qa = O.unpack_codes(a_codes[m:m + 1])[0]
    qb = O.unpack_codes(b_codes[e][n:n + 1])[0]
    mags = [Fraction(v).limit_denominator(4) for v in FMT["e2m1_magnitudes"]]

    def val(c):
        v = mags[int(c) & 7]
        return -v if int(c) & 8 else v
    tot = Fraction(0)
    for kk in range(K):
        sa = Fraction(float(O.e4m3_decode(a_sf[m, kk // 16])))
        sb = Fraction(float(O.e4m3_decode(b_sf[e][n, kk // 16])))
        tot += val(qa[kk]) * sa * val(qb[kk]) * sb
    return tot / (Fraction(float(a_g[m])) * Fraction(float(b_g[e])))


def test_grouped_gemm_brute_force_rational():
    rng = np.random.default_rng(18)
    for trial in range(6):
        E, N, K = int(rng.integers(1, 4)), int(rng.integers(1, 8)), 64
        counts = rng.integers(0, 5, E)
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        M = int(off[-1])
        if M == 0:
            continue
        xa = (rng.standard_normal((M, K)) * 3).astype(np.float32)
        ac, asf, ag = O.quantize_per_row(xa)
        wb = (rng.standard_normal((E, N, K)) * 0.05).astype(np.float32)
        bq = [O.quantize_per_tensor(wb[e]) for e in range(E)]
        bc = np.stack([q[0] for q in bq]); bsf = np.stack([q[1] for q in bq])
        bg = np.array([q[2] for q in bq], dtype=np.float32)
        y, bound = O.grouped_gemm_exact(ac, asf, ag, bc, bsf, bg, off)
        for m in range(M):
            for n in range(N):
                ex = _exact_rational(ac, asf, ag, bc, bsf, bg, off, m, n)
                assert abs(Fraction(y[m, n]) - ex) <= abs(ex) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)
        assert np.all(bound >= np.abs(y))


def _exact_rational_abs(a_codes, a_sf, a_g, b_codes, b_sf, b_g, off, m, n):
    """sum_k |ahat_k * bhat_k| of output (m, n), in rational arithmetic."""
    e = int(np.searchsorted(off, m, side="right") - 1)
    K = a_codes.shape[1] * 2
    qa = O.unpack_codes(a_codes[m:m + 1])[0]
    qb = O.unpack_codes(b_codes[e][n:n + 1])[0]
    mags = [Fraction(v).limit_denominator(4) for v in FMT["e2m1_magnitudes"]]
    tot = Fraction(0)
    for kk in range(K):
        sa = Fraction(float(O.e4m3_decode(a_sf[m, kk // 16])))
        sb = Fraction(float(O.e4m3_decode(b_sf[e][n, kk // 16])))
        tot += mags[int(qa[kk]) & 7] * sa * mags[int(qb[kk]) & 7] * sb
    return tot / (Fraction(float(a_g[m])) * Fraction(float(b_g[e])))


def _f32_nearest(q: Fraction) -> float:
    """The float32 nearest to the rational q (ties to even), by integer arithmetic."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    m = q / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(n * ulp)


def _fp32_gemm_case(rng, counts, N, K):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M = int(off[-1])
    xa = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-4, 5, (M, 1)))).astype(np.float32)
    ac, asf, ag = O.quantize_per_row(xa)
    wb = (rng.standard_normal((len(counts), N, K)) * 0.05).astype(np.float32)
    bq = [O.quantize_per_tensor(wb[e]) for e in range(len(counts))]
    bc = np.stack([q[0] for q in bq]); bsf = np.stack([q[1] for q in bq])
    bg = np.array([q[2] for q in bq], dtype=np.float32)
    return ac, asf, ag, bc, bsf, bg, off


def _fp32_accumulate_bound(K):
    # each dequantized operand is one float32 rounding of an exact value (its
    # product with the other: two roundings), then K products are summed in
    # float32 in some order: at most (K + 1) further roundings per term
    u = 2.0 ** -24
    return (K + 2) * u * (1 + 2.0 ** -20)


def test_grouped_gemm_fp32_accumulate_brute_force_rational():
    """The float32-accumulate GEMM (the timed CPU baseline) lies within the
    float32 summation bound of the exact rational result, row by row and
    expert by expert (including empty experts)."""
    rng = np.random.default_rng(61)
    for trial in range(5):
        counts = rng.integers(0, 5, int(rng.integers(1, 4)))
        if counts.sum() == 0:
            counts[0] = 2
        N, K = int(rng.integers(1, 8)), 64 * int(rng.integers(1, 3))
        ac, asf, ag, bc, bsf, bg, off = _fp32_gemm_case(rng, counts, N, K)
        y = O.grouped_gemm_fp32_accumulate(ac, asf, ag, bc, bsf, bg, off)
        assert y.dtype == np.float32 and y.shape == (int(off[-1]), N)
        lim = _fp32_accumulate_bound(K)
        for m in range(int(off[-1])):
            for n in range(N):
                ex = _exact_rational(ac, asf, ag, bc, bsf, bg, off, m, n)
                ab = _exact_rational_abs(ac, asf, ag, bc, bsf, bg, off, m, n)
                assert abs(Fraction(float(y[m, n])) - ex) <= Fraction(lim) * ab


def test_grouped_gemm_fp32_accumulate_one_hot_weights_give_float32_dequantized_activations():
    """One-hot weight rows of value 1 (quantized exactly: code 6, scale 448,
    global scale 2688) make each output a single product, so the result is
    the float32 nearest to the exact dequantized activation."""
    rng = np.random.default_rng(62)
    M, K, N = 12, 128, 8
    xa = (rng.standard_normal((M, K)) * 3).astype(np.float32)
    ac, asf, ag = O.quantize_per_row(xa)
    cols = rng.choice(K, N, replace=False)
    w = np.zeros((1, N, K), dtype=np.float32)
    w[0, np.arange(N), cols] = 1.0
    bc, bsf, _, bg = O.quantize_weights(O.f32_to_bf16(w))
    assert bg[0] == 2688.0
    y = O.grouped_gemm_fp32_accumulate(ac, asf, ag, bc, bsf, bg, np.array([0, M], dtype=np.int32))
    mags = [Fraction(v).limit_denominator(4) for v in FMT["e2m1_magnitudes"]]
    q = O.unpack_codes(ac)
    for m in range(M):
        for j, c in enumerate(cols):
            v = mags[int(q[m, c]) & 7] * (-1 if int(q[m, c]) & 8 else 1)
            xh = v * Fraction(float(O.e4m3_decode(asf[m, c // 16]))) / Fraction(float(ag[m]))
            assert float(y[m, j]) == _f32_nearest(xh)


def test_grouped_gemm_fp32_accumulate_within_bound_of_exact_at_larger_sizes():
    """Several experts (one empty), K = 512: within the float32 summation bound
    of the pinned exact grouped GEMM."""
    rng = np.random.default_rng(63)
    ac, asf, ag, bc, bsf, bg, off = _fp32_gemm_case(rng, [37, 0, 80, 5], 48, 512)
    y = O.grouped_gemm_fp32_accumulate(ac, asf, ag, bc, bsf, bg, off)
    ex, ab = O.grouped_gemm_exact(ac, asf, ag, bc, bsf, bg, off)
    assert np.all(np.abs(y.astype(np.float64) - ex) <= _fp32_accumulate_bound(512) * ab + 1e-300)
    # and it is not the exact result computed in float64 under another name
    assert not np.array_equal(y.astype(np.float64), ex)


# ---------------------------------------------------------------- weight gradient

def _token_operand_case(rng, counts, C, spread=True):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = rng.standard_normal((int(off[-1]), C)).astype(np.float32)
    if spread:  # experts far apart in magnitude: a scale applied to the wrong range shows
        for e in range(len(counts)):
            x[off[e]:off[e + 1]] *= np.float32(2.0 ** (6 * e - 6))
    return O.bf16_to_f32(O.f32_to_bf16(x)), off  # BF16 values, as the operands are


def test_token_operand_equals_weight_quantization_of_each_padded_expert_block():
    rng = np.random.default_rng(41)
    x, off = _token_operand_case(rng, [3, 0, 260, 17], 48)
    q = O.quantize_tokens_per_expert(x, off)
    kofs = q["kofs"]
    assert list(kofs) == [0, 256, 256, 768, 1024]
    for e in range(4):
        a, b, k0, k1 = int(off[e]), int(off[e + 1]), int(kofs[e]), int(kofs[e + 1])
        if b == a:
            assert q["g"][e] == 1.0
            continue
        blk = np.zeros((k1 - k0, 48), dtype=np.float32)
        blk[:b - a] = x[a:b]
        wc, ws, _, wg = O.quantize_weights(_as_bf16_exact(blk)[None], along_rows=True)
        assert np.array_equal(q["codes"][:, k0 // 2:k1 // 2], wc[0])
        assert np.array_equal(q["sf"][:, k0 // 16:k1 // 16], ws[0])
        assert q["g"][e] == wg[0]
    # padding columns hold code 0 and scale 0
    assert np.all(q["codes"][:, (3 + 1) // 2:128] == 0) and np.all(q["sf"][:, 1:16] == 0)


def _as_bf16_exact(x):
    """BF16 bits of float32 values that are already BF16-representable."""
    b = O.f32_to_bf16(x)
    assert np.array_equal(O.bf16_to_f32(b), x)
    return b


def test_token_operand_round_trip_of_scaled_grid_values():
    rng = np.random.default_rng(42)
    mags = np.array(FMT["e2m1_magnitudes"])
    counts = [32, 0, 48, 16]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    M, C = int(off[-1]), 40
    v = rng.choice(mags, size=(M, C)) * rng.choice([-1.0, 1.0], size=(M, C))
    x = np.zeros((M, C))
    for e, j in enumerate([-9, 0, 4, 13]):
        a, b = off[e], off[e + 1]
        blk = v[a:b].copy()
        # every 16-token block of every channel holds a +-6, so every block scale is 448
        for t0 in range(0, b - a, 16):
            blk[t0 + 5, :] = 6.0 * rng.choice([-1.0, 1.0], size=C)
        x[a:b] = blk * 2.0 ** j
    x = x.astype(np.float32)
    q = O.quantize_tokens_per_expert(x, off)
    kofs = q["kofs"]
    for e in range(4):
        a, b, k0 = int(off[e]), int(off[e + 1]), int(kofs[e])
        if b == a:
            continue
        xh = O.dequantize(q["codes"][:, k0 // 2:(k0 + b - a) // 2], q["sf"][:, k0 // 16:(k0 + b - a) // 16],
                          np.full(C, q["g"][e]))
        assert np.array_equal(xh, x[a:b].T.astype(np.float64))


def _wgrad_rational(a, b, e, n, i):
    mags = [Fraction(v).limit_denominator(4) for v in FMT["e2m1_magnitudes"]]

    def val(c):
        v = mags[int(c) & 7]
        return -v if int(c) & 8 else v
    k0, k1 = int(a["kofs"][e]), int(a["kofs"][e + 1])
    qa = O.unpack_codes(a["codes"][n:n + 1])[0]
    qb = O.unpack_codes(b["codes"][i:i + 1])[0]
    tot = Fraction(0)
    for kk in range(k0, k1):
        sa = Fraction(float(O.e4m3_decode(a["sf"][n, kk // 16])))
        sb = Fraction(float(O.e4m3_decode(b["sf"][i, kk // 16])))
        tot += val(qa[kk]) * sa * val(qb[kk]) * sb
    return tot / (Fraction(float(a["g"][e])) * Fraction(float(b["g"][e])))


def test_wgrad_brute_force_rational():
    rng = np.random.default_rng(43)
    xa, off = _token_operand_case(rng, [5, 0, 20], 3)
    xb = rng.standard_normal((int(off[-1]), 4)).astype(np.float32) * 0.1
    qa = O.quantize_tokens_per_expert(xa, off)
    qb = O.quantize_tokens_per_expert(xb, off)
    out, bound = O.wgrad_exact(qa, qb)
    assert out.shape == (3, 3, 4)
    assert np.all(out[1] == 0)
    for e in (0, 2):
        for n in range(3):
            for i in range(4):
                ex = _wgrad_rational(qa, qb, e, n, i)
                assert abs(Fraction(out[e, n, i]) - ex) <= abs(ex) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 200)
    assert np.all(bound >= np.abs(out))


def test_wgrad_equals_matmul_of_dequantized_tokens():
    """Each expert's gradient is the product of its dequantized rows, the
    definition of dW = sum over the expert's tokens of a_t (x) b_t."""
    rng = np.random.default_rng(44)
    xa, off = _token_operand_case(rng, [70, 300, 1], 32)
    xb = rng.standard_normal((int(off[-1]), 24)).astype(np.float32)
    qa = O.quantize_tokens_per_expert(xa, off)
    qb = O.quantize_tokens_per_expert(xb, off)
    out, _ = O.wgrad_exact(qa, qb)
    kofs = qa["kofs"]
    for e in range(3):
        a, b, k0 = int(off[e]), int(off[e + 1]), int(kofs[e])
        da = O.dequantize(qa["codes"][:, k0 // 2:(k0 + 256 * ((b - a + 255) // 256)) // 2],
                          qa["sf"][:, k0 // 16:(k0 + 256 * ((b - a + 255) // 256)) // 16], np.full(32, qa["g"][e]))
        db = O.dequantize(qb["codes"][:, k0 // 2:(k0 + 256 * ((b - a + 255) // 256)) // 2],
                          qb["sf"][:, k0 // 16:(k0 + 256 * ((b - a + 255) // 256)) // 16], np.full(24, qb["g"][e]))
        ref = da @ db.T
        assert np.allclose(out[e], ref, rtol=1e-12, atol=1e-300)
        # and the quantized gradient is close to the unquantized one
        exact = xa[a:b].astype(np.float64).T @ xb[a:b].astype(np.float64)
        assert np.linalg.norm(out[e] - exact) <= 0.25 * np.linalg.norm(exact)


def test_grouped_gemm_one_hot_weights_gather():
    """One-hot weight rows (each row selects column c with value 6 on a grid-exact
    quantization) make row n of the output equal xhat[:, c]."""
    rng = np.random.default_rng(19)
    M, K, N = 40, 128, 16
    xa = rng.standard_normal((M, K)).astype(np.float32)
    ac, asf, ag = O.quantize_per_row(xa)
    cols = rng.choice(K, N, replace=False)
    w = np.zeros((1, N, K), dtype=np.float32)
    w[0, np.arange(N), cols] = 6.0
    bc, bsf, _, bg = O.quantize_weights(O.f32_to_bf16(w))
    y, _ = O.grouped_gemm_exact(ac, asf, ag, bc, bsf, bg, np.array([0, M], dtype=np.int32))
    # the weight block holding the 6 gets scale 448 and global scale 2688/6 = 448
    assert bg[0] == 448.0
    xh = O.dequantize(ac, asf, ag)
    assert np.allclose(y, 6.0 * xh[:, cols], rtol=2.0 ** -50, atol=0)


def test_grouped_gemm_dense_case_equals_matmul_of_dequantized():
    rng = np.random.default_rng(20)
    M, N, K = 50, 24, 256
    xa = rng.standard_normal((M, K)).astype(np.float32)
    wb = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    ac, asf, ag = O.quantize_per_row(xa)
    bc, bsf, bg = O.quantize_per_tensor(wb)
    y, _ = O.grouped_gemm_exact(ac, asf, ag, bc[None], bsf[None], np.array([bg]), np.array([0, M]))
    ref = O.dequantize(ac, asf, ag) @ O.dequantize(bc, bsf, bg).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- SwiGLU exp

def _ulp_err_f32(got, ref64):
    ref32 = ref64.astype(np.float32)
    ulp = np.spacing(np.abs(ref32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - ref64) / ulp


def test_exp_spec_within_two_ulp():
    x = np.concatenate([np.linspace(-87, 88, 2_000_001, dtype=np.float32),
                        np.array([0.0, -0.0, 1e-8, -1e-8, 0.5, -0.5], dtype=np.float32)])
    got = O.exp_spec(x)
    ref = np.exp(x.astype(np.float64))
    assert np.max(_ulp_err_f32(got, ref)) <= 2.0
    assert O.exp_spec(np.array([0.0], dtype=np.float32))[0] == 1.0
    # clamping keeps every result finite
    assert np.all(np.isfinite(O.exp_spec(np.array([-1e30, 1e30, -100, 100], dtype=np.float32))))


def test_swiglu_matches_float64_formula():
    rng = np.random.default_rng(21)
    gu = (rng.standard_normal((64, 256)) * 4).astype(np.float32)
    w = rng.uniform(0, 1, 64).astype(np.float32)
    h = O.swiglu_weighted(gu, w)
    g, u = gu[:, :128].astype(np.float64), gu[:, 128:].astype(np.float64)
    ref = g / (1 + np.exp(-g)) * u * w[:, None]
    assert np.max(_ulp_err_f32(h, ref)) <= 6.0


def test_swiglu_backward_is_the_derivative_of_the_forward():
    """Central differences of the float64 forward h = g/(1+e^-g) * u * w
    (independent of the closed form typed in the oracle) against dg, and the
    float64 silu against du."""
    rng = np.random.default_rng(23)
    M, I = 48, 64
    gu = (rng.standard_normal((M, 2 * I)) * 3).astype(np.float32)
    dh = rng.standard_normal((M, I)).astype(np.float32)
    w = rng.uniform(0.1, 1, M).astype(np.float32)
    out = O.swiglu_backward(gu, dh, w)
    g, u = gu[:, :I].astype(np.float64), gu[:, I:].astype(np.float64)
    wd = w.astype(np.float64)[:, None]
    f = lambda gg: gg / (1 + np.exp(-gg)) * u * wd  # noqa: E731
    eps = 1e-6 * np.maximum(1.0, np.abs(g))
    dg_fd = dh.astype(np.float64) * (f(g + eps) - f(g - eps)) / (2 * eps)
    scale = np.abs(dh.astype(np.float64) * u * wd) + 1e-30
    assert np.max(np.abs(out[:, :I] - dg_fd) / scale) < 2e-5
    du_ref = dh.astype(np.float64) * (g / (1 + np.exp(-g))) * wd
    assert np.max(_ulp_err_f32(out[:, I:], du_ref)) <= 8.0


def test_swiglu_backward_special_gates():
    """g = 0: silu' = 1/2 exactly and du = 0; g = +-30: silu' -> 1 and -> 0."""
    I = 4
    g = np.array([[0.0, 0.0, 30.0, -30.0]], dtype=np.float32)
    u = np.array([[1.5, -2.0, 1.0, 1.0]], dtype=np.float32)
    dh = np.array([[1.0, 3.0, 2.0, 2.0]], dtype=np.float32)
    out = O.swiglu_backward(np.concatenate([g, u], axis=1), dh, None)
    assert out[0, 0] == np.float32(0.75) and out[0, 1] == np.float32(-3.0)
    assert out[0, I] == 0.0 and out[0, I + 1] == 0.0
    assert abs(out[0, 2] - 2.0) < 1e-5 and abs(out[0, 3]) < 1e-9
    assert abs(out[0, I + 2] - 60.0) < 1e-4 and abs(out[0, I + 3]) < 1e-9


# ---------------------------------------------------------------- combine

def test_combine_exact_cases():
    rng = np.random.default_rng(22)
    T, k, N = 30, 4, 64
    M = T * k
    D = rng.integers(-100, 100, (M, N)).astype(np.float32)
    perm = rng.permutation(M).reshape(T, k).astype(np.int32)
    perm[0, 1] = -1  # a dropped pair
    y = O.bf16_to_f32(O.moe_combine(O.f32_to_bf16(D), perm))
    ref = np.zeros((T, N))
    for t in range(T):
        for j in range(k):
            if perm[t, j] >= 0:
                ref[t] += D[perm[t, j]]
    assert np.array_equal(O.bf16_to_f32(O.f32_to_bf16(ref.astype(np.float32))), y)
    y1 = O.moe_combine(O.f32_to_bf16(D), perm[:, :1].copy())
    assert np.array_equal(y1[1:], O.f32_to_bf16(D)[perm[1:, 0]])


def test_combine_random_within_one_bf16_ulp_of_exact_sum():
    rng = np.random.default_rng(23)
    T, k, N = 40, 8, 128
    D = O.f32_to_bf16(rng.standard_normal((T * k, N)).astype(np.float32))
    perm = rng.permutation(T * k).reshape(T, k).astype(np.int32)
    y = O.bf16_to_f32(O.moe_combine(D, perm)).astype(np.float64)
    ref = O.bf16_to_f32(D).astype(np.float64)[perm].sum(axis=1)
    ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) * 2 ** 16
    assert np.all(np.abs(y - ref) <= ulp + 2 ** -30)


# ---------------------------------------------------------------- weights

def test_weight_orientations_share_global_scale():
    rng = np.random.default_rng(24)
    w = O.f32_to_bf16((rng.standard_normal((3, 64, 96)) * 0.02).astype(np.float32))
    c0, s0, sw0, g0 = O.quantize_weights(w)
    c1, s1, sw1, g1 = O.quantize_weights(w, along_rows=True)
    assert np.array_equal(g0, g1)
    assert c0.shape == (3, 64, 48) and c1.shape == (3, 96, 32)
    wf = O.bf16_to_f32(w)
    for e in range(3):
        c, s, g = O.quantize_per_tensor(wf[e].T.copy(), g0[e])
        assert np.array_equal(c, c1[e]) and np.array_equal(s, s1[e])


def test_tiny_chain_runs_and_is_finite():
    d = IN.make_moe_inputs("tiny")
    E = d["cfg"]["E"]
    wgu = O.quantize_weights(d["w_gate_up"])
    wd = O.quantize_weights(d["w_down"])
    out = O.moe_mlp_forward(d["x"], d["topk_ids"], d["topk_w"], E, wgu, wd)
    y = O.bf16_to_f32(out["y"])
    assert y.shape == (64, 64) and np.all(np.isfinite(y))
    assert np.abs(y).max() > 0
