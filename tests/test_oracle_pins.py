"""Pins for the CPU oracle (-m "not gpu").

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/*.json, each with its citation), closed forms,
invariants, an independent library (torch's float8_e5m2 and float16 casts), or
a brute-force float64 restatement written differently (explicit loops, complex
rotation, online softmax) on tiny inputs.  Each test names the mistake it
would catch.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
import synthetic as S

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ adaptive-range uint8 (P-5)
def test_u8_worked_example_from_page():
    """The page's worked example: min -1.2, max 2.8 -> scale ~0.0157, zp ~76.
    -min/scale is exactly 76.5 in fp32, so zp = 76 pins round-half-to-even
    (half-away would print 77)."""
    g = gold("adaptive_range_worked_example.json")
    seg = np.full(g["segment_tokens"], 0.5, np.float32)
    seg[0], seg[1] = np.float32(g["min"]), np.float32(g["max"])
    codes, scale, zp = O.u8_quantize(seg)
    assert round(float(scale), g["scale_printed_decimals"]) == g["scale_printed"]
    assert int(zp) == g["zero_point_printed"]
    assert float(np.float32(1.2) / scale) == 76.5  # the tie that decides the rounding rule
    assert codes[0] == 0                              # min maps to code 0
    assert codes[1] == 254                            # 178.5 rounds to even 178; 178 + 76


@pytest.mark.parametrize("seed", range(5))
def test_u8_roundtrip_bound(seed):
    """|x - x_hat| <= scale/2 (plus fp32 rounding) for every element; catches a
    wrong zero-point sign, an off-by-one in 255, or a dropped clamp."""
    x = S.outlier_f16(seed, 3, (128, 64)).astype(np.float32)
    codes, scale, zp = O.u8_quantize(x)
    xh = O.u8_dequantize(codes, scale, zp)
    err = np.abs(x - xh)
    assert err.max() <= float(scale) / 2 * (1 + 2 ** -20) + 4 * np.spacing(np.abs(x).max())
    assert codes.min() == 0 and codes.max() >= 254
    assert float(scale) == pytest.approx((x.max() - x.min()) / 255, rel=1e-6)


def test_u8_constant_segment():
    """max == min: scale 1, zp = round(-min); values come back exactly."""
    x = np.full((128, 8), -3.0, np.float32)
    codes, scale, zp = O.u8_quantize(x)
    assert float(scale) == 1.0 and int(zp) == 3
    assert np.all(O.u8_dequantize(codes, scale, zp) == x)


def test_u8_cache_tail_semantics():
    """Positions of an incomplete segment read back as fp16; the write that
    completes a segment quantises it (cache reads == u8 round trip)."""
    c = O.KVCache(1, 2, 8, 300, "u8")
    k = S.normal_f16(5, 1, (260, 2, 8), std=1.0)
    v = S.normal_f16(5, 2, (260, 2, 8), std=1.0)
    c.write(0, 0, k[:200], v[:200])
    # segment 0 complete, positions 128..199 are the tail
    np.testing.assert_array_equal(c.k[0][:, 128:200], k[128:200].astype(np.float32).transpose(1, 0, 2))
    codes, scale, zp = O.u8_quantize(k[:128, 1].astype(np.float32))
    np.testing.assert_array_equal(c.k[0][1, :128], O.u8_dequantize(codes, scale, zp))
    assert c.scale[0][0][1, 0] == scale and c.zp[0][0][1, 0] == zp
    for p in range(200, 256):
        c.write(0, p, k[p:p + 1], v[p:p + 1])
    codes, scale, zp = O.u8_quantize(v[128:256, 0].astype(np.float32))
    np.testing.assert_array_equal(c.v[0][0, 128:256], O.u8_dequantize(codes, scale, zp))


# ------------------------------------------------------------------ E5M2 (P-6)
def test_e5m2_all_fp16_patterns_vs_torch():
    """All 65,536 fp16 patterns: the oracle's bit-level RNE equals torch's
    float8_e5m2 cast wherever torch does not overflow (|x| <= 57344)."""
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = O.e5m2_from_f16_bits(bits)
    x16 = torch.from_numpy(bits.view(np.float16).copy())
    ref = x16.to(torch.float8_e5m2).view(torch.uint8).numpy()
    f = bits.view(np.float16).astype(np.float32)
    finite = np.isfinite(f) & (np.abs(f) <= 57344.0)
    np.testing.assert_array_equal(ours[finite], ref[finite])
    # NaN stays NaN, overflow and inf saturate to +-57344 (satfinite)
    back = O.e5m2_to_f16_bits(ours).view(np.float16).astype(np.float32)
    assert np.all(np.isnan(back[np.isnan(f)]))
    big = np.isfinite(f) & (np.abs(f) > 57344.0) | np.isinf(f)
    assert np.all(np.abs(back[big]) == 57344.0)
    assert np.all(np.sign(back[big]) == np.sign(f[big]))


def test_e5m2_range_from_page():
    g = gold("e5m2_range.json")
    assert O.E5M2_MAX == g["max_finite"]
    top = O.e5m2_to_f16_bits(np.array([0x7B], np.uint8)).view(np.float16)[0]
    assert float(top) == g["max_finite"]


def test_e5m2_ties_to_even():
    """1 + 2^-3 lies halfway between E5M2 neighbours 1 and 1.25: goes to even (1);
    1 + 3*2^-3 is halfway between 1.25 and 1.5: goes to even (1.5)."""
    v = np.array([1.125, 1.375, -1.125, 1.0 + 2 ** -10], np.float16)
    r = O.e5m2_round(v)
    np.testing.assert_array_equal(r, np.array([1.0, 1.5, -1.0, 1.0], np.float32))


# ------------------------------------------------------------------ scaled FP8 E5M2 cache (row F3)
def test_scaled_e5m2_first_slice_vs_torch():
    """Slice 0 is stored with the page's initial scales (K 0.0039, V 0.0042):
    each value reads back as e5m2(fp16(fp16(x) / s)) * s, with the fp16 and
    E5M2 roundings done by torch's casts instead of the oracle's encoder."""
    torch = pytest.importorskip("torch")
    H, h, n = 2, 8, 256
    k = S.normal_f16(41, 1, (n, H, h), 1.0)
    v = S.normal_f16(41, 2, (n, H, h), 3.0)
    c = O.KVCache(1, H, h, 512, "fp8_e5m2_scaled")
    c.write(0, 0, k, v)
    for which, x, s in ((0, k, 0.0039), (1, v, 0.0042)):
        t = torch.from_numpy(x.astype(np.float32))
        y = (t / torch.tensor(s, dtype=torch.float32)).to(torch.float16).to(torch.float8_e5m2)
        ref = (y.to(torch.float32) * torch.tensor(s, dtype=torch.float32)).numpy().transpose(1, 0, 2)
        got = (c.k if which == 0 else c.v)[0][:, :n]
        np.testing.assert_array_equal(got, ref)
    assert c.sc[0][0][0] == np.float32(0.0039) and c.sc[0][1][0] == np.float32(0.0042)


def test_scaled_e5m2_recalibration_hand_example():
    """Slice 0 holds a single nonzero K value 1.0: stored as e5m2(fp16(1 / 0.0039))
    = e5m2(256.5) = 256 (ties to even between 256 and 320), so the scale of slice
    1, fixed when position 256 is written, is 256 * 0.0039 / 127 in fp32; a
    slice of zeros keeps the scale before it (slice 2)."""
    H, h = 1, 4
    c = O.KVCache(1, H, h, 1024, "fp8_e5m2_scaled")
    k = np.zeros((256, H, h), np.float16)
    k[17, 0, 2] = 1.0
    c.write(0, 0, k, np.zeros_like(k))
    assert c.mcode[0][0][0] == np.float32(256.0)
    assert c.k[0][0, 17, 2] == np.float32(np.float32(256.0) * np.float32(0.0039))
    c.write(0, 256, np.zeros((256, H, h), np.float16), np.zeros((256, H, h), np.float16))
    s1 = np.float32(np.float32(np.float32(256.0) * np.float32(0.0039)) / np.float32(127.0))
    assert c.sc[0][0][1] == s1
    assert c.sc[0][1][1] == np.float32(0.0042)          # V slice 0 was all zero: the scale stays
    c.write(0, 512, np.ones((1, H, h), np.float16), np.ones((1, H, h), np.float16))
    assert c.sc[0][0][2] == s1                          # slice 1 was all zero: fallback
    assert c.k[0][0, 512, 0] == np.float32(1.0) or abs(c.k[0][0, 512, 0] - 1.0) <= 0.125


def test_scaled_e5m2_codec_closed_forms():
    """The scaled codec on values E5M2 holds exactly: 1.0 at scale 0.5 is stored as
    2.0 (code 0x40: sign 0, exponent 16, mantissa 0) and reads back as 1.0; -3.0
    at scale 0.25 is -12.0 (0xCA) and reads back as -3.0.  The next slice's scale
    maps the largest stored magnitude (in units of the previous scale) to 127:
    127 at scale 1 gives 1; a slice of zeros, or a non-finite maximum, keeps the
    previous scale."""
    c = O.e5m2s_quantize(np.array([1.0, -3.0], np.float16), np.float32(0.5))
    assert c[0] == 0x40
    c2 = O.e5m2s_quantize(np.array([-3.0], np.float16), np.float32(0.25))
    assert c2[0] == 0xCA
    assert O.e5m2s_dequantize(c[:1], np.float32(0.5))[0] == np.float32(1.0)
    assert O.e5m2s_dequantize(c2, np.float32(0.25))[0] == np.float32(-3.0)
    assert O.e5m2s_next_scale(127.0, np.float32(1.0)) == np.float32(1.0)
    assert O.e5m2s_next_scale(254.0, np.float32(0.5)) == np.float32(1.0)
    assert O.e5m2s_next_scale(0.0, np.float32(0.0039)) == np.float32(0.0039)
    assert O.e5m2s_next_scale(float("inf"), np.float32(0.0042)) == np.float32(0.0042)


def test_scaled_e5m2_round_trip_and_headroom():
    """Three slices whose magnitudes grow 4x per slice: every value reads back
    within E5M2's half step (2^-3 relative) of its fp16 value, and no code
    saturates (a scale maps the previous slice's largest value to 127, far
    below E5M2's 57344)."""
    H, h = 2, 16
    c = O.KVCache(1, H, h, 768, "fp8_e5m2_scaled")
    xs = [S.normal_f16(43, j, (256, H, h), 0.5 * 4.0 ** j) for j in range(3)]
    for j, x in enumerate(xs):
        c.write(0, 256 * j, x, x)
    got = c.k[0].transpose(1, 0, 2)
    ref = np.concatenate(xs).astype(np.float32)
    err = np.abs(got - ref)
    assert np.all(err <= 0.125 * np.abs(ref) + 1e-6)
    assert np.all(np.abs(O.e5m2_to_f16_bits(c.codes[0][0]).view(np.float16).astype(np.float32)) < 57344.0)
    assert c.sc[0][0][1] > 0 and c.sc[0][0][2] > c.sc[0][0][1]


def test_scaled_e5m2_byte_model_hand_count():
    """The 1.8B model over a 32,768-position scaled E5M2 cache at C = 32769: K and
    V of 16 heads x 128 one-byte codes per position and layer, plus one fp32
    scale per layer, K/V and attended 256-position slice (129 slices)."""
    w = S.WORKLOADS["1p8b_32k"].with_(kv_dtype="fp8_e5m2_scaled")
    assert O.decode_bytes_per_token(w, 32769)["kv"] == 25 * 2 * (32769 * 2048 + 4 * 129)


# ------------------------------------------------------------------ FP8 E4M3 weights (row F2)
def test_e4m3_all_codes_vs_torch():
    """Every one of the 256 E4M3 codes decodes to torch's float8_e4m3fn value
    (NaN where torch has NaN: S.1111.111)."""
    torch = pytest.importorskip("torch")
    b = np.arange(256, dtype=np.uint8)
    ours = O.e4m3_to_f32(b)
    ref = torch.from_numpy(b.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    np.testing.assert_array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert O.e4m3_to_f32(np.array([0x7E], np.uint8))[0] == O.E4M3_MAX == 448.0
    assert O.e4m3_to_f32(np.array([0x01], np.uint8))[0] == 2.0 ** -9      # smallest subnormal


def test_e4m3_encode_vs_torch_and_saturation():
    """fp32 -> E4M3 equals torch's round-to-nearest-even cast inside +-448;
    beyond it the encoder saturates (torch returns NaN there)."""
    torch = pytest.importorskip("torch")
    x = np.concatenate([S.normal_f32(21, 1, (200000,), std=60.0), S.normal_f32(21, 2, (100000,), std=0.01)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_from_f32(x), ref)
    sat = O.e4m3_from_f32(np.array([449.0, 1e6, -3000.0, np.inf], np.float32))
    np.testing.assert_array_equal(sat, np.array([0x7E, 0x7E, 0xFE, 0x7E], np.uint8))
    assert O.e4m3_from_f32(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_e4m3_ties_to_even():
    """1.0625 lies halfway between 1 (code 0x38) and 1.125 (0x39): even code, 1;
    1.1875 between 1.125 and 1.25 (0x3A): even code, 1.25."""
    r = O.e4m3_to_f32(O.e4m3_from_f32(np.array([1.0625, 1.1875, -1.0625], np.float32)))
    np.testing.assert_array_equal(r, np.array([1.0, 1.25, -1.0], np.float32))


def test_fp8_row_quantizer_bounds():
    """Row absmax maps to +-448 exactly; every weight is within half an E4M3
    step of its dequantised value (relative 2^-4 for normals, 2^-10 * s absolute
    for subnormals, plus the fp32 scale product); an all-zero row has s = 0."""
    w = S.normal_f32(22, 3, (64, 512), std=0.02).astype(np.float16)
    w[5] = 0
    codes, s = O.fp8_quantize_rows(w)
    assert s[5] == 0 and not codes[5].any()
    wf = w.astype(np.float32)
    rows = np.arange(64) != 5
    amax_idx = np.abs(wf).argmax(axis=1)
    top = codes[np.arange(64), amax_idx][rows]
    assert np.all((top & 0x7F) == 0x7E)
    back = O.fp8_dequantize_rows(codes, s)
    err = np.abs(back - wf)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, s[:, None] * 2.0 ** -10) * (1 + 1e-6) + 1e-12
    assert np.all(err <= bound)


def test_fp8_byte_model():
    """FP8 matrices cost one byte per weight plus a 4-byte scale per row."""
    w = S.WORKLOADS["1p8b_fp8"]
    b = O.decode_bytes_per_token(w, 1)["weights"]
    d, H, h, F, V, L = w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab, w.n_layers
    per_layer = (4 * d * H * h + 3 * F * d) + (3 * H * h + d + 2 * F + d) * 4 + 2 * d * 2
    assert b == L * per_layer + V * d + V * 4 + 2 * d * 2
    assert abs(b / O.decode_bytes_per_token(S.WORKLOADS["1p8b"], 1)["weights"] - 0.5) < 0.01


# ------------------------------------------------------------------ NVFP4 (E2M1 + E4M3 block scales)
# The E2M1 element of the OCP microscaling formats: sign, 2 exponent bits (bias
# 1), 1 mantissa bit; its eight magnitudes as the format publishes them.
E2M1_PUBLISHED = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_all_codes():
    """All 16 codes decode to the published magnitudes, the sign in bit 3."""
    vals = O.e2m1_to_f32(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(vals[:8], np.array(E2M1_PUBLISHED, np.float32))
    np.testing.assert_array_equal(vals[8:], -np.array(E2M1_PUBLISHED, np.float32))
    assert np.signbit(vals[8])


def test_e2m1_encode_brute_force():
    """Encoding equals an exhaustive nearest-value search (ties to the even
    code, beyond 6 saturating) on a grid holding every midpoint."""
    x = np.concatenate([np.arange(-7.0, 7.0001, 0.03125), [-100.0, 100.0, 6.5, -6.5]]).astype(np.float32)
    mags = np.array(E2M1_PUBLISHED)
    got = O.e2m1_from_f32(x)
    for xi, ci in zip(x.astype(np.float64), got):
        a = min(abs(xi), 6.0)
        dist = np.abs(mags - a)
        best = np.flatnonzero(dist == dist.min())
        code = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert (ci & 7) == code, (xi, ci)
        assert ((ci >> 3) & 1) == int(np.signbit(xi)), (xi, ci)


def test_e2m1_ties():
    """Midpoints go to the even code: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1,
    1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; 7 saturates to 6."""
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -5.0], np.float32)
    r = O.e2m1_to_f32(O.e2m1_from_f32(x))
    np.testing.assert_array_equal(r, np.array([0, 1, 1, 2, 2, 4, 4, 6, -4], np.float32))


def test_fp4_row_quantizer_bounds():
    """The block holding a row's absmax gets the largest E4M3 scale (448); every
    weight is within half the local E2M1 spacing of its dequantised value, in
    units of its block's scale times the row scale (saturation after the E4M3
    rounding of a block scale stays inside that bound); zero rows and zero
    blocks quantise to zero."""
    w = S.normal_f32(23, 4, (32, 256), std=0.02).astype(np.float16)
    w[3] = 0
    w[7, 16:32] = 0
    codes, bsc, rs = O.fp4_quantize_rows(w)
    assert rs[3] == 0 and not (codes[3] & 7).any()
    assert not (codes[7, 16:32] & 7).any()
    wf = w.astype(np.float32)
    rows = np.arange(32) != 3
    amax_block = np.abs(wf).argmax(axis=1) // 16
    assert np.all(O.e4m3_to_f32(bsc[np.arange(32), amax_block])[rows] == 448.0)
    back = O.fp4_dequantize_rows(codes, bsc, rs)
    unit = np.repeat(O.e4m3_to_f32(bsc) * rs[:, None], 16, axis=1)
    mags = np.array(E2M1_PUBLISHED)
    spacing = np.diff(mags)                                 # 0.5 0.5 0.5 0.5 1 1 2
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(unit > 0, np.abs(wf) / unit, 0.0)
    seg = np.clip(np.searchsorted(mags, q, side="right") - 1, 0, len(spacing) - 1)
    bound = 0.5 * spacing[seg] * unit * (1 + 1e-6) + 1e-12
    assert np.all(np.abs(back - wf) <= bound)


def test_fp4_byte_model():
    """NVFP4 matrices cost half a byte per weight, one scale byte per 16 weights
    and a 4-byte scale per row: 983,585,792 bytes for the 1.8B model."""
    w = S.WORKLOADS["1p8b"].with_(attn_wdtype="nvfp4", ffn_wdtype="nvfp4")
    n_weights = 25 * (4 * 2048 * 2048 + 3 * 2048 * 8192) + 32000 * 2048      # 1,743,257,600
    n_rows = 25 * (3 * 2048 + 2048 + 2 * 8192 + 2048) + 32000                 # 697,600
    gains_and_emb = 25 * 2 * 2048 * 2 + 2048 * 2 + 2048 * 2
    expect = n_weights // 2 + n_weights // 16 + n_rows * 4 + gains_and_emb
    assert expect == 983_585_792
    assert O.decode_bytes_per_token(w, 1)["weights"] == expect


# ------------------------------------------------------------------ fp16 rounding
def test_fp16_round_matches_torch_and_ties():
    torch = pytest.importorskip("torch")
    x = S.normal_f32(11, 1, (100000,), std=3.0)
    ours = O.fp16_round(x)
    ref = torch.from_numpy(x).to(torch.float16).to(torch.float32).numpy()
    np.testing.assert_array_equal(ours, ref)
    ties = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11], np.float32)
    np.testing.assert_array_equal(O.fp16_round(ties), np.array([1.0, 1 + 2 ** -9], np.float32))


# ------------------------------------------------------------------ INT4 (P-7)
def test_int4_hand_example():
    """absmax 0.7 -> s = fp16(0.1); codes round half to even."""
    w = np.zeros((1, 128), np.float16)
    w[0, :5] = [0.7, -0.7, 0.35, 0.25, -0.05]
    codes, s = O.int4_quantize_g128(w)
    s32 = float(s[0, 0])
    assert s32 == float(np.float16(np.float32(np.float16(0.7)) / np.float32(7)))
    expect = np.rint(w[0, :5].astype(np.float32) / np.float32(s32))
    np.testing.assert_array_equal(codes[0, :5], expect.astype(np.int8))
    assert codes[0, 0] == 7 and codes[0, 1] == -7
    assert np.all(codes[0, 5:] == 0)


def test_int4_bounds_and_zero_group():
    w = S.normal_f16(3, 4, (64, 512))
    w[3, 128:256] = 0
    codes, s = O.int4_quantize_g128(w)
    assert codes.min() >= -7 and codes.max() <= 7     # absmax/7 keeps |q| <= 7 (+-8 never used)
    assert np.all(codes[3, 128:256] == 0) and s[3, 1] == 0
    wd = O.int4_dequantize(codes, s)
    s_full = np.repeat(s.astype(np.float32), 128, axis=1)
    err = np.abs(w.astype(np.float32) - wd)
    # |w - q s| <= s/2 plus the fp16 rounding of s times |q| <= 7
    assert np.all(err <= s_full / 2 + 7 * s_full * 2 ** -11 + 1e-12)


# ------------------------------------------------------------------ RMSNorm (P-8)
def test_rmsnorm_closed_forms():
    c = np.float32(0.3)
    x = np.full(256, c, np.float32)
    g = np.linspace(0.5, 1.5, 256).astype(np.float32)
    y = O.rmsnorm(x, g, 1e-5)
    np.testing.assert_allclose(y, g * c / np.sqrt(c * c + 1e-5), rtol=1e-6)
    z = S.normal_f32(1, 1, (2048,), 5.0)
    yz = O.rmsnorm(z, np.ones(2048, np.float32), 0.0)
    assert float(np.sqrt(np.mean(yz.astype(np.float64) ** 2))) == pytest.approx(1.0, rel=1e-5)


# ------------------------------------------------------------------ RoPE (P-1)
def _rope_complex(x, p, theta):
    """Independent restatement: pair (i, i+h/2) as the complex number
    x_i + j x_{i+h/2}, multiplied by exp(j p theta^(-2i/h)), in complex128."""
    h = x.shape[-1]
    half = h // 2
    z = x[..., :half].astype(np.float64) + 1j * x[..., half:].astype(np.float64)
    ang = p * theta ** (-2.0 * np.arange(half) / h)
    r = z * np.exp(1j * ang)
    return np.concatenate([r.real, r.imag], axis=-1)


@pytest.mark.parametrize("p", [0, 1, 7, 1000, 32767])
def test_rope_vs_complex_rotation(p):
    x = S.normal_f32(2, 2, (4, 128), 1.0)
    c, s = O.rope_tables(128, [p], 10000.0)
    y = O.rope_apply(x, c, s)
    ref = _rope_complex(x, p, 10000.0)
    # the oracle rounds inv_freq and the angle to fp32 (the pinned reading); at
    # p = 32767 the fp32 angle differs from the exact one by up to ~2e-3 rad
    tol = 1e-5 + 4e-3 * (p >= 1000)
    np.testing.assert_allclose(y, ref, atol=tol * 4)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-6)
    if p == 0:
        np.testing.assert_array_equal(y, x)


def test_rope_frequencies_closed_form():
    """At p = 1 pair 0 turns by exactly 1 rad and pair h/4 by theta^(-1/2)."""
    c, s = O.rope_tables(128, [1], 10000.0)
    assert float(c[0, 0]) == pytest.approx(math.cos(1.0), abs=1e-7)
    assert float(s[0, 32]) == pytest.approx(math.sin(0.01), abs=1e-7)


def test_rope_relative_position():
    """<R(q,p), R(k,p')> depends only on p - p'."""
    q = S.normal_f32(3, 1, (1, 64), 1.0)
    k = S.normal_f32(3, 2, (1, 64), 1.0)
    def dot(p, pp):
        cq, sq = O.rope_tables(64, [p], 10000.0)
        ck, sk = O.rope_tables(64, [pp], 10000.0)
        return float(np.sum(O.rope_apply(q, cq, sq) * O.rope_apply(k, ck, sk)))
    assert dot(5, 2) == pytest.approx(dot(105, 102), abs=1e-4)
    assert dot(9, 9) == pytest.approx(float(np.sum(q * k)), abs=1e-5)


# ------------------------------------------------------------------ softmax / attention (P-2, P-3)
def test_softmax_invariants():
    s = S.normal_f32(4, 1, (8, 33), 4.0)
    a = O.softmax(s)
    np.testing.assert_allclose(a.sum(-1), 1.0, rtol=1e-6)
    np.testing.assert_allclose(O.softmax(s + 17.0), a, rtol=1e-5, atol=1e-7)
    np.testing.assert_allclose(O.softmax(np.array([0.0, math.log(3.0)], np.float32)), [0.25, 0.75], rtol=1e-6)


def test_silu_closed_forms():
    """silu(z) = z * sigmoid(z) (the SwiGLU gate): silu(0) = 0, silu(1) = e / (1 + e),
    silu(ln 3) = (3/4) ln 3, the odd-part identity silu(z) - silu(-z) = z, and the
    asymptotes silu(z) -> z (z >> 0) and -> 0 (z << 0).  A flipped exponent sign or
    a dropped factor fails the first three."""
    assert O.silu(np.float32(0.0)) == 0.0
    np.testing.assert_allclose(O.silu(np.float32(1.0)), math.e / (1.0 + math.e), rtol=1e-6)
    np.testing.assert_allclose(O.silu(np.float32(math.log(3.0))), 0.75 * math.log(3.0), rtol=1e-6)
    z = S.normal_f32(9, 0, (4096,), 3.0)
    np.testing.assert_allclose(O.silu(z) - O.silu(-z), z, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(O.silu(np.float32(40.0)), 40.0, rtol=1e-7)
    assert abs(float(O.silu(np.float32(-40.0)))) < 1e-15


def test_attention_single_key_and_equal_keys():
    q = S.normal_f32(5, 1, (3, 16), 1.0)
    K = S.normal_f32(5, 2, (3, 1, 16), 1.0)
    V = S.normal_f32(5, 3, (3, 1, 16), 1.0)
    np.testing.assert_array_equal(O.attention(q, K, V, 0.25), V[:, 0])
    K2 = np.repeat(K, 6, axis=1)
    V2 = S.normal_f32(5, 4, (3, 6, 16), 1.0)
    np.testing.assert_allclose(O.attention(q, K2, V2, 0.25), V2.mean(axis=1), rtol=1e-5, atol=1e-6)


def _attention_online_f64(q, K, V, scale):
    """Brute force, written as a single pass with a running max (the online
    form), in float64 — a different route to the same definition."""
    H, C, h = K.shape
    out = np.zeros((H, h))
    for hh in range(H):
        m, l, acc = -np.inf, 0.0, np.zeros(h)
        for j in range(C):
            s = float(np.dot(q[hh].astype(np.float64), K[hh, j].astype(np.float64))) * scale
            m_new = max(m, s)
            corr = math.exp(m - m_new) if m != -np.inf else 0.0
            e = math.exp(s - m_new)
            l = l * corr + e
            acc = acc * corr + e * V[hh, j].astype(np.float64)
            m = m_new
        out[hh] = acc / l
    return out


def test_attention_vs_online_brute_force():
    q = S.normal_f32(6, 1, (2, 8), 2.0)
    K = S.normal_f32(6, 2, (2, 9, 8), 2.0)
    V = S.normal_f32(6, 3, (2, 9, 8), 1.0)
    np.testing.assert_allclose(O.attention(q, K, V, 0.3), _attention_online_f64(q, K, V, 0.3), rtol=1e-5, atol=1e-6)


# ------------------------------------------------------------------ whole decoder (P-9)
MICRO = S.Workload("micro", 0, 2, 64, 2, 32, 128, 256, prompt_len=12, decode_steps=6)


def _decoder_f64(cfg, w, tokens):
    """Float64 brute force of the decoder, written with explicit per-head and
    per-position loops, complex RoPE and online softmax; keeps its own cache of
    fp16-rounded K/V (the storage format of an fp16 cache)."""
    L, d, H, h = cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.head_dim
    f = lambda a: np.asarray(a, np.float16).astype(np.float64)  # noqa: E731
    Kc = [[[] for _ in range(H)] for _ in range(L)]
    Vc = [[[] for _ in range(H)] for _ in range(L)]
    out = []
    def norm(x, g):
        return x * f(g) / math.sqrt(float(np.mean(x * x)) + cfg.rms_eps)
    for p, t in enumerate(tokens):
        x = f(w["tok_emb"][t])
        for l in range(L):
            lw = w["layers"][l]
            u = norm(x, lw["attn_norm"])
            q = f(lw["wq"]) @ u
            k = f(lw["wk"]) @ u
            v = f(lw["wv"]) @ u
            o = np.zeros(H * h)
            for hh in range(H):
                qh = _rope_complex(q[hh * h:(hh + 1) * h], p, cfg.rope_theta)
                kh = _rope_complex(k[hh * h:(hh + 1) * h], p, cfg.rope_theta)
                Kc[l][hh].append(np.float16(kh).astype(np.float64))
                Vc[l][hh].append(np.float16(v[hh * h:(hh + 1) * h]).astype(np.float64))
                o[hh * h:(hh + 1) * h] = _attention_online_f64(
                    qh[None], np.array(Kc[l][hh])[None], np.array(Vc[l][hh])[None], 1 / math.sqrt(h))[0]
            x = x + f(lw["wo"]) @ o
            u = norm(x, lw["ffn_norm"])
            gate = f(lw["w_gate"]) @ u
            act = gate / (1 + np.exp(-gate)) * (f(lw["w_up"]) @ u)
            x = x + f(lw["w_down"]) @ act
        out.append(f(w["lm_head"]) @ norm(x, w["final_norm"]))
    return np.array(out)


def test_decoder_vs_f64_brute_force():
    w = S.gen_weights(MICRO, seed=77)
    w["layers"][1]["attn_norm"] = S.normal_f16(9, 9, (64,), 0.5) + np.float16(1)  # non-unit gains
    toks = S.gen_prompt(MICRO, n=10, seed=78)
    ref = _decoder_f64(MICRO, w, toks)
    dec = O.OracleDecoder(MICRO, w, max_ctx=16)
    got = np.stack([dec.decode(int(t)) for t in toks])
    scale = np.abs(ref).max()
    assert np.abs(got - ref).max() <= 1e-4 * scale


def test_prefill_equals_stepwise_decode():
    w = S.gen_weights(MICRO, seed=79)
    toks = S.gen_prompt(MICRO, n=11, seed=80)
    for kv in ("fp16", "fp8_e5m2", "fp8_e5m2_scaled"):
        cfg = MICRO.with_(kv_dtype=kv)
        a = O.OracleDecoder(cfg, w, max_ctx=16)
        la = a.prefill(toks, q_block=4)
        b = O.OracleDecoder(cfg, w, max_ctx=16)
        for t in toks:
            lb = b.decode(int(t))
        np.testing.assert_allclose(la, lb, rtol=1e-4, atol=1e-4)
        # matmul vs matvec summation order can move a value across a rounding
        # boundary of the storage format: allow one step of that format, rarely
        ka, kb = a.cache.k[1], b.cache.k[1]
        step = 2.0 ** -10 if kv == "fp16" else 2.0 ** -2   # E5M2 (scaled or not): 2 mantissa bits
        diff = ka != kb
        assert diff.mean() < 0.01
        assert np.all(np.abs(ka - kb)[diff] <= step * np.abs(kb)[diff] + 1e-7)
        assert a.pos == b.pos == len(toks)


def test_greedy_chain_and_argmax_ties():
    assert O.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0], np.float32)) == 1
    w = S.gen_weights(MICRO, seed=81)
    d = O.OracleDecoder(MICRO, w, max_ctx=16)
    toks, logs = d.greedy(5, 4)
    d2 = O.OracleDecoder(MICRO, w, max_ctx=16)
    t = 5
    for i in range(4):
        lg = d2.decode(t)
        t = int(np.argmax(lg))
        assert t == toks[i]
        np.testing.assert_array_equal(lg, logs[i])


def test_int4_decoder_uses_dequantised_ffn():
    """With INT4 FFN the decoder equals an fp16-weight decoder whose FFN
    matrices are replaced by q * fp32(s) kept in fp32.  Those products need up
    to 14 significant bits, so rounding them to fp16 would lose precision (the
    Hunyuan page's section 5.2 lesson): check that the fp32 product is used."""
    cfg = S.Workload("micro4", 0, 1, 128, 2, 64, 256, 128, ffn_wdtype="int4_g128")
    w = S.gen_weights(cfg, seed=82)
    a = O.OracleDecoder(cfg, w, max_ctx=4)
    b = O.OracleDecoder(cfg.with_(ffn_wdtype="fp16"), w, max_ctx=4)
    lossy = False
    for k in ("w_gate", "w_up", "w_down"):
        codes, s = O.int4_quantize_g128(w["layers"][0][k])
        deq = O.int4_dequantize(codes, s)
        lossy |= bool(np.any(deq.astype(np.float16).astype(np.float32) != deq))
        b.layers[0][k] = deq
    assert lossy
    np.testing.assert_array_equal(a.decode(3), b.decode(3))


def test_int4_qkv_decoder_uses_dequantised_qkv_only():
    """With INT4 attention weights the decoder equals an fp16-weight decoder
    whose q, k and v matrices (and nothing else) are replaced by q * fp32(s) in
    fp32: the O projection and the LM head stay fp16 (xAI page, section 2.3:
    INT4 for the QKV projection; section 3.3 keeps lm_head fp16).  A planted
    INT4 O matrix must change the logits, so the check can tell the two apart."""
    cfg = S.Workload("micro4q", 0, 1, 128, 2, 64, 256, 128, attn_wdtype="int4_g128")
    w = S.gen_weights(cfg, seed=84)
    a = O.OracleDecoder(cfg, w, max_ctx=4)
    b = O.OracleDecoder(cfg.with_(attn_wdtype="fp16"), w, max_ctx=4)
    c = O.OracleDecoder(cfg.with_(attn_wdtype="fp16"), w, max_ctx=4)
    for k in ("wq", "wk", "wv"):
        b.layers[0][k] = c.layers[0][k] = O.int4_dequantize(*O.int4_quantize_g128(w["layers"][0][k]))
    c.layers[0]["wo"] = O.int4_dequantize(*O.int4_quantize_g128(w["layers"][0]["wo"]))
    la, lb, lc = a.decode(3), b.decode(3), c.decode(3)
    np.testing.assert_array_equal(la, lb)
    assert np.any(la != lc)
    np.testing.assert_array_equal(a.lm_head, w["lm_head"].astype(np.float32))


def test_int4_qkv_byte_model_hand_count():
    """The 1.8B model with INT4 q/k/v and FFN matrices and an E5M2 cache, per
    decode token, counted by hand: per layer 3 x 2048^2 INT4 q/k/v codes at half
    a byte (6,291,456 B) with one fp16 scale per 128 (196,608 B), the 2048^2 fp16
    O matrix (8,388,608 B), 3 x 8192 x 2048 INT4 FFN codes (25,165,824 B) with
    their scales (786,432 B) and two fp16 gain vectors (8,192 B); 25 layers; the
    32000 x 2048 fp16 LM head, the final gains and one embedding row; K and V of
    16 heads x 128 one-byte codes per position and layer."""
    w = S.WORKLOADS["1p8b_hpi"]
    b = O.decode_bytes_per_token(w, 2049)
    assert b["weights"] == 25 * 40_837_120 + 131_072_000 + 4_096 + 4_096 == 1_152_008_192
    assert b["kv"] == 25 * 4_096 * 2049


def test_fp8_decoder_matches_torch_quantised_weights():
    """With FP8 E4M3 weights the decoder equals an fp16-weight decoder whose
    matrices (q, k, v, o, gate, up, down and the LM head) are replaced by
    e4m3(w / s) * s, s = absmax(row) / 448 in fp32, with the E4M3 rounding done
    by torch's float8_e4m3fn cast instead of the oracle's own encoder."""
    torch = pytest.importorskip("torch")
    cfg = S.Workload("micro8", 0, 1, 128, 2, 64, 256, 160, ffn_wdtype="fp8_e4m3", attn_wdtype="fp8_e4m3")
    w = S.gen_weights(cfg, seed=83)
    a = O.OracleDecoder(cfg, w, max_ctx=4)
    b = O.OracleDecoder(cfg.with_(ffn_wdtype="fp16", attn_wdtype="fp16"), w, max_ctx=4)

    def torch_fp8(m16):
        wf = m16.astype(np.float32)
        s = (np.abs(wf).max(axis=1) / np.float32(448.0)).astype(np.float32)
        q = torch.from_numpy((wf / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).to(torch.float32)
        return (q.numpy() * s[:, None]).astype(np.float32)

    for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
        b.layers[0][k] = torch_fp8(w["layers"][0][k])
    b.lm_head = torch_fp8(w["lm_head"])
    for t in (3, 77, 5):
        np.testing.assert_array_equal(a.decode(t), b.decode(t))


def test_int4_byte_model_hand_count():
    """The 7B INT4 model's bytes per decode token, counted by hand: per layer
    4 x 4096^2 fp16 attention weights (134,217,728 B), 3 x 11008 x 4096 INT4
    codes at half a byte (67,633,152 B) with one fp16 scale per 128 (2,113,536 B)
    and two fp16 gain vectors (16,384 B); 32 layers; the 32000 x 4096 fp16 LM
    head, the final gains and one embedding row; K and V of 32 heads x 128 fp16
    per position and layer."""
    w = S.WORKLOADS["7b_int4"]
    b = O.decode_bytes_per_token(w, 4097)
    assert b["weights"] == 32 * 203_980_800 + 262_144_000 + 8_192 + 8_192 == 6_789_545_984
    assert b["kv"] == 524_288 * 4097


def test_u8_byte_model_hand_count():
    """The 1.8B uint8-cache model's KV bytes, counted by hand: at C = 8193 the
    64 complete 128-token segments are one byte per value (8192 x 16 x 128 B per
    layer, K and V), the open segment's one position stays fp16 (16 x 128 x 2 B)
    and each complete segment carries a fp32 scale and an int32 zero point per
    head (16 x 64 x 8 B); at C = 8320 segment 65 has just completed (65
    segments, no fp16 position)."""
    w = S.WORKLOADS["1p8b_u8"]
    assert O.decode_bytes_per_token(w, 8193)["kv"] == 25 * 2 * (16_777_216 + 4_096 + 8_192) == 839_475_200
    assert O.decode_bytes_per_token(w, 8320)["kv"] == 25 * 2 * (17_039_360 + 8_320) == 852_384_000
    assert O.decode_bytes_per_token(w, 8193)["weights"] == O.decode_bytes_per_token(S.WORKLOADS["1p8b"], 1)["weights"]


# ------------------------------------------------------------------ the bound (P-4) and shapes (P-12)
def test_kog_bound_arithmetic():
    g = gold("kog_bound_arithmetic.json")
    b = O.tokens_per_s_bound(g["h200_node_bandwidth"], g["fp16_2b_weights_bytes"])
    assert round(b, -2) == g["h200_ceiling_tok_s_printed"]
    b = O.tokens_per_s_bound(g["mi300x_node_bandwidth"], g["fp16_2b_weights_bytes"])
    assert round(b, -2) == g["mi300x_ceiling_tok_s_printed"]
    b = O.tokens_per_s_bound(g["h200_node_bandwidth"], g["fp4_moe_active_params"] * 0.5)
    assert round(b, -3) == g["fp4_ceiling_tok_s_printed"]
    us = 1e6 / g["budget_tok_s"]
    assert int(us) == g["budget_us_printed"]
    assert round(g["layers"] * 1.0 / us, 3) == g["one_us_per_layer_fraction_printed"]
    for kpl, ov, cap in zip(g["kernels_per_layer"], g["overhead_us_printed"], g["cap_tok_s_printed"]):
        o = g["launch_us"] * kpl * g["layers"]
        assert round(o) == ov or math.ceil(o) == ov
        assert round(1e6 / o, -1) == cap


def test_param_counts_and_bytes():
    def params(w):
        """Matrix parameters (norm gains excluded): ~1.8B and ~7B as named."""
        sh = S.weight_shapes(w)
        per_layer = sum(int(np.prod(sh[k])) for k in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"))
        return w.n_layers * per_layer + 2 * w.vocab * w.d_model
    assert params(S.WORKLOADS["1p8b"]) == 1_808_793_600
    assert params(S.WORKLOADS["7b_int4"]) == 6_738_149_376
    b = O.decode_bytes_per_token(S.WORKLOADS["1p8b"], 2048)
    assert b["kv"] == 204_800 * 2048
    assert abs(b["weights"] - 3.4867e9) < 1e6
