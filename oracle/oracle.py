"""Plain fp32 CPU restatement of the batch-1 decode step (TEST INFRASTRUCTURE ONLY).

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use this module.  It shares nothing with the CUDA engine.

Pages cited (titles as published):
  [Kog]     "Real-time LLM inference on standard GPUs: 3,000 tokens/s per request"
            (Kog Inference Engine blog) — sections "Memory bandwidth is the main
            bottleneck ..." (the bound tokens/s <= BW / (beta*W + KV)) and
            "Where standard inference stacks lose microseconds" (table rows
            "kernel boundaries", "CPU scheduling and sampling", "non-GEMM work").
  [xAI]     "How the xAI team pushed Grok Bot latency down to milliseconds"
            — section 2.3 (hybrid precision: INT4 W4A16 FFN, FP8-E5M2 KV cache
            dequantised to fp16 on load), section 3.3 (hpi_config: int4,
            group_size 128, symmetric), section 4.3 (E5M2 range +-57344).
  [Grok3]   "Grok-3 v3.2.4 hot-update deep dive" — section 3.2 (adaptive-range
            quantisation: per-128-token segment min/max -> scale, zero-point;
            worked example min -1.2, max 2.8 -> scale ~0.0157, zero-point ~76).
  [Hunyuan] Hunyuan serving re-architecture — section 5.2 (INT4 dequant: keep the
            scale product in fp32, round once at the end).
  [Kog] also, section "Memory bandwidth is the main bottleneck": an FP16 weight
            is 2 bytes for one multiply-add (~1 FLOP/byte), FP8 ~2, FP4 ~4 —
            the FP8 weight format below (E4M3, one fp32 scale per output row)
            and the NVFP4 format (E2M1, E4M3 scale per 16 columns, fp32 scale
            per row) are this module's readings; the page names only the byte
            width.

The decoder itself (RMSNorm, RoPE, SwiGLU, MHA, untied LM head) is fixed by the
workload description, not by the pages; where the pages leave a step open this
module takes the plain LLaMA-style reading listed below and in the design notes:
  - pre-norm RMSNorm, y = x * g / sqrt(mean(x^2) + eps), eps inside the root;
  - RoPE with half-split pairing (i, i + h/2), inv_freq_i = theta^(-2i/h);
  - attention scale 1/sqrt(h); decode attends to positions 0..p inclusive,
    the new K/V being written (through the cache's storage format) first;
  - SwiGLU: down(silu(gate u) * (up u)), silu(z) = z / (1 + e^-z);
  - argmax: lowest index on exact ties;
  - round-half-to-even wherever a value is rounded (pinned by [Grok3] 3.2's
    zero-point 76 for -min/scale = 76.5).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32

# ----------------------------------------------------------------------------------------------
# Storage formats
# ----------------------------------------------------------------------------------------------


def fp16_round(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 (round to nearest even) -> fp32: the fp16 KV cache and fp16
    weight storage ([xAI] 2.3: activations and cache are fp16 by default)."""
    return np.asarray(x, dtype=F32).astype(np.float16).astype(F32)


E5M2_MAX = 57344.0  # [xAI] 4.3: E5M2 covers +-57344


def e5m2_from_f16_bits(b16: np.ndarray) -> np.ndarray:
    """fp16 bit patterns -> FP8 E5M2 bytes, round to nearest even, saturating to
    +-57344 ([xAI] 2.3 stores K/V as E5M2; [xAI] 4.3 gives its range).

    E5M2 has the fp16 exponent field, so the conversion keeps the top byte and
    rounds away the low 8 mantissa bits.  NaN maps to a quiet NaN with the
    input's sign (sign | 0x7F); +-inf and finite overflow saturate to +-max."""
    b = np.asarray(b16, dtype=np.uint16).astype(np.uint32)
    sign = (b >> 15) & 1
    mag = b & 0x7FFF
    hi = mag >> 8
    lo = mag & 0xFF
    round_up = (lo > 0x80) | ((lo == 0x80) & ((hi & 1) == 1))
    r = hi + round_up.astype(np.uint32)
    is_nan = mag > 0x7C00
    is_inf = mag == 0x7C00
    r = np.where(r >= 0x7C, 0x7B, r)            # overflow (incl. inf) saturates to 57344
    r = np.where(is_inf, 0x7B, r)
    r = np.where(is_nan, 0x7F, r)
    return ((sign << 7) | r).astype(np.uint8)


def e5m2_to_f16_bits(b8: np.ndarray) -> np.ndarray:
    """E5M2 byte -> fp16 bits (exact: the byte is the fp16 top byte)."""
    return (np.asarray(b8, dtype=np.uint8).astype(np.uint16) << 8).astype(np.uint16)


def e5m2_round(x_f16: np.ndarray) -> np.ndarray:
    """fp16 values -> E5M2 -> fp16 -> fp32: the value an E5M2 cache returns when
    dequantised to fp16 on load ([xAI] 2.3)."""
    bits = np.asarray(x_f16, dtype=np.float16).view(np.uint16)
    return e5m2_to_f16_bits(e5m2_from_f16_bits(bits)).view(np.float16).astype(F32)


SEG = 128  # [Grok3] 3.2: "each 128-token segment", 128 found optimal

# Scaled FP8 E5M2 cache ([xAI] 3.3): per-tensor scales in hpi_config (k_cache
# 0.0039, v_cache 0.0042), recomputed every 256 tokens from the current cache
# slice; the scale maps the slice's largest magnitude to 127 ([xAI] 4.3's
# max|k| / 127).
KV_SLICE = 256
KV_SCALE0 = (0.0039, 0.0042)   # K, V: the scales slice 0 is stored with
KV_SCALE_TARGET = 127.0


def e5m2s_quantize(x16: np.ndarray, s) -> np.ndarray:
    """Scaled E5M2 codes of fp16 values with scale s: the fp16 value divided by
    s in fp32, rounded to fp16, then to E5M2 (round to nearest even,
    saturating) - the unscaled cache's fp16 -> E5M2 step applied to x / s."""
    y = (np.asarray(x16, dtype=np.float16).astype(F32) / F32(s)).astype(np.float16)
    return e5m2_from_f16_bits(y.view(np.uint16))


def e5m2s_dequantize(codes: np.ndarray, s) -> np.ndarray:
    """The value a scaled E5M2 cache returns: E5M2 -> fp16 (exact) -> fp32, times s."""
    return (e5m2_to_f16_bits(codes).view(np.float16).astype(F32) * F32(s)).astype(F32)


def e5m2s_next_scale(max_code: float, s_prev) -> np.float32:
    """Scale of slice j from slice j-1 (its scale s_prev and the largest
    magnitude max_code among its stored E5M2 values): the slice's largest
    dequantised magnitude max_code * s_prev, mapped to 127.  A slice with no
    usable magnitude (all zero, or not finite) keeps the previous scale (the
    page keeps recent scales as the fallback)."""
    amax = F32(F32(max_code) * F32(s_prev))
    if not np.isfinite(amax) or amax <= 0:
        return F32(s_prev)
    return F32(amax / F32(KV_SCALE_TARGET))


def u8_quantize(x: np.ndarray):
    """Adaptive-range uint8 quantisation of one segment ([Grok3] 3.2).

    x: the segment's values (any shape, fp16-representable), read as fp32.
    scale = (max - min) / 255 and zero_point = round(-min / scale), both in fp32
    (IEEE division), round = half-to-even; codes = clamp(round(x / scale) + zp,
    0, 255).  A constant segment (max == min) would divide by zero: it uses
    scale = 1 and zp = round(-min) instead.  zp is kept as an unclamped int32.
    Returns (codes uint8, scale float32, zp int32)."""
    xf = np.asarray(x, dtype=F32)
    mn = F32(xf.min())
    mx = F32(xf.max())
    if mx == mn:
        scale = F32(1.0)
        zp = np.int32(np.rint(-mn))
    else:
        scale = F32((mx - mn) / F32(255.0))
        zp = np.int32(np.rint(F32(-mn) / scale))
    q = np.rint(xf / scale).astype(np.int64) + int(zp)
    codes = np.clip(q, 0, 255).astype(np.uint8)
    return codes, scale, zp


def u8_dequantize(codes: np.ndarray, scale, zp) -> np.ndarray:
    """x_hat = (code - zp) * scale in fp32 ([Grok3] 3.2)."""
    return (np.asarray(codes, dtype=np.int64) - int(zp)).astype(F32) * F32(scale)


E4M3_MAX = 448.0  # largest finite FP8 E4M3 value (the variant without infinities)


def _e4m3_table() -> np.ndarray:
    """Values of the non-negative finite E4M3 codes 0x00..0x7E (float64, exact):
    code = eeee.mmm, e = 0 subnormal m/8 * 2^-6, else (1 + m/8) * 2^(e-7)."""
    c = np.arange(0x7F)
    e, m = c >> 3, c & 7
    return np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))


def e4m3_to_f32(b8: np.ndarray) -> np.ndarray:
    """FP8 E4M3 bytes -> fp32 (exact).  S.1111.111 is NaN; there is no infinity."""
    b = np.asarray(b8, dtype=np.uint8).astype(np.int64)
    mag = b & 0x7F
    val = np.where(mag == 0x7F, np.nan, _e4m3_table()[np.minimum(mag, 0x7E)])
    return np.where(b & 0x80, -val, val).astype(F32)


def e4m3_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> FP8 E4M3 bytes: the nearest representable value, ties to the even
    code, magnitudes beyond 448 saturating to +-448, NaN -> sign | 0x7F."""
    xf = np.asarray(x, dtype=F32).astype(np.float64)
    t = _e4m3_table()
    a = np.abs(xf)
    hi = np.clip(np.searchsorted(t, a, side="left"), 0, len(t) - 1)   # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - t[lo], t[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= t[-1], 0x7E, code)            # saturate (satfinite)
    code = np.where(np.isnan(xf), 0x7F, code)
    sign = np.signbit(xf).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def fp8_quantize_rows(w: np.ndarray):
    """FP8 E4M3 weights with one scale per output row (this module's reading of
    [Kog]'s "FP8 ~2 FLOP/byte"): s = absmax(row) / 448 in fp32, codes =
    e4m3(w / s) with the division in fp32, rounding to nearest even and
    saturation at +-448; an all-zero row gets s = 0 and codes 0.  Returns
    (codes uint8 [rows, cols], scales fp32 [rows])."""
    wf = np.asarray(w, dtype=np.float16).astype(F32)
    absmax = np.abs(wf).max(axis=1)
    s = (absmax / F32(E4M3_MAX)).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s[:, None] > 0, wf / s[:, None], F32(0.0)).astype(F32)
    return e4m3_from_f32(q), s


def fp8_dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """w' = e4m3(code) * s in fp32."""
    return (e4m3_to_f32(codes) * np.asarray(scales, dtype=F32)[:, None]).astype(F32)


# NVFP4 weights (this module's reading of [Kog]'s "FP4 ~4 FLOP/byte" for a
# Blackwell GPU, whose native 4-bit format is E2M1 with one FP8 E4M3 scale per
# block of 16 values): E2M1 codes, an E4M3 scale per 16 consecutive input
# columns of a row, and one fp32 scale per output row chosen so that the row's
# largest block scale is 448 (the largest E4M3 value).
E2M1_MAX = 6.0    # largest E2M1 magnitude
FP4_BLOCK = 16    # input columns sharing one E4M3 block scale


def _e2m1_table() -> np.ndarray:
    """Magnitudes of the E2M1 codes 0..7 (float64, exact): code = ee.m,
    e = 0 subnormal m/2, else (1 + m/2) * 2^(e-1): 0, 0.5, 1, 1.5, 2, 3, 4, 6."""
    c = np.arange(8)
    e, m = c >> 1, c & 1
    return np.where(e == 0, m / 2.0, (1.0 + m / 2.0) * 2.0 ** (e - 1.0))


def e2m1_to_f32(n4: np.ndarray) -> np.ndarray:
    """E2M1 codes (low 4 bits: sign, 2 exponent bits, 1 mantissa bit) -> fp32
    (exact; code 8 is -0)."""
    n = np.asarray(n4, dtype=np.uint8).astype(np.int64) & 0xF
    val = _e2m1_table()[n & 7]
    return np.where(n & 8, -val, val).astype(F32)


def e2m1_from_f32(x: np.ndarray) -> np.ndarray:
    """fp32 -> E2M1 codes: the nearest value, ties to the even code, magnitudes
    beyond 6 saturating to +-6; the sign bit follows the input's sign (also
    for zero).  E2M1 has no NaN; the input must be finite."""
    xf = np.asarray(x, dtype=F32).astype(np.float64)
    assert np.all(np.isfinite(xf)), "E2M1 has no NaN or infinity"
    t = _e2m1_table()
    a = np.abs(xf)
    hi = np.clip(np.searchsorted(t, a, side="left"), 0, len(t) - 1)   # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - t[lo], t[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a >= t[-1], 7, code)               # saturate
    sign = np.signbit(xf).astype(np.int64) << 3
    return (code | sign).astype(np.uint8)


def fp4_quantize_rows(w: np.ndarray):
    """NVFP4 weights of a [rows, cols] matrix (cols a multiple of 16), in fp32:
      rs   = absmax(row) / (6 * 448)                      one per row
      bs_b = e4m3(absmax(block b) / (6 * rs))             one per 16 columns
      code = e2m1(w / (bs_b * rs))                        ties to even, +-6 saturation
    An all-zero row gets rs = 0, and a block whose scale rounds to 0 gets
    codes 0.  Returns (codes uint8 [rows, cols] in 0..15, block scale codes
    uint8 [rows, cols/16], row scales fp32 [rows])."""
    wf = np.asarray(w, dtype=np.float16).astype(F32)
    rows, cols = wf.shape
    assert cols % FP4_BLOCK == 0
    rs = (np.abs(wf).max(axis=1) / F32(E2M1_MAX * E4M3_MAX)).astype(F32)
    wb = wf.reshape(rows, cols // FP4_BLOCK, FP4_BLOCK)
    amax_b = np.abs(wb).max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        bs_real = np.where(rs[:, None] > 0, amax_b / (F32(E2M1_MAX) * rs[:, None]), F32(0.0)).astype(F32)
        bs_codes = e4m3_from_f32(bs_real)
        denom = (e4m3_to_f32(bs_codes) * rs[:, None]).astype(F32)
        q = np.where(denom[:, :, None] > 0, wb / denom[:, :, None], F32(0.0)).astype(F32)
    codes = e2m1_from_f32(q).reshape(rows, cols)
    return codes, bs_codes, rs


def fp4_dequantize_rows(codes: np.ndarray, bs_codes: np.ndarray, rs: np.ndarray) -> np.ndarray:
    """w' = (e2m1(code) * e4m3(block scale)) * row scale in fp32 (the first
    product is exact: 2 and 4 significant bits)."""
    rows, cols = codes.shape
    v = e2m1_to_f32(codes).reshape(rows, cols // FP4_BLOCK, FP4_BLOCK)
    b = e4m3_to_f32(bs_codes)[:, :, None]
    return ((v * b).astype(F32) * np.asarray(rs, dtype=F32)[:, None, None]).astype(F32).reshape(rows, cols)


INT4_GROUP = 128  # [xAI] 3.3: int4, group_size 128, symmetric


def int4_quantize_g128(w: np.ndarray):
    """Symmetric INT4 quantisation per output row and per group of 128 input
    columns ([xAI] 2.3 W4A16 FFN; [xAI] 3.3 group_size 128, symmetric).

    s = fp16(absmax / 7) (the division in fp32, then round to nearest even
    fp16), q = clamp(round_half_even(w / fp32(s)), -8, 7); an all-zero group
    (s == 0) gets q = 0.  Returns (codes int8 [rows, cols], scales fp16
    [rows, cols/128])."""
    wf = np.asarray(w, dtype=np.float16).astype(F32)
    rows, cols = wf.shape
    if cols % INT4_GROUP:
        raise ValueError("cols must be a multiple of 128")
    g = wf.reshape(rows, cols // INT4_GROUP, INT4_GROUP)
    absmax = np.abs(g).max(axis=2)
    s16 = (absmax / F32(7.0)).astype(F32).astype(np.float16)
    s32 = s16.astype(F32)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(s32 > 0, np.rint(g / s32), F32(0.0))
    q = np.clip(q, -8, 7).astype(np.int8)
    return q.reshape(rows, cols), s16


def int4_dequantize(codes: np.ndarray, scales_f16: np.ndarray) -> np.ndarray:
    """w' = q * fp32(s): the product kept in fp32 ([Hunyuan] 5.2: an fp16 scale
    product truncates; compute the dequantised weight in fp32)."""
    rows, cols = codes.shape
    q = codes.astype(F32).reshape(rows, cols // INT4_GROUP, INT4_GROUP)
    return (q * scales_f16.astype(F32)[:, :, None]).reshape(rows, cols)


# ----------------------------------------------------------------------------------------------
# Decoder pieces
# ----------------------------------------------------------------------------------------------


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """y = x * g / sqrt(mean(x^2) + eps), fp32, over the last axis."""
    x = np.asarray(x, dtype=F32)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=F32)
    return (x / np.sqrt(ms + F32(eps))) * np.asarray(g, dtype=F32)


def rope_tables(head_dim: int, positions, theta: float):
    """cos/sin [len(positions), head_dim/2] for half-split RoPE.

    inv_freq_i = theta^(-2i/h) computed in double and rounded to fp32; the
    angle is fp32(p) * inv_freq_i in fp32; cos and sin of that fp32 angle are
    evaluated in double and rounded to fp32."""
    half = head_dim // 2
    inv = (float(theta) ** (-(2.0 * np.arange(half, dtype=np.float64)) / head_dim)).astype(F32)
    pos = np.asarray(positions, dtype=F32).reshape(-1, 1)
    ang = (pos * inv[None, :]).astype(F32)
    return np.cos(ang.astype(np.float64)).astype(F32), np.sin(ang.astype(np.float64)).astype(F32)


def rope_apply(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate pairs (i, i + h/2) of every head: x[..., H, h]; cos/sin broadcast
    as [..., 1, h/2]."""
    x = np.asarray(x, dtype=F32)
    half = x.shape[-1] // 2
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1).astype(F32)


def softmax(s: np.ndarray) -> np.ndarray:
    """Subtract the row max, exponentiate, normalise (fp32)."""
    s = np.asarray(s, dtype=F32)
    e = np.exp(s - s.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True, dtype=F32)).astype(F32)


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale) -> np.ndarray:
    """One query per head over C cached positions: s_j = (q . k_j) * scale,
    a = softmax(s), o = sum_j a_j v_j.  q [H, h], K/V [H, C, h] -> [H, h]."""
    s = np.einsum("hcd,hd->hc", K, q).astype(F32) * F32(scale)
    a = softmax(s)
    return np.einsum("hc,hcd->hd", a, V).astype(F32)


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=F32)
    return (z / (F32(1.0) + np.exp(-z))).astype(F32)


def argmax_lowest(logits: np.ndarray) -> int:
    """Greedy pick; np.argmax returns the first (lowest) index on ties."""
    return int(np.argmax(logits))


# ----------------------------------------------------------------------------------------------
# KV cache (holds the fp32 value each stored element represents)
# ----------------------------------------------------------------------------------------------


class KVCache:
    """Per-layer K and V caches in one of four storage formats.

    fp16:      stored value = fp16(k).
    fp8_e5m2:  stored value = E5M2(fp16(k)), read back as fp16 ([xAI] 2.3).
    fp8_e5m2_scaled: positions in slices of 256; slice j of a layer's K (or V)
               is stored as E5M2 codes of fp16(k) / s_j and read back as
               code * s_j ([xAI] 3.3).  s_0 is KV_SCALE0; s_j (j >= 1) comes
               from slice j-1's stored values (e5m2s_next_scale), fixed when
               slice j's first position is written.
    u8:        positions of a complete 128-token segment are stored as uint8
               codes with one (scale, zp) per (layer, K or V, head, segment)
               ([Grok3] 3.2); positions of the current, incomplete segment stay
               fp16 until the write that completes the segment, which quantises
               the whole segment once.
    ``k[l]``/``v[l]`` hold, as fp32 [H, max_ctx, h], the value a reader sees."""

    def __init__(self, n_layers, n_heads, head_dim, max_ctx, kv_dtype, kv_scale0=KV_SCALE0):
        if kv_dtype not in ("fp16", "fp8_e5m2", "u8", "fp8_e5m2_scaled"):
            raise ValueError(kv_dtype)
        self.kv_dtype = kv_dtype
        self.H, self.h, self.max_ctx = n_heads, head_dim, max_ctx
        self.k = [np.zeros((n_heads, max_ctx, head_dim), F32) for _ in range(n_layers)]
        self.v = [np.zeros((n_heads, max_ctx, head_dim), F32) for _ in range(n_layers)]
        self.raw16 = None  # fp16 values as written (kept only for u8 segment quantisation)
        if kv_dtype == "u8":
            self.raw16 = [[np.zeros((n_heads, max_ctx, head_dim), np.float16) for _ in range(2)]
                          for _ in range(n_layers)]
            nseg = (max_ctx + SEG - 1) // SEG
            self.codes = [[np.zeros((n_heads, max_ctx, head_dim), np.uint8) for _ in range(2)]
                          for _ in range(n_layers)]
            self.scale = [[np.zeros((n_heads, nseg), F32) for _ in range(2)] for _ in range(n_layers)]
            self.zp = [[np.zeros((n_heads, nseg), np.int32) for _ in range(2)] for _ in range(n_layers)]
        if kv_dtype == "fp8_e5m2_scaled":
            nsl = (max_ctx + KV_SLICE - 1) // KV_SLICE
            self.codes = [[np.zeros((n_heads, max_ctx, head_dim), np.uint8) for _ in range(2)]
                          for _ in range(n_layers)]
            # per layer, K/V, slice: its scale and the largest stored E5M2 magnitude
            self.sc = [[np.zeros(nsl, F32) for _ in range(2)] for _ in range(n_layers)]
            self.mcode = [[np.zeros(nsl, F32) for _ in range(2)] for _ in range(n_layers)]
            for lay in self.sc:
                lay[0][0], lay[1][0] = F32(kv_scale0[0]), F32(kv_scale0[1])

    def write(self, layer: int, pos: int, k: np.ndarray, v: np.ndarray):
        """Write positions pos .. pos+n-1 (k, v: fp32 or fp16 [n, H, h])."""
        k16 = np.asarray(k, dtype=F32).astype(np.float16)
        v16 = np.asarray(v, dtype=F32).astype(np.float16)
        n = k16.shape[0]
        sl = slice(pos, pos + n)
        if self.kv_dtype == "fp16":
            self.k[layer][:, sl] = k16.astype(F32).transpose(1, 0, 2)
            self.v[layer][:, sl] = v16.astype(F32).transpose(1, 0, 2)
        elif self.kv_dtype == "fp8_e5m2":
            self.k[layer][:, sl] = e5m2_round(k16).transpose(1, 0, 2)
            self.v[layer][:, sl] = e5m2_round(v16).transpose(1, 0, 2)
        elif self.kv_dtype == "fp8_e5m2_scaled":
            # slice by slice: a slice's scale is fixed when its first position is written
            p = pos
            while p < pos + n:
                j = p // KV_SLICE
                q = min(pos + n, (j + 1) * KV_SLICE)
                for which, x16 in ((0, k16), (1, v16)):
                    if p == j * KV_SLICE and j > 0:
                        self.sc[layer][which][j] = e5m2s_next_scale(self.mcode[layer][which][j - 1],
                                                                    self.sc[layer][which][j - 1])
                        self.mcode[layer][which][j] = F32(0)
                    s_j = self.sc[layer][which][j]
                    codes = e5m2s_quantize(x16[p - pos:q - pos], s_j).transpose(1, 0, 2)
                    self.codes[layer][which][:, p:q] = codes
                    mag = np.abs(e5m2_to_f16_bits(codes).view(np.float16).astype(F32))
                    self.mcode[layer][which][j] = max(self.mcode[layer][which][j], F32(mag.max()))
                    dst = self.k[layer] if which == 0 else self.v[layer]
                    dst[:, p:q] = e5m2s_dequantize(codes, s_j)
                p = q
        else:
            for which, x16 in ((0, k16), (1, v16)):
                self.raw16[layer][which][:, sl] = x16.transpose(1, 0, 2)
                dst = self.k[layer] if which == 0 else self.v[layer]
                dst[:, sl] = x16.astype(F32).transpose(1, 0, 2)
            # segments completed by this write are quantised once
            first_seg = pos // SEG
            last_full = (pos + n) // SEG  # segments [first_seg, last_full) are complete now
            for s in range(first_seg, last_full):
                self._quantize_segment(layer, s)

    def _quantize_segment(self, layer: int, s: int):
        sl = slice(s * SEG, (s + 1) * SEG)
        for which in (0, 1):
            dst = self.k[layer] if which == 0 else self.v[layer]
            for hh in range(self.H):
                codes, scale, zp = u8_quantize(self.raw16[layer][which][hh, sl])
                self.codes[layer][which][hh, sl] = codes
                self.scale[layer][which][hh, s] = scale
                self.zp[layer][which][hh, s] = zp
                dst[hh, sl] = u8_dequantize(codes, scale, zp)


# ----------------------------------------------------------------------------------------------
# The decoder
# ----------------------------------------------------------------------------------------------


class OracleDecoder:
    """Batch-1 decoder-only transformer, fp32, weights read from the given fp16.

    weights: dict as produced by ``synthetic.gen_weights`` (fp16 [out, in]).
    For ffn_wdtype == "int4_g128" the FFN matrices are quantised here with
    ``int4_quantize_g128`` and used dequantised in fp32 ([xAI] 2.3/3.3,
    [Hunyuan] 5.2).  attn_wdtype == "int4_g128" does the same for the q, k and
    v projections only ([xAI] 2.3: the attention's QKV projection weights in
    INT4); the O projection and the LM head stay fp16 ([xAI] 3.3 keeps
    lm_head in fp16 and lists no other attention matrix as INT4).  fp16 ->
    fp32 widening is exact, so widening every matrix once at construction
    equals widening it at each use."""

    def __init__(self, cfg, weights: dict, max_ctx: int | None = None):
        self.cfg = cfg
        self.L, self.d, self.H, self.h = cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.head_dim
        self.eps = cfg.rms_eps
        self.theta = cfg.rope_theta
        self.max_ctx = cfg.max_ctx if max_ctx is None else max_ctx
        f = lambda a: np.asarray(a, dtype=np.float16).astype(F32)  # noqa: E731
        wd = getattr(cfg, "attn_wdtype", "fp16")
        fp8 = lambda a: fp8_dequantize_rows(*fp8_quantize_rows(a))  # noqa: E731
        fp4 = lambda a: fp4_dequantize_rows(*fp4_quantize_rows(a))  # noqa: E731
        attn_w = {"fp8_e4m3": fp8, "nvfp4": fp4}.get(wd, f)          # q, k, v, o and the LM head
        i4 = lambda a: int4_dequantize(*int4_quantize_g128(a))  # noqa: E731
        qkv_w = i4 if wd == "int4_g128" else attn_w                    # INT4 reaches q, k, v only
        self.tok_emb = f(weights["tok_emb"])
        self.lm_head = attn_w(weights["lm_head"])
        self.final_norm = f(weights["final_norm"])
        self.layers = []
        self.int4 = []
        for lw in weights["layers"]:
            lay = {k: f(lw[k]) for k in ("attn_norm", "ffn_norm")}
            lay.update({k: qkv_w(lw[k]) for k in ("wq", "wk", "wv")})
            lay["wo"] = attn_w(lw["wo"])
            if cfg.ffn_wdtype in ("fp8_e4m3", "nvfp4"):
                for k in ("w_gate", "w_up", "w_down"):
                    lay[k] = (fp8 if cfg.ffn_wdtype == "fp8_e4m3" else fp4)(lw[k])
            elif cfg.ffn_wdtype == "int4_g128":
                q4 = {}
                for k in ("w_gate", "w_up", "w_down"):
                    codes, s16 = int4_quantize_g128(lw[k])
                    q4[k] = (codes, s16)
                    lay[k] = int4_dequantize(codes, s16)
                self.int4.append(q4)
            else:
                for k in ("w_gate", "w_up", "w_down"):
                    lay[k] = f(lw[k])
            self.layers.append(lay)
        self.cache = KVCache(self.L, self.H, self.h, self.max_ctx, cfg.kv_dtype,
                             getattr(cfg, "kv_scale0", KV_SCALE0))
        self.pos = 0
        self.scale = F32(1.0 / np.sqrt(self.h))

    # -- one position -----------------------------------------------------------------------
    def decode(self, tok: int) -> np.ndarray:
        """Consume token ``tok`` at position ``pos``; return logits fp32[V]."""
        if self.pos >= self.max_ctx:
            raise ValueError("context overflow")
        p = self.pos
        cos, sin = rope_tables(self.h, [p], self.theta)
        cos, sin = cos[:, None, :], sin[:, None, :]          # [1, 1, h/2]
        x = self.tok_emb[tok].copy()
        C = p + 1
        for l, lw in enumerate(self.layers):
            u = rmsnorm(x, lw["attn_norm"], self.eps)
            q = (lw["wq"] @ u).reshape(1, self.H, self.h)
            k = (lw["wk"] @ u).reshape(1, self.H, self.h)
            v = (lw["wv"] @ u).reshape(1, self.H, self.h)
            q = rope_apply(q, cos, sin)[0]
            k = rope_apply(k, cos, sin)
            self.cache.write(l, p, k, v)
            o = attention(q, self.cache.k[l][:, :C], self.cache.v[l][:, :C], self.scale).reshape(-1)
            x = (x + lw["wo"] @ o).astype(F32)
            u = rmsnorm(x, lw["ffn_norm"], self.eps)
            act = silu(lw["w_gate"] @ u) * (lw["w_up"] @ u)
            x = (x + lw["w_down"] @ act).astype(F32)
        logits = (self.lm_head @ rmsnorm(x, self.final_norm, self.eps)).astype(F32)
        self.pos += 1
        return logits

    # -- many positions ---------------------------------------------------------------------
    def prefill(self, tokens, q_block: int = 1024) -> np.ndarray:
        """Run ``decode`` for every prompt token; return the last logits.

        For fp16 and E5M2 caches the stored value of a position does not depend
        on later writes, so all positions are processed together (matmuls over
        the T rows, causal mask j <= t); row t's attention is the same
        computation ``decode`` does at position t.  Rows are processed in
        blocks of ``q_block`` only to bound memory.  The u8 cache changes the
        stored value of a segment when it completes, so it runs ``decode`` one
        position at a time."""
        tokens = np.asarray(tokens, dtype=np.int64)
        if self.cfg.kv_dtype == "u8" or len(tokens) == 1:
            logits = None
            for t in tokens:
                logits = self.decode(int(t))
            return logits
        T = len(tokens)
        p0 = self.pos
        if p0 + T > self.max_ctx:
            raise ValueError("context overflow")
        cos, sin = rope_tables(self.h, np.arange(p0, p0 + T), self.theta)
        cos, sin = cos[:, None, :], sin[:, None, :]          # [T, 1, h/2]
        X = self.tok_emb[tokens].astype(F32)                 # [T, d]
        for l, lw in enumerate(self.layers):
            U = rmsnorm(X, lw["attn_norm"], self.eps)
            Q = (U @ lw["wq"].T).reshape(T, self.H, self.h)
            Kn = (U @ lw["wk"].T).reshape(T, self.H, self.h)
            Vn = (U @ lw["wv"].T).reshape(T, self.H, self.h)
            Q = rope_apply(Q, cos, sin)
            Kn = rope_apply(Kn, cos, sin)
            self.cache.write(l, p0, Kn, Vn)
            K = self.cache.k[l][:, :p0 + T]                  # [H, C, h]
            V = self.cache.v[l][:, :p0 + T]
            O = np.empty((T, self.H, self.h), F32)
            for b0 in range(0, T, q_block):
                b1 = min(T, b0 + q_block)
                s = np.einsum("thd,hcd->htc", Q[b0:b1], K).astype(F32) * self.scale
                t_idx = p0 + np.arange(b0, b1)[:, None]
                mask = np.arange(p0 + T)[None, :] <= t_idx  # [tb, C]
                s = np.where(mask[None], s, F32(-np.inf))
                a = softmax(s)
                O[b0:b1] = np.einsum("htc,hcd->thd", a, V)
            X = (X + O.reshape(T, -1) @ lw["wo"].T).astype(F32)
            U = rmsnorm(X, lw["ffn_norm"], self.eps)
            act = silu(U @ lw["w_gate"].T) * (U @ lw["w_up"].T)
            X = (X + act @ lw["w_down"].T).astype(F32)
        self.pos = p0 + T
        return (self.lm_head @ rmsnorm(X[-1], self.final_norm, self.eps)).astype(F32)

    def set_kv(self, layer: int, k16: np.ndarray, v16: np.ndarray, pos: int = 0):
        """Load externally supplied post-RoPE K/V (fp16 [n, H, h]) at positions
        pos.. through the cache's storage format (synthetic contexts)."""
        self.cache.write(layer, pos, k16, v16)

    def greedy(self, first_tok: int, n: int):
        """n chained decode steps; returns (tokens, logits[n, V])."""
        toks, logs = [], []
        t = first_tok
        for _ in range(n):
            lg = self.decode(t)
            t = argmax_lowest(lg)
            toks.append(t)
            logs.append(lg)
        return np.array(toks, np.int32), np.stack(logs)


# ----------------------------------------------------------------------------------------------
# The bound ([Kog], "memory bandwidth is the main bottleneck")
# ----------------------------------------------------------------------------------------------


def tokens_per_s_bound(eff_bandwidth: float, active_weight_bytes: float, kv_bytes: float = 0.0,
                       beta: float = 1.0) -> float:
    """tokens/s <= effective_bandwidth / (beta * active_weight_bytes + KV bytes)."""
    return eff_bandwidth / (beta * active_weight_bytes + kv_bytes)


def decode_bytes_per_token(cfg, ctx_len: int) -> dict:
    """Algorithmic HBM bytes one decode step must read at context length C
    (C = positions attended, including the current one): every active weight
    once, plus the K and V of all C positions in every layer."""
    d, H, h, F, V, L = cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.ffn_dim, cfg.vocab, cfg.n_layers
    wd = getattr(cfg, "attn_wdtype", "fp16")
    fp8_attn, fp4_attn = wd == "fp8_e4m3", wd == "nvfp4"
    # FP8 matrices: one byte per weight plus a 4-byte scale per row; NVFP4: half
    # a byte per weight, one byte per 16 weights and a 4-byte scale per row
    n_attn, rows_attn = 3 * H * h * d + d * H * h, 3 * H * h + d
    if fp8_attn:
        attn_w = n_attn + rows_attn * 4
    elif fp4_attn:
        attn_w = n_attn // 2 + n_attn // FP4_BLOCK + rows_attn * 4
    elif wd == "int4_g128":   # q, k, v as INT4 codes + one fp16 scale per 128 weights; O in fp16
        attn_w = 3 * H * h * d // 2 + 3 * H * h * d // INT4_GROUP * 2 + d * H * h * 2
    else:
        attn_w = n_attn * 2
    if cfg.ffn_wdtype == "int4_g128":
        ffn_w = 3 * F * d // 2 + 3 * F * d // INT4_GROUP * 2
    elif cfg.ffn_wdtype == "fp8_e4m3":
        ffn_w = 3 * F * d + (2 * F + d) * 4
    elif cfg.ffn_wdtype == "nvfp4":
        ffn_w = 3 * F * d // 2 + 3 * F * d // FP4_BLOCK + (2 * F + d) * 4
    else:
        ffn_w = 3 * F * d * 2
    if fp8_attn:
        lm_w = V * d + V * 4
    elif fp4_attn:
        lm_w = V * d // 2 + V * d // FP4_BLOCK + V * 4
    else:
        lm_w = V * d * 2
    norms = 2 * d * 2
    weights = L * (attn_w + ffn_w + norms) + lm_w + d * 2 + d * 2  # LM head, final norm, embedding row
    if cfg.kv_dtype == "fp16":
        kv = L * 2 * C_bytes(ctx_len, H, h, 2)
    elif cfg.kv_dtype == "fp8_e5m2":
        kv = L * 2 * C_bytes(ctx_len, H, h, 1)
    elif cfg.kv_dtype == "fp8_e5m2_scaled":   # codes, plus the fp32 scale of every attended slice
        kv = L * 2 * (C_bytes(ctx_len, H, h, 1) + 4 * ((ctx_len + KV_SLICE - 1) // KV_SLICE))
    else:
        full = (ctx_len // SEG) * SEG
        tail = ctx_len - full
        kv = L * 2 * (C_bytes(full, H, h, 1) + C_bytes(tail, H, h, 2) + H * (full // SEG) * 8)
    return {"weights": weights, "kv": kv, "total": weights + kv}


def C_bytes(n_pos: int, H: int, h: int, elem: int) -> int:
    return n_pos * H * h * elem
