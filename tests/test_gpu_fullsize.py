"""Full-size parity: the four large workloads in the launch configuration the
bench times (persistent kernel, one CTA per SM), against the CPU oracle.

  1p8b      GPU prefill of the 2048-token prompt vs the oracle's prefill (last
            logits), then teacher-forced decode steps.
  1p8b_32k  FP8-E5M2 cache over a 32,768-position synthetic context (decode-only
            parity: the same fp16 K/V loaded into both sides).
  1p8b_u8   adaptive-range uint8 cache over the 8,192-position synthetic context
            (N(0,1) with 0.1% +-20 outliers); stored codes, scales and
            zero-points bit-exact on sampled layers.
  7b_int4   INT4 g128 FFN, fp16 cache over a 4,096-position synthetic context;
            INT4 codes and scales bit-exact on a sampled matrix.

Logits: max |delta| <= 5e-2 (fp16 paths) or 1.5e-1 (FP8 / uint8 / INT4), over
all vocab entries of every compared step; argmax equal where the oracle's
top-2 margin exceeds 0.1.
"""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from _common import engine_for, teacher_forced, tol_for
from autoregressive_decode_gb300 import kie

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 3


def _synthetic_context(w, e, o):
    for layer in range(w.n_layers):
        k, v = S.gen_kv(w, layer)
        e.set_kv(layer, k, v)
        o.set_kv(layer, k, v)
    e.set_pos(w.context_len)
    o.pos = w.context_len


def test_1p8b_prefill_and_decode():
    w = S.WORKLOADS["1p8b"]
    weights = S.gen_weights(w)
    e = engine_for(w, weights, max_ctx=w.prompt_len + STEPS)
    o = O.OracleDecoder(w, weights, max_ctx=w.prompt_len + STEPS)
    prompt = S.gen_prompt(w)
    lg = e.prefill(prompt)
    lo = o.prefill(prompt, q_block=512)
    assert np.abs(lg - lo).max() <= tol_for(w)
    teacher_forced(e, o, O.argmax_lowest(lo), STEPS, tol_for(w))


def test_1p8b_32k_fp8_decode():
    w = S.WORKLOADS["1p8b_32k"].with_(kv_source="synthetic", context_len=32768, prompt_len=0)
    weights = S.gen_weights(w)
    e = engine_for(w, weights, max_ctx=w.context_len + STEPS)
    o = O.OracleDecoder(w, weights, max_ctx=w.context_len + STEPS)
    _synthetic_context(w, e, o)
    # stored E5M2 bytes equal the oracle's conversion (sampled layer, K, first heads)
    data, _, _, _ = e.read_kv(7, 0, 0, 4096)
    k, _ = S.gen_kv(w, 7, n_pos=4096)
    ref = O.e5m2_from_f16_bits(k.view(np.uint16)).reshape(4096, w.n_heads, w.head_dim).transpose(1, 0, 2)
    np.testing.assert_array_equal(data, ref)
    teacher_forced(e, o, S.gen_first_token(w), STEPS, tol_for(w))


def test_1p8b_u8_decode():
    w = S.WORKLOADS["1p8b_u8"]
    weights = S.gen_weights(w)
    e = engine_for(w, weights, max_ctx=w.context_len + STEPS)
    o = O.OracleDecoder(w, weights, max_ctx=w.context_len + STEPS)
    _synthetic_context(w, e, o)
    for layer in (0, 13, 24):
        for which in (0, 1):
            data, _, sc, zp = e.read_kv(layer, which, 0, w.context_len)
            np.testing.assert_array_equal(data, o.cache.codes[layer][which][:, :w.context_len])
            np.testing.assert_array_equal(sc, o.cache.scale[layer][which][:, :w.context_len // 128])
            np.testing.assert_array_equal(zp, o.cache.zp[layer][which][:, :w.context_len // 128])
    teacher_forced(e, o, S.gen_first_token(w), STEPS, tol_for(w))


def test_7b_int4_decode():
    w = S.WORKLOADS["7b_int4"].with_(kv_source="synthetic", context_len=4096, prompt_len=0)
    weights = S.gen_weights(w)
    codes, sc = kie.quantize_int4_g128(weights["layers"][17]["w_down"])
    rc, rs = O.int4_quantize_g128(weights["layers"][17]["w_down"])
    np.testing.assert_array_equal(codes, rc)
    np.testing.assert_array_equal(sc.view(np.uint16), rs.view(np.uint16))
    e = engine_for(w, weights, max_ctx=w.context_len + STEPS)
    o = O.OracleDecoder(w, weights, max_ctx=w.context_len + STEPS)
    _synthetic_context(w, e, o)
    teacher_forced(e, o, S.gen_first_token(w), STEPS, tol_for(w))


def test_1p8b_fp8_weights_prefill_and_decode():
    """The 1.8B model with every GEMV matrix in FP8 E4M3 (the bench's 1p8b_fp8):
    2,048-token tensor-core prefill, then teacher-forced decode steps."""
    w = S.WORKLOADS["1p8b_fp8"]
    weights = S.gen_weights(w)
    e = engine_for(w, weights, max_ctx=w.prompt_len + STEPS)
    o = O.OracleDecoder(w, weights, max_ctx=w.prompt_len + STEPS)
    prompt = S.gen_prompt(w)
    lg = e.prefill(prompt)
    lo = o.prefill(prompt, q_block=512)
    assert np.abs(lg - lo).max() <= tol_for(w)
    teacher_forced(e, o, O.argmax_lowest(lo), STEPS, tol_for(w))
