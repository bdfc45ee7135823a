"""GPU decode parity against the CPU oracle on small models that still span
several slots per CTA and ragged tails (vocab and FFN sizes that do not divide
evenly over the grid), for every KV format, INT4 FFN weights, and both launch
modes (persistent cooperative kernel, CUDA graph of per-phase launches)."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from _common import check_free_running, engine_for, teacher_forced, tol_for

pytestmark = pytest.mark.gpu

TINY = S.WORKLOADS["tiny"]
# hd 128; the down projection's FFN 4608 = two whole 2048-column weight chunks (the
# GEMV fast path for full 4-row slots) plus a half chunk; ragged vocab (not a
# multiple of 4 rows x 152 CTAs)
MEDIUM = S.Workload("medium", 5, 2, 1024, 8, 128, 4608, 10007, prompt_len=100, decode_steps=24)
# d_model 2048: the fp16 GEMV phases run through the TMEM stage (whole 4-row x
# 2048-column slots); vocab 8002 leaves a 2-row tail slot in the LM phase,
# which goes through the shared-memory path of the same phase
WIDE = S.Workload("wide", 6, 2, 2048, 16, 128, 4096, 8002, prompt_len=40, decode_steps=16)


def _prefill_both(w, weights, mode="persistent", max_ctx=None):
    e = engine_for(w, weights, mode, max_ctx)
    o = O.OracleDecoder(w, weights, max_ctx=max_ctx or w.max_ctx)
    prompt = S.gen_prompt(w)
    lg = e.prefill(prompt)
    lo = o.prefill(prompt)
    return e, o, lg, lo


@pytest.mark.parametrize("w", [TINY, MEDIUM, WIDE], ids=lambda w: w.name)
@pytest.mark.parametrize("kv", ["fp16", "fp8_e5m2"])
def test_prefill_then_teacher_forced_decode(w, kv):
    w = w.with_(kv_dtype=kv)
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    tol = tol_for(w)
    assert np.abs(lg - lo).max() <= tol
    assert e.pos == o.pos == w.prompt_len
    worst, _ = teacher_forced(e, o, O.argmax_lowest(lo), w.decode_steps, tol)
    print(f"{w.name}/{kv}: max |dlogit| {worst:.3e}")


def test_kv_cache_contents_after_prefill():
    """Stored K/V equal the oracle's fp16 values up to fp16 rounding flips.
    Layer 0's K/V depend on the current token only, so flips there come from
    summation order alone (rare, one ulp); deeper layers also inherit earlier
    positions' flips through attention, so they are held to a relative bound."""
    w = TINY
    weights = S.gen_weights(w)
    e, o, _, _ = _prefill_both(w, weights)
    for layer in range(w.n_layers):
        for which in (0, 1):
            data, _, _, _ = e.read_kv(layer, which, 0, w.prompt_len)
            gpu = data.view(np.float16).astype(np.float32)
            ref = (o.cache.k if which == 0 else o.cache.v)[layer][:, :w.prompt_len]
            diff = gpu != ref
            if layer == 0:
                assert diff.mean() < 0.01
                # one fp16 ulp, or fp32 summation noise (~1e-6 absolute) near zero
                assert np.all(np.abs(gpu - ref)[diff] <= 2.0 ** -10 * np.abs(ref)[diff] + 1e-6)
            else:
                assert np.abs(gpu - ref).max() <= 1e-3 * np.abs(ref).max()


@pytest.mark.parametrize("w", [TINY, MEDIUM], ids=lambda w: w.name)
def test_free_running_greedy(w):
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    first = O.argmax_lowest(lo)
    toks, logs = e.generate_greedy(first, w.decode_steps, want_logits=True)
    check_free_running(o, first, toks, logs, tol_for(w))


@pytest.mark.parametrize("w", [TINY, MEDIUM, WIDE], ids=lambda w: w.name)
def test_graph_mode_bit_identical_to_persistent(w):
    weights = S.gen_weights(w)
    prompt = S.gen_prompt(w)
    res = {}
    for mode in ("persistent", "graph"):
        e = engine_for(w, weights, mode)
        lg = e.prefill(prompt)
        toks, logs = e.generate_greedy(int(np.argmax(lg)), 8, want_logits=True)
        nxt, lg1 = e.decode_step(int(toks[-1]))
        res[mode] = (lg, toks, logs, nxt, lg1)
        e.close()
    a, b = res["persistent"], res["graph"]
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])
    assert a[3] == b[3]
    np.testing.assert_array_equal(a[4], b[4])


@pytest.mark.parametrize("w", [TINY, WIDE], ids=lambda w: w.name)
def test_step_by_step_equals_generate(w):
    """n chained decode_step calls == one generate_greedy of n steps (bit-exact)."""
    weights = S.gen_weights(w)
    prompt = S.gen_prompt(w)
    e1 = engine_for(w, weights)
    first = int(np.argmax(e1.prefill(prompt)))
    toks, logs = e1.generate_greedy(first, 10, want_logits=True)
    e2 = engine_for(w, weights)
    e2.prefill(prompt)
    t = first
    for i in range(10):
        t, lg = e2.decode_step(t)
        assert t == toks[i]
        np.testing.assert_array_equal(lg, logs[i])


@pytest.mark.parametrize("w", [TINY, MEDIUM, WIDE], ids=lambda w: w.name)
def test_fp8_weights_prefill_and_decode(w):
    """Every GEMV matrix in FP8 E4M3 with row scales (decode: 8-row slots, the
    scale applied to the row sum; prefill: the codes' fp16 values in the MMA,
    the scale on the output column): logits match the oracle's model with the
    same quantised weights."""
    w = w.with_(ffn_wdtype="fp8_e4m3", attn_wdtype="fp8_e4m3")
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    tol = tol_for(w)
    assert np.abs(lg - lo).max() <= tol
    teacher_forced(e, o, O.argmax_lowest(lo), 8, tol)


@pytest.mark.parametrize("w", [TINY, MEDIUM, WIDE], ids=lambda w: w.name)
def test_nvfp4_weights_prefill_and_decode(w):
    """Every GEMV matrix in NVFP4 (E2M1 codes, an E4M3 scale per 16 columns, an
    fp32 scale per row): decode with 8-row slots and the block scale applied
    per 16-column block, prefill with the exact fp16 values code * block scale
    in the MMA and the row scale on the output column; logits match the
    oracle's model with the same quantised weights."""
    w = w.with_(ffn_wdtype="nvfp4", attn_wdtype="nvfp4")
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    tol = tol_for(w)
    assert np.abs(lg - lo).max() <= tol
    teacher_forced(e, o, O.argmax_lowest(lo), 8, tol)


@pytest.mark.parametrize("w", [TINY, MEDIUM, WIDE], ids=lambda w: w.name)
@pytest.mark.parametrize("ffn", ["fp16", "int4_g128"])
def test_int4_qkv_weights_decode(w, ffn):
    """q, k and v projections in INT4 g128 (O and the LM head fp16), with fp16
    or INT4 FFN weights and an E5M2 cache (the xAI page's mixed precision):
    the prompt goes through the decode kernel, teacher-forced, and the logits
    match the oracle's model with the same quantised weights."""
    w = w.with_(attn_wdtype="int4_g128", ffn_wdtype=ffn, kv_dtype="fp8_e5m2")
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    tol = tol_for(w)
    assert np.abs(lg - lo).max() <= tol
    teacher_forced(e, o, O.argmax_lowest(lo), 8, tol)


def test_int4_qkv_graph_equals_persistent():
    """INT4 q/k/v weights in both launch modes: bit-identical prompt logits,
    greedy tokens and logits."""
    w = MEDIUM.with_(attn_wdtype="int4_g128", ffn_wdtype="int4_g128")
    weights = S.gen_weights(w)
    prompt = S.gen_prompt(w)[:24]
    res = {}
    for mode in ("persistent", "graph"):
        e = engine_for(w, weights, mode)
        lg = e.prefill(prompt)
        toks, logs = e.generate_greedy(int(np.argmax(lg)), 6, want_logits=True)
        res[mode] = (lg, toks, logs)
        e.close()
    for a, b in zip(res["persistent"], res["graph"]):
        np.testing.assert_array_equal(a, b)


def _scaled(w):
    return w.with_(kv_dtype="fp8_e5m2_scaled")


def test_scaled_e5m2_prompt_crossing_slices():
    """Scaled E5M2 cache: a 300-token prompt through the decode kernel crosses
    the 256-position slice boundary (slice 1's scale derived in the kernel from
    slice 0's stored maximum), then 20 teacher-forced steps; slice 0's scales
    are the initial ones, slice 1's within one E5M2 step of the oracle's (the
    GEMV's summation order can move the slice maximum by a rounding step)."""
    w = _scaled(TINY).with_(prompt_len=300, decode_steps=20)
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights, max_ctx=340)
    assert np.abs(lg - lo).max() <= tol_for(w)
    for which in (0, 1):
        _, _, sc, _ = e.read_kv(1, which, 0, 300)
        ref = o.cache.sc[1][which][:2]
        assert sc[0] == ref[0] == np.float32(0.0039 if which == 0 else 0.0042)
        assert 0.79 <= sc[1] / ref[1] <= 1.26
    teacher_forced(e, o, O.argmax_lowest(lo), w.decode_steps, tol_for(w))


@pytest.mark.parametrize("w", [TINY, WIDE], ids=lambda w: w.name)
def test_scaled_e5m2_synthetic_context(w):
    """A 700-position synthetic context loaded slice by slice: codes and slice
    scales bit-exact against the oracle; 70 decode steps cross position 768
    (slice 3 begins in the kernel); a rewind to 700 and the same steps again
    give identical logits (the slice maximum is rebuilt from what stays)."""
    w = _scaled(w).with_(kv_source="synthetic", context_len=700, prompt_len=0, decode_steps=70)
    weights = S.gen_weights(w)
    e = engine_for(w, weights, max_ctx=800)
    o = O.OracleDecoder(w, weights, max_ctx=800)
    for layer in range(w.n_layers):
        k, v = S.gen_kv(w, layer)
        e.set_kv(layer, k, v)
        o.set_kv(layer, k, v)
    e.set_pos(700)
    o.pos = 700
    for which in (0, 1):
        data, _, sc, _ = e.read_kv(0, which, 0, 700)
        np.testing.assert_array_equal(data, o.cache.codes[0][which][:, :700])
        np.testing.assert_array_equal(sc, o.cache.sc[0][which][:3])
    first = S.gen_first_token(w)
    worst, toks = teacher_forced(e, o, first, w.decode_steps, tol_for(w))
    e.set_pos(700)
    t = first
    e2 = []
    for tk in [first] + toks[:-1]:
        _, lg = e.decode_step(tk)
        e2.append(lg)
    e.set_pos(700)
    for i, tk in enumerate([first] + toks[:-1]):
        _, lg = e.decode_step(tk)
        np.testing.assert_array_equal(lg, e2[i])


def test_scaled_e5m2_graph_equals_persistent():
    w = _scaled(MEDIUM).with_(kv_source="synthetic", context_len=500, prompt_len=0)
    weights = S.gen_weights(w)
    res = {}
    for mode in ("persistent", "graph"):
        e = engine_for(w, weights, mode, max_ctx=560)
        for layer in range(w.n_layers):
            k, v = S.gen_kv(w, layer)
            e.set_kv(layer, k, v)
        e.set_pos(500)
        res[mode] = e.generate_greedy(S.gen_first_token(w), 20, want_logits=True)
        e.close()
    for a, b in zip(res["persistent"], res["graph"]):
        np.testing.assert_array_equal(a, b)


def test_nvfp4_ffn_graph_equals_persistent_and_u8_cache():
    """NVFP4 FFN weights with fp16 attention weights, in both launch modes
    (bit-identical), with the uint8 cache (prefill through the decode kernel)."""
    w = WIDE.with_(ffn_wdtype="nvfp4", kv_dtype="u8")
    weights = S.gen_weights(w)
    prompt = S.gen_prompt(w)
    res = {}
    for mode in ("persistent", "graph"):
        e = engine_for(w, weights, mode)
        lg = e.prefill(prompt)
        toks, logs = e.generate_greedy(int(np.argmax(lg)), 6, want_logits=True)
        res[mode] = (lg, toks, logs)
    for a, b in zip(res["persistent"], res["graph"]):
        np.testing.assert_array_equal(a, b)
    o = O.OracleDecoder(w, weights)
    lo = o.prefill(prompt)
    assert np.abs(res["persistent"][0] - lo).max() <= tol_for(w)
    check_free_running(o, int(np.argmax(res["persistent"][0])), res["persistent"][1], res["persistent"][2], tol_for(w))


def test_fp8_weights_graph_equals_persistent_and_u8_cache():
    """FP8 weights in both launch modes (bit-identical), and with the uint8
    cache (prefill through the decode kernel)."""
    w = WIDE.with_(ffn_wdtype="fp8_e4m3", attn_wdtype="fp8_e4m3")
    weights = S.gen_weights(w)
    prompt = S.gen_prompt(w)
    res = {}
    for mode in ("persistent", "graph"):
        e = engine_for(w, weights, mode)
        lg = e.prefill(prompt)
        toks, logs = e.generate_greedy(int(np.argmax(lg)), 6, want_logits=True)
        res[mode] = (lg, toks, logs)
        e.close()
    for a, b in zip(res["persistent"], res["graph"]):
        np.testing.assert_array_equal(a, b)
    wu = w.with_(kv_dtype="u8")
    e, o, lg, lo = _prefill_both(wu, weights)
    assert np.abs(lg - lo).max() <= tol_for(wu)
    teacher_forced(e, o, O.argmax_lowest(lo), 4, tol_for(wu))


@pytest.mark.parametrize("kv", ["fp16", "fp8_e5m2"])
def test_long_chunks_synthetic_context(kv):
    """2,300 context positions over 9-10 CTAs per head: chunks of ~240 rows need
    more than one ring slot per consumer warp, so the last partial round of K/V
    slots is shared by all warps."""
    w = WIDE.with_(kv_dtype=kv, kv_source="synthetic", context_len=2300, prompt_len=0, decode_steps=4)
    weights = S.gen_weights(w)
    e = engine_for(w, weights)
    o = O.OracleDecoder(w, weights, max_ctx=w.max_ctx)
    for layer in range(w.n_layers):
        k, v = S.gen_kv(w, layer)
        e.set_kv(layer, k, v)
        o.set_kv(layer, k, v)
    e.set_pos(w.context_len)
    o.pos = w.context_len
    teacher_forced(e, o, S.gen_first_token(w), w.decode_steps, tol_for(w))


@pytest.mark.parametrize("ctx", [300, 383])
def test_u8_synthetic_context_crossing_segment_completion(ctx):
    """Synthetic N(0,1) K/V with 0.1% +-20 outliers; decoding fills the open
    segment and completes it (position 383) inside the run, then starts the
    next one."""
    w = TINY.with_(kv_dtype="u8", kv_source="synthetic", prompt_len=0, context_len=ctx, decode_steps=100)
    weights = S.gen_weights(w)
    e = engine_for(w, weights)
    o = O.OracleDecoder(w, weights)
    for layer in range(w.n_layers):
        k, v = S.gen_kv(w, layer)
        e.set_kv(layer, k, v)
        o.set_kv(layer, k, v)
    e.set_pos(ctx)
    o.pos = ctx
    # stored codes / scale / zp of the complete segments are bit-exact
    full = (ctx // 128) * 128
    data, _, sc, zp = e.read_kv(1, 0, 0, full)
    np.testing.assert_array_equal(data, o.cache.codes[1][0][:, :full])
    np.testing.assert_array_equal(sc, o.cache.scale[1][0][:, :full // 128])
    np.testing.assert_array_equal(zp, o.cache.zp[1][0][:, :full // 128])
    teacher_forced(e, o, S.gen_first_token(w), w.decode_steps, tol_for(w))
    # the segment completed during decoding was stored with the same codes
    seg = 383 // 128
    data, _, sc, zp = e.read_kv(0, 1, seg * 128, 128)
    np.testing.assert_array_equal(data, o.cache.codes[0][1][:, seg * 128:(seg + 1) * 128])
    assert np.array_equal(sc[:, 0], o.cache.scale[0][1][:, seg])


def test_int4_ffn_decode():
    w = TINY.with_(ffn_wdtype="int4_g128")
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    assert np.abs(lg - lo).max() <= tol_for(w)
    teacher_forced(e, o, O.argmax_lowest(lo), w.decode_steps, tol_for(w))


@pytest.mark.parametrize("w", [WIDE, MEDIUM.with_(kv_dtype="fp8_e5m2")], ids=lambda w: w.name + "/" + w.kv_dtype)
def test_prefill_in_pieces(w):
    """A prompt prefilled in three calls (the later pieces attend to the cache the
    earlier ones wrote) gives the oracle's logits after each piece, and then
    decodes like the oracle."""
    weights = S.gen_weights(w)
    e = engine_for(w, weights)
    o = O.OracleDecoder(w, weights, max_ctx=w.max_ctx)
    prompt = S.gen_prompt(w)
    tol = tol_for(w)
    for a, b in ((0, 7), (7, 8), (8, w.prompt_len)):
        lg = e.prefill(prompt[a:b])
        lo = o.prefill(prompt[a:b])
        assert np.abs(lg - lo).max() <= tol
        assert e.pos == o.pos == b
    teacher_forced(e, o, O.argmax_lowest(lo), 4, tol)


def test_context_edges():
    """Decode from position 0 (C = 1: attention returns V), fill the cache to
    max_ctx exactly, and reject one more step without writing."""
    w = TINY.with_(prompt_len=0, decode_steps=20)
    weights = S.gen_weights(w)
    e = engine_for(w, weights, max_ctx=20)
    o = O.OracleDecoder(w, weights, max_ctx=20)
    teacher_forced(e, o, 7, 20, tol_for(w))
    assert e.pos == 20
    from autoregressive_decode_gb300.kie import KieError
    with pytest.raises(KieError) as ei:
        e.decode_step(3)
    assert ei.value.status == -5
    assert e.pos == 20


def test_host_errors_on_gpu():
    from autoregressive_decode_gb300 import kie
    w = TINY
    cfg = kie.make_config(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab, 64)
    e = kie.Engine(cfg)
    with pytest.raises(kie.KieError) as ei:
        e.decode_step(1)
    assert ei.value.status == kie.KIE_ERR_NOT_LOADED
    e.load_weights(S.gen_weights(w))
    with pytest.raises(kie.KieError) as ei:
        e.decode_step(w.vocab)
    assert ei.value.status == kie.KIE_ERR_INVALID_ARG
    with pytest.raises(kie.KieError) as ei:
        e.prefill(np.array([1, -1], np.int32))
    assert ei.value.status == kie.KIE_ERR_INVALID_ARG
    assert e.pos == 0
    with pytest.raises(kie.KieError) as ei:
        e.generate_greedy(1, 65)
    assert ei.value.status == kie.KIE_ERR_CTX_OVERFLOW
    e.reset()
    t, lg = e.decode_step(1)
    assert 0 <= t < w.vocab and np.isfinite(lg).all()


def test_device_timeout_then_reset():
    """A bounded wait that runs out, made on purpose without any fault: one CTA
    skips its arrival at the first grid barrier of a launch, so every other
    CTA's wait there expires after the 50 ms limit.  The call returns
    KIE_ERR_DEVICE_TIMEOUT, the engine refuses further decode calls until
    kie_reset, and afterwards it matches the oracle again."""
    from autoregressive_decode_gb300 import kie
    w = TINY
    weights = S.gen_weights(w)
    e, o, lg, lo = _prefill_both(w, weights)
    first = O.argmax_lowest(lo)
    e.set_timeout_ms(50)
    e.debug_skip_grid_arrival(e.grid // 2)
    with pytest.raises(kie.KieError) as ei:
        e.generate_greedy(first, 4)
    assert ei.value.status == kie.KIE_ERR_DEVICE_TIMEOUT
    with pytest.raises(kie.KieError) as ei:
        e.decode_step(first)
    assert ei.value.status == kie.KIE_ERR_DEVICE_TIMEOUT
    e.reset()
    e.set_timeout_ms(2000)
    assert e.pos == 0
    lg2 = e.prefill(S.gen_prompt(w))
    np.testing.assert_array_equal(lg2, lg)
    # the injection was one-shot: a launch of several steps runs normally now
    toks, logs = e.generate_greedy(first, 6, want_logits=True)
    check_free_running(o, first, toks, logs, tol_for(w))
