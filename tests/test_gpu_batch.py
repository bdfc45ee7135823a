"""Low-batch decode: B independent requests share one pass over the weights
per step (a batched engine, kie_config.batch = B).  Every request is the
single-request model on its own KV cache, so each one is checked against its
own oracle decoder: prompt prefill per request (different prompts and lengths,
so the requests sit at different positions), then batched decode steps with
every request's logits within the tolerance and its token equal to the
oracle's argmax where the oracle's margin exceeds 0.1."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from _common import MARGIN, check_free_running, margin, tol_for
from autoregressive_decode_gb300 import kie

pytestmark = pytest.mark.gpu

TINY = S.WORKLOADS["tiny"]
MEDIUM = S.Workload("medium", 5, 2, 1024, 8, 128, 4608, 10007, prompt_len=100, decode_steps=24)
WIDE = S.Workload("wide", 6, 2, 2048, 16, 128, 4096, 8002, prompt_len=40, decode_steps=16)


def batched_engine(w, weights, B, max_ctx=None):
    cfg = kie.make_config(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab, max_ctx or w.max_ctx,
                          w.rms_eps, w.rope_theta, w.kv_dtype, w.ffn_wdtype, "persistent",
                          attn_wdtype=w.attn_wdtype, batch=B)
    e = kie.Engine(cfg)
    e.load_weights(weights)
    return e


def request_prompt(w, b):
    """Request b's prompt: its own seed, and 3 tokens shorter per request."""
    return S.gen_prompt(w, n=max(4, w.prompt_len - 3 * b), seed=w.prompt_seed + 7919 * b)


def prefill_all(e, oracles, w, B):
    firsts = []
    tol = tol_for(w)
    for b in range(B):
        p = request_prompt(w, b)
        e.select_request(b)
        lg = e.prefill(p)
        lo = oracles[b].prefill(p)
        assert np.abs(lg - lo).max() <= tol, f"request {b} prefill"
        assert e.pos == len(p)
        firsts.append(O.argmax_lowest(lo))
    return firsts


@pytest.mark.parametrize("w", [TINY, MEDIUM, WIDE], ids=lambda w: w.name)
@pytest.mark.parametrize("B", [2, 8])
@pytest.mark.parametrize("kv", ["fp16", "fp8_e5m2"])
def test_batched_teacher_forced(w, B, kv):
    w = w.with_(kv_dtype=kv)
    weights = S.gen_weights(w)
    e = batched_engine(w, weights, B)
    oracles = [O.OracleDecoder(w, weights) for _ in range(B)]
    toks = prefill_all(e, oracles, w, B)
    tol = tol_for(w)
    worst = 0.0
    for step in range(8):
        nxt, lg = e.decode_batch(toks)
        new = []
        for b in range(B):
            lo = oracles[b].decode(toks[b])
            dl = float(np.abs(lg[b] - lo).max())
            worst = max(worst, dl)
            assert dl <= tol, f"step {step} request {b}: max |dlogit| {dl}"
            if margin(lo) > MARGIN:
                assert nxt[b] == int(np.argmax(lo)), f"step {step} request {b}: argmax"
            new.append(O.argmax_lowest(lo))
        toks = new
    print(f"{w.name}/{kv}/B={B}: max |dlogit| {worst:.3e}")


@pytest.mark.parametrize("B", [3, 8])
def test_batched_generate_free_running(B):
    """One launch of n greedy steps for all requests (the bench's call), every
    request's chain validated against its oracle fed the GPU's tokens; the
    host-logits path (chunked launches) and the device path agree bit for bit."""
    torch = pytest.importorskip("torch")
    w = MEDIUM
    weights = S.gen_weights(w)
    n = 12
    e = batched_engine(w, weights, B)
    oracles = [O.OracleDecoder(w, weights) for _ in range(B)]
    firsts = prefill_all(e, oracles, w, B)
    toks, logs = e.generate_greedy_batch(firsts, n, want_logits=True)
    assert toks.shape == (n, B) and logs.shape == (n, B, w.vocab)
    for b in range(B):
        check_free_running(oracles[b], firsts[b], toks[:, b], logs[:, b], tol_for(w))
    # the same chain through the device-output call on a fresh engine
    e2 = batched_engine(w, weights, B)
    for b in range(B):
        e2.select_request(b)
        e2.prefill(request_prompt(w, b), want_logits=False)
    d_tok = torch.zeros((n, B), dtype=torch.int32, device="cuda")
    d_log = torch.zeros((n, B, w.vocab), dtype=torch.float32, device="cuda")
    e2.generate_greedy_batch_device(firsts, n, d_tok, d_log)
    e2.sync()
    np.testing.assert_array_equal(d_tok.cpu().numpy(), toks)
    np.testing.assert_array_equal(d_log.cpu().numpy(), logs)
    for b in range(B):
        e2.select_request(b)
        assert e2.pos == len(request_prompt(w, b)) + n


def test_batched_identical_requests_agree():
    """Eight copies of one request give bit-identical tokens and logits (the
    requests' arithmetic does not depend on their slot in the batch)."""
    w = WIDE
    weights = S.gen_weights(w)
    B = 8
    e = batched_engine(w, weights, B)
    p = S.gen_prompt(w)
    for b in range(B):
        e.select_request(b)
        lg = e.prefill(p)
    first = int(np.argmax(lg))
    toks, logs = e.generate_greedy_batch([first] * B, 6, want_logits=True)
    for b in range(1, B):
        np.testing.assert_array_equal(toks[:, b], toks[:, 0])
        np.testing.assert_array_equal(logs[:, b], logs[:, 0])


def test_batched_synthetic_long_contexts():
    """Requests over different synthetic contexts (2,300 and 700 positions):
    long attention chunks per (request, head) pair."""
    B = 2
    w = WIDE.with_(kv_source="synthetic", prompt_len=0, decode_steps=4)
    weights = S.gen_weights(w)
    ctx = [2300, 700]
    e = batched_engine(w, weights, B, max_ctx=2400)
    oracles = [O.OracleDecoder(w, weights, max_ctx=2400) for _ in range(B)]
    for b in range(B):
        e.select_request(b)
        for layer in range(w.n_layers):
            k, v = S.gen_kv(w, layer, n_pos=ctx[b], seed=w.kv_seed + 7919 * b)
            e.set_kv(layer, k, v)
            oracles[b].set_kv(layer, k, v)
        e.set_pos(ctx[b])
        oracles[b].pos = ctx[b]
    toks = [S.gen_first_token(w, seed=w.prompt_seed + 7919 * b) for b in range(B)]
    for step in range(4):
        nxt, lg = e.decode_batch(toks)
        new = []
        for b in range(B):
            lo = oracles[b].decode(toks[b])
            assert np.abs(lg[b] - lo).max() <= tol_for(w)
            new.append(O.argmax_lowest(lo))
        toks = new


def test_batched_engine_rules():
    """Single-request calls are refused on a batched engine; select_request
    bounds; configs outside the batched kernel's scope are refused."""
    w = TINY
    weights = S.gen_weights(w)
    e = batched_engine(w, weights, 2)
    with pytest.raises(kie.KieError) as ei:
        e.decode_step(1)
    assert ei.value.status == -8
    with pytest.raises(kie.KieError):
        e.select_request(2)
    with pytest.raises(kie.KieError) as ei:
        kie.Engine(kie.make_config(2, 256, 4, 64, 1024, 4096, 64, ffn_wdtype="int4_g128", batch=2))
    assert ei.value.status == -1
    with pytest.raises(kie.KieError) as ei:   # batch * n_heads above the SM count
        kie.Engine(kie.make_config(1, 4096, 32, 128, 1024, 4096, 64, batch=8))
    assert ei.value.status == -8
    single = kie.Engine(kie.make_config(2, 256, 4, 64, 1024, 4096, 64))
    with pytest.raises(kie.KieError) as ei:
        single.decode_batch([1])
    assert ei.value.status == -8
