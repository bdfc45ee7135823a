"""The allocation-free decode step (kie_decode_step_static_scratch).

Some callers may not allocate device memory while decoding: code hosted inside
another framework's allocator, plugins without allocation rights, services that
forbid allocation after start-up.  This entry point runs the decode step with
its scratch in a fixed array inside the library.  Here it must give the same
tokens and logits as the ordinary kie_decode_step on two calls in a row, and
neither call may change the device's free memory or torch's reserved memory
(the array's device memory is committed when the engine is created, not by the
step).  A config whose scratch does not fit the array is refused.

Kept in a file that pytest collects last, so a failure here stops a run only
after every other test has run.
"""
import numpy as np
import pytest

import synthetic as S
from _common import TOL_FP16, engine_for
from autoregressive_decode_gb300 import kie

pytestmark = pytest.mark.gpu

# d_model 4096 with a 32 x 128 attention and FFN 11008 (the 7B shape) at one
# layer: the step's scratch is about 278 KiB of the array's 320 KiB
NEAR_BOUND = S.Workload("near_bound", 4, 1, 4096, 32, 128, 11008, 4096, prompt_len=12, decode_steps=4)


@pytest.mark.parametrize("w", [S.WORKLOADS["tiny"], NEAR_BOUND], ids=lambda w: w.name)
def test_static_scratch_step_matches_decode_step(w):
    torch = pytest.importorskip("torch")
    weights = S.gen_weights(w)
    prompt = S.gen_prompt(w)
    ref = engine_for(w, weights)
    eng = engine_for(w, weights)
    first = int(np.argmax(ref.prefill(prompt)))
    eng.prefill(prompt)

    d_tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_log = torch.zeros(w.vocab, dtype=torch.float32, device="cuda")
    t_ref = t_new = first
    for call in range(2):
        nxt_ref, lg_ref = ref.decode_step(t_ref)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        reserved_before = torch.cuda.memory_reserved()
        eng.decode_step_static_scratch(t_new, d_tok, d_log)
        eng.sync()
        assert torch.cuda.mem_get_info()[0] == free_before, f"call {call} changed the device's free memory"
        assert torch.cuda.memory_reserved() == reserved_before
        nxt_new = int(d_tok.cpu().item())
        lg_new = d_log.cpu().numpy()
        assert np.abs(lg_new - lg_ref).max() <= TOL_FP16
        assert nxt_new == nxt_ref
        assert eng.pos == ref.pos == w.prompt_len + call + 1
        t_ref, t_new = nxt_ref, nxt_new
    # the engine's own path continues from the state the static-scratch steps left
    nxt_a, lg_a = ref.decode_step(t_ref)
    nxt_b, lg_b = eng.decode_step(t_new)
    assert nxt_a == nxt_b and np.abs(lg_a - lg_b).max() <= TOL_FP16


def test_static_scratch_rejects_oversized_config():
    """d_model 4096, 32 x 128 heads, FFN 24576: the step's scratch (about 384
    KiB: two copies each of the residual, the attention output and the SwiGLU
    output, q, current K/V, 152 attention partials, argmax partials, control
    block) exceeds the 320 KiB array, so the call is refused without
    launching."""
    torch = pytest.importorskip("torch")
    w = S.Workload("wide_ffn", 0, 1, 4096, 32, 128, 24576, 4096, prompt_len=4, decode_steps=2)
    weights = S.gen_weights(w)
    eng = engine_for(w, weights)
    d_tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(kie.KieError) as ei:
        eng.decode_step_static_scratch(1, d_tok)
    assert ei.value.status == -8          # KIE_ERR_UNSUPPORTED
    assert eng.pos == 0
    # the engine is not poisoned: the ordinary step still runs
    nxt, lg = eng.decode_step(1)
    assert 0 <= nxt < w.vocab and np.isfinite(lg).all()
