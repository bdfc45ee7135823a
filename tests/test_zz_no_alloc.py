"""The allocation-free decode step (kie_decode_step_static_scratch).

Some callers may not allocate device memory while decoding: code hosted inside
another framework's allocator, plugins without allocation rights, services that
forbid allocation after start-up.  This entry point runs the decode step with
its scratch in a fixed array inside the library.  Here it must give the same
tokens and logits as the ordinary kie_decode_step on two calls in a row, and the
second call must leave the device's free memory unchanged.

Kept in a file that pytest collects last, so a failure here stops a run only
after every other test has run.
"""
import numpy as np
import pytest

import synthetic as S
from _common import TOL_FP16, engine_for

pytestmark = pytest.mark.gpu


def test_static_scratch_step_matches_decode_step():
    torch = pytest.importorskip("torch")
    w = S.WORKLOADS["tiny"]
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
        if call == 1:
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
        eng.decode_step_static_scratch(t_new, d_tok, d_log)
        eng.sync()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before
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
