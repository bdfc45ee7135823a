"""Helpers shared by the GPU parity tests: build an engine and an oracle on the
same seeded inputs, and compare them."""
from __future__ import annotations

import numpy as np

import oracle as O
import synthetic as S
from autoregressive_decode_gb300 import kie

# Tolerances fixed by the decode-engine specification: max |delta logit| <= 5e-2
# on fp16 paths, <= 1.5e-1 on FP8 / uint8 / INT4 paths; argmax bit-exact where
# the oracle's top-1/top-2 margin exceeds 0.1.
TOL_FP16 = 5e-2
TOL_QUANT = 1.5e-1
MARGIN = 0.1


def tol_for(w: S.Workload) -> float:
    return TOL_FP16 if (w.kv_dtype == "fp16" and w.ffn_wdtype == "fp16" and w.attn_wdtype == "fp16") else TOL_QUANT


def engine_for(w: S.Workload, weights: dict, mode: str = "persistent", max_ctx: int | None = None) -> kie.Engine:
    cfg = kie.make_config(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab,
                          max_ctx or w.max_ctx, w.rms_eps, w.rope_theta, w.kv_dtype, w.ffn_wdtype, mode,
                          attn_wdtype=w.attn_wdtype)
    e = kie.Engine(cfg)
    e.load_weights(weights)
    return e


def margin(logits: np.ndarray) -> float:
    top2 = np.partition(logits, -2)[-2:]
    return float(top2[1] - top2[0])


def teacher_forced(e: kie.Engine, o: O.OracleDecoder, first: int, n: int, tol: float):
    """Feed both the oracle's own greedy tokens; compare logits at every step.
    Returns (max |delta logit|, tokens)."""
    t = first
    worst = 0.0
    toks = []
    for _ in range(n):
        lo = o.decode(t)
        nxt, lg = e.decode_step(t)
        d = float(np.abs(lg - lo).max())
        worst = max(worst, d)
        assert d <= tol, f"step pos={o.pos - 1}: max |dlogit| {d} > {tol}"
        if margin(lo) > MARGIN:
            assert nxt == int(np.argmax(lo)), "argmax differs where the oracle margin > 0.1"
        t = O.argmax_lowest(lo)
        toks.append(t)
    return worst, toks


def check_free_running(o: O.OracleDecoder, first: int, gpu_toks, gpu_logits, tol: float) -> int:
    """Validate a free-running GPU greedy chain: feed the oracle the GPU's own
    tokens, compare logits at every step, and require each GPU token to be the
    oracle's argmax where the margin exceeds 0.1, and otherwise a token whose
    oracle logit is within 2*tol of the maximum (several answers are correct
    there).  Returns the number of steps decided by a clear margin."""
    t = first
    clear = 0
    for g, lg in zip(gpu_toks, gpu_logits):
        lo = o.decode(int(t))
        assert float(np.abs(lg - lo).max()) <= tol
        if margin(lo) > MARGIN:
            assert int(g) == int(np.argmax(lo))
            clear += 1
        else:
            assert lo[int(g)] >= lo.max() - 2 * tol
        t = int(g)
    return clear
