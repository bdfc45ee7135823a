"""The bench's byte model (autoregressive_decode_gb300.traffic) against the
oracle's restatement of the same bound (Kog Inference Engine page, section
"memory bandwidth is the main bottleneck"): the two are written separately and
must agree byte for byte on every workload, KV format and weight format."""
import pytest

import oracle as O
import synthetic as S
from autoregressive_decode_gb300 import traffic


@pytest.mark.parametrize("name", sorted(S.WORKLOADS))
def test_step_bytes_match_oracle(name):
    w = S.WORKLOADS[name]
    for ctx in (1, 127, 128, 129, 2049, w.max_ctx):
        assert traffic.step_bytes(w, ctx) == O.decode_bytes_per_token(w, ctx)


@pytest.mark.parametrize("fmt", ["fp8_e4m3", "nvfp4"])
def test_step_bytes_match_oracle_weight_formats(fmt):
    w = S.WORKLOADS["1p8b"].with_(attn_wdtype=fmt, ffn_wdtype=fmt)
    for ctx in (1, 2049):
        assert traffic.step_bytes(w, ctx) == O.decode_bytes_per_token(w, ctx)


def test_launch_bytes_sum_of_steps():
    w = S.WORKLOADS["1p8b"]
    total = traffic.launch_bytes(w, 2048, 4)
    assert total == sum(O.decode_bytes_per_token(w, c)["total"] for c in range(2049, 2053))


def test_1p8b_weight_bytes():
    # 1,808,793,600 parameters; the decode step reads all but the embedding
    # table (one row), i.e. 3,486,728,192 bytes of fp16 weights and gains
    w = S.WORKLOADS["1p8b"]
    assert traffic.step_bytes(w, 1)["weights"] == 3_486_728_192


def test_batch_launch_bytes():
    """A batched step reads the weights once and every request's own cache."""
    w = S.WORKLOADS["1p8b_b8"]
    pos = [2048, 100, 700]
    total = traffic.batch_launch_bytes(w, pos, 3)
    ref = sum(O.decode_bytes_per_token(w, pos[0] + t + 1)["weights"]
              + sum(O.decode_bytes_per_token(w, p + t + 1)["kv"] for p in pos) for t in range(3))
    assert total == ref
    assert traffic.batch_launch_bytes(w, [2048], 4) == traffic.launch_bytes(w, 2048, 4)
