"""Algorithmic HBM bytes of one decode step: the roofline's numerator.

A batch-1 decode step has to read every active weight once and the K and V of
every attended position in every layer (Kog Inference Engine page, section
"memory bandwidth is the main bottleneck": tokens/s is bounded by bandwidth
divided by the bytes read per token).  This module counts those bytes from the
model shape and storage formats, for the bench's GB/s and roofline fraction.

Storage formats counted:
  * fp16 matrices: 2 bytes per weight;
  * FP8 E4M3 matrices: 1 byte per weight plus one fp32 scale per output row;
  * INT4 g128 matrices (the FFN, or the q/k/v projections): half a byte per
    weight plus one fp16 scale per 128-column group of a row;
  * NVFP4 matrices: half a byte per weight, one E4M3 scale byte per 16-column
    block of a row and one fp32 scale per row;
  * KV cache: fp16 (2 bytes), FP8 E5M2 (1 byte; the scaled variant adds one
    fp32 scale per layer, K/V and 256-position slice), or uint8 codes for completed
    128-token segments (1 byte, plus an fp32 scale and an int32 zero point per
    segment, layer, K/V and head) with the open segment's tail in fp16;
  * RMSNorm gains (two per layer), the final gain and the embedding row read
    for the input token, counted at 2 bytes per element.
"""
from __future__ import annotations

SEGMENT = 128     # uint8 KV segment (tokens)
SLICE = 256       # scaled FP8 KV: positions sharing one scale
INT4_GROUP = 128  # INT4 scale group (columns)
FP4_BLOCK = 16    # NVFP4 scale block (columns)


def _matrix(rows: int, cols: int, fmt: str) -> int:
    if fmt == "fp16":
        return rows * cols * 2
    if fmt == "fp8_e4m3":
        return rows * cols + rows * 4
    if fmt == "int4_g128":
        return rows * cols // 2 + rows * (cols // INT4_GROUP) * 2
    if fmt == "nvfp4":
        return rows * cols // 2 + rows * (cols // FP4_BLOCK) + rows * 4
    raise ValueError(f"unknown weight format {fmt}")


def _kv_layer(ctx: int, heads: int, head_dim: int, kv_dtype: str) -> int:
    """K and V bytes of one layer for `ctx` attended positions."""
    per_pos = heads * head_dim
    if kv_dtype == "fp16":
        return 2 * ctx * per_pos * 2
    if kv_dtype == "fp8_e5m2":
        return 2 * ctx * per_pos
    if kv_dtype == "fp8_e5m2_scaled":   # one byte per value, one fp32 scale per 256-position slice
        return 2 * (ctx * per_pos + 4 * ((ctx + SLICE - 1) // SLICE))
    if kv_dtype == "u8":
        done = ctx - ctx % SEGMENT
        meta = heads * (done // SEGMENT) * 8
        return 2 * (done * per_pos + (ctx - done) * per_pos * 2 + meta)
    raise ValueError(f"unknown KV format {kv_dtype}")


def step_bytes(w, ctx: int) -> dict:
    """Bytes of one decode step of workload shape `w` (attributes n_layers,
    d_model, n_heads, head_dim, ffn_dim, vocab, kv_dtype, ffn_wdtype and
    optionally attn_wdtype) attending `ctx` positions including its own."""
    d, qkv = w.d_model, w.n_heads * w.head_dim
    attn_fmt = getattr(w, "attn_wdtype", "fp16")
    # INT4 attention weights cover q, k and v; O and the LM head stay fp16
    o_fmt = "fp16" if attn_fmt == "int4_g128" else attn_fmt
    layer = (_matrix(3 * qkv, d, attn_fmt) + _matrix(d, qkv, o_fmt)
             + 2 * _matrix(w.ffn_dim, d, w.ffn_wdtype) + _matrix(d, w.ffn_dim, w.ffn_wdtype)
             + 2 * d * 2)
    weights = w.n_layers * layer + _matrix(w.vocab, d, o_fmt) + d * 2 + d * 2
    kv = w.n_layers * _kv_layer(ctx, w.n_heads, w.head_dim, w.kv_dtype)
    return {"weights": weights, "kv": kv, "total": weights + kv}


def launch_bytes(w, first_pos: int, n_steps: int) -> int:
    """Bytes of n_steps consecutive decode steps, the first at position
    first_pos (so it attends first_pos + 1 positions)."""
    return sum(step_bytes(w, p + 1)["total"] for p in range(first_pos, first_pos + n_steps))


def batch_launch_bytes(w, first_pos, n_steps: int) -> int:
    """Bytes of n_steps steps of a batched engine: every weight once per step
    and each request's own K and V; first_pos: each request's first position."""
    total = 0
    for t in range(n_steps):
        total += step_bytes(w, first_pos[0] + t + 1)["weights"]
        total += sum(step_bytes(w, p + t + 1)["kv"] for p in first_pos)
    return total
