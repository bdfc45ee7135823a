"""Seeded synthetic inputs shared by the oracle and the GPU tests.

This module only draws numbers (weights, prompt ids, synthetic KV activations)
and describes the workload shapes.  It holds none of the decoder's arithmetic,
so neither side can borrow the other's maths through it.

The five workloads are the batch-1 decode cases the pages' discussion centres
on (the Kog Inference Engine page, "memory bandwidth is the main bottleneck"
section, takes a ~2B fp16 dense model; the xAI page, section 2.3, adds FP8-E5M2
KV and INT4 W4A16 FFN weights; the Grok-3 hot-update page, section 3.2, adds
adaptive-range uint8 KV):

  tiny      2 layers, d 256, 4x64 heads, FFN 1024, vocab 4096, 16-token prompt, 32 steps, fp16 KV
  1p8b      25 layers, d 2048, 16x128, FFN 8192, vocab 32000, 2048-token prompt, 256 steps, fp16 KV
  1p8b_32k  as 1p8b, 32768-token context, FP8-E5M2 KV, 128 steps
  1p8b_u8   as 1p8b, 8192 synthetic KV positions, adaptive-range uint8 KV, 128 steps
  7b_int4   32 layers, d 4096, 32x128, FFN 11008, vocab 32000, 4096-token prompt, 256 steps,
            FFN weights INT4 (group 128, symmetric, fp16 scales), fp16 KV

Weights are fp16 ~ N(0, 0.02) drawn by the counter-based generator in
``synth.c``; RMSNorm gains are 1.  Seeds: weights 1000 + workload index,
prompt ids +1, synthetic KV +2.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libkie_synth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the generator (host C, OpenMP).  Returns the library path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_normal_f16.argtypes = [u64, u64, dbl, i64, vp]
            lib.synth_normal_f32.argtypes = [u64, u64, dbl, i64, vp]
            lib.synth_uniform_int.argtypes = [u64, u64, i64, i64, vp]
            lib.synth_outlier_f16.argtypes = [u64, u64, dbl, dbl, i64, vp]
            for f in (lib.synth_normal_f16, lib.synth_normal_f32, lib.synth_uniform_int, lib.synth_outlier_f16):
                f.restype = None
            _lib = lib
    return _lib


def normal_f16(seed: int, tid: int, shape, std: float = 0.02) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    _load().synth_normal_f16(seed, tid, std, out.size, out.ctypes.data)
    return out


def normal_f32(seed: int, tid: int, shape, std: float = 1.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    _load().synth_normal_f32(seed, tid, std, out.size, out.ctypes.data)
    return out


def uniform_int(seed: int, tid: int, n: int, m: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_uniform_int(seed, tid, n, m, out.ctypes.data)
    return out


def outlier_f16(seed: int, tid: int, shape, p_out: float = 1e-3, mag: float = 20.0) -> np.ndarray:
    out = np.empty(shape, dtype=np.float16)
    _load().synth_outlier_f16(seed, tid, p_out, mag, out.size, out.ctypes.data)
    return out


# ----------------------------------------------------------------------------------------------
# workload shapes
# ----------------------------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # position in the workload list; seeds derive from it
    n_layers: int
    d_model: int
    n_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    kv_dtype: str = "fp16"          # "fp16" | "fp8_e5m2" | "u8" | "fp8_e5m2_scaled"
    ffn_wdtype: str = "fp16"        # "fp16" | "int4_g128" | "fp8_e4m3"
    attn_wdtype: str = "fp16"       # q/k/v/o and LM head: "fp16" | "fp8_e4m3"
    prompt_len: int = 16            # prompt tokens (kv_source == "prefill")
    context_len: int = 0            # synthetic KV positions (kv_source == "synthetic")
    decode_steps: int = 32
    kv_source: str = "prefill"      # "prefill" | "synthetic"
    batch: int = 1                  # requests decoded together (batched engine); each has its own seeds

    @property
    def start_pos(self) -> int:
        return self.prompt_len if self.kv_source == "prefill" else self.context_len

    @property
    def max_ctx(self) -> int:
        return self.start_pos + self.decode_steps

    @property
    def weight_seed(self) -> int:
        return 1000 + self.index

    @property
    def prompt_seed(self) -> int:
        return 1001 + self.index

    @property
    def kv_seed(self) -> int:
        return 1002 + self.index

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def request_seed(self, base: int, b: int) -> int:
        """Seed of request b's prompt / first token (base = prompt_seed) or
        synthetic KV (base = kv_seed); request 0 keeps the workload's own."""
        return base + 7919 * b


WORKLOADS = {
    "tiny": Workload("tiny", 0, 2, 256, 4, 64, 1024, 4096, prompt_len=16, decode_steps=32),
    "1p8b": Workload("1p8b", 1, 25, 2048, 16, 128, 8192, 32000, prompt_len=2048, decode_steps=256),
    "1p8b_32k": Workload("1p8b_32k", 2, 25, 2048, 16, 128, 8192, 32000, kv_dtype="fp8_e5m2",
                         prompt_len=32768, decode_steps=128),
    "1p8b_u8": Workload("1p8b_u8", 3, 25, 2048, 16, 128, 8192, 32000, kv_dtype="u8",
                        kv_source="synthetic", prompt_len=0, context_len=8192, decode_steps=128),
    "7b_int4": Workload("7b_int4", 4, 32, 4096, 32, 128, 11008, 32000, ffn_wdtype="int4_g128",
                        prompt_len=4096, decode_steps=256),
    # the 1.8B fp16 model (same seeds, index 1) with every GEMV matrix in FP8 E4M3
    "1p8b_fp8": Workload("1p8b_fp8", 1, 25, 2048, 16, 128, 8192, 32000, ffn_wdtype="fp8_e4m3",
                         attn_wdtype="fp8_e4m3", prompt_len=2048, decode_steps=256),
    # ... and in NVFP4 (E2M1 codes, E4M3 scale per 16 columns, fp32 scale per row)
    "1p8b_nvfp4": Workload("1p8b_nvfp4", 1, 25, 2048, 16, 128, 8192, 32000, ffn_wdtype="nvfp4",
                           attn_wdtype="nvfp4", prompt_len=2048, decode_steps=256),
    # ... and in the xAI page's mixed precision: INT4 g128 q/k/v and FFN matrices,
    # fp16 O projection and LM head, an FP8 E5M2 KV cache
    "1p8b_hpi": Workload("1p8b_hpi", 1, 25, 2048, 16, 128, 8192, 32000, ffn_wdtype="int4_g128",
                         attn_wdtype="int4_g128", kv_dtype="fp8_e5m2", prompt_len=2048, decode_steps=256),
    # the 32K workload with the scaled FP8 E5M2 cache (a scale per layer, K/V and
    # 256-position slice), over a synthetic 32,768-position context
    "1p8b_32k_scaled": Workload("1p8b_32k_scaled", 2, 25, 2048, 16, 128, 8192, 32000,
                                kv_dtype="fp8_e5m2_scaled", kv_source="synthetic", prompt_len=0,
                                context_len=32768, decode_steps=128),
    # the 1.8B fp16 model decoding 8 requests at once (low-batch decode), each over
    # its own synthetic 2048-position context, 256 steps
    "1p8b_b8": Workload("1p8b_b8", 1, 25, 2048, 16, 128, 8192, 32000, kv_source="synthetic", prompt_len=0,
                        context_len=2048, decode_steps=256, batch=8),
}

# tensor ids for the generator: per layer base 64*(layer+1) + slot
_LAYER_SLOTS = {"wq": 1, "wk": 2, "wv": 3, "wo": 4, "w_gate": 6, "w_up": 7, "w_down": 8}
TID_TOK_EMB, TID_LM_HEAD = 1, 3


def layer_tid(layer: int, name: str) -> int:
    return 64 * (layer + 1) + _LAYER_SLOTS[name]


def weight_shapes(w: Workload) -> dict:
    d, f, v = w.d_model, w.ffn_dim, w.vocab
    hd = w.n_heads * w.head_dim
    return {"wq": (hd, d), "wk": (hd, d), "wv": (hd, d), "wo": (d, hd),
            "w_gate": (f, d), "w_up": (f, d), "w_down": (d, f),
            "tok_emb": (v, d), "lm_head": (v, d)}


def gen_weights(w: Workload, seed: int | None = None) -> dict:
    """fp16 weights, PyTorch Linear layout [out, in].  Keys: 'tok_emb', 'lm_head',
    'final_norm', and 'layers' = list of dicts with attn_norm, wq, wk, wv, wo,
    ffn_norm, w_gate, w_up, w_down."""
    seed = w.weight_seed if seed is None else seed
    sh = weight_shapes(w)
    ones = np.ones(w.d_model, dtype=np.float16)
    layers = []
    for l in range(w.n_layers):
        layer = {"attn_norm": ones.copy(), "ffn_norm": ones.copy()}
        for name in _LAYER_SLOTS:
            layer[name] = normal_f16(seed, layer_tid(l, name), sh[name])
        layers.append(layer)
    return {"tok_emb": normal_f16(seed, TID_TOK_EMB, sh["tok_emb"]),
            "lm_head": normal_f16(seed, TID_LM_HEAD, sh["lm_head"]),
            "final_norm": ones.copy(),
            "layers": layers}


def gen_prompt(w: Workload, n: int | None = None, seed: int | None = None) -> np.ndarray:
    seed = w.prompt_seed if seed is None else seed
    return uniform_int(seed, 0, w.prompt_len if n is None else n, w.vocab)


def gen_first_token(w: Workload, seed: int | None = None) -> int:
    """A seeded uniform id used as the first decode input when the context is synthetic."""
    seed = w.prompt_seed if seed is None else seed
    return int(uniform_int(seed, 7, 1, w.vocab)[0])


def gen_kv(w: Workload, layer: int, n_pos: int | None = None, seed: int | None = None):
    """Synthetic post-RoPE K and V for one layer, fp16 [n_pos, n_heads, head_dim]:
    N(0,1) with 0.1% of the entries replaced by +-20."""
    seed = w.kv_seed if seed is None else seed
    n = w.context_len if n_pos is None else n_pos
    shape = (n, w.n_heads, w.head_dim)
    k = outlier_f16(seed, 2 * layer + 1, shape)
    v = outlier_f16(seed, 2 * layer + 2, shape)
    return k, v
