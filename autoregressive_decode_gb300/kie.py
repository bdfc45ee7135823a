"""Thin ctypes binding of libkie.so (argument marshalling only).

Every entry point of include/kie.h is exposed under the same name on ``lib``;
``Engine`` wraps one engine handle.  All computation happens in the CUDA
library: if the library cannot be loaded this module raises instead of falling
back to anything else.

Arrays may be numpy arrays (host memory) or torch tensors; torch CUDA tensors
are passed as device pointers where the C entry point takes device pointers
(kie_generate_greedy_device, kie_load_weights with on_device = 1, the
workspace of kie_create).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import _build

KIE_OK, KIE_ERR_INVALID_ARG, KIE_ERR_OOM, KIE_ERR_CUDA = 0, -1, -2, -3
KIE_ERR_NOT_LOADED, KIE_ERR_CTX_OVERFLOW, KIE_ERR_DEVICE_TIMEOUT = -4, -5, -6
KIE_ERR_LAUNCH, KIE_ERR_UNSUPPORTED = -7, -8
KV_DTYPES = {"fp16": 0, "fp8_e5m2": 1, "u8": 2, "fp8_e5m2_scaled": 3}
W_DTYPES = {"fp16": 0, "int4_g128": 1, "fp8_e4m3": 2, "nvfp4": 3}
MODES = {"persistent": 0, "graph": 1}

STATUS_NAMES = {0: "KIE_OK", -1: "KIE_ERR_INVALID_ARG", -2: "KIE_ERR_OOM", -3: "KIE_ERR_CUDA",
                -4: "KIE_ERR_NOT_LOADED", -5: "KIE_ERR_CTX_OVERFLOW", -6: "KIE_ERR_DEVICE_TIMEOUT",
                -7: "KIE_ERR_LAUNCH", -8: "KIE_ERR_UNSUPPORTED"}


class KieError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class kie_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
                ("head_dim", C.c_int32), ("ffn_dim", C.c_int32), ("vocab", C.c_int32),
                ("max_ctx", C.c_int32), ("rms_eps", C.c_float), ("rope_theta", C.c_float),
                ("kv_dtype", C.c_int32), ("ffn_wdtype", C.c_int32), ("mode", C.c_int32),
                ("device", C.c_int32), ("attn_wdtype", C.c_int32), ("batch", C.c_int32),
                ("kv_scale_k", C.c_float), ("kv_scale_v", C.c_float)]


class kie_layer_weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm",
                                         "w_gate", "w_up", "w_down")]


class kie_weights(C.Structure):
    _fields_ = [("tok_emb", C.c_void_p), ("final_norm", C.c_void_p), ("lm_head", C.c_void_p),
                ("layers", C.POINTER(kie_layer_weights)), ("on_device", C.c_int32)]


EXPORTS = {
    # name: (restype, argtypes)
    "kie_workspace_bytes": (C.c_size_t, [C.POINTER(kie_config)]),
    "kie_create": (C.c_int, [C.POINTER(kie_config), C.c_void_p, C.c_size_t, C.c_void_p, C.POINTER(C.c_void_p)]),
    "kie_load_weights": (C.c_int, [C.c_void_p, C.POINTER(kie_weights)]),
    "kie_prefill": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p]),
    "kie_decode_step": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int32), C.c_void_p]),
    "kie_generate_greedy": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_generate_greedy_device": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_sync": (C.c_int, [C.c_void_p]),
    "kie_decode_step_static_scratch": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_trace_decode": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_size_t]),
    "kie_select_request": (C.c_int, [C.c_void_p, C.c_int32]),
    "kie_decode_batch": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "kie_generate_greedy_batch": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_generate_greedy_batch_device": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_reset": (C.c_int, [C.c_void_p]),
    "kie_get_pos": (C.c_int32, [C.c_void_p]),
    "kie_set_pos": (C.c_int, [C.c_void_p, C.c_int32]),
    "kie_set_timeout_ms": (C.c_int, [C.c_void_p, C.c_int32]),
    "kie_debug_skip_grid_arrival": (C.c_int, [C.c_void_p, C.c_int32]),
    "kie_get_stream": (C.c_void_p, [C.c_void_p]),
    "kie_grid_size": (C.c_int32, [C.c_void_p]),
    "kie_last_error": (C.c_char_p, [C.c_void_p]),
    "kie_destroy": (None, [C.c_void_p]),
    "kie_set_kv": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_int32]),
    "kie_read_kv": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                              C.c_void_p, C.c_void_p, C.c_void_p]),
    "kie_quantize_kv_u8": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "kie_quantize_int4_g128": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_quantize_fp8_rows": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p]),
    "kie_quantize_nvfp4_rows": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]),
    "kie_convert_fp8_e5m2": (C.c_int, [C.c_void_p, C.c_size_t, C.c_void_p]),
}

_lib = None


def load(build: bool = True):
    """Load libkie.so (building it first if missing or stale)."""
    global _lib
    if _lib is None:
        path = _build.build() if build else _build.LIB
        if not os.path.exists(path):
            raise OSError(f"libkie.so not found at {path}")
        lib = C.CDLL(path)
        for name, (res, args) in EXPORTS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _ptr(a):
    """Address of a numpy array or torch tensor (None -> NULL)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return a.ctypes.data
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return a.data_ptr()
    raise TypeError(f"unsupported buffer type {type(a)}")


def _check(st, eng=None):
    if st != KIE_OK:
        msg = load().kie_last_error(eng)
        raise KieError(st, msg.decode() if msg else "")


def make_config(n_layers, d_model, n_heads, head_dim, ffn_dim, vocab, max_ctx, rms_eps=1e-5, rope_theta=10000.0,
                kv_dtype="fp16", ffn_wdtype="fp16", mode="persistent", device=0, attn_wdtype="fp16",
                batch=1, kv_scale=(0.0, 0.0)) -> kie_config:
    return kie_config(n_layers, d_model, n_heads, head_dim, ffn_dim, vocab, max_ctx, rms_eps, rope_theta,
                      KV_DTYPES[kv_dtype], W_DTYPES[ffn_wdtype], MODES[mode], device, W_DTYPES[attn_wdtype],
                      int(batch), float(kv_scale[0]), float(kv_scale[1]))


class Engine:
    """One engine handle (kie_create .. kie_destroy)."""

    def __init__(self, cfg: kie_config, stream=None, workspace=None):
        lib = load()
        self.cfg = cfg
        self._ws = workspace                 # kept alive for the engine's lifetime
        h = C.c_void_p()
        ws_ptr = _ptr(workspace)
        ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        st_ptr = None if stream is None else (stream if isinstance(stream, int) else stream.cuda_stream)
        _check(lib.kie_create(C.byref(cfg), ws_ptr, ws_bytes, st_ptr, C.byref(h)))
        self.h = h
        self.vocab = cfg.vocab
        self.batch = max(1, cfg.batch)

    # -- lifetime -------------------------------------------------------------------------
    def close(self):
        if getattr(self, "h", None):
            load().kie_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- API --------------------------------------------------------------------------------
    def load_weights(self, w: dict):
        """w: dict as from synthetic.gen_weights (numpy fp16 arrays, or torch CUDA fp16 tensors)."""
        layers = w["layers"]
        on_dev = int(not isinstance(w["tok_emb"], np.ndarray) and getattr(w["tok_emb"], "is_cuda", False))
        arr = (kie_layer_weights * len(layers))()
        keep = []
        for i, lw in enumerate(layers):
            for n in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down"):
                setattr(arr[i], n, _ptr(lw[n]))
                keep.append(lw[n])
        kw = kie_weights(_ptr(w["tok_emb"]), _ptr(w["final_norm"]), _ptr(w["lm_head"]),
                         C.cast(arr, C.POINTER(kie_layer_weights)), on_dev)
        _check(load().kie_load_weights(self.h, C.byref(kw)), self.h)

    def prefill(self, tokens, want_logits: bool = True):
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty(self.vocab, np.float32) if want_logits else None
        _check(load().kie_prefill(self.h, _ptr(toks), len(toks), _ptr(out)), self.h)
        return out

    def decode_step(self, token: int, want_logits: bool = True):
        nxt = C.c_int32()
        out = np.empty(self.vocab, np.float32) if want_logits else None
        _check(load().kie_decode_step(self.h, int(token), C.byref(nxt), _ptr(out)), self.h)
        return nxt.value, out

    def generate_greedy(self, first_token: int, n: int, want_logits: bool = False):
        toks = np.empty(n, np.int32)
        logs = np.empty((n, self.vocab), np.float32) if want_logits else None
        _check(load().kie_generate_greedy(self.h, int(first_token), int(n), _ptr(toks), _ptr(logs)), self.h)
        return toks, logs

    def generate_greedy_device(self, first_token: int, n: int, d_tokens, d_logits=None):
        _check(load().kie_generate_greedy_device(self.h, int(first_token), int(n), _ptr(d_tokens), _ptr(d_logits)),
               self.h)

    def trace_decode(self, first_token: int, n: int):
        """n greedy steps with per-phase stamps: (uint64 [n, 5L+1, 6, grid],
        ring trace of CTA 0 [32768, 4]) in ns."""
        shape = (n, 5 * self.cfg.n_layers + 1, 6, self.grid)
        nph = int(np.prod(shape))
        buf = np.zeros(nph + 32768 * 4, np.uint64)
        _check(load().kie_trace_decode(self.h, int(first_token), int(n), _ptr(buf), buf.size), self.h)
        return buf[:nph].reshape(shape), buf[nph:].reshape(32768, 4)

    def decode_step_static_scratch(self, token: int, d_next_token, d_logits=None):
        """kie_decode_step_static_scratch: device outputs, no allocation, no sync."""
        _check(load().kie_decode_step_static_scratch(self.h, int(token), _ptr(d_next_token), _ptr(d_logits)), self.h)

    # -- batched engines --------------------------------------------------------------------
    def select_request(self, b: int):
        """Address request b with prefill / set_kv / read_kv / set_pos / pos."""
        _check(load().kie_select_request(self.h, int(b)), self.h)

    def decode_batch(self, tokens, want_logits: bool = True):
        """One step of every request: (next tokens [batch], logits [batch, vocab] or None)."""
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        nxt = np.empty(self.batch, np.int32)
        out = np.empty((self.batch, self.vocab), np.float32) if want_logits else None
        _check(load().kie_decode_batch(self.h, _ptr(t), _ptr(nxt), _ptr(out)), self.h)
        return nxt, out

    def generate_greedy_batch(self, first_tokens, n: int, want_logits: bool = False):
        """n greedy steps of every request: (tokens [n, batch], logits [n, batch, vocab] or None)."""
        f = np.ascontiguousarray(first_tokens, dtype=np.int32)
        toks = np.empty((n, self.batch), np.int32)
        logs = np.empty((n, self.batch, self.vocab), np.float32) if want_logits else None
        _check(load().kie_generate_greedy_batch(self.h, _ptr(f), int(n), _ptr(toks), _ptr(logs)), self.h)
        return toks, logs

    def generate_greedy_batch_device(self, first_tokens, n: int, d_tokens, d_logits=None):
        f = np.ascontiguousarray(first_tokens, dtype=np.int32)
        _check(load().kie_generate_greedy_batch_device(self.h, _ptr(f), int(n), _ptr(d_tokens), _ptr(d_logits)),
               self.h)

    def sync(self):
        _check(load().kie_sync(self.h), self.h)

    def reset(self):
        _check(load().kie_reset(self.h), self.h)

    @property
    def pos(self) -> int:
        return load().kie_get_pos(self.h)

    def set_pos(self, pos: int):
        _check(load().kie_set_pos(self.h, int(pos)), self.h)

    def set_timeout_ms(self, ms: int):
        _check(load().kie_set_timeout_ms(self.h, int(ms)), self.h)

    def debug_skip_grid_arrival(self, cta: int):
        """Failure injection (tests): CTA `cta` skips its first grid-barrier
        arrival in the next persistent launch of several steps."""
        _check(load().kie_debug_skip_grid_arrival(self.h, int(cta)), self.h)

    @property
    def stream(self) -> int:
        return load().kie_get_stream(self.h) or 0

    @property
    def grid(self) -> int:
        return load().kie_grid_size(self.h)

    def set_kv(self, layer: int, k16: np.ndarray, v16: np.ndarray):
        k = np.ascontiguousarray(k16, dtype=np.float16)
        v = np.ascontiguousarray(v16, dtype=np.float16)
        _check(load().kie_set_kv(self.h, int(layer), _ptr(k), _ptr(v), k.shape[0]), self.h)

    def read_kv(self, layer: int, which: int, p0: int, n: int):
        """Raw storage of K (which=0) or V (1): (data [H, n, h], tail fp16 or None,
        scale [H, nseg] (uint8) / [nslices] (scaled E5M2) or None, zp [H, nseg] or None)."""
        H, h = self.cfg.n_heads, self.cfg.head_dim
        kv = self.cfg.kv_dtype
        data = np.empty((H, n, h), np.uint16 if kv == 0 else np.uint8)
        tail = sc = zp = None
        if kv == 3:   # scaled E5M2: the scales of the slices the range meets
            sc = np.zeros((p0 + n + 255) // 256 - p0 // 256, np.float32)
        if kv == 2:
            tail = np.zeros((H, n, h), np.uint16)
            nseg = (p0 + n + 127) // 128 - p0 // 128
            sc = np.zeros((H, nseg), np.float32)
            zp = np.zeros((H, nseg), np.int32)
        _check(load().kie_read_kv(self.h, int(layer), int(which), int(p0), int(n), _ptr(data), _ptr(tail), _ptr(sc),
                                  _ptr(zp)), self.h)
        return data, tail, sc, zp


# ---- stateless routines ----------------------------------------------------------------------
def quantize_kv_u8(x16: np.ndarray, n_seg: int):
    x = np.ascontiguousarray(x16, dtype=np.float16).reshape(-1)
    seg = x.size // n_seg
    codes = np.empty(x.size, np.uint8)
    scale = np.empty(n_seg, np.float32)
    zp = np.empty(n_seg, np.int32)
    _check(load().kie_quantize_kv_u8(_ptr(x), n_seg, seg, _ptr(codes), _ptr(scale), _ptr(zp)))
    return codes.reshape(n_seg, seg), scale, zp


def quantize_int4_g128(w16: np.ndarray):
    w = np.ascontiguousarray(w16, dtype=np.float16)
    rows, cols = w.shape
    codes = np.empty((rows, cols), np.int8)
    sc = np.empty((rows, cols // 128), np.uint16)
    _check(load().kie_quantize_int4_g128(_ptr(w), rows, cols, _ptr(codes), _ptr(sc)))
    return codes, sc.view(np.float16)


def quantize_fp8_rows(w16: np.ndarray):
    """kie_quantize_fp8_rows: (codes uint8 [rows, cols], scales fp32 [rows])."""
    w = np.ascontiguousarray(w16, dtype=np.float16)
    rows, cols = w.shape
    codes = np.empty((rows, cols), np.uint8)
    sc = np.empty(rows, np.float32)
    _check(load().kie_quantize_fp8_rows(_ptr(w), rows, cols, _ptr(codes), _ptr(sc)))
    return codes, sc


def quantize_nvfp4_rows(w16: np.ndarray):
    """kie_quantize_nvfp4_rows: (E2M1 codes uint8 [rows, cols] in 0..15,
    E4M3 block-scale bytes uint8 [rows, cols/16], row scales fp32 [rows])."""
    w = np.ascontiguousarray(w16, dtype=np.float16)
    rows, cols = w.shape
    codes = np.empty((rows, cols), np.uint8)
    bs = np.empty((rows, cols // 16), np.uint8)
    rs = np.empty(rows, np.float32)
    _check(load().kie_quantize_nvfp4_rows(_ptr(w), rows, cols, _ptr(codes), _ptr(bs), _ptr(rs)))
    return codes, bs, rs


def convert_fp8_e5m2(x16: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x16, dtype=np.float16).reshape(-1)
    out = np.empty(x.size, np.uint8)
    _check(load().kie_convert_fp8_e5m2(_ptr(x), x.size, _ptr(out)))
    return out
