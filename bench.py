"""Batch-1 decode benchmark.

Workload (default): the ~1.8B dense decoder (25 layers, d 2048, 16 heads x 128,
SwiGLU FFN 8192, vocab 32000, fp16 weights ~N(0, 0.02), RMSNorm gains 1), a
2048-token uniform-random prompt prefilled on the GPU (untimed), then steps of
256 greedy decode tokens at positions 2048..2303 (fp16 KV cache).  One bench
step = one kie_generate_greedy of 256 tokens from position 2048.

value   decode tokens/s with every input resident in HBM, timed with CUDA events
        on the engine's stream (one persistent cooperative launch per step).
e2e     the same metric through the host API (kie_generate_greedy with host
        output buffers), wall clock, including the token copy back.
roofline  achieved HBM GB/s of the decode kernel = algorithmic bytes per launch
        (every weight once per token + K/V of all attended positions) / launch
        time, against the measured copy bandwidth.
cpu_baseline  the CPU oracle (numpy fp32) timed on this host's cores on a short
        bounded sample of the same workload.

Multi-GPU (torchrun): independent replicas, one engine per rank, no
collective on the data path; value = tokens of all ranks / max rank time.

workloads  (1 GPU, default run) a compact record for each of the other
        workloads -- 1.8B decoding 8 requests at once (low-batch decode), 1.8B with FP8 E4M3 weights, 1.8B with NVFP4 weights, 1.8B with
        INT4 q/k/v and FFN weights over an E5M2 cache, 1.8B over a 32K FP8-E5M2 cache,
        1.8B over a 32K scaled FP8-E5M2 cache, 1.8B over an 8K adaptive uint8 cache,
        7B with INT4 FFN -- with its
        decode tokens/s, roofline fraction and a CPU-oracle figure.

`--impl reference` times the CPU oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402
from autoregressive_decode_gb300 import traffic  # noqa: E402

METRIC = "batch-1 decode tokens/s per request; achieved HBM GB/s (MBU) vs GB300 peak"
REF_TOKENS = 8       # oracle decode steps per reference-arm bench step


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="1p8b", choices=sorted(S.WORKLOADS))
    ap.add_argument("--mode", default="persistent", choices=["persistent", "graph"])
    ap.add_argument("--decode-tokens", type=int, default=None,
                    help="decode tokens per step (default: the workload's decode steps)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the compact records of the other workloads (1 GPU runs only)")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: the workload with this many layers (a small case of the same "
                         "kernels for multi-pass ncu captures); the line's config records the depth")
    return ap.parse_args()


def workload_desc(w: S.Workload) -> str:
    ctx = (f"{w.prompt_len}-token prompt" if w.kv_source == "prefill" else f"{w.context_len} synthetic KV positions")
    names = {"int4_g128": "INT4 g128", "fp8_e4m3": "FP8 E4M3 (row scales)", "fp16": "fp16",
             "nvfp4": "NVFP4 (E2M1, E4M3 scale per 16 columns, fp32 row scales)"}
    ffn = f"{names[w.ffn_wdtype]} FFN"
    attn = ("" if w.attn_wdtype == "fp16" else ", INT4 g128 q/k/v (fp16 O and LM head)" if w.attn_wdtype == "int4_g128"
            else f", {names[w.attn_wdtype]} q/k/v/o and LM head")
    req = f", {w.batch} requests decoded together (each its own context)" if w.batch > 1 else ""
    return (f"{w.name}: {w.n_layers} layers, d {w.d_model}, {w.n_heads}x{w.head_dim} heads, FFN {w.ffn_dim}, "
            f"vocab {w.vocab}, {ctx}, {w.decode_steps} greedy decode steps, {w.kv_dtype} KV, {ffn}{attn}{req}")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


KERNEL_SOURCES = ["autoregressive_decode_gb300/csrc/kie_decode.cu", "autoregressive_decode_gb300/csrc/kie_decode_core.cuh",
                  "autoregressive_decode_gb300/csrc/kie_device.cuh", "autoregressive_decode_gb300/csrc/kie_internal.h"]


def measured_traffic(w: S.Workload, bpl: float):
    """DRAM bytes per launch from the committed ncu capture, scaled from the
    captured launch to this one by algorithmic bytes; None if the kernel sources
    changed since the capture or the capture is for another workload."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"kie_decode_kernel_{w.name}_traffic.json")
    try:
        rec = json.load(open(path))
        h = hashlib.sha256()
        for p in rec["kernel_sources"]:
            h.update(open(os.path.join(ROOT, p), "rb").read())
        if h.hexdigest() != rec["kernel_sources_sha256"]:
            return None
        return (rec["dram_bytes_read"] + rec["dram_bytes_write"]) * bpl / rec["algorithmic_bytes"]
    except Exception:
        return None


def bytes_per_launch(w: S.Workload, p0: int, n: int) -> float:
    return float(traffic.launch_bytes(w, p0, n))


class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class OracleSample:
    """The oracle decoding the workload on this host: a synthetic fp16 context
    of p0 positions (prefill cost excluded, as for the GPU metric), then timed
    samples of n decode steps from position p0."""

    def __init__(self, w: S.Workload, weights: dict, p0: int, n_steps: int):
        import oracle as O
        self.O = O
        self.p0, self.n = p0, n_steps
        self.dec = O.OracleDecoder(w, weights, max_ctx=p0 + n_steps + 1)
        for layer in range(w.n_layers):
            k, v = S.gen_kv(w.with_(context_len=p0), layer)
            self.dec.set_kv(layer, k, v)
        self.first = S.gen_first_token(w)
        self.dec.pos = p0
        self.dec.decode(self.first)          # warm-up step (page-in, BLAS threads)

    def time(self) -> float:
        """Seconds for n greedy decode steps at positions p0 .. p0 + n - 1."""
        self.dec.pos = self.p0
        tok = self.first
        t0 = time.perf_counter()
        for _ in range(self.n):
            tok = self.O.argmax_lowest(self.dec.decode(tok))
        return time.perf_counter() - t0


def cpu_baseline(w: S.Workload, weights: dict, p0: int, n_steps: int = 8):
    """Time the oracle's decode on this host over n_steps decode steps."""
    threads = len(os.sched_getaffinity(0))
    dt = OracleSample(w, weights, p0, n_steps).time()
    return {"value": n_steps / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_steps} timed decode steps (after 1 warm-up) at positions {p0}..{p0 + n_steps - 1} "
                      f"of {w.name} over a synthetic {p0}-position KV context; numpy fp32 with OpenBLAS"}


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (timing: the slowest replica sets
    the whole job's time); x itself when not distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world_size: int, tokens_per_step: int, ms_per_step: float) -> float:
    """Whole-job throughput of world_size independent replicas (weak scaling:
    every replica decodes tokens_per_step per step) timed by the slowest one."""
    return world_size * tokens_per_step / (ms_per_step / 1e3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def gpu_config(w: S.Workload, n_dec: int, mode: str, replicas: int) -> dict:
    p0 = w.start_pos
    return {"workload": workload_desc(w), "decode_tokens_per_step": n_dec,
            "positions": f"{p0}..{p0 + n_dec - 1}", "mode": mode,
            "l2": "inputs larger than L2 (all weights streamed from HBM every token)",
            "replicas": replicas}


def run_reference(args, w: S.Workload):
    """The reference arm: the CPU oracle as it stands, on this host's cores.
    One bench step = one timed sample of REF_TOKENS greedy decode steps of the
    same workload (its full 256-token chain would take minutes per step on the
    CPU); ms_per_step is that sample's measured time."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    n_ref = REF_TOKENS
    weights = S.gen_weights(w)
    sample = OracleSample(w, weights, w.start_pos, n_ref)
    times = []
    for i in range(args.warmup + args.steps):
        dt = sample.time()
        if i >= args.warmup:
            times.append(dt)
    sec = statistics.median(times)
    val = n_ref / sec
    cores = len(os.sched_getaffinity(0))
    desc = (f"{n_ref} greedy decode steps per bench step at positions {w.start_pos}..{w.start_pos + n_ref - 1} of "
            f"{w.name} over a synthetic {w.start_pos}-position KV context (prefill excluded); numpy fp32 with "
            f"OpenBLAS; median of {args.steps} timed samples after {args.warmup} warm-up")
    cfg = gpu_config(w, n_ref, "oracle (CPU)", 1)
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_by_depth(w: S.Workload, weights: dict, p0: int, n_steps: int = 3):
    """The oracle on this host for a large workload, from a bounded sample: its
    first one and first two layers (same weights, LM head and a synthetic
    p0-position context) each decode n_steps tokens; the per-layer time (the
    difference) extrapolates linearly to the workload's full depth."""
    per = []
    for depth in (1, 2):
        wd = w.with_(n_layers=depth)
        wt = dict(weights, layers=weights["layers"][:depth])
        sample = OracleSample(wd, wt, p0, n_steps)
        per.append(statistics.median(sample.time() / n_steps for _ in range(2)))
        del sample
    t_layer = max(per[1] - per[0], 0.0)
    t_full = per[0] + (w.n_layers - 1) * t_layer
    return {"value": 1.0 / t_full, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{n_steps} decode steps at positions {p0}..{p0 + n_steps - 1} of {w.name} at depth 1 "
                      f"({per[0] * 1e3:.0f} ms/token) and depth 2 ({per[1] * 1e3:.0f} ms/token), extrapolated "
                      f"linearly to {w.n_layers} layers; numpy fp32 with OpenBLAS"}


def time_decode(eng, torch, stream, first: int, p0: int, n_dec: int, steps: int, warmup: int, device):
    """Mean ms of `steps` device-timed generate launches of n_dec tokens from p0."""
    d_tok = torch.empty(n_dec, dtype=torch.int32, device=device)
    for _ in range(warmup):
        eng.set_pos(p0)
        eng.generate_greedy_device(first, n_dec, d_tok)
    eng.sync()
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in per:
        eng.set_pos(p0)
        a.record(stream)
        eng.generate_greedy_device(first, n_dec, d_tok)
        b.record(stream)
    eng.sync()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in per)


def time_decode_batch(eng, torch, stream, firsts, p0: int, n_dec: int, steps: int, warmup: int, device):
    """Mean ms of `steps` device-timed batched launches of n_dec tokens per
    request, every request restarting from position p0."""
    B = len(firsts)
    d_tok = torch.empty((n_dec, B), dtype=torch.int32, device=device)

    def restart():
        for b in range(B):
            eng.select_request(b)
            eng.set_pos(p0)

    for _ in range(warmup):
        restart()
        eng.generate_greedy_batch_device(firsts, n_dec, d_tok)
    eng.sync()
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in per:
        restart()
        a.record(stream)
        eng.generate_greedy_batch_device(firsts, n_dec, d_tok)
        b.record(stream)
    eng.sync()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in per)


def batched_record(args, local, kie, torch, w, weights, peak, peak_kind):
    """Low-batch decode: w.batch requests, each over its own synthetic context
    (request b's KV and first token from its own seeds), decoded together."""
    B, p0, n_dec = w.batch, w.context_len, w.decode_steps
    cfg = kie.make_config(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab, p0 + n_dec,
                          w.rms_eps, w.rope_theta, w.kv_dtype, w.ffn_wdtype, "persistent", local,
                          attn_wdtype=w.attn_wdtype, batch=B)
    stream = torch.cuda.Stream(device=local)
    eng = kie.Engine(cfg, stream=stream)
    eng.load_weights(weights)
    for b in range(B):
        eng.select_request(b)
        for layer in range(w.n_layers):
            k, v = S.gen_kv(w, layer, seed=w.request_seed(w.kv_seed, b))
            eng.set_kv(layer, k, v)
        eng.set_pos(p0)
    firsts = [S.gen_first_token(w, seed=w.request_seed(w.prompt_seed, b)) for b in range(B)]
    ms = time_decode_batch(eng, torch, stream, firsts, p0, n_dec, 3, 2, f"cuda:{local}")
    eng.close()
    bpl = float(traffic.batch_launch_bytes(w, [p0] * B, n_dec))
    achieved = bpl / (ms / 1e3) / 1e9
    rec = {"context": f"synthetic, {p0} positions per request (own seeds)", "requests": B,
           "value": B * n_dec / (ms / 1e3), "unit": "tokens/s (all requests)",
           "per_request_tokens_per_s": n_dec / (ms / 1e3), "steps": 3, "warmup": 2, "ms_per_step": ms,
           "decode_tokens_per_step": B * n_dec, "positions": f"{p0}..{p0 + n_dec - 1} in every request",
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                        "frac": achieved / peak, "peak_source": peak_kind, "kernel": "kie_decode_batch_kernel",
                        "algorithmic_bytes_per_launch": bpl, "launch_ms": ms,
                        "bytes": "every weight once per step plus each request's own K and V"}}
    if not args.no_cpu_baseline:
        cb = cpu_baseline_by_depth(w.with_(batch=1), weights, p0)
        cb["sample"] += "; per request: the oracle decodes the requests one after another, so its rate over " \
                        "all requests is the same"
        rec["cpu_baseline"] = cb
    return rec


# The other workloads (a compact record each): their decode steps over the
# context the workload names, prefilled on the GPU where the tensor-core path
# covers it and otherwise (uint8 cache; the 7B model, whose decode bytes do not
# depend on how its 4,096-position context was made) a synthetic one.
EXTRA = ("1p8b_b8", "1p8b_fp8", "1p8b_nvfp4", "1p8b_hpi", "1p8b_32k", "1p8b_32k_scaled", "1p8b_u8", "7b_int4")


def extra_workloads(args, local, kie, torch, weights_1p8b):
    peak, peak_kind = peaks()
    out = {}
    w7 = None
    for name in EXTRA:
        w = S.WORKLOADS[name]
        rec = {"workload": workload_desc(w)}
        try:
            if w.d_model == 2048:
                weights = weights_1p8b
                rec["weights"] = "the 1p8b workload's seeded weights (the 1.8B variants share one weight set here)"
            else:
                w7 = w7 or S.gen_weights(w)
                weights = w7
            if w.batch > 1:
                rec.update(batched_record(args, local, kie, torch, w, weights, peak, peak_kind))
                out[name] = rec
                continue
            synth = w.kv_source == "synthetic" or w.ffn_wdtype == "int4_g128"
            if synth and w.kv_source == "prefill":
                w = w.with_(kv_source="synthetic", context_len=w.prompt_len, prompt_len=0)
            p0, n_dec = w.start_pos, w.decode_steps
            cfg = kie.make_config(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab, p0 + n_dec,
                                  w.rms_eps, w.rope_theta, w.kv_dtype, w.ffn_wdtype, "persistent", local,
                                  attn_wdtype=w.attn_wdtype)
            stream = torch.cuda.Stream(device=local)
            eng = kie.Engine(cfg, stream=stream)
            eng.load_weights(weights)
            if synth:
                for layer in range(w.n_layers):
                    k, v = S.gen_kv(w, layer)
                    eng.set_kv(layer, k, v)
                eng.set_pos(p0)
                first = S.gen_first_token(w)
                rec["context"] = f"synthetic, {p0} positions"
            else:
                prompt = S.gen_prompt(w)
                torch.cuda.synchronize()
                t0 = time.perf_counter()
                first = int(np.argmax(eng.prefill(prompt)))
                pf_ms = (time.perf_counter() - t0) * 1e3
                rec["context"] = f"GPU prefill of the {p0}-token prompt"
                rec["prefill"] = {"tokens": p0, "ms": pf_ms, "tokens_per_s": p0 / (pf_ms / 1e3),
                                  "path": "tcgen05 GEMM"}
            ms = time_decode(eng, torch, stream, first, p0, n_dec, 3, 2, f"cuda:{local}")
            eng.close()
            bpl = bytes_per_launch(w, p0, n_dec)
            achieved = bpl / (ms / 1e3) / 1e9
            rec.update({"value": n_dec / (ms / 1e3), "unit": "tokens/s", "steps": 3, "warmup": 2,
                        "ms_per_step": ms, "decode_tokens_per_step": n_dec,
                        "positions": f"{p0}..{p0 + n_dec - 1}",
                        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                                     "frac": achieved / peak, "peak_source": peak_kind,
                                     "kernel": "kie_decode_kernel", "algorithmic_bytes_per_launch": bpl,
                                     "launch_ms": ms}})
            if not args.no_cpu_baseline:
                rec["cpu_baseline"] = cpu_baseline_by_depth(w, weights, p0)
        except Exception as ex:  # report, never hide
            rec["error"] = repr(ex)
        out[name] = rec
    return out


def main():
    args = parse()
    w = S.WORKLOADS[args.workload]
    if args.layers:
        w = w.with_(n_layers=args.layers)
    if w.batch > 1 and args.impl != "reference":
        # the batched workload is reported as a record of the default run
        if not args.no_workloads:
            raise SystemExit(f"{w.name}: run the default workload; its record is under 'workloads'")
        import torch

        from autoregressive_decode_gb300 import kie
        torch.cuda.set_device(0)
        peak, kind = peaks()
        rec = batched_record(args, 0, kie, torch, w, S.gen_weights(w), peak, kind)
        print(json.dumps({"workload": workload_desc(w), **rec}))
        return
    if args.impl == "reference":
        return run_reference(args, w)
    import torch

    from autoregressive_decode_gb300 import kie

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    n_dec = args.decode_tokens or w.decode_steps
    p0 = w.start_pos
    weights = S.gen_weights(w)
    cfg = kie.make_config(w.n_layers, w.d_model, w.n_heads, w.head_dim, w.ffn_dim, w.vocab, p0 + n_dec,
                          w.rms_eps, w.rope_theta, w.kv_dtype, w.ffn_wdtype, args.mode, local,
                          attn_wdtype=w.attn_wdtype)
    stream = torch.cuda.Stream(device=local)
    eng = kie.Engine(cfg, stream=stream)
    eng.load_weights(weights)
    # context: GPU prefill of the prompt (untimed), or synthetic KV
    prefill_info = None
    if w.kv_source == "prefill":
        prompt = S.gen_prompt(w)
        lg = eng.prefill(prompt)
        first = int(np.argmax(lg))
        # the prompt once more, timed (row a0, not on the decode metric's clock):
        # it rewrites the same cache positions with the same values
        eng.set_pos(0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        lg2 = eng.prefill(prompt)
        pf_ms = (time.perf_counter() - t0) * 1e3
        assert int(np.argmax(lg2)) == first
        prefill_info = {"tokens": len(prompt), "ms": pf_ms, "tokens_per_s": len(prompt) / (pf_ms / 1e3),
                        "path": "tcgen05 GEMM" if w.ffn_wdtype != "int4_g128" and w.kv_dtype != "u8"
                        else "decode kernel"}
    else:
        for layer in range(w.n_layers):
            k, v = S.gen_kv(w, layer)
            eng.set_kv(layer, k, v)
        eng.set_pos(p0)
        first = S.gen_first_token(w)
    d_tok = torch.empty(n_dec, dtype=torch.int32, device=f"cuda:{local}")

    def step():
        eng.set_pos(p0)
        eng.generate_greedy_device(first, n_dec, d_tok)

    for _ in range(args.warmup):
        step()
    eng.sync()
    # device-timed region
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        ev0.record(stream)
        for a, b in per:
            eng.set_pos(p0)
            a.record(stream)
            eng.generate_greedy_device(first, n_dec, d_tok)
            b.record(stream)
        ev1.record(stream)
        eng.sync()
        torch.cuda.synchronize()
    total_ms = ev0.elapsed_time(ev1)
    launch_ms = [a.elapsed_time(b) for a, b in per]
    if ws > 1:
        total_ms = max_over_ranks(total_ms, f"cuda:{local}")
        dist.barrier()
    tokens_gpu = list(d_tok.cpu().numpy())

    # end to end through the host API
    e2e_ms = []
    for i in range(max(2, args.steps // 2) + 1):
        eng.set_pos(p0)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        toks, _ = eng.generate_greedy(first, n_dec)
        dt = (time.perf_counter() - t0) * 1e3
        if i > 0:
            e2e_ms.append(dt)
    assert list(toks) == tokens_gpu, "host-API tokens differ from the device-timed run"
    if ws > 1:
        e2e_max = max_over_ranks(max(e2e_ms), f"cuda:{local}")
    else:
        e2e_max = statistics.median(e2e_ms)

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    ms_per_step = total_ms / args.steps
    value = job_tokens_per_s(ws, n_dec, ms_per_step)
    peak, peak_kind = peaks()
    bpl = bytes_per_launch(w, p0, n_dec)
    launch_avg = statistics.mean(launch_ms)
    achieved = bpl / (launch_avg / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "storage": f"weights attn {w.attn_wdtype} / FFN {w.ffn_wdtype}, KV {w.kv_dtype}",
        "data": "synthetic",
        "config": gpu_config(w, n_dec, args.mode, ws),
        # per step: the control-block kernel of set_pos, then one cooperative decode launch
        # (persistent) or a control kernel plus (5L+1) phase kernels per token (graph)
        "gpu_launches": args.steps * (2 if args.mode == "persistent" else 2 + (5 * w.n_layers + 1) * n_dec),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": measured_traffic(w, bpl), "peak_source": peak_kind, "kernel": "kie_decode_kernel",
                     "algorithmic_bytes_per_launch": bpl, "launch_ms": launch_avg},
        "e2e": {"value": job_tokens_per_s(ws, n_dec, e2e_max), "unit": "tokens/s", "h2d_bytes_per_step": 4,
                "d2h_bytes_per_step": 4 * n_dec},
        "clocks": clk.summary(),
    }
    if prefill_info:
        line["prefill"] = prefill_info
    if not args.no_cpu_baseline and ws >= 1:
        try:
            line["cpu_baseline"] = cpu_baseline(w, weights, p0)
        except Exception as ex:  # report, never hide
            line["cpu_baseline"] = {"error": repr(ex)}
    eng.close()
    if ws == 1 and not args.no_workloads and not args.layers and args.workload == "1p8b" and args.mode == "persistent":
        line["workloads"] = extra_workloads(args, local, kie, torch, weights)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
