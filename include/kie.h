/*
 * kie.h — C ABI of the batch-1 decode engine (libkie.so) for one GB300 (sm_103a).
 *
 * What it computes.  The single-request autoregressive decode step of a dense
 * decoder-only transformer (pre-norm RMSNorm, RoPE, multi-head attention over a
 * KV cache, SwiGLU FFN, untied LM head, greedy argmax).  The Kog page "Real-time
 * LLM inference on standard GPUs: 3,000 tokens/s per request", section "Memory
 * bandwidth is the main bottleneck", frames this step as bandwidth bound:
 * tokens/s <= effective_bandwidth / (beta * active_weight_bytes + KV bytes); its
 * table "Where standard inference stacks lose microseconds" asks for one
 * persistent GPU program over the whole decode path (row "kernel boundaries"),
 * LM head and sampling kept on the GPU (row "CPU scheduling and sampling"), and
 * prefetch across non-GEMM work (row "non-GEMM work").  KV storage formats:
 * fp16; FP8 E5M2 converted from fp16 and dequantised to fp16 on load (xAI page
 * "How the xAI team pushed Grok Bot latency down to milliseconds", section 2.3);
 * adaptive-range uint8 with per-128-token-segment scale/zero-point (Grok-3
 * v3.2.4 hot-update page, section 3.2).  FFN weights fp16 or INT4 W4A16, group
 * 128, symmetric (xAI page sections 2.3 and 3.3).
 *
 * Numeric contract.  Weights are fp16 (or INT4 codes + fp16 scales); every
 * product, sum, norm, softmax and residual is fp32; K/V are rounded to fp16
 * (round to nearest even) before storage and, for FP8, converted from that fp16
 * to E5M2 (round to nearest even, saturating to +-57344).
 *
 * Conventions (all entry points).
 *  - Every call returns a kie_status; KIE_OK == 0, errors are negative.  The
 *    message of the last failure is available from kie_last_error().
 *  - An engine is used from one host thread at a time and runs all its GPU work
 *    on the stream given at creation.  Calls that take host output pointers
 *    synchronise that stream before returning; the *_device variants do not.
 *  - Pointers are host pointers unless the name or comment says device.  The
 *    caller owns every buffer it passes; the engine never keeps a caller's
 *    pointer after the call returns.
 *  - Token ids are int32 in [0, vocab); any other id gives KIE_ERR_INVALID_ARG
 *    and nothing is written.
 *  - A call that would take the position past max_ctx returns
 *    KIE_ERR_CTX_OVERFLOW and writes nothing.
 *  - Every wait inside the GPU program is bounded (default 2 s, see
 *    kie_set_timeout_ms); when one expires the program stops, the call returns
 *    KIE_ERR_DEVICE_TIMEOUT and the engine refuses further decode calls until
 *    kie_reset().
 */
#ifndef KIE_H
#define KIE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KIE_OK = 0,
    KIE_ERR_INVALID_ARG = -1,   /* bad pointer, size, token id, layer index or config      */
    KIE_ERR_OOM = -2,           /* device allocation failed, or the workspace is too small  */
    KIE_ERR_CUDA = -3,          /* a CUDA runtime call failed (message has the CUDA error)  */
    KIE_ERR_NOT_LOADED = -4,    /* decode/prefill before kie_load_weights                  */
    KIE_ERR_CTX_OVERFLOW = -5,  /* pos + n > max_ctx                                       */
    KIE_ERR_DEVICE_TIMEOUT = -6,/* a bounded wait inside the GPU program expired          */
    KIE_ERR_LAUNCH = -7,        /* the persistent grid cannot be co-resident on this GPU   */
    KIE_ERR_UNSUPPORTED = -8    /* shape or option outside what this build implements      */
} kie_status;

/* KV cache storage.  FP16.  FP8_E5M2: E5M2 of the fp16 value, no scale (xAI
 * page section 2.3).  U8_ADAPTIVE: uint8 codes with a scale and zero point per
 * 128-token segment and head (Grok-3 hot-update page section 3.2).
 * FP8_E5M2_SCALED: E5M2 codes of fp16(v) / s, read back as code * s, with one
 * scale s per layer, K or V and 256-position slice (xAI page section 3.3's
 * per-tensor k_cache / v_cache scales, recomputed every 256 tokens from the
 * cache): slice 0 uses kv_scale_k / kv_scale_v; slice j >= 1 takes, when its
 * first position is written, the largest magnitude m of slice j-1's stored
 * codes and s_j = (m * s_{j-1}) / 127, or s_{j-1} when that is zero or not
 * finite.  Prompts prefill through the decode kernel for this format. */
typedef enum { KIE_KV_FP16 = 0, KIE_KV_FP8_E5M2 = 1, KIE_KV_U8_ADAPTIVE = 2, KIE_KV_FP8_E5M2_SCALED = 3 } kie_kv_dtype;
/* Weight storage of the GEMV matrices.  FP16: as given.  INT4_G128: symmetric
 * INT4, group 128 (xAI page sections 2.3, 3.3); as ffn_wdtype it covers the
 * three FFN matrices, as attn_wdtype the q, k and v projections only (the same
 * page's section 2.3 names the QKV projection), with wo and the LM head kept
 * in fp16.  FP8_E4M3: one byte
 * per weight with one fp32 scale per output row, s = absmax/448, codes = E4M3
 * of w/s rounded to nearest even, saturating (the Kog page's "FP8 ~2 FLOP per
 * byte", section "Memory bandwidth is the main bottleneck"; the format and the
 * scale granularity are this engine's reading).  NVFP4: E2M1 codes (half a
 * byte per weight), an E4M3 scale per 16 consecutive input columns and an fp32
 * scale per output row (the same page's "FP4 ~4 FLOP per byte"; the format is
 * this engine's reading: Blackwell's native 4-bit layout), quantised as
 * kie_quantize_nvfp4_rows describes; the matrices' input dimension must be a
 * multiple of 16. */
typedef enum { KIE_W_FP16 = 0, KIE_W_INT4_G128 = 1, KIE_W_FP8_E4M3 = 2, KIE_W_NVFP4 = 3 } kie_w_dtype;
/* PERSISTENT: one cooperative launch runs all requested tokens (a grid-wide
 * barrier between steps; the phases of a step are ordered by tagged
 * activations).  GRAPH: the same phases as separate launches,
 * captured once into a CUDA graph per engine and replayed once per token.
 * Both give bit-identical tokens and logits (same partitioning and reduction
 * order). */
typedef enum { KIE_MODE_PERSISTENT = 0, KIE_MODE_GRAPH = 1 } kie_mode;

typedef struct {
    int32_t n_layers;
    int32_t d_model;      /* multiple of 8 (of 128 for INT4 attention weights)      */
    int32_t n_heads;      /* query heads == KV heads (multi-head attention)         */
    int32_t head_dim;     /* 64 or 128                                              */
    int32_t ffn_dim;      /* multiple of 8 (of 128 for INT4 FFN)                    */
    int32_t vocab;
    int32_t max_ctx;      /* KV positions to allocate                               */
    float rms_eps;
    float rope_theta;
    int32_t kv_dtype;     /* kie_kv_dtype                                           */
    int32_t ffn_wdtype;   /* kie_w_dtype of w_gate, w_up, w_down                     */
    int32_t mode;         /* kie_mode                                               */
    int32_t device;       /* CUDA device ordinal                                    */
    int32_t attn_wdtype;  /* kie_w_dtype of wq, wk, wv, wo and the LM head (INT4_G128: of wq, wk, wv) */
    int32_t batch;        /* 0 or 1: one request.  2..KIE_MAX_BATCH_REQUESTS: a batched engine (see
                           * kie_decode_batch): that many independent requests, each with its
                           * own KV cache (max_ctx positions) and position, decoded together
                           * so that every weight byte is read once per step for all of them.
                           * Needs PERSISTENT mode, FP16 weights, an FP16 or FP8_E5M2 cache,
                           * d_model, ffn_dim and n_heads*head_dim multiples of 64, and
                           * batch * n_heads <= the GPU's SM count. */
    float kv_scale_k;     /* FP8_E5M2_SCALED: slice 0's K and V scales (<= 0: the xAI page's   */
    float kv_scale_v;     /* hpi_config values, 0.0039 and 0.0042)                              */
} kie_config;

#define KIE_MAX_BATCH_REQUESTS 8

/* Per-layer weights, fp16 bit patterns, PyTorch Linear layout [out][in], row major.
 *   attn_norm[d]  wq,wk,wv[H*h][d]  wo[d][H*h]  ffn_norm[d]
 *   w_gate,w_up[F][d]  w_down[d][F]
 * For ffn_wdtype == KIE_W_INT4_G128 the engine quantises w_gate/w_up/w_down
 * itself (kie_quantize_int4_g128 below), and wq/wk/wv for attn_wdtype ==
 * KIE_W_INT4_G128; for KIE_W_FP8_E4M3 or KIE_W_NVFP4
 * (ffn_wdtype or attn_wdtype) it quantises the matrices concerned as
 * kie_quantize_fp8_rows or kie_quantize_nvfp4_rows do. */
typedef struct {
    const uint16_t *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} kie_layer_weights;

typedef struct {
    const uint16_t* tok_emb;          /* [vocab][d]           */
    const uint16_t* final_norm;       /* [d]                  */
    const uint16_t* lm_head;          /* [vocab][d]           */
    const kie_layer_weights* layers;  /* [n_layers]           */
    int32_t on_device;                /* 1: all pointers above are device pointers */
} kie_weights;

typedef struct kie_engine kie_engine;  /* opaque */

/* Bytes of device memory kie_create needs for this config (weights, KV cache,
 * activations, plan tables), for a caller that wants to pass its own workspace.
 * Returns 0 for an invalid config. */
size_t kie_workspace_bytes(const kie_config* cfg);

/* Create an engine.  workspace: NULL (the engine allocates with cudaMalloc and
 * frees on destroy) or a device buffer of at least kie_workspace_bytes(cfg)
 * bytes, 256-byte aligned, owned by the caller and kept alive until
 * kie_destroy.  cuda_stream: a cudaStream_t (NULL = the legacy default stream).
 * It also resolves the device address of the library's static scratch array
 * (see kie_decode_step_static_scratch), which loads the device code holding it.
 * On failure *out is NULL and kie_last_error(NULL) has the reason. */
kie_status kie_create(const kie_config* cfg, void* workspace, size_t ws_bytes, void* cuda_stream,
                      kie_engine** out);

/* Copy, repack (per-SM contiguous weight streams) and, for INT4 FFN, quantise
 * the weights.  The caller keeps ownership of w's buffers.  Resets pos to 0. */
kie_status kie_load_weights(kie_engine* e, const kie_weights* w);

/* Consume n prompt tokens at positions pos .. pos+n-1 (teacher-forced, causal),
 * appending their K/V to the cache.  last_logits: NULL or host fp32[vocab],
 * receives the logits after the last prompt token.  pos += n. */
kie_status kie_prefill(kie_engine* e, const int32_t* tokens, int32_t n, float* last_logits);

/* One step: consume `token` at position pos, append its K/V, write the argmax
 * of the logits (lowest id on ties) to *next_token; logits: NULL or host
 * fp32[vocab].  pos += 1. */
kie_status kie_decode_step(kie_engine* e, int32_t token, int32_t* next_token, float* logits);

/* n greedy steps equal to n chained kie_decode_step calls: out_tokens[i] is the
 * argmax after consuming token i, where token 0 is first_token and token i is
 * out_tokens[i-1].  out_logits: NULL or host fp32[n][vocab].  pos += n. */
kie_status kie_generate_greedy(kie_engine* e, int32_t first_token, int32_t n, int32_t* out_tokens,
                               float* out_logits);

/* Same as kie_generate_greedy with DEVICE output buffers (out_logits may be
 * NULL), enqueued on the engine's stream without synchronising: the call that
 * timing and graph capture by the caller use.  Errors detected inside the GPU
 * program are reported by the next synchronising call (or kie_sync). */
kie_status kie_generate_greedy_device(kie_engine* e, int32_t first_token, int32_t n,
                                      int32_t* d_out_tokens, float* d_out_logits);

/* ---- batched engines (kie_config.batch >= 2) ------------------------------------------------
 * Low-batch decode (the Kog page's TL;DR: batch 1 for its preview, larger
 * batches for production): the requests share one pass over the weights per
 * step.  Each request is the single-request model on its own cache: the same
 * tokens and logits as a one-request engine up to fp32 summation order (the
 * batched GEMV runs on the tensor cores with the activations split into fp16
 * hi + lo parts, about 2^-22 relative).
 *
 * kie_select_request chooses the request that kie_prefill, kie_set_kv,
 * kie_read_kv, kie_set_pos and kie_get_pos address (default 0; on a
 * one-request engine only 0 is valid).  kie_decode_step, kie_generate_greedy
 * and their variants are refused on a batched engine (KIE_ERR_UNSUPPORTED):
 * use the calls below, which advance every request by the same number of
 * tokens from its own position. */
kie_status kie_select_request(kie_engine* e, int32_t request);

/* One step for every request: tokens[b] (host, [batch]) is consumed at
 * request b's position; next_tokens[b] (host) receives its argmax (lowest id
 * on ties); logits: NULL or host fp32[batch][vocab].  Every position += 1. */
kie_status kie_decode_batch(kie_engine* e, const int32_t* tokens, int32_t* next_tokens, float* logits);

/* n greedy steps for every request, equal to n chained kie_decode_batch
 * calls: out_tokens (host, [n][batch]) and out_logits (NULL or host
 * fp32[n][batch][vocab]).  first_tokens: host [batch]. */
kie_status kie_generate_greedy_batch(kie_engine* e, const int32_t* first_tokens, int32_t n, int32_t* out_tokens,
                                     float* out_logits);

/* The same with DEVICE output buffers (d_out_logits may be NULL), enqueued on
 * the engine's stream without synchronising (first_tokens stays a host array,
 * read before the call returns). */
kie_status kie_generate_greedy_batch_device(kie_engine* e, const int32_t* first_tokens, int32_t n,
                                            int32_t* d_out_tokens, float* d_out_logits);

/* Synchronise the engine's stream and report any error the GPU program set. */
kie_status kie_sync(kie_engine* e);

/* pos = 0 (the cache contents become unreachable) and clear a sticky device
 * error (a scaled E5M2 cache restarts from its initial scales). */
kie_status kie_reset(kie_engine* e);
int32_t kie_get_pos(const kie_engine* e);
/* Set pos (0 <= pos <= max_ctx), e.g. after loading a context with kie_set_kv. */
kie_status kie_set_pos(kie_engine* e, int32_t pos);
/* Bound on every wait inside the GPU program (default 2000 ms). */
kie_status kie_set_timeout_ms(kie_engine* e, int32_t ms);
/* Failure injection for tests of the device-timeout path: the next
 * persistent launch that reaches a grid barrier lets CTA `cta` (0 <= cta <
 * kie_grid_size) skip its arrival at the first one, so every other CTA's
 * bounded wait there runs out after the kie_set_timeout_ms limit; the launch
 * then ends with KIE_ERR_DEVICE_TIMEOUT and the engine stays poisoned until
 * kie_reset.  The injection applies to one launch only; cta = -1 cancels it.
 * Nothing hangs: every wait in the GPU program is bounded. */
kie_status kie_debug_skip_grid_arrival(kie_engine* e, int32_t cta);
/* The engine's stream (cudaStream_t) and number of CTAs of the persistent grid. */
void* kie_get_stream(const kie_engine* e);
int32_t kie_grid_size(const kie_engine* e);
/* Message of the last failure on this engine (e == NULL: of the last failed
 * kie_create or stateless call).  Engine-owned; valid until the next call. */
const char* kie_last_error(const kie_engine* e);
/* Free everything the engine allocated.  NULL-safe. */
void kie_destroy(kie_engine* e);

/* ---- diagnostics ------------------------------------------------------------------------------ */

/* Run n greedy steps like kie_generate_greedy (persistent mode only) while the
 * GPU program records %globaltimer stamps (ns) into
 * stamps[n][5*n_layers+1][6][grid]: per step and phase (per layer QKV,
 * attention, O, gate/up, down; then LM head) and per CTA: 0 phase start (after
 * the grid barrier), 1 activation staged, 2 GEMV or attention done, 3 epilogue
 * done, 4 first weight slot of the phase issued, 5 last slot issued (0 where
 * an event does not occur); followed by a ring trace of CTA 0, [32768][4]: per
 * shared-memory ring slot of the launch, 0 bulk copy issued, 1 data seen by the
 * consuming warp, 2 slot released (3 unused).  cap: entries available in
 * stamps.  The engine allocates a temporary device buffer for the call.
 * pos += n. */
kie_status kie_trace_decode(kie_engine* e, int32_t first_token, int32_t n, uint64_t* stamps, size_t cap);

/* ---- decode step without any allocation ------------------------------------------------------ */

/* The pages have no counterpart to this call; it serves callers that may not
 * allocate device memory while decoding (code hosted inside another
 * framework's allocator, a plugin without allocation rights, a service that
 * forbids allocation after start-up, or a device already fully committed).
 * Together with an engine created on a caller-provided workspace it performs
 * no cudaMalloc, cudaFree or other allocating call.
 *
 * One greedy step like kie_decode_step (consume `token` at pos, append its
 * K/V, pos += 1) in persistent mode, enqueued on the engine's stream without
 * synchronising.  d_next_token: DEVICE int32 receiving the argmax; d_logits:
 * NULL or DEVICE fp32[vocab].  The step's scratch (activations, attention and
 * argmax partials, control block) is a fixed 320 KiB array inside the library
 * that every GPU loading the library keeps until the process exits; configs
 * whose scratch would exceed it (roughly 2*d_model + 5*n_heads*head_dim +
 * 2*ffn_dim + grid*(head_dim+6) floats) return KIE_ERR_UNSUPPORTED.  The array
 * is part of the library's device code: kie_create looks up its device address
 * with the engine's device current, which (under CUDA's lazy module loading)
 * is when the array's device memory is committed, so this call itself commits
 * nothing.  A device reset invalidates the engine and the address with it.
 * All calls on a device share
 * the array and it keeps the last call's contents: calls that may overlap on
 * the GPU (several engines, several streams) race and must be serialised by
 * the caller.  A device error of the step is reported by the engine's next
 * synchronising call (e.g. kie_sync). */
kie_status kie_decode_step_static_scratch(kie_engine* e, int32_t token, int32_t* d_next_token, float* d_logits);

/* ---- context loading and inspection (synthetic contexts, tests) ---------------------------- */

/* Write post-RoPE K and V for positions 0 .. n-1 of one layer through the
 * cache's storage format (fp16 as given; E5M2 converted from it; uint8: every
 * complete 128-token segment quantised, the rest kept fp16 as the open
 * segment; scaled E5M2: slice by slice, each slice's scale from the one
 * before as in decoding).  k_fp16, v_fp16: host fp16 [n][n_heads][head_dim].
 * pos is not changed (see kie_set_pos). */
kie_status kie_set_kv(kie_engine* e, int32_t layer, const uint16_t* k_fp16, const uint16_t* v_fp16,
                      int32_t n);

/* Read back the stored K (which=0) or V (which=1) of one layer, positions
 * [p0, p0+n), as raw storage: fp16 bits (2 bytes/elem), E5M2 bytes or uint8
 * codes (1 byte/elem), layout [n_heads][n][head_dim].  For scaled E5M2 caches
 * `scale` receives the scales of the 256-position slices the range meets
 * ([nslices], NULL allowed).  For uint8 caches the
 * positions of the open segment are returned as their fp16 values in
 * `tail_fp16` ([n_heads][n][head_dim], NULL allowed; other positions are left
 * untouched) -- when pos is a positive multiple of 128 no position of the new
 * open segment exists yet, and the fp16 values returned are those of the
 * segment [pos-128, pos) that was quantised last -- and scale/zp of the
 * segments covering the range in scale[n_heads][nseg], zp[n_heads][nseg]
 * (nseg = segments overlapping [p0, p0+n); NULL allowed). */
kie_status kie_read_kv(kie_engine* e, int32_t layer, int32_t which, int32_t p0, int32_t n, void* out,
                       uint16_t* tail_fp16, float* scale, int32_t* zp);

/* ---- stateless device routines (host in, host out; used for bit-exact checks) -------------- */

/* Adaptive-range uint8 quantisation of n_seg independent segments of
 * seg_elems fp16 values each (Grok-3 page, section 3.2): scale = (max-min)/255,
 * zp = round_half_even(-min/scale) (fp32 IEEE division, unclamped int32),
 * code = clamp(round_half_even(x/scale) + zp, 0, 255); a constant segment uses
 * scale 1, zp = round(-min).  codes[n_seg*seg_elems], scale[n_seg], zp[n_seg]. */
kie_status kie_quantize_kv_u8(const uint16_t* x_fp16, int32_t n_seg, int32_t seg_elems, uint8_t* codes,
                              float* scale, int32_t* zp);

/* Symmetric INT4, per row and group of 128 columns (xAI page, sections 2.3,
 * 3.3): s = fp16_rne(absmax/7), q = clamp(round_half_even(w/s), -8, 7), q = 0
 * when s == 0.  codes: int8 [rows][cols] (one code per byte), scale_fp16:
 * [rows][cols/128].  cols must be a multiple of 128. */
kie_status kie_quantize_int4_g128(const uint16_t* w_fp16, int32_t rows, int32_t cols, int8_t* codes,
                                  uint16_t* scale_fp16);

/* FP8 E4M3 weight quantisation with one fp32 scale per output row (see
 * kie_w_dtype): s = absmax(row)/448 in fp32; codes = E4M3(w/s), the division in
 * fp32, round to nearest even, saturating at +-448; an all-zero row gets s = 0
 * and codes 0.  Host pointers: w_fp16 [rows][cols] in, codes [rows][cols] and
 * scales [rows] out.  Runs on the current CUDA device and synchronises it. */
kie_status kie_quantize_fp8_rows(const uint16_t* w_fp16, int32_t rows, int32_t cols, uint8_t* codes, float* scales);

/* NVFP4 weight quantisation (see kie_w_dtype), every step in fp32 with IEEE
 * division and each product rounded once:
 *   rs = absmax(row) / 2688                  (2688 = 6 * 448)
 *   bs = E4M3(absmax(block) / (6 * rs))      per 16 consecutive columns, nearest even, saturating
 *   code = E2M1(w / (bs * rs))               nearest even, saturating at +-6; the sign
 *                                            bit follows w's sign (also for a zero)
 * An all-zero row gets rs = 0, block scales 0 and codes 0.  Host pointers:
 * w_fp16 [rows][cols] in (cols a multiple of 16); codes [rows][cols] out, one
 * E2M1 code (0..15: sign, two exponent bits, one mantissa bit) per byte;
 * block_scales [rows][cols/16] E4M3 bytes; row_scales [rows] fp32.  Runs on
 * the current CUDA device and synchronises it. */
kie_status kie_quantize_nvfp4_rows(const uint16_t* w_fp16, int32_t rows, int32_t cols, uint8_t* codes,
                                   uint8_t* block_scales, float* row_scales);

/* fp16 -> FP8 E5M2, round to nearest even, saturating to +-57344 (the cache's
 * conversion; xAI page sections 2.3 and 4.3).  NaN stays NaN. */
kie_status kie_convert_fp8_e5m2(const uint16_t* x_fp16, size_t n, uint8_t* out);

#ifdef __cplusplus
}
#endif
#endif /* KIE_H */
