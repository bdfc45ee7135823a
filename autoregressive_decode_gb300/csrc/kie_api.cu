// Host side of libkie: the C ABI declared in include/kie.h.
//
// The engine owns one device workspace (its own cudaMalloc, or a buffer the
// caller passes), carved into: per-CTA weight streams, embedding table, norm
// gains, KV cache, activations, plan tables and output staging.  All GPU work
// runs on the stream given at creation.
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "../../include/kie.h"
#include "kie_internal.h"

extern "C" void* kie_decode_kernel_ptr(int hd, int kv);
extern "C" void* kie_decode_batch_kernel_ptr(int hd, int kv);
extern "C" cudaError_t kie_launch_slot_chunk_major(uint8_t* stream, const uint4* table, int nslots, cudaStream_t st);
extern "C" cudaError_t kie_launch_ctl(KieControl* c, int tok, int pos, int clear, cudaStream_t st);
extern "C" cudaError_t kie_launch_err_merge(const KieControl* src, KieControl* dst, cudaStream_t st);
extern "C" cudaError_t kie_launch_copy_desc(uint8_t* dst, const uint8_t* src, const void* desc, int n,
                                            cudaStream_t st);
// tensor-core prefill (kie_prefill.cu)
extern "C" cudaError_t kie_pf_gemm(const __half* Ahi, const __half* Alo, const __half* W, float* C, int ldc,
                                   int M_pad, int N_pad, int K, int m_valid, const float* col_scale, int ksplit,
                                   size_t c_stride, uint64_t timeout_ns, int* err, cudaStream_t st);
extern "C" cudaError_t kie_pf_pack_e4m3(const uint8_t* codes, int n, int K, int row0, __half* dst, cudaStream_t st);
extern "C" cudaError_t kie_pf_pack_fp4(const uint8_t* codes, const uint8_t* bscales, int n, int K, int row0, __half* dst,
                                       cudaStream_t st);
extern "C" cudaError_t kie_launch_quant_fp8(const uint16_t* w, int rows, int cols, uint8_t* codes, float* scales,
                                            cudaStream_t st);
extern "C" cudaError_t kie_pf_pack(const __half* src, int n, int K, int row0, __half* dst, cudaStream_t st);
extern "C" cudaError_t kie_pf_embed(const int32_t* tokens, int T, const uint16_t* emb, int d, float* x,
                                    cudaStream_t st);
extern "C" cudaError_t kie_pf_norm_split(const float* x, int ld, const float* g, float eps, int T, int T_pad, int d,
                                         __half* hi, __half* lo, cudaStream_t st);
extern "C" cudaError_t kie_pf_split(const float* src, int ld, int T, int T_pad, int K, __half* hi, __half* lo,
                                    cudaStream_t st);
extern "C" cudaError_t kie_pf_swiglu_split(const float* C, int ldc, int T, int T_pad, int F, __half* hi, __half* lo,
                                           cudaStream_t st);
extern "C" cudaError_t kie_pf_residual(float* x, const float* C, int ldc, int T, int d, int ns, size_t c_stride,
                                       cudaStream_t st);
extern "C" cudaError_t kie_pf_qkv_post(const float* C, int ldc, int T, int pos0, int H, int hd, const float* inv_freq,
                                       int kvfmt, uint8_t* kc, uint8_t* vc, int layer, int max_ctx, float* Q, int ns,
                                       size_t c_stride, cudaStream_t st);
extern "C" cudaError_t kie_pf_attention(const float* Q, const uint8_t* kc, const uint8_t* vc, int layer, int H,
                                        int hd, int kvfmt, int max_ctx, int pos0, int T, float scale, float* O,
                                        uint64_t timeout_ns, int* err, cudaStream_t st);
extern "C" cudaError_t kie_launch_quant_fp4(const uint16_t* w, int rows, int cols, uint8_t* packed, uint8_t* codes,
                                            uint8_t* bscales, float* rscales, cudaStream_t st);
extern "C" cudaError_t kie_launch_quant_int4(const uint16_t* w, int rows, int cols, uint8_t* packed,
                                             int8_t* codes_i8, uint16_t* scales, cudaStream_t st);
extern "C" cudaError_t kie_launch_quant_u8(const uint16_t* src, int n_seg, int64_t src_seg, int64_t src_row,
                                           int rows, int row_elems, uint8_t* codes, int64_t dst_seg,
                                           int64_t dst_row, float* scale, int32_t* zp, int64_t meta_stride,
                                           cudaStream_t st);
extern "C" cudaError_t kie_launch_e5m2(const uint16_t* x, size_t n, uint8_t* out, cudaStream_t st);
extern "C" cudaError_t kie_launch_kv_slice(const uint16_t* src, int p0, int p1, int H, int hd, int max_ctx, float* sc,
                                           uint32_t* mx, int j, uint8_t* dst, cudaStream_t st);
extern "C" cudaError_t kie_launch_kv_rescan(const uint8_t* kc, const uint8_t* vc, uint32_t* mx, int L, int H, int hd,
                                            int max_ctx, int nslice, int pos, cudaStream_t st);
extern "C" cudaError_t kie_launch_set_kv(const uint16_t* src, int n, int H, int hd, int max_ctx, int fmt,
                                         uint8_t* dst, uint16_t* tail, int first_tail, cudaStream_t st);

namespace {

struct CopyDesc {
    uint64_t dst, src;
    uint32_t len, pad;
};

thread_local std::string g_last_error;

constexpr int kLogitChunk = 64;      // steps per launch when logits are copied to the host
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kSmemLimit = 232448;   // 227 KB opt-in shared memory per block

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Plan of one GEMV phase type (host copy).
struct HostPhase {
    int K = 0, KC = 0, nK = 0, rpu = 1, wfmt = WF_F16, n_units = 0, R = KIE_R, cpb = 0;
    std::vector<int32_t> unit_begin;   // G+1
    std::vector<uint32_t> bytes;       // G
    std::vector<uint32_t> nslots;      // G
};

uint32_t slot_bytes_host(int wfmt, int rows_g, int kc) {
    if (wfmt == WF_F16) return uint32_t(rows_g) * uint32_t(kc) * 2u;
    if (wfmt == WF_F8) return (uint32_t(rows_g) * uint32_t(kc) + 15u) & ~15u;
    if (wfmt == WF_F4) return (uint32_t(rows_g) * uint32_t(kc / 2 + kc / 16) + 15u) & ~15u;
    uint32_t b = uint32_t(rows_g) * uint32_t(kc / 2) + uint32_t(rows_g) * uint32_t(kc / 64);
    return (b + 15u) & ~15u;
}

struct Layout {  // byte offsets into the workspace
    size_t wstream, wstream_bytes;
    size_t emb, norms, inv_freq;
    size_t kc, vc, kv_bytes, tail, seg_scale, seg_zp;
    size_t kv_sc, kv_mx;              // scaled E5M2: [L][2][nslice] slice scales and running maxima
    int nslice;
    // FP8 row scales (floats): per layer [QKV | O | GU | D] in each phase's row order, then the LM head
    size_t wsc, wsc_layer, wsc_off[PH_NTYPES];
    size_t x, kcur, vcur, zero_bytes, q, a, o, att_part, par_bytes, amax_val, amax_idx, ctl;
    size_t req;                       // batched: [2][KIE_MAX_BATCH] int32 request tokens, then positions
    size_t plan_i32, plan_u32, cta_base, cta_layer;
    size_t out_tokens, out_logits, forced, step_token, step_logits;
    // tensor-core prefill: weight tiles (per layer: Wqkv, Wo, Wgu, Wd; then Wlm) and scratch
    bool pf = false;
    int pf_tc = 0;                    // prompt rows per prefill chunk (a multiple of 128)
    size_t pf_w, pf_layer_elems, pf_qkv, pf_o, pf_gu, pf_d, pf_lm;   // element offsets within a layer / of Wlm
    size_t pf_x, pf_ahi, pf_alo, pf_c, pf_q, pf_att, pf_err;
    size_t pf_c_elems = 0;            // floats in pf_c
    size_t pf_sc, pf_sc_layer;        // FP8: output-column scales (floats) per layer [QKV | O | GU | D], then Wlm
    size_t total;
    int nseg;
};

int pad256(int n) { return (n + 255) / 256 * 256; }

// Weight formats stored with one fp32 scale per output row (FP8 E4M3, NVFP4).
bool scaled_fmt(int32_t wdtype) { return wdtype == KIE_W_FP8_E4M3 || wdtype == KIE_W_NVFP4; }

// The tensor-core prefill covers non-INT4 weights with an fp16 or E5M2 cache
// (the uint8 cache changes stored values when a segment completes, the scaled
// E5M2 cache's slice scales follow each other, and INT4 weights have no fp16
// copy); every GEMM K must be a multiple of 64.
bool prefill_tc_ok(const kie_config& c) {
    return c.ffn_wdtype != KIE_W_INT4_G128 && c.attn_wdtype != KIE_W_INT4_G128 && c.kv_dtype != KIE_KV_U8_ADAPTIVE &&
           c.kv_dtype != KIE_KV_FP8_E5M2_SCALED &&
           c.d_model % 64 == 0 &&
           (c.n_heads * c.head_dim) % 64 == 0 && c.ffn_dim % 64 == 0;
}

struct Plan {
    int G = 0;
    int nb = 0;   // batched engine: requests (0: the single-request kernel)
    HostPhase ph[PH_NTYPES];
    std::vector<uint64_t> cta_base, cta_layer;
    uint64_t stream_bytes = 0;
    int nslot = 0, act_floats = 0, part_floats = 0;
    size_t smem = 0;
};

bool valid_cfg(const kie_config* c, std::string& why) {
    if (!c) { why = "config is NULL"; return false; }
    if (c->n_layers < 1 || c->d_model < 8 || c->n_heads < 1 || c->ffn_dim < 8 || c->vocab < 2 || c->max_ctx < 1) {
        why = "non-positive model dimension";
        return false;
    }
    if (c->head_dim != 64 && c->head_dim != 128) { why = "head_dim must be 64 or 128"; return false; }
    if (c->d_model % 8 || c->ffn_dim % 8 || (c->n_heads * c->head_dim) % 8) { why = "dims must be multiples of 8"; return false; }
    if (c->kv_dtype < 0 || c->kv_dtype > 3) { why = "bad kv_dtype"; return false; }
    if (c->ffn_wdtype < 0 || c->ffn_wdtype > 3) { why = "bad ffn_wdtype"; return false; }
    if (c->attn_wdtype < 0 || c->attn_wdtype > 3) { why = "bad attn_wdtype"; return false; }
    if (c->attn_wdtype == KIE_W_INT4_G128 && c->d_model % 128) {
        why = "INT4 q/k/v weights need d_model a multiple of 128";
        return false;
    }
    if ((c->ffn_wdtype == KIE_W_NVFP4 || c->attn_wdtype == KIE_W_NVFP4) &&
        (c->d_model % 16 || c->ffn_dim % 16 || (c->n_heads * c->head_dim) % 16)) {
        why = "NVFP4 weights need d_model, ffn_dim and n_heads*head_dim multiples of 16";
        return false;
    }
    if (c->ffn_wdtype == KIE_W_INT4_G128 && (c->d_model % 128 || c->ffn_dim % 128)) {
        why = "INT4 FFN needs d_model and ffn_dim multiples of 128";
        return false;
    }
    if (c->mode < 0 || c->mode > 1) { why = "bad mode"; return false; }
    if (c->batch < 0 || c->batch > KIE_MAX_BATCH) { why = "batch outside [0, 8]"; return false; }
    if (c->batch > 1) {
        if (c->mode != KIE_MODE_PERSISTENT) { why = "a batched engine needs the persistent mode"; return false; }
        if (c->attn_wdtype != KIE_W_FP16 || c->ffn_wdtype != KIE_W_FP16) { why = "a batched engine needs fp16 weights"; return false; }
        if (c->kv_dtype == KIE_KV_U8_ADAPTIVE || c->kv_dtype == KIE_KV_FP8_E5M2_SCALED) {
            why = "a batched engine needs an fp16 or E5M2 cache";
            return false;
        }
        if (c->d_model % 64 || c->ffn_dim % 64 || (c->n_heads * c->head_dim) % 64) {
            why = "a batched engine needs d_model, ffn_dim and n_heads*head_dim multiples of 64";
            return false;
        }
    }
    if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) { why = "bad rms_eps or rope_theta"; return false; }
    return true;
}

// Partition every phase over G CTAs, balancing each CTA's cumulative stream bytes.
void build_plan(const kie_config& c, int G, Plan& pl) {
    pl.G = G;
    pl.nb = c.batch > 1 ? c.batch : 0;
    const bool bat = pl.nb > 0;
    const int d = c.d_model, H = c.n_heads, hd = c.head_dim, F = c.ffn_dim, V = c.vocab;
    const int ffn_fmt = c.ffn_wdtype == KIE_W_INT4_G128 ? WF_I4 : c.ffn_wdtype == KIE_W_FP8_E4M3 ? WF_F8
                        : c.ffn_wdtype == KIE_W_NVFP4 ? WF_F4 : WF_F16;
    const int attn_fmt = c.attn_wdtype == KIE_W_FP8_E4M3 ? WF_F8 : c.attn_wdtype == KIE_W_NVFP4 ? WF_F4 : WF_F16;
    const int qkv_fmt = c.attn_wdtype == KIE_W_INT4_G128 ? WF_I4 : attn_fmt;   // INT4 reaches q, k, v only
    auto setp = [&](int t, int K, int rpu, int units, int wfmt) {
        HostPhase& p = pl.ph[t];
        p.K = K; p.rpu = rpu; p.n_units = units; p.wfmt = wfmt;
        // a slot: 4 rows x 2048 fp16, 8 rows x 2048 FP8, or 4 rows x 4096 INT4 (+ scales), 16 KB;
        // KIE_R4 rows x 2048 NVFP4 (+ block scales)
        p.KC = std::min(K, wfmt == WF_I4 ? KIE_KC_I4 : KIE_KC_F16);
        p.R = wfmt == WF_F8 ? KIE_R8 : wfmt == WF_F4 ? KIE_R4 : KIE_R;
        if (bat) {   // batched kernel: 16-row x 512-column fp16 slots, staged 2048 columns at a time
            p.KC = std::min(K, KIE_KCB);
            p.R = KIE_RB;
        }
        p.nK = (K + p.KC - 1) / p.KC;
        p.cpb = bat ? KIE_KBLK / KIE_KCB : p.nK;
    };
    setp(PH_QKV, d, 2, 3 * H * (hd / 2), qkv_fmt);
    setp(PH_O, H * hd, 1, d, attn_fmt);
    setp(PH_GU, d, 2, F, ffn_fmt);
    setp(PH_D, F, 1, d, ffn_fmt);
    setp(PH_LM, d, 1, V, attn_fmt);

    std::vector<uint64_t> cum(G, 0);
    auto assign = [&](int t, std::vector<uint64_t>& acc, uint64_t weight) {
        HostPhase& p = pl.ph[t];
        const int base = p.n_units / G, rem = p.n_units % G;
        std::vector<int> order(G);
        std::iota(order.begin(), order.end(), 0);
        std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return acc[a] < acc[b]; });
        std::vector<int> cnt(G, base);
        for (int k = 0; k < rem; ++k) cnt[order[k]] += 1;
        p.unit_begin.assign(G + 1, 0);
        for (int i = 0; i < G; ++i) p.unit_begin[i + 1] = p.unit_begin[i] + cnt[i];
        p.bytes.assign(G, 0);
        p.nslots.assign(G, 0);
        for (int i = 0; i < G; ++i) {
            const int rows = cnt[i] * p.rpu;
            const int groups = (rows + p.R - 1) / p.R;
            uint64_t b = 0;
            for (int g = 0; g < groups; ++g) {
                const int rg = std::min(p.R, rows - g * p.R);
                for (int ch = 0; ch < p.nK; ++ch) {
                    const int kc = std::min(p.KC, p.K - ch * p.KC);
                    b += slot_bytes_host(p.wfmt, rg, kc);
                }
            }
            p.bytes[i] = uint32_t(b);
            p.nslots[i] = uint32_t(groups * p.nK);
            acc[i] += b * weight;
        }
    };
    for (int t : {PH_QKV, PH_O, PH_GU, PH_D}) assign(t, cum, 1);
    for (auto& v : cum) v *= uint64_t(c.n_layers);
    assign(PH_LM, cum, 1);

    pl.cta_base.assign(G, 0);
    pl.cta_layer.assign(G, 0);
    uint64_t off = 0;
    for (int i = 0; i < G; ++i) {
        uint64_t lb = 0;
        for (int t : {PH_QKV, PH_O, PH_GU, PH_D}) lb += pl.ph[t].bytes[i];
        pl.cta_layer[i] = lb;
        pl.cta_base[i] = off;
        off += lb * uint64_t(c.n_layers) + pl.ph[PH_LM].bytes[i];
    }
    pl.stream_bytes = off;

    // shared memory
    int64_t part = 0;
    for (int t = 0; t < PH_NTYPES; ++t) {
        const HostPhase& p = pl.ph[t];
        for (int i = 0; i < G; ++i) {
            const int rows = (p.unit_begin[i + 1] - p.unit_begin[i]) * p.rpu;
            part = std::max<int64_t>(part, int64_t((rows + p.R - 1) / p.R) * p.R * std::max(p.nK, 1));
        }
    }
    // attention: head h gets floor((h+1)G/H) - floor(hG/H) >= floor(G/H) CTAs; a
    // chunk holds at most ceil(max_ctx / floor(G/H)) rows (scores in the act
    // buffer) and, for uint8 caches, meets at most rows/128 + 2 segments whose
    // scale/zp (K and V) are staged in the partial buffer.
    const int64_t min_heads_cta = std::max(1, G / H);
    const int64_t max_seg = (int64_t(c.max_ctx) + min_heads_cta - 1) / min_heads_cta + 2;
    part = std::max<int64_t>(part, 4 * (max_seg / KIE_SEG + 2));
    part = std::max<int64_t>(part, 2 * (max_seg / KIE_KV_SLICE + 2));   // scaled E5M2: the chunk's slice scales
    part = std::max<int64_t>(part, G + H);   // O-phase combine: per-CTA weights and per-head 1/L
    int act = std::max({d, F, H * hd, int(std::min<int64_t>(max_seg, 1 << 30))});
    if (bat) {
        // batched: a phase staged in several blocks keeps each row tile's running
        // sums in the part buffer (128 floats a tile), and one with fewer row
        // tiles than consumer warps each slot's sums of a block (128 floats a
        // (tile, chunk)); the activations are one block of MMA fragments (2048
        // columns x 8 requests x hi/lo fp16)
        part = std::max<int64_t>(G + H, 4);
        for (int t = 0; t < PH_NTYPES; ++t) {
            const HostPhase& p = pl.ph[t];
            const int nblk = (p.K + KIE_KBLK - 1) / KIE_KBLK;
            for (int i = 0; i < G; ++i) {
                const int64_t tiles = ((p.unit_begin[i + 1] - p.unit_begin[i]) * p.rpu + KIE_RB - 1) / KIE_RB;
                const int64_t need = (nblk > 1 ? tiles * 128 : 0) + (tiles < KIE_NW ? tiles * p.cpb * 128 : 0);
                part = std::max<int64_t>(part, need);
            }
        }
        act = (KIE_KBLK / 16) * 132;   // k-steps of 128 fragment words, 4 words of padding each
    }
    pl.part_floats = int(align_up(size_t(std::max<int64_t>(part, 4)), 4));
    pl.act_floats = int(align_up(act, 8));
    const KieSmemLayout l0 = kie_smem_layout(pl.part_floats, pl.act_floats, 0, pl.nb);
    const long avail = long(kSmemLimit) - long(l0.total);
    pl.nslot = int(std::max<long>(0, std::min<long>(KIE_MAX_SLOTS, avail / KIE_SLOT_BYTES)));
    pl.smem = kie_smem_layout(pl.part_floats, pl.act_floats, pl.nslot, pl.nb).total;
}

void compute_layout(const kie_config& c, const Plan& pl, Layout& L) {
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = align_up(o, 256); o = at + bytes; return at; };
    const int G = pl.G, d = c.d_model, H = c.n_heads, hd = c.head_dim, F = c.ffn_dim, V = c.vocab;
    L.wstream = take(pl.stream_bytes);
    L.wstream_bytes = pl.stream_bytes;
    L.emb = take(size_t(V) * d * 2);
    L.norms = take((size_t(c.n_layers) * 2 + 1) * d * 4);
    L.inv_freq = take(size_t(hd / 2) * 4);
    const size_t esz = c.kv_dtype == KIE_KV_FP16 ? 2 : 1;
    {
        const size_t rows[PH_NTYPES] = {size_t(3) * H * hd, size_t(d), size_t(2) * F, size_t(d), size_t(V)};
        const bool f8 = scaled_fmt(c.attn_wdtype) || scaled_fmt(c.ffn_wdtype);
        size_t o8 = 0;
        for (int t : {PH_QKV, PH_O, PH_GU, PH_D}) { L.wsc_off[t] = o8; o8 += rows[t]; }
        L.wsc_layer = o8;
        L.wsc_off[PH_LM] = o8 * c.n_layers;
        L.wsc = take(f8 ? (L.wsc_off[PH_LM] + rows[PH_LM]) * 4 : 0);
    }
    // one request's cache (a batched engine keeps pl.nb of them back to back)
    const size_t nbq = pl.nb > 0 ? size_t(pl.nb) : 1;
    L.kv_bytes = size_t(c.n_layers) * H * c.max_ctx * hd * esz;
    L.kc = take(nbq * L.kv_bytes);
    L.vc = take(nbq * L.kv_bytes);
    L.nseg = (c.max_ctx + KIE_SEG - 1) / KIE_SEG;
    const bool u8 = c.kv_dtype == KIE_KV_U8_ADAPTIVE;
    L.tail = take(u8 ? size_t(c.n_layers) * 2 * H * KIE_SEG * hd * 2 : 0);
    L.seg_scale = take(u8 ? size_t(c.n_layers) * 2 * H * L.nseg * 4 : 0);
    L.seg_zp = take(u8 ? size_t(c.n_layers) * 2 * H * L.nseg * 4 : 0);
    const bool e5s = c.kv_dtype == KIE_KV_FP8_E5M2_SCALED;
    L.nslice = (c.max_ctx + KIE_KV_SLICE - 1) / KIE_KV_SLICE;
    L.kv_sc = take(e5s ? size_t(c.n_layers) * 2 * L.nslice * 4 : 0);
    L.kv_mx = take(e5s ? size_t(c.n_layers) * 2 * L.nslice * 4 : 0);
    // tagged activations, reset before each launch sequence (reset_tags):
    // x .. vcur to zero, q .. att_part to one parity
    L.x = take(size_t(KIE_REPL) * nbq * d * 4);
    L.kcur = take(nbq * H * hd * 4);
    L.vcur = take(nbq * H * hd * 4);
    L.zero_bytes = L.vcur + nbq * H * hd * 4 - L.x;
    L.q = take(nbq * H * hd * 4);
    L.a = take(size_t(KIE_REPL) * nbq * F * 4);
    L.o = take(size_t(KIE_REPL) * nbq * H * hd * 4);
    L.att_part = take(size_t(G) * (hd + 4) * 4);
    L.par_bytes = L.att_part + size_t(G) * (hd + 4) * 4 - L.q;
    L.amax_val = take(nbq * G * 4);
    L.amax_idx = take(nbq * G * 4);
    L.ctl = take(sizeof(KieControl));
    L.req = take(size_t(2) * KIE_MAX_BATCH * 4);
    L.plan_i32 = take(size_t(PH_NTYPES) * (G + 1) * 4);
    L.plan_u32 = take(size_t(PH_NTYPES) * 2 * G * 4);
    L.cta_base = take(size_t(G) * 8);
    L.cta_layer = take(size_t(G) * 8);
    L.out_tokens = take(size_t(c.max_ctx) * nbq * 4);
    L.out_logits = take(size_t(kLogitChunk) * nbq * V * 4);
    L.forced = take(size_t(c.max_ctx) * 4);
    L.step_token = take(4);
    L.step_logits = take(size_t(V) * 4);
    L.pf = prefill_tc_ok(c);
    if (L.pf) {
        const int HD = H * hd;
        L.pf_qkv = 0;
        L.pf_o = L.pf_qkv + size_t(pad256(3 * HD)) * d;
        L.pf_gu = L.pf_o + size_t(pad256(d)) * HD;
        L.pf_d = L.pf_gu + size_t(pad256(2 * F)) * d;
        L.pf_layer_elems = L.pf_d + size_t(pad256(d)) * F;
        L.pf_lm = L.pf_layer_elems * c.n_layers;
        L.pf_w = take((L.pf_lm + size_t(pad256(V)) * d) * 2);
        L.pf_tc = std::min(1024, (c.max_ctx + 127) / 128 * 128);
        const size_t kmax = std::max({d, HD, F});
        const size_t nmax = std::max<size_t>(size_t(L.pf_tc) * std::max({pad256(3 * HD), pad256(2 * F), pad256(d)}),
                                             size_t(128) * pad256(V));
        L.pf_x = take(size_t(L.pf_tc) * d * 4);
        L.pf_ahi = take(size_t(L.pf_tc) * kmax * 2);
        L.pf_alo = take(size_t(L.pf_tc) * kmax * 2);
        L.pf_c = take(nmax * 4);
        L.pf_c_elems = nmax;
        L.pf_q = take(size_t(L.pf_tc) * HD * 4);
        L.pf_att = take(size_t(L.pf_tc) * HD * 4);
        L.pf_err = take(16);
        const bool f8 = scaled_fmt(c.attn_wdtype) || scaled_fmt(c.ffn_wdtype);
        L.pf_sc_layer = size_t(3) * HD + d + 2 * size_t(F) + d;
        L.pf_sc = take(f8 ? (L.pf_sc_layer * c.n_layers + size_t(V)) * 4 : 0);
    }
    L.total = align_up(o, 256);
}

int query_grid(int device, std::string& why) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) { why = "cudaGetDeviceProperties failed"; return 0; }
    return prop.multiProcessorCount;
}

}  // namespace

struct kie_engine {
    kie_config cfg{};
    int G = 0;
    cudaStream_t stream = nullptr;
    void* ws = nullptr;
    bool own_ws = false;
    Layout lay{};
    Plan plan;
    KieParams P{};
    void* kernel = nullptr;
    bool loaded = false;
    int pos = 0;                      // position of the selected request
    int cur = 0;                      // batched engine: the request kie_prefill, kie_set_kv, ... address
    int rpos[KIE_MAX_BATCH] = {};     // batched engine: every request's position (rpos[cur] is stale; pos is current)
    int sticky = 0;
    uint64_t timeout_ns = kDefaultTimeoutNs;
    cudaGraphExec_t graph[2] = {nullptr, nullptr};   // graph mode, by tag_fill of the step's position
    KieControl* h_ctl = nullptr;  // pinned staging
    void* static_scratch = nullptr;   // device address of the library's static scratch array on this device
    int skip_arrival_cta = -1;        // failure injection for the next persistent launch (tests)
    std::string err;

    uint8_t* dev(size_t off) const { return static_cast<uint8_t*>(ws) + off; }
    // byte offset of the selected request's K (or V) cache inside the cache arrays
    size_t kv_off() const { return size_t(cur) * lay.kv_bytes; }
    bool batched() const { return plan.nb > 0; }
};

namespace {

kie_status fail(kie_engine* e, kie_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    if (e) e->err = buf;
    g_last_error = buf;
    return st;
}

#define KIE_CUDA(e, call)                                                                        \
    do {                                                                                         \
        cudaError_t _r = (call);                                                                 \
        if (_r != cudaSuccess) return fail((e), KIE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(_r)); \
    } while (0)

kie_status check_tokens(kie_engine* e, const int32_t* t, int n) {
    for (int i = 0; i < n; ++i)
        if (t[i] < 0 || t[i] >= e->cfg.vocab) return fail(e, KIE_ERR_INVALID_ARG, "token id %d out of range", t[i]);
    return KIE_OK;
}

kie_status ready(kie_engine* e, int n) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    if (!e->loaded) return fail(e, KIE_ERR_NOT_LOADED, "weights not loaded");
    if (e->sticky) return fail(e, KIE_ERR_DEVICE_TIMEOUT, "engine poisoned by an earlier device error; call kie_reset");
    if (n < 0) return fail(e, KIE_ERR_INVALID_ARG, "negative count");
    if (int64_t(e->pos) + n > e->cfg.max_ctx) return fail(e, KIE_ERR_CTX_OVERFLOW, "pos %d + %d > max_ctx %d", e->pos, n, e->cfg.max_ctx);
    return KIE_OK;
}

// Read the control block after a sync; a device error poisons the engine.
kie_status check_device(kie_engine* e) {
    KIE_CUDA(e, cudaMemcpyAsync(e->h_ctl, e->dev(e->lay.ctl), sizeof(KieControl), cudaMemcpyDeviceToHost, e->stream));
    KIE_CUDA(e, cudaStreamSynchronize(e->stream));
    if (e->h_ctl->err != KERR_NONE) {
        e->sticky = e->h_ctl->err;
        return fail(e, KIE_ERR_DEVICE_TIMEOUT, "device error %d (info %d)", e->h_ctl->err, e->h_ctl->err_info);
    }
    return KIE_OK;
}

// Scaled E5M2 cache, emptied: every slice's maximum zero, slice 0 of every
// (layer, K or V) at the configured initial scale (the xAI page's hpi_config
// values 0.0039 for K and 0.0042 for V unless the config gives others).
kie_status init_kv_scales(kie_engine* e) {
    const kie_config& c = e->cfg;
    if (c.kv_dtype != KIE_KV_FP8_E5M2_SCALED) return KIE_OK;
    const Layout& L = e->lay;
    const float s0[2] = {c.kv_scale_k > 0.f ? c.kv_scale_k : 0.0039f, c.kv_scale_v > 0.f ? c.kv_scale_v : 0.0042f};
    std::vector<float> sc(size_t(c.n_layers) * 2 * L.nslice, 0.f);
    for (int l = 0; l < c.n_layers; ++l)
        for (int kv = 0; kv < 2; ++kv) sc[(size_t(l) * 2 + kv) * L.nslice] = s0[kv];
    KIE_CUDA(e, cudaMemcpyAsync(e->dev(L.kv_sc), sc.data(), sc.size() * 4, cudaMemcpyHostToDevice, e->stream));
    KIE_CUDA(e, cudaMemsetAsync(e->dev(L.kv_mx), 0, sc.size() * 4, e->stream));
    KIE_CUDA(e, cudaStreamSynchronize(e->stream));
    return KIE_OK;
}

kie_status set_ctl(kie_engine* e, int tok, int pos, bool clear) {
    KIE_CUDA(e, kie_launch_ctl(reinterpret_cast<KieControl*>(e->dev(e->lay.ctl)), tok, pos, clear ? 1 : 0, e->stream));
    return KIE_OK;
}

KieLaunch base_launch(kie_engine* e) {
    KieLaunch l{};
    l.n_steps = 1;
    l.phase_begin = 0;
    l.phase_end = 5 * e->cfg.n_layers + 1;
    l.first_tok = -1;
    l.pos0 = -1;
    l.forced = nullptr;
    l.lm_from_step = 0;
    l.out_tokens = nullptr;
    l.out_logits = nullptr;
    l.timeout_ns = e->timeout_ns;
    l.use_grid_barrier = 1;
    l.skip_arrival_cta = -1;
    return l;
}

// Fill byte of q, a, o before a launch sequence starting at position pos: its
// words carry the parity opposite to the first write's, (pos * L + 1) & 1.
int tag_fill(const kie_config& c, int pos) {
    return ((int64_t(pos) * c.n_layers + 1) & 1) ? 0x00 : 0x01;
}

// Reset the tagged activations before a launch sequence starting at pos
// (x, kcur, vcur to tag 0; q, a, o, att_part to the parity before the first write).
cudaError_t reset_tags(const kie_config& c, uint8_t* x, size_t zero_bytes, uint8_t* q, size_t par_bytes, int pos,
                       cudaStream_t s) {
    cudaError_t r = cudaMemsetAsync(x, 0, zero_bytes, s);
    if (r == cudaSuccess) r = cudaMemsetAsync(q, tag_fill(c, pos), par_bytes, s);
    return r;
}

kie_status launch_persistent(kie_engine* e, const KieLaunch& l) {
    KIE_CUDA(e, cudaMemsetAsync(e->dev(e->lay.ctl) + offsetof(KieControl, bar), 0, 4, e->stream));
    KIE_CUDA(e, reset_tags(e->cfg, e->dev(e->lay.x), e->lay.zero_bytes, e->dev(e->lay.q), e->lay.par_bytes,
                           l.pos0 >= 0 ? l.pos0 : e->pos, e->stream));
    void* args[] = {(void*)&e->P, (void*)&l};
    cudaError_t r = cudaLaunchCooperativeKernel(e->kernel, dim3(e->G), dim3(KIE_THREADS), args, e->plan.smem, e->stream);
    if (r == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        return fail(e, KIE_ERR_LAUNCH, "persistent grid of %d CTAs cannot be co-resident", e->G);
    }
    if (r != cudaSuccess) return fail(e, KIE_ERR_CUDA, "cooperative launch: %s", cudaGetErrorString(r));
    return KIE_OK;
}

void drop_graphs(kie_engine* e) {
    for (auto& g : e->graph)
        if (g) { cudaGraphExecDestroy(g); g = nullptr; }
}

// Graph mode: one captured graph = one decode step = the tag reset and 5L+1
// single-phase launches.  The reset's fill byte depends on the step position's
// parity, so there is one graph per fill byte.
kie_status ensure_graph(kie_engine* e, int fill) {
    if (e->graph[fill]) return KIE_OK;
    cudaStream_t cap;
    KIE_CUDA(e, cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
    cudaGraph_t g = nullptr;
    cudaError_t r = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
    if (r != cudaSuccess) { cudaStreamDestroy(cap); return fail(e, KIE_ERR_CUDA, "begin capture: %s", cudaGetErrorString(r)); }
    const int P_ = 5 * e->cfg.n_layers + 1;
    // every step starts from reset activation tags
    r = cudaMemsetAsync(e->dev(e->lay.x), 0, e->lay.zero_bytes, cap);
    if (r == cudaSuccess) r = cudaMemsetAsync(e->dev(e->lay.q), fill, e->lay.par_bytes, cap);
    for (int phi = 0; phi < P_ && r == cudaSuccess; ++phi) {
        KieLaunch l = base_launch(e);
        l.phase_begin = phi;
        l.phase_end = phi + 1;
        l.use_grid_barrier = 0;
        l.out_tokens = reinterpret_cast<int32_t*>(e->dev(e->lay.step_token));
        l.out_logits = reinterpret_cast<float*>(e->dev(e->lay.step_logits));
        void* args[] = {(void*)&e->P, (void*)&l};
        r = cudaLaunchKernel(e->kernel, dim3(e->G), dim3(KIE_THREADS), args, e->plan.smem, cap);
    }
    cudaError_t r2 = cudaStreamEndCapture(cap, &g);
    cudaStreamDestroy(cap);
    if (r != cudaSuccess || r2 != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return fail(e, KIE_ERR_CUDA, "graph capture: %s", cudaGetErrorString(r != cudaSuccess ? r : r2));
    }
    r = cudaGraphInstantiate(&e->graph[fill], g, 0);
    cudaGraphDestroy(g);
    if (r != cudaSuccess) { e->graph[fill] = nullptr; return fail(e, KIE_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(r)); }
    return KIE_OK;
}

// Run n steps.  Step 0 consumes first_tok (>= 0) or the forced/ctl token; the
// step inputs after that are forced[t] (prefill) or the previous argmax.
// d_tokens/d_logits: device outputs (may be null).  lm_from: LM head only from that step.
kie_status run_steps(kie_engine* e, int n, int first_tok, const int32_t* d_forced, int lm_from, int32_t* d_tokens,
                     float* d_logits) {
    if (n <= 0) return KIE_OK;
    kie_status st;
    if (e->cfg.mode == KIE_MODE_PERSISTENT) {
        KieLaunch l = base_launch(e);
        l.n_steps = n;
        l.first_tok = d_forced ? -1 : first_tok;
        l.pos0 = e->pos;
        l.forced = d_forced;
        l.lm_from_step = lm_from;
        l.out_tokens = d_tokens;
        l.out_logits = d_logits;
        if (n > 1) {   // only a launch of several steps meets a grid barrier
            l.skip_arrival_cta = e->skip_arrival_cta;
            e->skip_arrival_cta = -1;
        }
        if ((st = launch_persistent(e, l)) != KIE_OK) return st;
    } else {
        for (int f = 0; f < 2; ++f)
            if ((st = ensure_graph(e, f)) != KIE_OK) return st;
        if ((st = set_ctl(e, first_tok >= 0 ? first_tok : 0, e->pos, false)) != KIE_OK) return st;
        int32_t* ctl_tok = reinterpret_cast<int32_t*>(e->dev(e->lay.ctl) + offsetof(KieControl, tok));
        for (int t = 0; t < n; ++t) {
            if (d_forced)
                KIE_CUDA(e, cudaMemcpyAsync(ctl_tok, d_forced + t, 4, cudaMemcpyDeviceToDevice, e->stream));
            KIE_CUDA(e, cudaGraphLaunch(e->graph[tag_fill(e->cfg, e->pos + t)], e->stream));
            if (d_tokens)
                KIE_CUDA(e, cudaMemcpyAsync(d_tokens + t, e->dev(e->lay.step_token), 4, cudaMemcpyDeviceToDevice, e->stream));
            if (d_logits && t >= lm_from)
                KIE_CUDA(e, cudaMemcpyAsync(d_logits + size_t(t - lm_from) * e->cfg.vocab, e->dev(e->lay.step_logits),
                                            size_t(e->cfg.vocab) * 4, cudaMemcpyDeviceToDevice, e->stream));
        }
    }
    e->pos += n;
    return KIE_OK;
}

// Split-K factor of a prefill GEMM with `tiles` output tiles (128 rows x
// KIE_PF_BN columns) and KB 64-column K tiles, on G resident CTA slots: s CTAs
// per output tile each take KB / s of the K tiles and store a partial of
// c_elems floats; the s partials must fit the cap_elems of the output buffer.
// Chosen to minimise the modelled time: waves of tiles * s CTAs x K tiles per
// CTA x the time of one K tile on a CTA slot (hi and lo MMAs: about 0.8 us,
// measured on the 1.8B prompt), plus writing and re-reading each extra
// partial at about 6 TB/s.  The O and down projections of a 1,024-row chunk
// have few output tiles for the GPU's slots and are split.
int pf_ksplit(int tiles, int KB, size_t c_elems, size_t cap_elems, int G) {
    constexpr double kKTileUs = 0.8, kBytesPerUs = 6.0e6;
    double best = 0.0;
    int bs = 1;
    for (int s = 1; s <= 8 && s <= KB; ++s) {
        if (size_t(s) * c_elems > cap_elems) break;
        const double waves = double((int64_t(tiles) * s + G - 1) / G);
        const double t = waves * std::ceil(double(KB) / s) * kKTileUs + double(s - 1) * double(c_elems) * 8.0 / kBytesPerUs;
        if (s == 1 || t < best) { best = t; bs = s; }
    }
    return bs;
}

// Prompt prefill through the tensor-core path (kie_prefill.cu): chunks of up
// to pf_tc prompt rows, each through all layers; the last row's logits.
kie_status prefill_tensor_cores(kie_engine* e, const int32_t* tokens, int n, float* last_logits) {
    const kie_config& c = e->cfg;
    const Layout& L = e->lay;
    cudaStream_t st = e->stream;
    const int d = c.d_model, H = c.n_heads, hd = c.head_dim, HD = H * hd, F = c.ffn_dim, V = c.vocab;
    const __half* pfw = reinterpret_cast<const __half*>(e->dev(L.pf_w));
    float* x = reinterpret_cast<float*>(e->dev(L.pf_x));
    __half* ahi = reinterpret_cast<__half*>(e->dev(L.pf_ahi));
    __half* alo = reinterpret_cast<__half*>(e->dev(L.pf_alo));
    float* C = reinterpret_cast<float*>(e->dev(L.pf_c));
    float* Q = reinterpret_cast<float*>(e->dev(L.pf_q));
    float* O = reinterpret_cast<float*>(e->dev(L.pf_att));
    int* err = reinterpret_cast<int*>(e->dev(L.pf_err));
    const float* norms = reinterpret_cast<const float*>(e->dev(L.norms));
    const float* inv_freq = reinterpret_cast<const float*>(e->dev(L.inv_freq));
    const uint16_t* emb = reinterpret_cast<const uint16_t*>(e->dev(L.emb));
    int32_t* d_tok = reinterpret_cast<int32_t*>(e->dev(L.forced));
    uint8_t* kc = e->dev(L.kc) + e->kv_off();   // the selected request's cache
    uint8_t* vc = e->dev(L.vc) + e->kv_off();
    const int kvf = c.kv_dtype == KIE_KV_FP16 ? KV_F16 : KV_E5M2;
    const float scale = 1.0f / std::sqrt(float(hd));
    const int nqkv = pad256(3 * HD), ngu = pad256(2 * F), nd = pad256(d), nv = pad256(V);
    const uint64_t to = e->timeout_ns;
    // FP8 matrices: the GEMM output columns take their row scales
    const float* pfsc = reinterpret_cast<const float*>(e->dev(L.pf_sc));
    const bool a8 = scaled_fmt(c.attn_wdtype), f8 = scaled_fmt(c.ffn_wdtype);
    auto colsc = [&](bool on, size_t off) -> const float* { return on ? pfsc + off : nullptr; };
    KIE_CUDA(e, cudaMemsetAsync(err, 0, 4, st));
    KIE_CUDA(e, cudaMemcpyAsync(d_tok, tokens, size_t(n) * 4, cudaMemcpyHostToDevice, st));
    const int pos_start = e->pos;
    int Tn = 0;
    for (int c0 = 0; c0 < n; c0 += L.pf_tc) {
        Tn = std::min(L.pf_tc, n - c0);
        const int Tp = (Tn + 127) / 128 * 128, pos = pos_start + c0;
        // split K where the output tiles alone leave SMs idle (partials Tp x N apart in C)
        const size_t cap = L.pf_c_elems;
        const int slots = e->G * (KIE_PF_BN == 128 ? 2 : 1);   // GEMM CTAs resident at once
        const int s_qkv = pf_ksplit((nqkv / KIE_PF_BN) * (Tp / 128), d / 64, size_t(Tp) * nqkv, cap, slots);
        const int s_o = pf_ksplit((nd / KIE_PF_BN) * (Tp / 128), HD / 64, size_t(Tp) * nd, cap, slots);
        const int s_d = pf_ksplit((nd / KIE_PF_BN) * (Tp / 128), F / 64, size_t(Tp) * nd, cap, slots);
        KIE_CUDA(e, kie_pf_embed(d_tok + c0, Tn, emb, d, x, st));
        for (int l = 0; l < c.n_layers; ++l) {
            const __half* W = pfw + L.pf_layer_elems * l;
            const size_t sb = L.pf_sc_layer * l;
            const float* g1 = norms + size_t(2 * l) * d;
            const float* g2 = g1 + d;
            KIE_CUDA(e, kie_pf_norm_split(x, d, g1, c.rms_eps, Tn, Tp, d, ahi, alo, st));
            KIE_CUDA(e, kie_pf_gemm(ahi, alo, W + L.pf_qkv, C, nqkv, Tp, nqkv, d, Tn, colsc(a8, sb), s_qkv,
                                    size_t(Tp) * nqkv, to, err, st));
            KIE_CUDA(e, kie_pf_qkv_post(C, nqkv, Tn, pos, H, hd, inv_freq, kvf, kc, vc, l,
                                        c.max_ctx, Q, s_qkv, size_t(Tp) * nqkv, st));
            KIE_CUDA(e, kie_pf_attention(Q, kc, vc, l, H, hd, kvf, c.max_ctx, pos, Tn, scale, O, to, err, st));
            KIE_CUDA(e, kie_pf_split(O, HD, Tn, Tp, HD, ahi, alo, st));
            KIE_CUDA(e, kie_pf_gemm(ahi, alo, W + L.pf_o, C, nd, Tp, nd, HD, Tn, colsc(a8, sb + 3 * HD), s_o,
                                    size_t(Tp) * nd, to, err, st));
            KIE_CUDA(e, kie_pf_residual(x, C, nd, Tn, d, s_o, size_t(Tp) * nd, st));
            KIE_CUDA(e, kie_pf_norm_split(x, d, g2, c.rms_eps, Tn, Tp, d, ahi, alo, st));
            KIE_CUDA(e, kie_pf_gemm(ahi, alo, W + L.pf_gu, C, ngu, Tp, ngu, d, Tn, colsc(f8, sb + 3 * HD + d), 1, 0,
                                    to, err, st));
            KIE_CUDA(e, kie_pf_swiglu_split(C, ngu, Tn, Tp, F, ahi, alo, st));
            KIE_CUDA(e, kie_pf_gemm(ahi, alo, W + L.pf_d, C, nd, Tp, nd, F, Tn,
                                    colsc(f8, sb + 3 * HD + d + 2 * size_t(F)), s_d, size_t(Tp) * nd, to, err, st));
            KIE_CUDA(e, kie_pf_residual(x, C, nd, Tn, d, s_d, size_t(Tp) * nd, st));
        }
    }
    // logits of the last prompt row
    KIE_CUDA(e, kie_pf_norm_split(x + size_t(Tn - 1) * d, d, norms + size_t(2 * c.n_layers) * d, c.rms_eps, 1, 128, d,
                                  ahi, alo, st));
    KIE_CUDA(e, kie_pf_gemm(ahi, alo, pfw + L.pf_lm, C, nv, 128, nv, d, 1, colsc(a8, L.pf_sc_layer * c.n_layers), 1, 0,
                            to, err, st));
    int herr = 0;
    KIE_CUDA(e, cudaMemcpyAsync(&herr, err, 4, cudaMemcpyDeviceToHost, st));
    KIE_CUDA(e, cudaStreamSynchronize(st));
    if (herr) return fail(e, KIE_ERR_DEVICE_TIMEOUT, "prefill GEMM wait expired");
    if (last_logits) KIE_CUDA(e, cudaMemcpy(last_logits, C, size_t(V) * 4, cudaMemcpyDeviceToHost));
    e->pos = pos_start + n;
    return set_ctl(e, 0, e->pos, false);
}

}  // namespace

// ---- scratch in a static device array (for the allocation-free decode step) -------------------
//
// For callers that must not allocate device memory while decoding: code running
// inside another framework's memory pool or an allocator-less plugin host, a
// real-time service that forbids allocation after start-up, or a process whose
// device memory is already fully committed.  Together with an engine created on
// a caller-provided workspace, kie_decode_step_static_scratch performs no
// cudaMalloc, cudaFree or other allocating call.  The decode kernel's scratch
// (residual stream, q, attention output and partials, SwiGLU output, argmax
// partials, control block) lives in the array below; weights and the KV cache
// stay in the engine.

#define KIE_STATIC_SCRATCH_BYTES (320u * 1024u)

// The array belongs to this file's device module.  With CUDA's lazy module
// loading the module (and so the array's device memory) is loaded the first
// time its address is looked up; kie_create does that, with the engine's
// device current, so the decode step itself never triggers the load.  Host
// code must not use the array's name as an address.
static __device__ __align__(256) uint8_t kie_static_scratch[KIE_STATIC_SCRATCH_BYTES];

namespace {

struct StaticScratchLayout {
    size_t x, kcur, vcur, zero_bytes, q, a, o, att_part, par_bytes, amax_val, amax_idx, ctl, total;
};

StaticScratchLayout static_scratch_layout(const kie_config& c, int G) {
    StaticScratchLayout l;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = align_up(o, 256); o = at + bytes; return at; };
    const size_t hq = size_t(c.n_heads) * c.head_dim * 4;
    // tagged activations, reset per step as in the engine's workspace
    l.x = take(size_t(KIE_REPL) * c.d_model * 4);
    l.kcur = take(hq);
    l.vcur = take(hq);
    l.zero_bytes = l.vcur + hq - l.x;
    l.q = take(hq);
    l.a = take(size_t(KIE_REPL) * c.ffn_dim * 4);
    l.o = take(size_t(KIE_REPL) * hq);
    l.att_part = take(size_t(G) * (c.head_dim + 4) * 4);
    l.par_bytes = l.att_part + size_t(G) * (c.head_dim + 4) * 4 - l.q;
    l.amax_val = take(size_t(G) * 4);
    l.amax_idx = take(size_t(G) * 4);
    l.ctl = take(sizeof(KieControl));
    l.total = align_up(o, 256);
    return l;
}

// Device address of kie_static_scratch on the current device (the caller has
// made the engine's device current).  This loads the module that holds it.
cudaError_t static_scratch_address(void** out) {
    *out = nullptr;
    return cudaGetSymbolAddress(out, kie_static_scratch);
}

}  // namespace

// =============================================================================================
// C ABI
// =============================================================================================
extern "C" {

size_t kie_workspace_bytes(const kie_config* cfg) {
    std::string why;
    if (!valid_cfg(cfg, why)) return 0;
    const int G = query_grid(cfg->device, why);
    if (G <= 0) return 0;
    Plan pl;
    build_plan(*cfg, G, pl);
    Layout L;
    compute_layout(*cfg, pl, L);
    return L.total;
}

kie_status kie_create(const kie_config* cfg, void* workspace, size_t ws_bytes, void* cuda_stream, kie_engine** out) {
    if (!out) return fail(nullptr, KIE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    std::string why;
    if (!valid_cfg(cfg, why)) return fail(nullptr, KIE_ERR_INVALID_ARG, "invalid config: %s", why.c_str());
    if (cudaSetDevice(cfg->device) != cudaSuccess) return fail(nullptr, KIE_ERR_CUDA, "cudaSetDevice(%d) failed", cfg->device);
    const int G = query_grid(cfg->device, why);
    if (G <= 0) return fail(nullptr, KIE_ERR_CUDA, "%s", why.c_str());
    if (G < cfg->n_heads) return fail(nullptr, KIE_ERR_UNSUPPORTED, "need at least n_heads SMs");
    if (G > KIE_MAX_GRID) return fail(nullptr, KIE_ERR_UNSUPPORTED, "more than %d SMs", KIE_MAX_GRID);
    if (cfg->d_model > 4096) return fail(nullptr, KIE_ERR_UNSUPPORTED, "d_model above 4096");
    if (uint64_t(cfg->n_heads) * uint64_t(cfg->max_ctx) * uint64_t(G) >= (1ull << 32))
        return fail(nullptr, KIE_ERR_UNSUPPORTED, "n_heads * max_ctx too large for this grid");
    kie_engine* e = new kie_engine();
    e->cfg = *cfg;
    e->G = G;
    e->stream = static_cast<cudaStream_t>(cuda_stream);
    build_plan(*cfg, G, e->plan);
    // The ring protocol needs at least as many slots as consumer warps (see the
    // full-barrier note in kie_decode.cu).
    if (e->plan.nslot < KIE_NW) { delete e; return fail(nullptr, KIE_ERR_UNSUPPORTED, "shared memory too small for the weight ring"); }
    compute_layout(*cfg, e->plan, e->lay);
    if (workspace) {
        if (ws_bytes < e->lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
            delete e;
            return fail(nullptr, KIE_ERR_OOM, "workspace too small or misaligned (need %zu bytes)", e->lay.total);
        }
        e->ws = workspace;
    } else {
        if (cudaMalloc(&e->ws, e->lay.total) != cudaSuccess) {
            cudaGetLastError();
            delete e;
            return fail(nullptr, KIE_ERR_OOM, "cudaMalloc of %zu bytes failed", e->lay.total);
        }
        e->own_ws = true;
    }
    if (cudaMallocHost(&e->h_ctl, sizeof(KieControl)) != cudaSuccess) {
        kie_destroy(e);
        return fail(nullptr, KIE_ERR_OOM, "cudaMallocHost failed");
    }
    if (e->batched() && cfg->batch * cfg->n_heads > G) {
        kie_destroy(e);
        return fail(nullptr, KIE_ERR_UNSUPPORTED, "batch * n_heads = %d exceeds the %d SMs", cfg->batch * cfg->n_heads, G);
    }
    e->kernel = e->batched() ? kie_decode_batch_kernel_ptr(cfg->head_dim, cfg->kv_dtype)
                             : kie_decode_kernel_ptr(cfg->head_dim, cfg->kv_dtype);
    cudaError_t r = cudaFuncSetAttribute(e->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(e->plan.smem));
    if (r != cudaSuccess) { kie_destroy(e); return fail(nullptr, KIE_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(r)); }
    int per_sm = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, e->kernel, KIE_THREADS, e->plan.smem);
    if (r != cudaSuccess || per_sm < 1) { kie_destroy(e); return fail(nullptr, KIE_ERR_LAUNCH, "decode kernel does not fit on an SM"); }
    // the static scratch array of the allocation-free decode step: looked up
    // now, so that its module is loaded here and never by that step
    r = static_scratch_address(&e->static_scratch);
    if (r != cudaSuccess) { kie_destroy(e); return fail(nullptr, KIE_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(r)); }

    // plan tables and parameters
    const Layout& L = e->lay;
    const Plan& pl = e->plan;
    std::vector<int32_t> pi32(size_t(PH_NTYPES) * (G + 1));
    std::vector<uint32_t> pu32(size_t(PH_NTYPES) * 2 * G);
    for (int t = 0; t < PH_NTYPES; ++t) {
        std::copy(pl.ph[t].unit_begin.begin(), pl.ph[t].unit_begin.end(), pi32.begin() + size_t(t) * (G + 1));
        std::copy(pl.ph[t].bytes.begin(), pl.ph[t].bytes.end(), pu32.begin() + size_t(t) * 2 * G);
        std::copy(pl.ph[t].nslots.begin(), pl.ph[t].nslots.end(), pu32.begin() + size_t(t) * 2 * G + G);
    }
    std::vector<float> invf(cfg->head_dim / 2);
    for (int i = 0; i < cfg->head_dim / 2; ++i)
        invf[i] = float(std::pow(double(cfg->rope_theta), -(2.0 * i) / cfg->head_dim));
    cudaStream_t st = e->stream;
    bool ok = cudaMemcpyAsync(e->dev(L.plan_i32), pi32.data(), pi32.size() * 4, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(e->dev(L.plan_u32), pu32.data(), pu32.size() * 4, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(e->dev(L.cta_base), pl.cta_base.data(), G * 8, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(e->dev(L.cta_layer), pl.cta_layer.data(), G * 8, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemcpyAsync(e->dev(L.inv_freq), invf.data(), invf.size() * 4, cudaMemcpyHostToDevice, st) == cudaSuccess &&
              cudaMemsetAsync(e->dev(L.x), 0, L.plan_i32 - L.x, st) == cudaSuccess &&
              cudaStreamSynchronize(st) == cudaSuccess;
    if (!ok) { kie_destroy(e); return fail(nullptr, KIE_ERR_CUDA, "initialising device tables failed"); }
    if (init_kv_scales(e) != KIE_OK) { kie_destroy(e); return fail(nullptr, KIE_ERR_CUDA, "initialising KV scales failed"); }

    KieParams& P = e->P;
    P.L = cfg->n_layers; P.d = cfg->d_model; P.H = cfg->n_heads; P.hd = cfg->head_dim; P.F = cfg->ffn_dim;
    P.V = cfg->vocab; P.max_ctx = cfg->max_ctx; P.G = G;
    P.eps = cfg->rms_eps;
    P.attn_scale = float(1.0 / std::sqrt(double(cfg->head_dim)));
    P.kv = cfg->kv_dtype;
    P.nseg = L.nseg;
    P.wstream = e->dev(L.wstream);
    P.cta_base = reinterpret_cast<const uint64_t*>(e->dev(L.cta_base));
    P.cta_layer = reinterpret_cast<const uint64_t*>(e->dev(L.cta_layer));
    for (int t = 0; t < PH_NTYPES; ++t) {
        KiePhasePlan& q = P.ph[t];
        const HostPhase& h = pl.ph[t];
        q.K = h.K; q.KC = h.KC; q.nK = h.nK; q.rows_per_unit = h.rpu; q.wfmt = h.wfmt; q.n_units = h.n_units;
        q.R = h.R;
        q.cpb = h.cpb;
        q.wscale = (h.wfmt == WF_F8 || h.wfmt == WF_F4) ? reinterpret_cast<const float*>(e->dev(L.wsc)) + L.wsc_off[t]
                                                         : nullptr;
        q.wscale_layer = int64_t(L.wsc_layer);
        q.unit_begin = reinterpret_cast<const int32_t*>(e->dev(L.plan_i32)) + size_t(t) * (G + 1);
        q.bytes = reinterpret_cast<const uint32_t*>(e->dev(L.plan_u32)) + size_t(t) * 2 * G;
        q.nslots = q.bytes + G;
    }
    P.emb = reinterpret_cast<const uint16_t*>(e->dev(L.emb));
    P.norms = reinterpret_cast<const float*>(e->dev(L.norms));
    P.inv_freq = reinterpret_cast<const float*>(e->dev(L.inv_freq));
    P.kc = e->dev(L.kc);
    P.vc = e->dev(L.vc);
    P.tail = reinterpret_cast<uint16_t*>(e->dev(L.tail));
    P.seg_scale = reinterpret_cast<float*>(e->dev(L.seg_scale));
    P.seg_zp = reinterpret_cast<int32_t*>(e->dev(L.seg_zp));
    P.kv_sc = reinterpret_cast<float*>(e->dev(L.kv_sc));
    P.kv_mx = reinterpret_cast<uint32_t*>(e->dev(L.kv_mx));
    P.nslice = L.nslice;
    P.x = reinterpret_cast<float*>(e->dev(L.x));
    P.q = reinterpret_cast<float*>(e->dev(L.q));
    P.a = reinterpret_cast<float*>(e->dev(L.a));
    P.o = reinterpret_cast<float*>(e->dev(L.o));
    P.kcur = reinterpret_cast<uint32_t*>(e->dev(L.kcur));
    P.vcur = reinterpret_cast<uint32_t*>(e->dev(L.vcur));
    P.att_part = reinterpret_cast<float*>(e->dev(L.att_part));
    P.amax_val = reinterpret_cast<float*>(e->dev(L.amax_val));
    P.amax_idx = reinterpret_cast<int32_t*>(e->dev(L.amax_idx));
    P.ctl = reinterpret_cast<KieControl*>(e->dev(L.ctl));
    P.nb = pl.nb;
    P.kv_req = int64_t(L.kv_bytes / (cfg->kv_dtype == KIE_KV_FP16 ? 2 : 1));
    P.req_tok = reinterpret_cast<int32_t*>(e->dev(L.req));
    P.req_pos = P.req_tok + KIE_MAX_BATCH;
    P.nslot = pl.nslot;
    P.act_floats = pl.act_floats;
    P.part_floats = pl.part_floats;
    *out = e;
    return KIE_OK;
}

kie_status kie_load_weights(kie_engine* e, const kie_weights* w) {
    if (!e || !w || !w->tok_emb || !w->final_norm || !w->lm_head || !w->layers)
        return fail(e, KIE_ERR_INVALID_ARG, "NULL engine or weight pointer");
    const kie_config& c = e->cfg;
    const int d = c.d_model, H = c.n_heads, hd = c.head_dim, F = c.ffn_dim, V = c.vocab, G = e->G;
    for (int l = 0; l < c.n_layers; ++l) {
        const kie_layer_weights& lw = w->layers[l];
        if (!lw.attn_norm || !lw.wq || !lw.wk || !lw.wv || !lw.wo || !lw.ffn_norm || !lw.w_gate || !lw.w_up || !lw.w_down)
            return fail(e, KIE_ERR_INVALID_ARG, "NULL weight pointer in layer %d", l);
    }
    cudaStream_t st = e->stream;
    const Layout& L = e->lay;
    const Plan& pl = e->plan;
    const cudaMemcpyKind kind = w->on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    e->loaded = false;
    drop_graphs(e);

    // embedding (as given) and norm gains (fp32)
    KIE_CUDA(e, cudaMemcpyAsync(e->dev(L.emb), w->tok_emb, size_t(V) * d * 2, kind, st));
    {
        std::vector<uint16_t> g16(size_t(c.n_layers * 2 + 1) * d);
        for (int l = 0; l < c.n_layers; ++l) {
            KIE_CUDA(e, cudaMemcpy(g16.data() + size_t(2 * l) * d, w->layers[l].attn_norm, size_t(d) * 2, w->on_device ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost));
            KIE_CUDA(e, cudaMemcpy(g16.data() + size_t(2 * l + 1) * d, w->layers[l].ffn_norm, size_t(d) * 2, w->on_device ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost));
        }
        KIE_CUDA(e, cudaMemcpy(g16.data() + size_t(2 * c.n_layers) * d, w->final_norm, size_t(d) * 2, w->on_device ? cudaMemcpyDeviceToHost : cudaMemcpyHostToHost));
        std::vector<float> g32(g16.size());
        for (size_t i = 0; i < g16.size(); ++i) {
            // fp16 -> fp32, exact (IEEE half layout)
            const uint16_t h = g16[i];
            const uint32_t s = uint32_t(h >> 15) << 31, ex = (h >> 10) & 31, m = h & 1023;
            float f;
            if (ex == 0) f = std::ldexp(float(m), -24);
            else if (ex == 31) f = m ? NAN : INFINITY;
            else f = std::ldexp(float(m | 1024), int(ex) - 25);
            uint32_t b;
            std::memcpy(&b, &f, 4);
            b |= s;
            std::memcpy(&g32[i], &b, 4);
        }
        KIE_CUDA(e, cudaMemcpyAsync(e->dev(L.norms), g32.data(), g32.size() * 4, cudaMemcpyHostToDevice, st));
        KIE_CUDA(e, cudaStreamSynchronize(st));
    }

    // staging buffer on the device for one source matrix (plus INT4 codes/scales)
    const size_t max_mat = std::max({size_t(H) * hd * d, size_t(F) * d, size_t(V) * d}) * 2;
    size_t i4_elems = 0;   // the largest INT4 matrix: F x d (FFN) or H*h x d (q, k, v)
    if (c.ffn_wdtype == KIE_W_INT4_G128) i4_elems = size_t(F) * d;
    if (c.attn_wdtype == KIE_W_INT4_G128) i4_elems = std::max(i4_elems, size_t(H) * hd * d);
    const size_t i4_bytes = i4_elems ? i4_elems / 2 + i4_elems / 128 * 2 + 256 : 0;
    uint8_t* stage = nullptr;
    uint8_t* i4 = nullptr;
    CopyDesc* ddesc = nullptr;
    size_t desc_cap = 0;
    if (!w->on_device && cudaMalloc(&stage, max_mat) != cudaSuccess) return fail(e, KIE_ERR_OOM, "staging cudaMalloc failed");
    if (i4_bytes && cudaMalloc(&i4, i4_bytes) != cudaSuccess) { cudaFree(stage); return fail(e, KIE_ERR_OOM, "INT4 staging cudaMalloc failed"); }
    kie_status result = KIE_OK;
    std::vector<CopyDesc> desc;

    auto free_all = [&]() {
        if (stage) cudaFree(stage);
        if (i4) cudaFree(i4);
        if (ddesc) cudaFree(ddesc);
    };
    auto flush = [&](const uint8_t* src_base) -> bool {
        if (desc.empty()) return true;
        if (desc.size() > desc_cap) {
            if (ddesc) cudaFree(ddesc);
            desc_cap = desc.size() * 2;
            if (cudaMalloc(&ddesc, desc_cap * sizeof(CopyDesc)) != cudaSuccess) { ddesc = nullptr; return false; }
        }
        if (cudaMemcpyAsync(ddesc, desc.data(), desc.size() * sizeof(CopyDesc), cudaMemcpyHostToDevice, st) != cudaSuccess) return false;
        if (kie_launch_copy_desc(e->dev(L.wstream), src_base, ddesc, int(desc.size()), st) != cudaSuccess) return false;
        if (cudaStreamSynchronize(st) != cudaSuccess) return false;
        desc.clear();
        return true;
    };
    // Emit copies of every row of phase `t` whose source is matrix `mat` (selector).
    // row_of(unit, half) -> (matrix id, source row) ; base offset of the layer's phase in each CTA stream.
    auto emit = [&](int t, int layer, int mat, auto row_of, bool int4, uint64_t codes_off, uint64_t scales_off) {
        const HostPhase& p = pl.ph[t];
        const int K = p.K;
        for (int i = 0; i < G; ++i) {
            uint64_t off = pl.cta_base[i];
            if (t == PH_LM) off += uint64_t(c.n_layers) * pl.cta_layer[i];
            else {
                off += uint64_t(layer) * pl.cta_layer[i];
                for (int tt = 0; tt < t; ++tt) off += pl.ph[tt].bytes[i];
            }
            const int u0 = p.unit_begin[i], nu = p.unit_begin[i + 1] - u0;
            const int rows = nu * p.rpu;
            const int groups = (rows + p.R - 1) / p.R;
            // slots in the order (staging block, row group, chunk); a block is the whole row
            // except in the batched kernel (KIE_KBLK columns)
            for (int ch0 = 0; ch0 < p.nK; ch0 += p.cpb)
            for (int g = 0; g < groups; ++g) {
                const int rg = std::min(p.R, rows - g * p.R);
                for (int ch = ch0; ch < std::min(p.nK, ch0 + p.cpb); ++ch) {
                    const int kc = std::min(p.KC, K - ch * p.KC);
                    for (int r = 0; r < rg; ++r) {
                        const int lr = g * p.R + r;
                        int m, srow;
                        row_of(u0 + lr / p.rpu, lr % p.rpu, m, srow);
                        if (m != mat) continue;
                        if (p.wfmt == WF_F8) {   // source: the matrix's E4M3 codes [rows][K]
                            desc.push_back({off + uint64_t(r) * kc, uint64_t(srow) * K + uint64_t(ch) * p.KC,
                                            uint32_t(kc), 0});
                        } else if (p.wfmt == WF_F4) {   // source: packed E2M1 codes [rows][K/2], then block scales [rows][K/16]
                            desc.push_back({off + uint64_t(r) * (kc / 2),
                                            uint64_t(srow) * (K / 2) + uint64_t(ch) * (p.KC / 2), uint32_t(kc / 2), 0});
                            desc.push_back({off + uint64_t(rg) * (kc / 2) + uint64_t(r) * (kc / 16),
                                            scales_off + uint64_t(srow) * (K / 16) + uint64_t(ch) * (p.KC / 16),
                                            uint32_t(kc / 16), 0});
                        } else if (!int4) {
                            desc.push_back({off + uint64_t(r) * kc * 2, uint64_t(srow) * K * 2 + uint64_t(ch) * p.KC * 2,
                                            uint32_t(kc * 2), 0});
                        } else {
                            desc.push_back({off + uint64_t(r) * (kc / 2),
                                            codes_off + uint64_t(srow) * (K / 2) + uint64_t(ch) * (p.KC / 2), uint32_t(kc / 2), 0});
                            desc.push_back({off + uint64_t(rg) * (kc / 2) + uint64_t(r) * (kc / 64),
                                            scales_off + uint64_t(srow) * (K / 128) * 2 + uint64_t(ch) * (p.KC / 128) * 2,
                                            uint32_t(kc / 64), 0});
                        }
                    }
                    off += slot_bytes_host(p.wfmt, rg, kc);
                }
            }
        }
    };
    auto src_of = [&](const uint16_t* ptr, size_t bytes) -> const uint8_t* {
        if (w->on_device) return reinterpret_cast<const uint8_t*>(ptr);
        if (cudaMemcpyAsync(stage, ptr, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return nullptr;
        return stage;
    };
    const int hh = hd / 2, per = H * hh;
    auto qkv_row = [&](int U, int half, int& m, int& srow) {
        const int which = U / per, rem = U % per, h = rem / hh, i = rem % hh;
        m = which;
        srow = h * hd + i + half * hh;
    };
    auto plain_row = [&](int U, int, int& m, int& srow) { m = 0; srow = U; };
    auto gu_row = [&](int U, int half, int& m, int& srow) { m = half; srow = U; };

    // tensor-core prefill copy of the weights (tiles; padding rows stay zero)
    __half* pfw = reinterpret_cast<__half*>(e->dev(L.pf_w));
    if (L.pf && cudaMemsetAsync(pfw, 0, (L.pf_lm + size_t(pad256(V)) * d) * 2, st) != cudaSuccess)
        result = fail(e, KIE_ERR_CUDA, "prefill weight clear failed");
    const int HDm = H * hd;
    // FP8 staging: one matrix's codes and row scales; host copies of the scales
    const bool any_f8 = scaled_fmt(c.attn_wdtype) || scaled_fmt(c.ffn_wdtype);
    const size_t max_rows = std::max({size_t(HDm), size_t(F), size_t(d), size_t(V)});
    uint8_t* f8codes = nullptr;
    float* f8sc = nullptr;
    if (any_f8 && (cudaMalloc(&f8codes, max_mat / 2 + 256) != cudaSuccess || cudaMalloc(&f8sc, max_rows * 4) != cudaSuccess)) {
        if (f8codes) cudaFree(f8codes);
        f8codes = nullptr;
        result = fail(e, KIE_ERR_OOM, "FP8 staging cudaMalloc failed");
    }
    std::vector<float> sc_host(max_rows), wsc_phase, pfsc;
    if (L.pf && any_f8) pfsc.assign(L.pf_sc_layer * c.n_layers + size_t(V), 0.f);
    // One matrix of phase t (source fp16 `s`, n rows x K): into the decode stream
    // (fp16 as given or FP8 codes) and, for the prefill, into its weight tiles
    // at rows [pf_row0, pf_row0 + n) of the tile array at pf_off (with its
    // column scales at pf_sc_off + pf_row0 for FP8).
    auto put_matrix = [&](int t, int l, int m, auto row_of, const uint8_t* s, int n, int K, size_t pf_off, int pf_row0,
                          size_t pf_sc_off) -> bool {
        const HostPhase& p = pl.ph[t];
        if (p.wfmt == WF_I4) {   // INT4 g128: codes [n][K/2], then fp16 group scales [n][K/128] at sc_off
            const uint64_t sc_off = align_up(size_t(n) * K / 2, 256);
            if (kie_launch_quant_int4(reinterpret_cast<const uint16_t*>(s), n, K, i4, nullptr,
                                      reinterpret_cast<uint16_t*>(i4 + sc_off), st) != cudaSuccess)
                return false;
            emit(t, l, m, row_of, true, 0, sc_off);
            return flush(i4);
        }
        if (p.wfmt != WF_F8 && p.wfmt != WF_F4) {
            if (L.pf && kie_pf_pack(reinterpret_cast<const __half*>(s), n, K, pf_row0, pfw + pf_off, st) != cudaSuccess)
                return false;
            emit(t, l, m, row_of, false, 0, 0);
            return flush(s);
        }
        if (p.wfmt == WF_F8) {
            if (kie_launch_quant_fp8(reinterpret_cast<const uint16_t*>(s), n, K, f8codes, f8sc, st) != cudaSuccess) return false;
            if (L.pf && kie_pf_pack_e4m3(f8codes, n, K, pf_row0, pfw + pf_off, st) != cudaSuccess) return false;
            emit(t, l, m, row_of, false, 0, 0);
        } else {   // NVFP4: packed codes [n][K/2], then block scales [n][K/16] at bs_off
            const uint64_t bs_off = align_up(size_t(n) * K / 2, 256);
            if (kie_launch_quant_fp4(reinterpret_cast<const uint16_t*>(s), n, K, f8codes, nullptr, f8codes + bs_off, f8sc,
                                     st) != cudaSuccess)
                return false;
            if (L.pf && kie_pf_pack_fp4(f8codes, f8codes + bs_off, n, K, pf_row0, pfw + pf_off, st) != cudaSuccess)
                return false;
            emit(t, l, m, row_of, false, 0, bs_off);
        }
        if (!flush(f8codes)) return false;
        if (cudaMemcpy(sc_host.data(), f8sc, size_t(n) * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return false;
        // scales in the phase's row order (phase row = unit * rows_per_unit + half)
        for (int U = 0; U < p.n_units; ++U)
            for (int half = 0; half < p.rpu; ++half) {
                int mm, srow;
                row_of(U, half, mm, srow);
                if (mm == m) wsc_phase[size_t(U) * p.rpu + half] = sc_host[srow];
            }
        if (L.pf) std::copy(sc_host.begin(), sc_host.begin() + n, pfsc.begin() + pf_sc_off + pf_row0);
        return true;
    };
    auto put_scales = [&](int t, int l) -> bool {   // the phase's FP8 row scales, once all its matrices are in
        const HostPhase& p = pl.ph[t];
        if (p.wfmt != WF_F8 && p.wfmt != WF_F4) return true;
        const size_t at = t == PH_LM ? L.wsc_off[PH_LM] : L.wsc_layer * l + L.wsc_off[t];
        return cudaMemcpy(e->dev(L.wsc) + at * 4, wsc_phase.data(), size_t(p.n_units) * p.rpu * 4,
                          cudaMemcpyHostToDevice) == cudaSuccess;
    };
    for (int l = 0; l < c.n_layers && result == KIE_OK; ++l) {
        const kie_layer_weights& lw = w->layers[l];
        const uint16_t* qkv[3] = {lw.wq, lw.wk, lw.wv};
        const size_t lb = L.pf_layer_elems * l, sb = L.pf_sc_layer * l;
        wsc_phase.assign(size_t(3) * HDm, 0.f);
        for (int m = 0; m < 3 && result == KIE_OK; ++m) {
            const uint8_t* s = src_of(qkv[m], size_t(H) * hd * d * 2);
            if (!s) { result = fail(e, KIE_ERR_CUDA, "weight upload failed"); break; }
            if (!put_matrix(PH_QKV, l, m, qkv_row, s, HDm, d, lb + L.pf_qkv, m * HDm, sb))
                result = fail(e, KIE_ERR_CUDA, "repack failed");
        }
        if (result == KIE_OK && !put_scales(PH_QKV, l)) result = fail(e, KIE_ERR_CUDA, "scale upload failed");
        if (result != KIE_OK) break;
        {
            wsc_phase.assign(size_t(d), 0.f);
            const uint8_t* s = src_of(lw.wo, size_t(d) * H * hd * 2);
            if (!s) { result = fail(e, KIE_ERR_CUDA, "weight upload failed"); break; }
            if (!put_matrix(PH_O, l, 0, plain_row, s, d, HDm, lb + L.pf_o, 0, sb + size_t(3) * HDm) ||
                !put_scales(PH_O, l)) { result = fail(e, KIE_ERR_CUDA, "repack failed"); break; }
        }
        const uint16_t* gu[2] = {lw.w_gate, lw.w_up};
        wsc_phase.assign(size_t(2) * F, 0.f);
        for (int m = 0; m < 2 && result == KIE_OK; ++m) {
            const uint8_t* s = src_of(gu[m], size_t(F) * d * 2);
            if (!s) { result = fail(e, KIE_ERR_CUDA, "weight upload failed"); break; }
            if (!put_matrix(PH_GU, l, m, gu_row, s, F, d, lb + L.pf_gu, m * F, sb + size_t(3) * HDm + d))
                result = fail(e, KIE_ERR_CUDA, "repack failed");
        }
        if (result == KIE_OK && !put_scales(PH_GU, l)) result = fail(e, KIE_ERR_CUDA, "scale upload failed");
        if (result != KIE_OK) break;
        {
            wsc_phase.assign(size_t(d), 0.f);
            const uint8_t* s = src_of(lw.w_down, size_t(d) * F * 2);
            if (!s) { result = fail(e, KIE_ERR_CUDA, "weight upload failed"); break; }
            if (!put_matrix(PH_D, l, 0, plain_row, s, d, F, lb + L.pf_d, 0, sb + size_t(3) * HDm + d + 2 * size_t(F)) ||
                !put_scales(PH_D, l)) {
                result = fail(e, KIE_ERR_CUDA, "repack failed");
            }
        }
    }
    if (result == KIE_OK) {
        wsc_phase.assign(size_t(V), 0.f);
        const uint8_t* s = src_of(w->lm_head, size_t(V) * d * 2);
        if (!s) result = fail(e, KIE_ERR_CUDA, "weight upload failed");
        else if (!put_matrix(PH_LM, 0, 0, plain_row, s, V, d, L.pf_lm, 0, L.pf_sc_layer * c.n_layers) ||
                 !put_scales(PH_LM, 0))
            result = fail(e, KIE_ERR_CUDA, "repack failed");
    }
    if (result == KIE_OK && L.pf && any_f8 &&
        cudaMemcpy(e->dev(L.pf_sc), pfsc.data(), pfsc.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess)
        result = fail(e, KIE_ERR_CUDA, "prefill scale upload failed");
    if (result == KIE_OK && e->batched()) {
        // the batched kernel reads its fp16 slots chunk-major: rewrite every slot in place
        std::vector<uint4> tab;
        for (int i = 0; i < G; ++i) {
            uint64_t off = pl.cta_base[i];
            for (int l = 0; l <= c.n_layers; ++l) {
                for (int t : {PH_QKV, PH_O, PH_GU, PH_D, PH_LM}) {
                    if ((l == c.n_layers) != (t == PH_LM)) continue;
                    const HostPhase& p = pl.ph[t];
                    const int rows = (p.unit_begin[i + 1] - p.unit_begin[i]) * p.rpu;
                    const int groups = (rows + p.R - 1) / p.R;
                    for (int ch0 = 0; ch0 < p.nK; ch0 += p.cpb)
                        for (int g = 0; g < groups; ++g)
                            for (int ch = ch0; ch < std::min(p.nK, ch0 + p.cpb); ++ch) {
                                const int rg = std::min(p.R, rows - g * p.R), kc = std::min(p.KC, p.K - ch * p.KC);
                                tab.push_back(make_uint4(uint32_t(off), uint32_t(off >> 32), uint32_t(rg), uint32_t(kc)));
                                off += slot_bytes_host(p.wfmt, rg, kc);
                            }
                }
            }
        }
        uint4* dtab = nullptr;
        if (cudaMalloc(&dtab, tab.size() * sizeof(uint4)) != cudaSuccess) result = fail(e, KIE_ERR_OOM, "slot table cudaMalloc failed");
        else {
            if (cudaMemcpyAsync(dtab, tab.data(), tab.size() * sizeof(uint4), cudaMemcpyHostToDevice, st) != cudaSuccess ||
                kie_launch_slot_chunk_major(e->dev(L.wstream), dtab, int(tab.size()), st) != cudaSuccess ||
                cudaStreamSynchronize(st) != cudaSuccess)
                result = fail(e, KIE_ERR_CUDA, "slot layout pass failed");
            cudaFree(dtab);
        }
    }
    if (f8codes) cudaFree(f8codes);
    if (f8sc) cudaFree(f8sc);
    cudaStreamSynchronize(st);
    free_all();
    if (result != KIE_OK) return result;
    e->loaded = true;
    e->pos = 0;
    std::fill(std::begin(e->rpos), std::end(e->rpos), 0);
    e->sticky = 0;
    if ((result = init_kv_scales(e)) != KIE_OK) return result;
    return set_ctl(e, 0, 0, true);
}

kie_status kie_prefill(kie_engine* e, const int32_t* tokens, int32_t n, float* last_logits) {
    kie_status st = ready(e, n);
    if (st != KIE_OK) return st;
    if (n == 0) return KIE_OK;
    if (!tokens) return fail(e, KIE_ERR_INVALID_ARG, "tokens is NULL");
    if ((st = check_tokens(e, tokens, n)) != KIE_OK) return st;
    if (e->lay.pf) return prefill_tensor_cores(e, tokens, n, last_logits);
    int32_t* d_forced = reinterpret_cast<int32_t*>(e->dev(e->lay.forced));
    KIE_CUDA(e, cudaMemcpyAsync(d_forced, tokens, size_t(n) * 4, cudaMemcpyHostToDevice, e->stream));
    float* d_log = reinterpret_cast<float*>(e->dev(e->lay.out_logits));
    const int pos0 = e->pos;
    if ((st = run_steps(e, n, -1, d_forced, n - 1, nullptr, d_log)) != KIE_OK) { e->pos = pos0; return st; }
    if ((st = check_device(e)) != KIE_OK) return st;
    if (last_logits)
        KIE_CUDA(e, cudaMemcpy(last_logits, d_log, size_t(e->cfg.vocab) * 4, cudaMemcpyDeviceToHost));
    return KIE_OK;
}

kie_status kie_generate_greedy_device(kie_engine* e, int32_t first_token, int32_t n, int32_t* d_out_tokens,
                                      float* d_out_logits) {
    kie_status st = ready(e, n);
    if (st != KIE_OK) return st;
    if (e->batched()) return fail(e, KIE_ERR_UNSUPPORTED, "a batched engine decodes with kie_generate_greedy_batch");
    if (n == 0) return KIE_OK;
    if (!d_out_tokens) return fail(e, KIE_ERR_INVALID_ARG, "d_out_tokens is NULL");
    if ((st = check_tokens(e, &first_token, 1)) != KIE_OK) return st;
    return run_steps(e, n, first_token, nullptr, 0, d_out_tokens, d_out_logits);
}

kie_status kie_generate_greedy(kie_engine* e, int32_t first_token, int32_t n, int32_t* out_tokens, float* out_logits) {
    kie_status st = ready(e, n);
    if (st != KIE_OK) return st;
    if (e->batched()) return fail(e, KIE_ERR_UNSUPPORTED, "a batched engine decodes with kie_generate_greedy_batch");
    if (n == 0) return KIE_OK;
    if (!out_tokens) return fail(e, KIE_ERR_INVALID_ARG, "out_tokens is NULL");
    if ((st = check_tokens(e, &first_token, 1)) != KIE_OK) return st;
    int32_t* d_tok = reinterpret_cast<int32_t*>(e->dev(e->lay.out_tokens));
    float* d_log = reinterpret_cast<float*>(e->dev(e->lay.out_logits));
    if (!out_logits) {
        if ((st = run_steps(e, n, first_token, nullptr, 0, d_tok, nullptr)) != KIE_OK) return st;
    } else {
        int done = 0, tok = first_token;
        while (done < n) {
            const int m = std::min(kLogitChunk, n - done);
            if ((st = run_steps(e, m, tok, nullptr, 0, d_tok + done, d_log)) != KIE_OK) return st;
            KIE_CUDA(e, cudaMemcpyAsync(out_logits + size_t(done) * e->cfg.vocab, d_log, size_t(m) * e->cfg.vocab * 4,
                                        cudaMemcpyDeviceToHost, e->stream));
            if ((st = check_device(e)) != KIE_OK) return st;
            KIE_CUDA(e, cudaMemcpy(&tok, d_tok + done + m - 1, 4, cudaMemcpyDeviceToHost));
            done += m;
        }
    }
    KIE_CUDA(e, cudaMemcpyAsync(out_tokens, d_tok, size_t(n) * 4, cudaMemcpyDeviceToHost, e->stream));
    return check_device(e);
}

kie_status kie_decode_step(kie_engine* e, int32_t token, int32_t* next_token, float* logits) {
    if (!next_token) return fail(e, KIE_ERR_INVALID_ARG, "next_token is NULL");
    return kie_generate_greedy(e, token, 1, next_token, logits);
}

kie_status kie_select_request(kie_engine* e, int32_t request) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    const int nbq = e->batched() ? e->plan.nb : 1;
    if (request < 0 || request >= nbq) return fail(e, KIE_ERR_INVALID_ARG, "request %d outside [0, %d)", request, nbq);
    e->rpos[e->cur] = e->pos;
    e->cur = request;
    e->pos = e->rpos[request];
    return KIE_OK;
}

}  // extern "C"

namespace {

kie_status ready_batch(kie_engine* e, int n) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    if (!e->batched()) return fail(e, KIE_ERR_UNSUPPORTED, "not a batched engine (kie_config.batch < 2)");
    if (!e->loaded) return fail(e, KIE_ERR_NOT_LOADED, "weights not loaded");
    if (e->sticky) return fail(e, KIE_ERR_DEVICE_TIMEOUT, "engine poisoned by an earlier device error; call kie_reset");
    if (n < 0) return fail(e, KIE_ERR_INVALID_ARG, "negative count");
    e->rpos[e->cur] = e->pos;
    for (int b = 0; b < e->plan.nb; ++b)
        if (int64_t(e->rpos[b]) + n > e->cfg.max_ctx)
            return fail(e, KIE_ERR_CTX_OVERFLOW, "request %d: pos %d + %d > max_ctx %d", b, e->rpos[b], n, e->cfg.max_ctx);
    return KIE_OK;
}

// n steps of every request of a batched engine, one persistent launch.  first:
// host tokens [nb], or null to continue from the tokens the device holds.
kie_status run_batch(kie_engine* e, const int32_t* first, int n, int32_t* d_tokens, float* d_logits) {
    if (n <= 0) return KIE_OK;
    const int nb = e->plan.nb;
    int32_t h[2 * KIE_MAX_BATCH] = {};
    for (int b = 0; b < nb; ++b) {
        h[b] = first ? first[b] : 0;
        h[KIE_MAX_BATCH + b] = e->rpos[b];
    }
    int32_t* dreq = reinterpret_cast<int32_t*>(e->dev(e->lay.req));
    if (first) KIE_CUDA(e, cudaMemcpyAsync(dreq, h, sizeof(h), cudaMemcpyHostToDevice, e->stream));
    else KIE_CUDA(e, cudaMemcpyAsync(dreq + KIE_MAX_BATCH, h + KIE_MAX_BATCH, KIE_MAX_BATCH * 4, cudaMemcpyHostToDevice, e->stream));
    KieLaunch l = base_launch(e);
    l.n_steps = n;
    l.pos0 = e->rpos[0];   // the tags number writes by request 0's position
    l.out_tokens = d_tokens;
    l.out_logits = d_logits;
    kie_status st = launch_persistent(e, l);
    if (st != KIE_OK) return st;
    for (int b = 0; b < nb; ++b) e->rpos[b] += n;
    e->pos = e->rpos[e->cur];
    return KIE_OK;
}

kie_status check_batch_tokens(kie_engine* e, const int32_t* t) {
    if (!t) return fail(e, KIE_ERR_INVALID_ARG, "token array is NULL");
    return check_tokens(e, t, e->plan.nb);
}

}  // namespace

extern "C" {

kie_status kie_generate_greedy_batch_device(kie_engine* e, const int32_t* first_tokens, int32_t n,
                                            int32_t* d_out_tokens, float* d_out_logits) {
    kie_status st = ready_batch(e, n);
    if (st != KIE_OK) return st;
    if (n == 0) return KIE_OK;
    if (!d_out_tokens) return fail(e, KIE_ERR_INVALID_ARG, "d_out_tokens is NULL");
    if ((st = check_batch_tokens(e, first_tokens)) != KIE_OK) return st;
    return run_batch(e, first_tokens, n, d_out_tokens, d_out_logits);
}

kie_status kie_generate_greedy_batch(kie_engine* e, const int32_t* first_tokens, int32_t n, int32_t* out_tokens,
                                     float* out_logits) {
    kie_status st = ready_batch(e, n);
    if (st != KIE_OK) return st;
    if (n == 0) return KIE_OK;
    if (!out_tokens) return fail(e, KIE_ERR_INVALID_ARG, "out_tokens is NULL");
    if ((st = check_batch_tokens(e, first_tokens)) != KIE_OK) return st;
    const int nb = e->plan.nb;
    const size_t V = size_t(e->cfg.vocab);
    int32_t* d_tok = reinterpret_cast<int32_t*>(e->dev(e->lay.out_tokens));
    float* d_log = reinterpret_cast<float*>(e->dev(e->lay.out_logits));
    if (!out_logits) {
        if ((st = run_batch(e, first_tokens, n, d_tok, nullptr)) != KIE_OK) return st;
    } else {
        for (int done = 0; done < n;) {
            const int m = std::min(kLogitChunk, n - done);
            if ((st = run_batch(e, done == 0 ? first_tokens : nullptr, m, d_tok + size_t(done) * nb, d_log)) != KIE_OK)
                return st;
            KIE_CUDA(e, cudaMemcpyAsync(out_logits + size_t(done) * nb * V, d_log, size_t(m) * nb * V * 4,
                                        cudaMemcpyDeviceToHost, e->stream));
            if ((st = check_device(e)) != KIE_OK) return st;
            done += m;
        }
    }
    KIE_CUDA(e, cudaMemcpyAsync(out_tokens, d_tok, size_t(n) * nb * 4, cudaMemcpyDeviceToHost, e->stream));
    return check_device(e);
}

kie_status kie_decode_batch(kie_engine* e, const int32_t* tokens, int32_t* next_tokens, float* logits) {
    if (!next_tokens) return fail(e, KIE_ERR_INVALID_ARG, "next_tokens is NULL");
    return kie_generate_greedy_batch(e, tokens, 1, next_tokens, logits);
}

kie_status kie_trace_decode(kie_engine* e, int32_t first_token, int32_t n, uint64_t* stamps, size_t cap) {
    kie_status st = ready(e, n);
    if (st != KIE_OK) return st;
    if (e->cfg.mode != KIE_MODE_PERSISTENT) return fail(e, KIE_ERR_UNSUPPORTED, "tracing needs the persistent mode");
    if ((st = check_tokens(e, &first_token, 1)) != KIE_OK) return st;
    const size_t nphase = size_t(n) * (5 * e->cfg.n_layers + 1) * KIE_PROF_EVENTS * e->G;
    const size_t need = nphase + size_t(KIE_PROF_SLOTS) * 4;
    if (!stamps || cap < need) return fail(e, KIE_ERR_INVALID_ARG, "stamp buffer needs %zu entries", need);
    uint64_t* d = nullptr;
    if (cudaMalloc(&d, need * 8) != cudaSuccess) return fail(e, KIE_ERR_OOM, "trace buffer cudaMalloc failed");
    KieLaunch l = base_launch(e);
    l.n_steps = n;
    l.first_tok = first_token;
    l.pos0 = e->pos;
    if (e->batched()) {   // every request starts from first_token at its own position
        e->rpos[e->cur] = e->pos;
        int32_t h[2 * KIE_MAX_BATCH] = {};
        for (int b = 0; b < e->plan.nb; ++b) {
            if (int64_t(e->rpos[b]) + n > e->cfg.max_ctx) { cudaFree(d); return fail(e, KIE_ERR_CTX_OVERFLOW, "request %d overflows", b); }
            h[b] = first_token;
            h[KIE_MAX_BATCH + b] = e->rpos[b];
        }
        cudaMemcpyAsync(e->dev(e->lay.req), h, sizeof(h), cudaMemcpyHostToDevice, e->stream);
        l.first_tok = -1;
        l.pos0 = e->rpos[0];
    }
    l.out_tokens = reinterpret_cast<int32_t*>(e->dev(e->lay.out_tokens));
    l.prof = d;
    l.prof_slots = d + nphase;
    cudaMemsetAsync(d, 0, need * 8, e->stream);
    st = launch_persistent(e, l);
    if (st == KIE_OK) {
        if (e->batched()) {
            for (int b = 0; b < e->plan.nb; ++b) e->rpos[b] += n;
            e->pos = e->rpos[e->cur];
        } else {
            e->pos += n;
        }
        st = check_device(e);
    }
    if (st == KIE_OK && cudaMemcpy(stamps, d, need * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(e, KIE_ERR_CUDA, "trace copy failed");
    cudaFree(d);
    return st;
}

kie_status kie_sync(kie_engine* e) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    return check_device(e);
}

kie_status kie_reset(kie_engine* e) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    cudaStreamSynchronize(e->stream);
    e->sticky = 0;
    e->pos = 0;
    std::fill(std::begin(e->rpos), std::end(e->rpos), 0);
    kie_status st0 = init_kv_scales(e);
    if (st0 != KIE_OK) return st0;
    KIE_CUDA(e, reset_tags(e->cfg, e->dev(e->lay.x), e->lay.zero_bytes, e->dev(e->lay.q), e->lay.par_bytes, 0,
                           e->stream));
    return set_ctl(e, 0, 0, true);
}

int32_t kie_get_pos(const kie_engine* e) { return e ? e->pos : -1; }

kie_status kie_set_pos(kie_engine* e, int32_t pos) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    if (pos < 0 || pos > e->cfg.max_ctx) return fail(e, KIE_ERR_INVALID_ARG, "pos %d outside [0, %d]", pos, e->cfg.max_ctx);
    e->pos = pos;
    if (e->cfg.kv_dtype == KIE_KV_FP8_E5M2_SCALED) {
        // positions >= pos leave the cache: pos's slice keeps the maximum of what stays
        const kie_config& c = e->cfg;
        KIE_CUDA(e, kie_launch_kv_rescan(e->dev(e->lay.kc), e->dev(e->lay.vc), reinterpret_cast<uint32_t*>(e->dev(e->lay.kv_mx)),
                                         c.n_layers, c.n_heads, c.head_dim, c.max_ctx, e->lay.nslice, pos, e->stream));
    }
    return set_ctl(e, 0, pos, false);
}

kie_status kie_set_timeout_ms(kie_engine* e, int32_t ms) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    if (ms <= 0) return fail(e, KIE_ERR_INVALID_ARG, "timeout must be positive");
    e->timeout_ns = uint64_t(ms) * 1000000ull;
    drop_graphs(e);
    return KIE_OK;
}

kie_status kie_debug_skip_grid_arrival(kie_engine* e, int32_t cta) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    if (cta < -1 || cta >= e->G) return fail(e, KIE_ERR_INVALID_ARG, "cta %d outside [-1, %d)", cta, e->G);
    e->skip_arrival_cta = cta;
    return KIE_OK;
}

void* kie_get_stream(const kie_engine* e) { return e ? static_cast<void*>(e->stream) : nullptr; }
int32_t kie_grid_size(const kie_engine* e) { return e ? e->G : 0; }

const char* kie_last_error(const kie_engine* e) { return e ? e->err.c_str() : g_last_error.c_str(); }

void kie_destroy(kie_engine* e) {
    if (!e) return;
    if (e->stream) cudaStreamSynchronize(e->stream);
    else cudaDeviceSynchronize();
    drop_graphs(e);
    if (e->own_ws && e->ws) cudaFree(e->ws);
    if (e->h_ctl) cudaFreeHost(e->h_ctl);
    delete e;
}

kie_status kie_set_kv(kie_engine* e, int32_t layer, const uint16_t* k_fp16, const uint16_t* v_fp16, int32_t n) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    const kie_config& c = e->cfg;
    if (layer < 0 || layer >= c.n_layers) return fail(e, KIE_ERR_INVALID_ARG, "layer %d out of range", layer);
    if (!k_fp16 || !v_fp16) return fail(e, KIE_ERR_INVALID_ARG, "NULL K or V");
    if (n < 0 || n > c.max_ctx) return fail(e, KIE_ERR_CTX_OVERFLOW, "n %d outside [0, max_ctx]", n);
    if (n == 0) return KIE_OK;
    const int H = c.n_heads, hd = c.head_dim;
    const size_t elems = size_t(n) * H * hd;
    uint16_t* stage = nullptr;
    if (cudaMalloc(&stage, elems * 2) != cudaSuccess) return fail(e, KIE_ERR_OOM, "staging cudaMalloc failed");
    kie_status result = KIE_OK;
    cudaStream_t st = e->stream;
    const Layout& L = e->lay;
    for (int kv = 0; kv < 2 && result == KIE_OK; ++kv) {
        const uint16_t* src = kv ? v_fp16 : k_fp16;
        uint8_t* base = e->dev(kv ? L.vc : L.kc) + e->kv_off();
        if (cudaMemcpyAsync(stage, src, elems * 2, cudaMemcpyHostToDevice, st) != cudaSuccess) { result = fail(e, KIE_ERR_CUDA, "upload failed"); break; }
        const size_t esz = c.kv_dtype == KIE_KV_FP16 ? 2 : 1;
        uint8_t* dst = base + size_t(layer) * H * c.max_ctx * hd * esz;
        cudaError_t r = cudaSuccess;
        if (c.kv_dtype == KIE_KV_FP8_E5M2_SCALED) {
            // slice by slice: each slice's scale comes from the slice before it
            const size_t ent = (size_t(layer) * 2 + kv) * L.nslice;
            float* sc = reinterpret_cast<float*>(e->dev(L.kv_sc)) + ent;
            uint32_t* mx = reinterpret_cast<uint32_t*>(e->dev(L.kv_mx)) + ent;
            for (int j = 0; j * KIE_KV_SLICE < n && r == cudaSuccess; ++j)
                r = kie_launch_kv_slice(stage, j * KIE_KV_SLICE, std::min(n, (j + 1) * KIE_KV_SLICE), H, hd, c.max_ctx,
                                        sc, mx, j, dst, st);
        } else if (c.kv_dtype != KIE_KV_U8_ADAPTIVE) {
            r = kie_launch_set_kv(stage, n, H, hd, c.max_ctx, c.kv_dtype == KIE_KV_FP16 ? 0 : 1, dst, nullptr, 0, st);
        } else {
            const int full = n / KIE_SEG;
            uint16_t* tail = reinterpret_cast<uint16_t*>(e->dev(L.tail)) + (size_t(layer) * 2 + kv) * H * KIE_SEG * hd;
            float* sc = reinterpret_cast<float*>(e->dev(L.seg_scale)) + (size_t(layer) * 2 + kv) * H * L.nseg;
            int32_t* zp = reinterpret_cast<int32_t*>(e->dev(L.seg_zp)) + (size_t(layer) * 2 + kv) * H * L.nseg;
            r = cudaSuccess;
            for (int h = 0; h < H && r == cudaSuccess; ++h) {
                // segment s of head h: rows p = s*128 .. +127, row stride H*hd in the source
                r = kie_launch_quant_u8(stage + size_t(h) * hd, full, int64_t(KIE_SEG) * H * hd, int64_t(H) * hd, KIE_SEG, hd,
                                        dst + size_t(h) * c.max_ctx * hd, int64_t(KIE_SEG) * hd, hd, sc + size_t(h) * L.nseg,
                                        zp + size_t(h) * L.nseg, 1, st);
            }
            if (r == cudaSuccess) r = kie_launch_set_kv(stage, n, H, hd, c.max_ctx, 2, nullptr, tail, full * KIE_SEG, st);
        }
        if (r != cudaSuccess) result = fail(e, KIE_ERR_CUDA, "set_kv kernel: %s", cudaGetErrorString(r));
        if (cudaStreamSynchronize(st) != cudaSuccess) result = fail(e, KIE_ERR_CUDA, "set_kv sync failed");
    }
    cudaFree(stage);
    return result;
}

kie_status kie_read_kv(kie_engine* e, int32_t layer, int32_t which, int32_t p0, int32_t n, void* out,
                       uint16_t* tail_fp16, float* scale, int32_t* zp) {
    if (!e) return fail(nullptr, KIE_ERR_INVALID_ARG, "engine is NULL");
    const kie_config& c = e->cfg;
    if (layer < 0 || layer >= c.n_layers || (which != 0 && which != 1)) return fail(e, KIE_ERR_INVALID_ARG, "bad layer/which");
    if (p0 < 0 || n < 0 || int64_t(p0) + n > c.max_ctx) return fail(e, KIE_ERR_INVALID_ARG, "bad range");
    if (!out) return fail(e, KIE_ERR_INVALID_ARG, "out is NULL");
    KIE_CUDA(e, cudaStreamSynchronize(e->stream));
    const Layout& L = e->lay;
    const int H = c.n_heads, hd = c.head_dim;
    const size_t esz = c.kv_dtype == KIE_KV_FP16 ? 2 : 1;
    const uint8_t* base = e->dev(which ? L.vc : L.kc) + e->kv_off() + size_t(layer) * H * c.max_ctx * hd * esz;
    for (int h = 0; h < H; ++h)
        KIE_CUDA(e, cudaMemcpy(static_cast<uint8_t*>(out) + size_t(h) * n * hd * esz,
                               base + (size_t(h) * c.max_ctx + p0) * hd * esz, size_t(n) * hd * esz, cudaMemcpyDeviceToHost));
    if (c.kv_dtype == KIE_KV_FP8_E5M2_SCALED && scale) {   // the scales of the slices [p0, p0 + n) meets
        const int s0 = p0 / KIE_KV_SLICE, s1 = (p0 + n + KIE_KV_SLICE - 1) / KIE_KV_SLICE;
        if (s1 > s0)
            KIE_CUDA(e, cudaMemcpy(scale, e->dev(L.kv_sc) + ((size_t(layer) * 2 + which) * L.nslice + s0) * 4,
                                   size_t(s1 - s0) * 4, cudaMemcpyDeviceToHost));
    }
    if (c.kv_dtype == KIE_KV_U8_ADAPTIVE) {
        const int s0 = p0 / KIE_SEG, s1 = (p0 + n + KIE_SEG - 1) / KIE_SEG;
        for (int h = 0; h < H; ++h) {
            const size_t mi = (size_t(layer) * 2 + which) * H * L.nseg + size_t(h) * L.nseg + s0;
            if (scale && s1 > s0)
                KIE_CUDA(e, cudaMemcpy(scale + size_t(h) * (s1 - s0), e->dev(L.seg_scale) + mi * 4, size_t(s1 - s0) * 4, cudaMemcpyDeviceToHost));
            if (zp && s1 > s0)
                KIE_CUDA(e, cudaMemcpy(zp + size_t(h) * (s1 - s0), e->dev(L.seg_zp) + mi * 4, size_t(s1 - s0) * 4, cudaMemcpyDeviceToHost));
        }
        if (tail_fp16) {
            // positions of [p0, p0+n) in the open segment (the one holding
            // pos); when pos sits on a segment boundary nothing of the new
            // open segment is written yet and the tail still holds the fp16
            // values of the segment that has just been quantised
            const int open0 = (e->pos % KIE_SEG == 0 && e->pos > 0) ? e->pos - KIE_SEG : (e->pos / KIE_SEG) * KIE_SEG;
            std::vector<uint16_t> t(size_t(H) * KIE_SEG * hd);
            KIE_CUDA(e, cudaMemcpy(t.data(), e->dev(L.tail) + (size_t(layer) * 2 + which) * H * KIE_SEG * hd * 2, t.size() * 2, cudaMemcpyDeviceToHost));
            for (int h = 0; h < H; ++h)
                for (int p = p0; p < p0 + n; ++p) {
                    if (p < open0 || p >= open0 + KIE_SEG) continue;
                    std::memcpy(tail_fp16 + (size_t(h) * n + (p - p0)) * hd, t.data() + (size_t(h) * KIE_SEG + (p - open0)) * hd, size_t(hd) * 2);
                }
        }
    }
    return KIE_OK;
}

// ---- stateless routines -----------------------------------------------------------------------
kie_status kie_quantize_kv_u8(const uint16_t* x_fp16, int32_t n_seg, int32_t seg_elems, uint8_t* codes, float* scale,
                              int32_t* zp) {
    if (!x_fp16 || !codes || !scale || !zp || n_seg < 0 || seg_elems <= 0) return fail(nullptr, KIE_ERR_INVALID_ARG, "bad arguments");
    if (n_seg == 0) return KIE_OK;
    const size_t n = size_t(n_seg) * seg_elems;
    uint8_t* buf = nullptr;
    const size_t o_codes = align_up(n * 2, 256), o_sc = o_codes + align_up(n, 256), o_zp = o_sc + align_up(size_t(n_seg) * 4, 256);
    if (cudaMalloc(&buf, o_zp + size_t(n_seg) * 4) != cudaSuccess) return fail(nullptr, KIE_ERR_OOM, "cudaMalloc failed");
    kie_status st = KIE_OK;
    if (cudaMemcpy(buf, x_fp16, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        kie_launch_quant_u8(reinterpret_cast<uint16_t*>(buf), n_seg, seg_elems, seg_elems, 1, seg_elems, buf + o_codes,
                            seg_elems, seg_elems, reinterpret_cast<float*>(buf + o_sc), reinterpret_cast<int32_t*>(buf + o_zp),
                            1, nullptr) != cudaSuccess ||
        cudaMemcpy(codes, buf + o_codes, n, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(scale, buf + o_sc, size_t(n_seg) * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(zp, buf + o_zp, size_t(n_seg) * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(nullptr, KIE_ERR_CUDA, "uint8 quantisation failed: %s", cudaGetErrorString(cudaGetLastError()));
    cudaFree(buf);
    return st;
}

kie_status kie_quantize_int4_g128(const uint16_t* w_fp16, int32_t rows, int32_t cols, int8_t* codes, uint16_t* scale_fp16) {
    if (!w_fp16 || !codes || !scale_fp16 || rows <= 0 || cols <= 0 || cols % 128) return fail(nullptr, KIE_ERR_INVALID_ARG, "bad arguments");
    const size_t n = size_t(rows) * cols;
    uint8_t* buf = nullptr;
    const size_t o_codes = align_up(n * 2, 256), o_sc = o_codes + align_up(n, 256);
    if (cudaMalloc(&buf, o_sc + n / 128 * 2) != cudaSuccess) return fail(nullptr, KIE_ERR_OOM, "cudaMalloc failed");
    kie_status st = KIE_OK;
    if (cudaMemcpy(buf, w_fp16, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        kie_launch_quant_int4(reinterpret_cast<uint16_t*>(buf), rows, cols, nullptr, reinterpret_cast<int8_t*>(buf + o_codes),
                              reinterpret_cast<uint16_t*>(buf + o_sc), nullptr) != cudaSuccess ||
        cudaMemcpy(codes, buf + o_codes, n, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(scale_fp16, buf + o_sc, n / 128 * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(nullptr, KIE_ERR_CUDA, "INT4 quantisation failed: %s", cudaGetErrorString(cudaGetLastError()));
    cudaFree(buf);
    return st;
}

kie_status kie_quantize_fp8_rows(const uint16_t* w_fp16, int32_t rows, int32_t cols, uint8_t* codes, float* scales) {
    if (!w_fp16 || !codes || !scales || rows <= 0 || cols <= 0 || cols % 2)
        return fail(nullptr, KIE_ERR_INVALID_ARG, "bad arguments");
    const size_t n = size_t(rows) * cols;
    uint8_t* buf = nullptr;
    const size_t o_codes = align_up(n * 2, 256), o_sc = o_codes + align_up(n, 256);
    if (cudaMalloc(&buf, o_sc + size_t(rows) * 4) != cudaSuccess) return fail(nullptr, KIE_ERR_OOM, "cudaMalloc failed");
    kie_status st = KIE_OK;
    if (cudaMemcpy(buf, w_fp16, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        kie_launch_quant_fp8(reinterpret_cast<uint16_t*>(buf), rows, cols, buf + o_codes,
                             reinterpret_cast<float*>(buf + o_sc), nullptr) != cudaSuccess ||
        cudaMemcpy(codes, buf + o_codes, n, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(scales, buf + o_sc, size_t(rows) * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(nullptr, KIE_ERR_CUDA, "FP8 quantisation failed: %s", cudaGetErrorString(cudaGetLastError()));
    cudaFree(buf);
    return st;
}

kie_status kie_quantize_nvfp4_rows(const uint16_t* w_fp16, int32_t rows, int32_t cols, uint8_t* codes,
                                   uint8_t* block_scales, float* row_scales) {
    if (!w_fp16 || !codes || !block_scales || !row_scales || rows <= 0 || cols <= 0 || cols % 16)
        return fail(nullptr, KIE_ERR_INVALID_ARG, "bad arguments");
    const size_t n = size_t(rows) * cols;
    uint8_t* buf = nullptr;
    const size_t o_codes = align_up(n * 2, 256), o_bs = o_codes + align_up(n, 256), o_rs = o_bs + align_up(n / 16, 256);
    if (cudaMalloc(&buf, o_rs + size_t(rows) * 4) != cudaSuccess) return fail(nullptr, KIE_ERR_OOM, "cudaMalloc failed");
    kie_status st = KIE_OK;
    if (cudaMemcpy(buf, w_fp16, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        kie_launch_quant_fp4(reinterpret_cast<uint16_t*>(buf), rows, cols, nullptr, buf + o_codes, buf + o_bs,
                             reinterpret_cast<float*>(buf + o_rs), nullptr) != cudaSuccess ||
        cudaMemcpy(codes, buf + o_codes, n, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(block_scales, buf + o_bs, n / 16, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(row_scales, buf + o_rs, size_t(rows) * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(nullptr, KIE_ERR_CUDA, "NVFP4 quantisation failed: %s", cudaGetErrorString(cudaGetLastError()));
    cudaFree(buf);
    return st;
}

kie_status kie_convert_fp8_e5m2(const uint16_t* x_fp16, size_t n, uint8_t* out) {
    if (!x_fp16 || !out) return fail(nullptr, KIE_ERR_INVALID_ARG, "bad arguments");
    if (n == 0) return KIE_OK;
    uint8_t* buf = nullptr;
    const size_t o_out = align_up(n * 2, 256);
    if (cudaMalloc(&buf, o_out + n) != cudaSuccess) return fail(nullptr, KIE_ERR_OOM, "cudaMalloc failed");
    kie_status st = KIE_OK;
    if (cudaMemcpy(buf, x_fp16, n * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
        kie_launch_e5m2(reinterpret_cast<uint16_t*>(buf), n, buf + o_out, nullptr) != cudaSuccess ||
        cudaMemcpy(out, buf + o_out, n, cudaMemcpyDeviceToHost) != cudaSuccess)
        st = fail(nullptr, KIE_ERR_CUDA, "E5M2 conversion failed: %s", cudaGetErrorString(cudaGetLastError()));
    cudaFree(buf);
    return st;
}

extern "C" kie_status kie_decode_step_static_scratch(kie_engine* e, int32_t token, int32_t* d_next_token,
                                                     float* d_logits) {
    kie_status st = ready(e, 1);
    if (st != KIE_OK) return st;
    if (e->batched()) return fail(e, KIE_ERR_UNSUPPORTED, "a batched engine decodes with kie_decode_batch");
    if (!d_next_token) return fail(e, KIE_ERR_INVALID_ARG, "d_next_token is NULL");
    if ((st = check_tokens(e, &token, 1)) != KIE_OK) return st;
    if (e->cfg.mode != KIE_MODE_PERSISTENT) return fail(e, KIE_ERR_UNSUPPORTED, "static-scratch step needs the persistent mode");
    const StaticScratchLayout sl = static_scratch_layout(e->cfg, e->G);
    if (sl.total > KIE_STATIC_SCRATCH_BYTES)
        return fail(e, KIE_ERR_UNSUPPORTED, "scratch of %zu bytes exceeds the static maximum of %u bytes", sl.total,
                    KIE_STATIC_SCRATCH_BYTES);
    uint8_t* b = static_cast<uint8_t*>(e->static_scratch);
    // the control block (barrier count, error word, argmax arrivals) starts at
    // zero and the activation tags are reset; everything else is written
    // before it is read
    KIE_CUDA(e, cudaMemsetAsync(b + sl.ctl, 0, sizeof(KieControl), e->stream));
    KIE_CUDA(e, reset_tags(e->cfg, b + sl.x, sl.zero_bytes, b + sl.q, sl.par_bytes, e->pos, e->stream));
    KieParams P = e->P;
    P.x = reinterpret_cast<float*>(b + sl.x);
    P.q = reinterpret_cast<float*>(b + sl.q);
    P.o = reinterpret_cast<float*>(b + sl.o);
    P.a = reinterpret_cast<float*>(b + sl.a);
    P.kcur = reinterpret_cast<uint32_t*>(b + sl.kcur);
    P.vcur = reinterpret_cast<uint32_t*>(b + sl.vcur);
    P.att_part = reinterpret_cast<float*>(b + sl.att_part);
    P.amax_val = reinterpret_cast<float*>(b + sl.amax_val);
    P.amax_idx = reinterpret_cast<int32_t*>(b + sl.amax_idx);
    P.ctl = reinterpret_cast<KieControl*>(b + sl.ctl);
    KieLaunch l = base_launch(e);
    l.n_steps = 1;
    l.first_tok = token;
    l.pos0 = e->pos;
    l.out_tokens = d_next_token;
    l.out_logits = d_logits;
    void* args[] = {(void*)&P, (void*)&l};
    const cudaError_t r = cudaLaunchCooperativeKernel(e->kernel, dim3(e->G), dim3(KIE_THREADS), args, e->plan.smem, e->stream);
    if (r == cudaErrorCooperativeLaunchTooLarge) {
        cudaGetLastError();
        return fail(e, KIE_ERR_LAUNCH, "persistent grid of %d CTAs cannot be co-resident", e->G);
    }
    if (r != cudaSuccess) return fail(e, KIE_ERR_CUDA, "cooperative launch: %s", cudaGetErrorString(r));
    // a device error of this step is reported by the engine's next synchronising call
    KIE_CUDA(e, kie_launch_err_merge(P.ctl, reinterpret_cast<KieControl*>(e->dev(e->lay.ctl)), e->stream));
    e->pos += 1;
    return KIE_OK;
}

}  // extern "C"
