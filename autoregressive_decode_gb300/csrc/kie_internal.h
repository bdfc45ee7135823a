// Internal structures shared by the host engine and the device program.
//
// The decode step is cut into phases; per layer:
//   QKV  RMSNorm + fused q/k/v GEMV + RoPE + K/V append      (weights streamed)
//   ATT  split-KV attention partials + per-head combine        (KV streamed)
//   O    O-projection GEMV + residual                           (weights streamed)
//   GU   RMSNorm + gate/up GEMV + SwiGLU                        (weights streamed)
//   D    down GEMV + residual                                   (weights streamed)
// and once per token LM (final RMSNorm + LM-head GEMV + argmax).
//
// Every GEMV phase partitions its output "units" (a row, or a pair of rows that
// one epilogue needs together: the RoPE pair (i, i+h/2) of q or k, or the
// matching gate/up rows) over the G CTAs of the grid.  Each CTA's weights for
// all phases of all layers are laid out as ONE contiguous byte stream in HBM,
// cut into slots of at most R rows x KC input columns; a producer warp copies
// the stream slot by slot into a shared-memory ring with bulk async copies and
// never waits for activations, so HBM streaming continues across grid barriers
// and non-GEMM work.
#pragma once
#include <stdint.h>

#ifndef KIE_NW
#define KIE_NW 7                 // consumer warps per CTA (with the producer: 2 warps per SM sub-partition, no register cap below 255)
#endif
#define KIE_THREADS ((KIE_NW + 1) * 32)
#define KIE_R 4                  // rows per slot
#ifndef KIE_KC_F16
#define KIE_KC_F16 2048          // input columns per slot, fp16 weights
#endif
#define KIE_KC_I4 (2 * KIE_KC_F16)  // input columns per slot, INT4 weights
#ifndef KIE_F16_UNROLL
#define KIE_F16_UNROLL 8         // unroll of the full-slot fp16 GEMV loop (KIE_KC_F16 / 256 iterations)
#endif
#ifndef KIE_I4_UNROLL
#define KIE_I4_UNROLL 2          // unroll of the full-slot INT4 GEMV loop (KIE_KC_I4 / 256 iterations); 4 and 8 measured slower
#endif
#ifndef KIE_F8_UNROLL
#define KIE_F8_UNROLL 1          // unroll of the full-slot FP8 GEMV loop (KIE_KC_F16 / 256 iterations); 2 and 4 measured slower
#endif
#ifndef KIE_SLOT_BYTES
#define KIE_SLOT_BYTES 16384     // slot capacity (KIE_R rows x KIE_KC_F16 fp16); 8 KB slots measured slower
#endif
#define KIE_MAX_SLOTS 16
// prefill GEMM output tile columns: 256 (one CTA per SM) or 128 (two CTAs per
// SM; measured slower, 1.8B 2,048-token prompt 25.0 vs 23.4 ms)
#ifndef KIE_PF_BN
#define KIE_PF_BN 256
#endif
#ifndef KIE_REPL
#define KIE_REPL 2               // copies of the activations x, a, o that CTAs exchange (readers poll copy cta % KIE_REPL)
#endif
#define KIE_MAX_BATCH 8          // requests of a batched engine (one tensor-core fragment holds 8 requests' hi and lo)
#define KIE_RB 16                // batched kernel: rows per slot (two 8-row MMA column groups)
#define KIE_KCB 512              // batched kernel: input columns per slot (16 rows x 512 fp16 = 16 KB)
#define KIE_KBLK 2048            // batched kernel: input columns staged at once (4 slots of a row tile)
#define KIE_SEG 128              // adaptive-range uint8 KV segment (tokens)
#define KIE_XRES 64              // residual rows per CTA whose old x is kept in shared memory
#define KIE_MAX_HEAD_DIM 128
#define KIE_MAX_GRID 256         // CTAs of the persistent grid (one per SM)
#define KIE_PROF_EVENTS 6        // trace stamps per (step, phase, CTA)
#define KIE_PROF_SLOTS 32768     // ring-slot trace entries (CTA 0)

#if defined(__CUDACC__)
#define KIE_HD __host__ __device__
#else
#define KIE_HD
#endif

// Dynamic shared-memory layout of the decode kernel; host (allocation size) and
// device (carving) both use this one function.  Offsets are relative to the
// dynamic shared-memory base; the ring starts on a 128-byte boundary.
struct KieSmemLayout {
    uint32_t full, empty, cbase, flags, plan, clist, rope, red, xres, wsc, cnt, part, act, ring, total;
};
KIE_HD inline uint32_t kie_align(uint32_t x, uint32_t a) { return (x + a - 1u) / a * a; }
// nb > 0 (the batched kernel): per-request cos/sin tables, norm partials,
// argmax partials and kept x rows for nb requests.
KIE_HD inline KieSmemLayout kie_smem_layout(int part_floats, int act_floats, int nslot, int nb = 0) {
    KieSmemLayout l;
    uint32_t o = 0;
    const uint32_t req = nb > 0 ? uint32_t(nb) : 1u;
    l.full = o;  o += KIE_MAX_SLOTS * 2 * 8;   // two per slot: even / odd generations
    l.empty = o; o += KIE_MAX_SLOTS * 8;
    l.cbase = o; o += 16;
    l.flags = o; o += 64;
    l.plan = o;  o += 5 * 4 * 4;
    l.clist = o; o += KIE_MAX_GRID * 4;
    l.rope = o;  o += req * KIE_MAX_HEAD_DIM * 4;     // cos/sin of the step's position, [req][2][hd/2]
    l.red = o;   o += (KIE_NW * (KIE_MAX_HEAD_DIM + 2) + 64 + (nb > 0 ? 3 * KIE_MAX_BATCH * KIE_NW : 0)) * 4;
    l.xres = o;  o += req * KIE_XRES * 4;
    // FP8 row scales of the phase (part_floats >= rows); batched: the staged block's RMSNorm gains
    l.wsc = nb > 0 ? kie_align(o, 16) : o;
    o = l.wsc + (nb > 0 ? uint32_t(KIE_KBLK) * 4 : uint32_t(part_floats) * 4);
    l.cnt = o;   o += nb > 0 ? 0u : (uint32_t(part_floats) / KIE_R + 4) * 4;   // per row group: chunks done (>= groups)
    l.part = o;  o += uint32_t(part_floats) * 4;
    l.act = kie_align(o, 16); o = l.act + uint32_t(act_floats) * 4;
    l.ring = kie_align(o, 128);
    l.total = l.ring + uint32_t(nslot) * KIE_SLOT_BYTES;
    return l;
}

enum KiePhaseType { PH_QKV = 0, PH_O = 1, PH_GU = 2, PH_D = 3, PH_LM = 4, PH_NTYPES = 5 };
enum KieWFmt { WF_F16 = 0, WF_I4 = 1, WF_F8 = 2, WF_F4 = 3 };
#define KIE_R8 8                 // rows per FP8 slot (8 rows x KIE_KC_F16 one-byte weights)
#ifndef KIE_R4
#define KIE_R4 8                 // rows per NVFP4 slot (8 rows x KIE_KC_F16 half-byte codes + block scales: 9 KB);
#endif                           // measured 1.8B NVFP4: 4 rows 985, 8 rows 1022, 14 rows 915 tok/s
enum KieKv { KV_F16 = 0, KV_E5M2 = 1, KV_U8 = 2, KV_E5M2S = 3 };
#define KIE_KV_SLICE 256         // scaled E5M2 cache: positions sharing one scale (per layer, K or V)
#define KIE_KV_SCALE_TARGET 127.0f   // a new slice's scale maps the previous slice's largest magnitude here

enum KieErr {
    KERR_NONE = 0,
    KERR_TIMEOUT_GRID = 1,    // grid barrier wait expired
    KERR_TIMEOUT_FULL = 2,    // consumer wait for a weight slot expired
    KERR_TIMEOUT_EMPTY = 3,   // producer wait for a free slot expired
    KERR_BAD_TOKEN = 4,       // input token id out of range
    KERR_SMEM = 5,            // launched with less dynamic shared memory than the layout needs
    KERR_TIMEOUT_PROGRESS = 6, // producer wait for the consumers' progress expired
    KERR_TIMEOUT_DATA = 7     // wait for another CTA's tagged activations expired
};

// Partition of one GEMV phase type over the grid (identical for every layer).
struct KiePhasePlan {
    int32_t K;               // input columns
    int32_t KC;              // columns per slot
    int32_t nK;              // chunks per row = ceil(K / KC)
    int32_t rows_per_unit;   // 1 or 2
    int32_t wfmt;            // KieWFmt
    int32_t R;               // rows per slot: KIE_R, KIE_R8 for FP8, KIE_R4 for NVFP4, KIE_RB batched
    int32_t cpb;             // chunks per staging block (batched: KIE_KBLK / KIE_KCB; single: nK)
    int32_t n_units;         // units over the grid
    const float* wscale;     // FP8 / NVFP4: fp32 row scales of layer 0 in the phase's row order (null otherwise)
    int64_t wscale_layer;    // FP8 / NVFP4: floats between consecutive layers' scales
    const int32_t* unit_begin;   // [G+1] device: CTA i owns units [unit_begin[i], unit_begin[i+1])
    const uint32_t* bytes;       // [G]   device: stream bytes of this phase for CTA i
    const uint32_t* nslots;      // [G]   device: slots of this phase for CTA i
};

struct KieControl {
    int32_t tok;             // input token of the next step
    int32_t pos;             // its position
    uint32_t bar;            // grid barrier counter (zeroed before each persistent launch)
    int32_t err;             // KieErr of the first failure
    int32_t err_info;        // CTA or phase of the first failure
    uint32_t amax_cnt;       // arrivals at the LM argmax reduction
    int32_t pad[2];
};

struct KieParams {
    // model
    int32_t L, d, H, hd, F, V, max_ctx, G;
    float eps, attn_scale;
    int32_t kv;              // KieKv
    int32_t nseg;            // segments per (layer, kv, head) for uint8 caches
    // weights
    const uint8_t* wstream;
    const uint64_t* cta_base;    // [G] byte offset of CTA i's stream
    const uint64_t* cta_layer;   // [G] bytes of one layer of CTA i's stream
    KiePhasePlan ph[PH_NTYPES];
    const uint16_t* emb;         // [V][d] fp16
    const float* norms;          // [L][2][d] then final [d], fp32
    const float* inv_freq;       // [hd/2] fp32
    // KV cache: [L][H][max_ctx][hd] of 2 (fp16) or 1 (E5M2, u8 codes) bytes
    uint8_t* kc;
    uint8_t* vc;
    uint16_t* tail;              // u8: [L][2][H][SEG][hd] fp16, the open segment
    float* seg_scale;            // u8: [L][2][H][nseg]
    int32_t* seg_zp;             // u8: [L][2][H][nseg]
    float* kv_sc;                // scaled E5M2: [L][2][nslice] scale of each slice (slice 0 set by the host)
    uint32_t* kv_mx;             // scaled E5M2: [L][2][nslice] largest stored magnitude (fp32 bits), by red.max
    int32_t nslice;
    // Activations passed between CTAs inside a step carry their own validity
    // tag, so no grid barrier separates the phases of a layer: fp32 vectors
    // hold a parity bit in the least significant mantissa bit; the current
    // position's K and V hold (storage bits << 16 | 16-bit epoch).  The host
    // resets x, kcur, vcur (to zero) and q, a, o, att_part (to one parity)
    // before every launch sequence.
    float* x;                    // [KIE_REPL][d] residual stream
    uint32_t* kcur;              // [H*hd] K of the current position, as stored, tagged
    uint32_t* vcur;              // [H*hd] V of the current position, as stored, tagged
    float* q;                    // [H*hd] rotated query
    float* a;                    // [KIE_REPL][F] SwiGLU output
    float* o;                    // [KIE_REPL][H*hd] attention output
    float* att_part;             // [G][hd+4] per-CTA attention partial: m, l, -, -, o[hd]
    float* amax_val;             // [G]
    int32_t* amax_idx;           // [G]
    KieControl* ctl;
    // batched kernel (kie_decode_batch.cu); the single-request kernel has nb == 0.
    // Activations gain a request index after their copy index: x [KIE_REPL][nb][d],
    // kcur, vcur, q [nb][H*hd], a [KIE_REPL][nb][F], o [KIE_REPL][nb][H*hd],
    // amax_val/idx [nb][G]; the KV cache of request b starts kv_req elements
    // after request b-1's.
    int32_t nb;
    int64_t kv_req;
    int32_t* req_tok;            // [nb] input token of each request's next step
    int32_t* req_pos;            // [nb] its position
    // shared-memory layout
    int32_t nslot;               // ring slots
    int32_t act_floats;          // activation buffer (floats)
    int32_t part_floats;         // GEMV partial buffer (floats)
};

struct KieLaunch {
    int32_t n_steps;             // tokens processed by this launch
    int32_t phase_begin;         // phases [phase_begin, phase_end) of each step (5L+1 per step)
    int32_t phase_end;
    int32_t first_tok;           // >= 0: input token of step 0; < 0: read ctl->tok
    int32_t pos0;                // >= 0: position of step 0; < 0: read ctl->pos
    const int32_t* forced;       // device [n_steps] input tokens (prefill), or null
    int32_t lm_from_step;        // LM head only for steps >= this
    int32_t* out_tokens;         // device [n_steps] (batched: [n_steps][nb]) or null
    float* out_logits;           // device [n_steps - lm_from_step][V] (batched: [..][nb][V]) or null
    uint64_t timeout_ns;
    int32_t use_grid_barrier;    // 1 in the persistent (cooperative) launch
    int32_t skip_arrival_cta;    // failure injection: this CTA skips its arrival at the first grid barrier (-1: none)
    // Optional trace: %globaltimer stamps [n_steps][5L+1][KIE_PROF_EVENTS][G]:
    // 0 phase start (after the grid barrier), 1 activation staged, 2 GEMV /
    // attention done, 3 epilogue done, 4 producer issued the phase's first slot
    // (attention: q arrived), 5 producer issued its last slot (attention: warp 0
    // done with its ring slots).  Null: no tracing.
    uint64_t* prof;
    // Optional ring trace of CTA 0: [KIE_PROF_SLOTS][4] stamps per slot index of
    // the launch: 0 copy issued, 1 data seen by the consumer warp, 2 released.
    uint64_t* prof_slots;
};
