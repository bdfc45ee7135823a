// Device building blocks of the decode program, shared by the single-request
// kernel (kie_decode.cu) and the batched kernel (kie_decode_batch.cu): the
// shared-memory carve-up, the weight ring and its producer warp, tagged
// activations, the GEMV slot routines and epilogues, split-KV attention and
// the grid barrier.  Everything is in an anonymous namespace: each
// translation unit that includes this file gets its own copy.
#pragma once
#include <cfloat>

#include "kie_device.cuh"
#include "kie_internal.h"

using namespace kie;

namespace {

constexpr int NW = KIE_NW;
constexpr int NCT = NW * 32;  // consumer threads

// Ring protocol.  Global slot index g lives in ring slot s = g % nslot as
// generation q = g / nslot.  "full" barriers are doubled per slot: generation q
// completes on full[2*s + (q & 1)] as that barrier's phase q/2, so a consumer
// waiting for generation q can only meet that barrier in phase q/2 (data in
// flight) or q/2 + 1 (data landed): generation q-2 was released before q-1 was
// issued, and q+2 cannot be issued before this consumer releases q.  With a
// single barrier per slot a consumer could arrive while generation q-1 is still
// in flight, and the parity of q would then name an already completed phase.
// Slot j of a phase goes to consumer warp j % NW, and every phase starts after
// a consumer-wide barrier, so all slots of earlier phases have landed.  The
// claim about q-2 then holds when nslot >= NW: for j < NW, g - 2*nslot lies in
// an earlier phase; for j >= NW the warp's previous slot g - NW landed, so every
// index <= g - NW was issued and every index <= g - NW - nslot was released
// (landed), g - 2*nslot among them.  Attention's last partial round is shared
// by all warps: before such a slot g a warp has waited for g - 1 (an earlier
// shared slot) or for its own last slot, at most NW before g; either way
// g - nslot was issued, so g - 2*nslot was released.
// "empty[s]" completes once per release (NW arrivals: the slot's warp arrives
// with count NW, each warp of a shared slot with 1), in generation order (the
// producer re-arms a slot only after its release), so one barrier suffices.
struct Smem {
    uint64_t* full;
    uint64_t* empty;
    int32_t* flags;   // [0]: abort, [1]: last-arriver flag, [2]: token, [3]: contributor count,
                      // [4]: consumers' progress (index of the phase they started, within the launch)
    int32_t* plan;    // [PH_NTYPES][4]: first unit, units, slots, stream bytes of this CTA
    uint64_t* cbase;  // [0]: this CTA's stream offset, [1]: bytes of one layer of it
    int32_t* clist;   // attention: contributors (2*cta + segment) of the head being combined
    float* rope;      // [2][hd/2] cos, sin of the current step's position
    float* red;       // reduction scratch: NW*(KIE_MAX_HEAD_DIM+2) + 64 floats
    float* xres;      // [KIE_XRES] old x of the rows the next residual epilogue updates
    float* wsc;       // FP8 phases: the row scales of this CTA's rows
    int32_t* cnt;     // GEMV phases with several column chunks: chunks done per row group
    float* part;      // GEMV partial sums
    float* act;       // activation (piece-split layout) / attention scores
    uint8_t* ring;
};

template <bool BAT = false>
__device__ __forceinline__ Smem carve(uint8_t* base, const KieParams& P) {
    const KieSmemLayout l = kie_smem_layout(P.part_floats, P.act_floats, P.nslot, BAT ? P.nb : 0);
    Smem s;
    s.full = reinterpret_cast<uint64_t*>(base + l.full);
    s.empty = reinterpret_cast<uint64_t*>(base + l.empty);
    s.cbase = reinterpret_cast<uint64_t*>(base + l.cbase);
    s.flags = reinterpret_cast<int32_t*>(base + l.flags);
    s.plan = reinterpret_cast<int32_t*>(base + l.plan);
    s.clist = reinterpret_cast<int32_t*>(base + l.clist);
    s.rope = reinterpret_cast<float*>(base + l.rope);
    s.red = reinterpret_cast<float*>(base + l.red);
    s.xres = reinterpret_cast<float*>(base + l.xres);
    s.wsc = reinterpret_cast<float*>(base + l.wsc);
    s.cnt = reinterpret_cast<int32_t*>(base + l.cnt);
    s.part = reinterpret_cast<float*>(base + l.part);
    s.act = reinterpret_cast<float*>(base + l.act);
    s.ring = base + l.ring;
    return s;
}

__device__ __forceinline__ uint32_t dynamic_smem_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
    return r;
}

// Index of element k in the piece-split activation layout: pieces of 8
// elements, first 4 of each piece in the low plane, last 4 in the high plane,
// so that a lane reading "its" piece loads two conflict-free float4s.
__device__ __forceinline__ int act_idx(int k, int half) {
    return ((k & 4) ? half : 0) + (k >> 3) * 4 + (k & 3);
}

struct Cursor {  // geometry of one GEMV phase for this CTA
    int K, KC, nK, rpu, wfmt, R;
    int unit0, n_units, rows;
    uint32_t nslots;
};

__device__ __forceinline__ Cursor cursor(const KieParams& P, const Smem& S, int type) {
    const KiePhasePlan& pp = P.ph[type];
    Cursor c;
    c.K = pp.K; c.KC = pp.KC; c.nK = pp.nK; c.rpu = pp.rows_per_unit; c.wfmt = pp.wfmt; c.R = pp.R;
    c.unit0 = S.plan[type * 4 + 0];
    c.n_units = S.plan[type * 4 + 1];
    c.rows = c.n_units * c.rpu;
    c.nslots = uint32_t(S.plan[type * 4 + 2]);
    return c;
}

__device__ __forceinline__ uint32_t slot_bytes(int wfmt, int rows_g, int kc) {
    if (wfmt == WF_F16) return uint32_t(rows_g) * uint32_t(kc) * 2u;
    if (wfmt == WF_F8) return (uint32_t(rows_g) * uint32_t(kc) + 15u) & ~15u;
    if (wfmt == WF_F4) return (uint32_t(rows_g) * uint32_t(kc / 2 + kc / 16) + 15u) & ~15u;
    uint32_t b = uint32_t(rows_g) * uint32_t(kc / 2) + uint32_t(rows_g) * uint32_t(kc / 64);
    return (b + 15u) & ~15u;
}

__device__ __forceinline__ void slot_geom(const Cursor& c, uint32_t j, int& g, int& ch, int& rows_g, int& kc) {
    g = int(j / uint32_t(c.nK));
    ch = int(j % uint32_t(c.nK));
    rows_g = min(c.R, c.rows - g * c.R);
    kc = min(c.KC, c.K - ch * c.KC);
}

// phase index within a step -> (layer, sub); sub: 0 QKV, 1 ATT, 2 O, 3 GU, 4 D, 5 LM
__device__ __forceinline__ void phase_of(int phi, int L, int& layer, int& sub) {
    if (phi >= 5 * L) { layer = L; sub = 5; }
    else { layer = phi / 5; sub = phi % 5; }
}
__device__ __forceinline__ int gemv_type(int sub) {
    return sub == 0 ? PH_QKV : sub == 2 ? PH_O : sub == 3 ? PH_GU : sub == 4 ? PH_D : sub == 5 ? PH_LM : -1;
}
__device__ __forceinline__ uint64_t stream_offset(const KieParams& P, const Smem& S, int layer, int type) {
    uint64_t off = S.cbase[0];
    if (type == PH_LM) return off + uint64_t(P.L) * S.cbase[1];
    off += uint64_t(layer) * S.cbase[1];
    for (int t = 0; t < type; ++t) off += uint32_t(S.plan[t * 4 + 3]);
    return off;
}

__device__ __forceinline__ void slot_stamp(const KieLaunch& Lc, int cta, uint32_t g, int ev) {
    if (Lc.prof_slots && cta == 0 && g < KIE_PROF_SLOTS) Lc.prof_slots[size_t(g) * 4 + ev] = globaltimer_stamp();
}

__device__ __forceinline__ void stamp(const KieParams& P, const KieLaunch& Lc, int t, int phi, int ev, int cta) {
    if (Lc.prof) {
        const size_t nph = size_t(5 * P.L + 1);
        Lc.prof[((size_t(t) * nph + phi) * KIE_PROF_EVENTS + ev) * P.G + cta] = globaltimer_stamp();
    }
}

__device__ void set_error(const KieParams& P, int code, int info) {
    if (atomicCAS(&P.ctl->err, 0, code) == 0) P.ctl->err_info = info;
}

// ---------------------------------------------------------------------------------------------
// tagged activations
// ---------------------------------------------------------------------------------------------
// Inside a step no grid barrier separates the phases.  Every activation that
// one CTA writes and others read carries a tag of the write that produced it,
// and a reader polls until the tag it expects is there.  Writes are numbered
// by n = pos * L + layer, the same in every launch mode:
//  * q, a and o (fp32, written once per layer): the parity of n + 1 in the
//    least significant mantissa bit (a relative change of at most 2^-23,
//    applied identically in every mode);
//  * x (fp32): parity 1 after an O epilogue, 0 after a D epilogue;
//  * K and V of the current position: (storage bits << 16) | (n mod 65535) + 1.
// Before every launch sequence the host sets x, K, V to tag 0 and q, a, o to
// the parity opposite to the first write's, so the initial state never
// matches.  One parity bit suffices because every reader of a write has read
// the write before it at the same address (read-read coherence: what it sees
// is that write or the one it waits for): every CTA stages all of x after each
// epilogue that writes it, and reads its head's q and the whole of a and o
// every layer.  No write can overtake a pending read: the next write of a
// buffer needs the layer's whole data flow, which needs every reader of the
// current value to be past it.
__device__ __forceinline__ uint32_t tag_seq(const KieParams& P, int pos, int layer) {
    return uint32_t(pos) * uint32_t(P.L) + uint32_t(layer);
}
__device__ __forceinline__ uint32_t tag_par(uint32_t n) { return (n + 1u) & 1u; }
__device__ __forceinline__ uint32_t tag_ep16(uint32_t n) { return n % 65535u + 1u; }
__device__ __forceinline__ float tag_f32(float v, uint32_t par) {
    return __uint_as_float((__float_as_uint(v) & ~1u) | par);
}
__device__ __forceinline__ bool has_tag4(const float4& v, uint32_t par) {
    return (((__float_as_uint(v.x) ^ par) | (__float_as_uint(v.y) ^ par) | (__float_as_uint(v.z) ^ par) |
             (__float_as_uint(v.w) ^ par)) & 1u) == 0u;
}
__device__ __forceinline__ bool has_ep4(const uint4& v, uint32_t ep16) {
    return ((v.x & 0xFFFFu) == ep16) & ((v.y & 0xFFFFu) == ep16) & ((v.z & 0xFFFFu) == ep16) & ((v.w & 0xFFFFu) == ep16);
}

// Bounded poll of one thread: false once the launch's timeout has passed
// (recorded as KERR_TIMEOUT_DATA) or another thread or CTA has failed.
struct TagWait {
    uint64_t t0;
    uint32_t spins;
    __device__ TagWait() : t0(globaltimer()), spins(0) {}
    __device__ __forceinline__ bool again(const KieParams& P, const KieLaunch& Lc, const Smem& S, int cta) {
        if ((++spins & 15u) != 0u) return true;
        if (ld_volatile_i32(&S.flags[0]) != 0 || ld_volatile_i32(&P.ctl->err) != 0) return false;
        if (globaltimer() - t0 > Lc.timeout_ns) {
            set_error(P, KERR_TIMEOUT_DATA, cta);
            S.flags[0] = 1;
            return false;
        }
        return true;
    }
};

// One tagged fp32 element (scalar poll).
__device__ __forceinline__ float wait_f32(const KieParams& P, const KieLaunch& Lc, const Smem& S, const float* p,
                                          uint32_t par, int cta) {
    float v = ld_relaxed_f32(p);
    if (((__float_as_uint(v) ^ par) & 1u) == 0u) return v;
    TagWait w;
    do {
        v = ld_relaxed_f32(p);
        if (((__float_as_uint(v) ^ par) & 1u) == 0u) break;
    } while (w.again(P, Lc, S, cta));
    return v;
}
// One tagged K/V word of the current position; returns its storage bits.
__device__ __forceinline__ uint32_t wait_cur(const KieParams& P, const KieLaunch& Lc, const Smem& S,
                                             const uint32_t* p, uint32_t ep16, int cta) {
    uint32_t v = ld_relaxed_u32(p);
    if ((v & 0xFFFFu) != ep16) {
        TagWait w;
        do {
            v = ld_relaxed_u32(p);
            if ((v & 0xFFFFu) == ep16) break;
        } while (w.again(P, Lc, S, cta));
    }
    return v >> 16;
}

// ---------------------------------------------------------------------------------------------
// KV cache access
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ size_t kv_elem_index(const KieParams& P, int layer, int h, int pos) {
    return ((size_t(layer) * P.H + h) * P.max_ctx + pos) * P.hd;
}
__device__ __forceinline__ size_t tail_index(const KieParams& P, int layer, int kv, int h, int slot) {
    return (((size_t(layer) * 2 + kv) * P.H + h) * KIE_SEG + slot) * P.hd;
}
__device__ __forceinline__ size_t meta_index(const KieParams& P, int layer, int kv, int h, int seg) {
    return ((size_t(layer) * 2 + kv) * P.H + h) * P.nseg + seg;
}

// Attention work: head h owns CTAs [c0(h), c0(h+1)) with c0(h) = floor(h*G/H);
// CTA k of them takes positions [floor(k*C/n_h), floor((k+1)*C/n_h)) of the C
// attended ones.  Rows [j0, jt) were written in earlier steps and reach shared
// memory through the weight ring, K and V of the same rows in one slot; rows
// [jt, j1) (the current position, and for a uint8 cache the open segment kept
// in fp16) are read directly.
struct AttChunk {
    int h, c0, nh, j0, j1, jt;
    int b, pos;   // batched kernel: the request and its position (single kernel: 0 and the step's position)
};
__device__ __forceinline__ AttChunk att_chunk(const KieParams& P, int cta, int pos) {
    AttChunk a;
    const uint32_t H = uint32_t(P.H), G = uint32_t(P.G), C = uint32_t(pos) + 1u;
    a.h = int(((uint32_t(cta) + 1u) * H - 1u) / G);
    a.c0 = int(uint32_t(a.h) * G / H);
    a.nh = int((uint32_t(a.h) + 1u) * G / H) - a.c0;
    const uint32_t k = uint32_t(cta - a.c0);
    a.j0 = int(k * C / uint32_t(a.nh));
    a.j1 = int((k + 1u) * C / uint32_t(a.nh));
    const int tma_end = (P.kv == KV_U8) ? (pos / KIE_SEG) * KIE_SEG : pos;
    a.jt = max(a.j0, min(a.j1, tma_end));
    a.b = 0;
    a.pos = pos;
    return a;
}
// Batched kernel: the nb * H (request, head) pairs take the CTAs the way heads
// do above (pair p = b * H + h owns [floor(p G / np), floor((p+1) G / np)),
// np = nb * H <= G), each pair over its own request's positions; request b's
// position at step t is S.flags[8 + b] + t.
__device__ __forceinline__ AttChunk att_chunk_b(const KieParams& P, const int32_t* pos0, int cta, int t) {
    AttChunk a;
    const uint32_t np = uint32_t(P.nb * P.H), G = uint32_t(P.G);
    const int p = int(((uint32_t(cta) + 1u) * np - 1u) / G);
    a.c0 = int(uint32_t(p) * G / np);
    a.nh = int((uint32_t(p) + 1u) * G / np) - a.c0;
    a.b = p / P.H;
    a.h = p - a.b * P.H;
    a.pos = pos0[a.b] + t;
    const uint32_t C = uint32_t(a.pos) + 1u, k = uint32_t(cta - a.c0);
    a.j0 = int(k * C / uint32_t(a.nh));
    a.j1 = int((k + 1u) * C / uint32_t(a.nh));
    a.jt = max(a.j0, min(a.j1, a.pos));
    return a;
}
__device__ __forceinline__ int att_row_bytes(const KieParams& P) { return P.hd * (P.kv == KV_F16 ? 2 : 1); }
// Rows per slot (its K rows, then the same rows of V at offset rows * row bytes):
// a chunk that fits one slot per consumer warp is spread over them (at least 8
// rows a slot); a longer one uses full slots (half a slot of K, half of V),
// whole rounds of them one per warp and the last partial round shared by all.
__device__ __forceinline__ int att_rows_per_slot(const KieParams& P, const AttChunk& a) {
    const int full = KIE_SLOT_BYTES / (2 * att_row_bytes(P));
    const int nt = a.jt - a.j0;
    if (nt > NW * full) return full;
    return min(full, max(8, (nt + NW - 1) / NW));
}
__device__ __forceinline__ uint32_t att_nslots(const KieParams& P, const AttChunk& a) {
    const int rps = att_rows_per_slot(P, a);
    return uint32_t((a.jt - a.j0 + rps - 1) / rps);
}

// Producer: wait until ring slot `slot` was released by its previous user
// (the phase of parity `par` of its "empty" barrier).
__device__ __forceinline__ bool producer_wait_slot(const KieParams& P, const KieLaunch& Lc, const Smem& S,
                                                   uint32_t slot, uint32_t par, int cta) {
    if (mbar_test_wait(&S.empty[slot], par)) return true;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&S.empty[slot], par)) {
        if (ld_volatile_i32(&S.flags[0]) != 0 || ld_volatile_i32(&P.ctl->err) != 0) return false;
        if (globaltimer() - t0 > Lc.timeout_ns) {
            set_error(P, KERR_TIMEOUT_EMPTY, cta);
            return false;
        }
    }
    return true;
}

// Consumer warp: wait until global slot gidx has landed.  Every lane probes the
// barrier (each lane needs the acquire of the bulk-copy data) but the decision
// to continue or abort is warp-uniform, so no lane can leave the slot loop while
// others go on to the warp's shuffles.
__device__ __forceinline__ bool warp_wait_full(const KieParams& P, const KieLaunch& Lc, const Smem& S,
                                               uint32_t gidx, int cta, int lane) {
    const uint32_t nslot = uint32_t(P.nslot);
    const uint32_t slot = gidx % nslot, q = gidx / nslot;
    uint64_t* fb = &S.full[2 * slot + (q & 1u)];
    const uint32_t par = (q >> 1) & 1u;
    const uint64_t t0 = globaltimer();
    while (true) {
        const bool done = mbar_try_wait(fb, par);
        if (__all_sync(0xffffffffu, done)) return true;
        int bad = 0;
        if (lane == 0) {
            if (ld_volatile_i32(&S.flags[0]) != 0 || ld_volatile_i32(&P.ctl->err) != 0) bad = 1;
            else if (globaltimer() - t0 > Lc.timeout_ns) { set_error(P, KERR_TIMEOUT_FULL, cta); bad = 1; }
        }
        if (__shfl_sync(0xffffffffu, bad, 0)) return false;
    }
}

// ---------------------------------------------------------------------------------------------
// producer warp: stream every slot of this CTA, in consumption order, into the ring
// ---------------------------------------------------------------------------------------------
// BAT (the batched kernel): attention copies its (request, head) pair's rows
// from that request's cache, GEMV slots go in staging-block order (block,
// row tile, chunk), and every issue is published in S.flags[5] (slots issued so
// far in the launch) for the consumers' gate.
template <bool BAT>
__device__ void producer(const KieParams& P, const KieLaunch& Lc, const Smem& S, int cta) {
    const uint64_t pol = policy_evict_first();
    const uint32_t nslot = uint32_t(P.nslot);
    uint32_t g = 0, rs = 0, rq = 0;   // global slot index, its ring slot and generation
    bool abort = false;
    const uint64_t pol_kv = policy_evict_first();
    const int pos0 = Lc.pos0 >= 0 ? Lc.pos0 : ld_volatile_i32(&P.ctl->pos);
    for (int t = 0; t < Lc.n_steps && !abort; ++t) {
        for (int phi = Lc.phase_begin; phi < Lc.phase_end && !abort; ++phi) {
            int layer, sub;
            phase_of(phi, P.L, layer, sub);
            const int type = gemv_type(sub);
            if (sub == 1) {
                // attention: this CTA's K rows then V rows written in earlier steps.
                // Rows up to pos-1 were written by step t-1 (K/V at its QKV phase,
                // uint8 codes of a completed segment during its attention), so the
                // copies may start only once this block's consumers have started
                // step t, i.e. passed the grid barrier that publishes those writes.
                // With a ring much smaller than one step's stream this never
                // waits; it bounds the run-ahead of deep rings.
                if (t >= 1) {
                    const int32_t need = t * (Lc.phase_end - Lc.phase_begin);
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire_cta_shared(&S.flags[4]) < need) {
                        if (ld_volatile_i32(&S.flags[0]) != 0 || ld_volatile_i32(&P.ctl->err) != 0) { abort = true; break; }
                        if (globaltimer() - t0 > Lc.timeout_ns) { set_error(P, KERR_TIMEOUT_PROGRESS, cta); abort = true; break; }
                        __nanosleep(64);
                    }
                    if (abort) break;
                    fence_proxy_async_global();
                }
                const int pos = pos0 + t;
                const AttChunk a = BAT ? att_chunk_b(P, S.flags + 8, cta, t) : att_chunk(P, cta, pos);
                const uint32_t nsl = att_nslots(P, a);
                const int rps = att_rows_per_slot(P, a), rb = att_row_bytes(P);
                for (uint32_t j = 0; j < nsl && !abort; ++j, ++g) {
                    const uint32_t slot = rs;
                    if (g >= nslot && !producer_wait_slot(P, Lc, S, rs, (rq - 1u) & 1u, cta)) { abort = true; break; }
                    const int r0 = int(j) * rps;
                    const int rows = min(rps, a.jt - a.j0 - r0);
                    size_t el = kv_elem_index(P, layer, a.h, a.j0 + r0);
                    if (BAT) el += size_t(a.b) * size_t(P.kv_req);
                    const size_t off = el * size_t(rb / P.hd);
                    const uint32_t bytes = uint32_t(rows * rb);
                    uint64_t* fb = &S.full[2 * slot + (rq & 1u)];
                    uint8_t* dst = S.ring + size_t(slot) * KIE_SLOT_BYTES;
                    mbar_arrive_expect_tx(fb, 2u * bytes);
                    bulk_g2s(dst, P.kc + off, bytes, fb, pol_kv);
                    bulk_g2s(dst + size_t(rps) * rb, P.vc + off, bytes, fb, pol_kv);
                    slot_stamp(Lc, cta, g, 0);
                    if (BAT) st_release_cta_shared(&S.flags[5], int32_t(g + 1u));
                    if (++rs == nslot) { rs = 0; ++rq; }
                }
                continue;
            }
            if (type < 0) continue;
            if (type == PH_LM && t < Lc.lm_from_step) continue;
            const Cursor c = cursor(P, S, type);
            const uint8_t* src = P.wstream + stream_offset(P, S, layer, type);
            if (BAT) {   // fp16 slots of KIE_RB rows, in the order (staging block, row tile, chunk)
                const int nblk = (c.K + KIE_KBLK - 1) / KIE_KBLK;
                uint32_t j = 0;
                for (int blk = 0; blk < nblk && !abort; ++blk) {
                    const int kb = min(KIE_KBLK, c.K - blk * KIE_KBLK);
                    const int nch = (kb + c.KC - 1) / c.KC;
                    for (int gg = 0; gg * c.R < c.rows && !abort; ++gg) {
                        const int rows_g = min(c.R, c.rows - gg * c.R);
                        for (int ch = 0; ch < nch; ++ch, ++j) {
                            if (g >= nslot && !producer_wait_slot(P, Lc, S, rs, (rq - 1u) & 1u, cta)) { abort = true; break; }
                            const uint32_t bytes = uint32_t(rows_g) * uint32_t(min(c.KC, kb - ch * c.KC)) * 2u;
                            uint64_t* fb = &S.full[2 * rs + (rq & 1u)];
                            mbar_arrive_expect_tx(fb, bytes);
                            bulk_g2s(S.ring + size_t(rs) * KIE_SLOT_BYTES, src, bytes, fb, pol);
                            slot_stamp(Lc, cta, g, 0);
                            src += bytes;
                            if (j == 0) stamp(P, Lc, t, phi, 4, cta);
                            if (j + 1 == c.nslots) stamp(P, Lc, t, phi, 5, cta);
                            ++g;
                            st_release_cta_shared(&S.flags[5], int32_t(g));
                            if (++rs == nslot) { rs = 0; ++rq; }
                        }
                    }
                }
                continue;
            }
            // slots j = group * nK + chunk, walked without divisions; the ring
            // position (rs, rq) = (g % nslot, g / nslot) is kept incrementally
            const uint32_t j_end = c.nslots;
            uint32_t j = 0;
            for (int gg = 0; j < j_end && !abort; ++gg) {
                const int rows_g = min(c.R, c.rows - gg * c.R);
                for (int ch = 0; ch < c.nK; ++ch, ++j) {
                    if (g >= nslot && !producer_wait_slot(P, Lc, S, rs, (rq - 1u) & 1u, cta)) { abort = true; break; }
                    const int kc = min(c.KC, c.K - ch * c.KC);
                    const uint32_t bytes = slot_bytes(c.wfmt, rows_g, kc);
                    uint64_t* fb = &S.full[2 * rs + (rq & 1u)];
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s(S.ring + size_t(rs) * KIE_SLOT_BYTES, src, bytes, fb, pol);
                    slot_stamp(Lc, cta, g, 0);
                    src += bytes;
                    if (j == 0) stamp(P, Lc, t, phi, 4, cta);
                    if (j + 1 == j_end) stamp(P, Lc, t, phi, 5, cta);
                    ++g;
                    if (++rs == nslot) { rs = 0; ++rq; }
                }
            }
        }
    }
    // Wait until every copy issued into the ring has landed before the CTA may exit.
    const uint32_t issued = g;
    const uint32_t first = issued > nslot ? issued - nslot : 0u;
    for (uint32_t k = first; k < issued; ++k) {
        const uint32_t slot = k % nslot, q = k / nslot;
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(&S.full[2 * slot + (q & 1u)], (q >> 1) & 1u)) {
            if (globaltimer() - t0 > Lc.timeout_ns) { set_error(P, KERR_TIMEOUT_FULL, cta); break; }
        }
    }
}

// ---------------------------------------------------------------------------------------------
// consumer helpers
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float block_sum(float v, float* red, int tid) {
    v = warp_sum(v);
    if ((tid & 31) == 0) red[tid >> 5] = v;
    consumer_sync(NCT);
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += red[w];
    consumer_sync(NCT);
    return s;
}

__device__ __forceinline__ float block_max(float v, float* red, int tid) {
    v = warp_max(v);
    if ((tid & 31) == 0) red[tid >> 5] = v;
    consumer_sync(NCT);
    float m = red[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) m = fmaxf(m, red[w]);
    consumer_sync(NCT);
    return m;
}

// RMSNorm folded into the GEMV: act <- src * g, and each warp leaves its part of
// sum(src^2) in S.red[NORM_SLOT + warp]; the epilogue divides every output by
// sqrt(mean(src^2) + eps) (norm_r).  W (x g / r) = (W (x g)) / r, so no
// block-wide reduction sits between the barrier and the first slot.
// src = x (fp32, global) or an embedding row (fp16).
constexpr int NORM_SLOT = NW * (KIE_MAX_HEAD_DIM + 2) + 8;
// scaled E5M2 cache: the current position's K and V slice scales, set while the QKV phase stages
constexpr int KVS_SLOT = NW * (KIE_MAX_HEAD_DIM + 2) + 16;
// x is tagged with parity `par` (polled until every element carries it).  The
// raw values of elements [cap0, cap0 + ncap) (the rows this CTA's next residual
// epilogue updates) are also kept in S.xres.
__device__ void act_scaled(const KieParams& P, const KieLaunch& Lc, const Smem& S, const float* x,
                           const uint16_t* emb_row, const float* g, uint32_t par, int tid, int cta, int cap0,
                           int ncap) {
    const int d = P.d, half = P.act_floats / 2, ng = d >> 2;
    float ss = 0.f;
    for (int q0 = tid; q0 < ng; q0 += 4 * NCT) {
        float4 v[4], gg[4];
        uint32_t bad = 0;
        // the gains first: their loads do not depend on x, so their latency
        // passes while x is polled instead of after it has arrived
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (q0 + u * NCT < ng) gg[u] = __ldg(reinterpret_cast<const float4*>(g + 4 * (q0 + u * NCT)));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int q = q0 + u * NCT;
            if (q < ng) {
                if (x) {
                    v[u] = ld_relaxed_f4(x + 4 * q);
                    if (!has_tag4(v[u], par)) bad |= 1u << u;
                } else {
                    const uint2 hv = *reinterpret_cast<const uint2*>(emb_row + 4 * q);
                    const float2 a = h2_to_f2(hv.x), b = h2_to_f2(hv.y);
                    v[u] = make_float4(a.x, a.y, b.x, b.y);
                }
            }
        }
        if (bad) {
            TagWait w;
            do {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if ((bad >> u) & 1u) {
                        v[u] = ld_relaxed_f4(x + 4 * (q0 + u * NCT));
                        if (has_tag4(v[u], par)) bad &= ~(1u << u);
                    }
                }
            } while (bad && w.again(P, Lc, S, cta));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int q = q0 + u * NCT;
            if (q < ng) {
                ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
                const int k4 = 4 * q - cap0;
                if (k4 > -4 && k4 < ncap) {
                    const float vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (k4 + e >= 0 && k4 + e < ncap) S.xres[k4 + e] = vv[e];
                }
                // 4 consecutive elements share one plane of one 8-element piece
                *reinterpret_cast<float4*>(S.act + act_idx(4 * q, half)) =
                    make_float4(v[u].x * gg[u].x, v[u].y * gg[u].y, v[u].z * gg[u].z, v[u].w * gg[u].w);
            }
        }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) S.red[NORM_SLOT + (tid >> 5)] = ss;
    consumer_sync(NCT);
}

// sqrt(mean(src^2) + eps) of the phase's act_scaled input (after the phase's
// final consumer barrier).
__device__ __forceinline__ float norm_r(const KieParams& P, const Smem& S) {
    float ss = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) ss += S.red[NORM_SLOT + w];
    return sqrtf(ss / float(P.d) + P.eps);
}

// cos / sin of pos * inv_freq_i, i < hd/2, into S.rope (visible after the next
// consumer barrier).
__device__ __forceinline__ void rope_table(const KieParams& P, const Smem& S, int pos, int tid) {
    const int hh = P.hd / 2;
    if (tid < hh) {
        float sn, cs;
        sincosf(float(pos) * P.inv_freq[tid], &sn, &cs);
        S.rope[tid] = cs;
        S.rope[hh + tid] = sn;
    }
}

// src is tagged with parity `par` (polled until every element carries it).
__device__ void act_copy(const KieParams& P, const KieLaunch& Lc, const Smem& S, const float* src, int n,
                         uint32_t par, int tid, int cta) {
    const int half = P.act_floats / 2, ng = n >> 2;
    constexpr int U = 10;   // loads in flight per thread: 10 x 224 float4 cover an 8192-float vector in one poll round
    for (int q0 = tid; q0 < ng; q0 += U * NCT) {
        float4 v[U];
        uint32_t bad = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (q0 + u * NCT < ng) {
                v[u] = ld_relaxed_f4(src + 4 * (q0 + u * NCT));
                if (!has_tag4(v[u], par)) bad |= 1u << u;
            }
        }
        if (bad) {
            TagWait w;
            do {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if ((bad >> u) & 1u) {
                        v[u] = ld_relaxed_f4(src + 4 * (q0 + u * NCT));
                        if (has_tag4(v[u], par)) bad &= ~(1u << u);
                    }
                }
            } while (bad && w.again(P, Lc, S, cta));
        }
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (q0 + u * NCT < ng) *reinterpret_cast<float4*>(S.act + act_idx(4 * (q0 + u * NCT), half)) = v[u];
    }
    consumer_sync(NCT);
}

// The GEMV loops keep a float2 partial sum per row.  With KIE_FFMA2 they use
// the packed fp32 FMA (fma.rn.f32x2) on even and odd elements of each
// 8-element piece (half the FMA instructions, two chains per row, added once
// at the end of the slot); otherwise one fp32 chain per row in .x.
#ifndef KIE_FFMA2
#define KIE_FFMA2 1              // measured: fp16 1061 -> 1072, FP8 1122 -> 1151 tok/s on the 1.8B model
#endif
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// acc += w[0..7] * (xl, xh) for one 8-element piece; w as four fp16 pairs.
__device__ __forceinline__ float2 piece_f16(const uint4& w, const float4& xl, const float4& xh, float2 s) {
#if KIE_FFMA2
    s = ffma2(h2_to_f2(w.x), make_float2(xl.x, xl.y), s);
    s = ffma2(h2_to_f2(w.y), make_float2(xl.z, xl.w), s);
    s = ffma2(h2_to_f2(w.z), make_float2(xh.x, xh.y), s);
    s = ffma2(h2_to_f2(w.w), make_float2(xh.z, xh.w), s);
#else
    const float2 a = h2_to_f2(w.x), b = h2_to_f2(w.y), c = h2_to_f2(w.z), e = h2_to_f2(w.w);
    float t = s.x;
    t = fmaf(a.x, xl.x, t); t = fmaf(a.y, xl.y, t); t = fmaf(b.x, xl.z, t); t = fmaf(b.y, xl.w, t);
    t = fmaf(c.x, xh.x, t); t = fmaf(c.y, xh.y, t); t = fmaf(e.x, xh.z, t); t = fmaf(e.y, xh.w, t);
    s.x = t;
#endif
    return s;
}

// y-partials of one fp16 slot: rows_g rows x kc columns, row-major; columns start at k0.
__device__ __forceinline__ void slot_f16(const uint8_t* slot, int rows_g, int kc, int k0, const float* act,
                                         int half, int lane, float* acc) {
    const int npc = kc >> 3;
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
    float2 a2[KIE_R];
#pragma unroll
    for (int r = 0; r < KIE_R; ++r) a2[r] = make_float2(0.f, 0.f);
    for (int p = lane; p < npc; p += 32) {
        const float4 xl = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh = *reinterpret_cast<const float4*>(ahi + p * 4);
#pragma unroll
        for (int r = 0; r < KIE_R; ++r) {
            if (r < rows_g) {
                const uint4 w = *reinterpret_cast<const uint4*>(slot + size_t(r) * kc * 2 + size_t(p) * 16);
                a2[r] = piece_f16(w, xl, xh, a2[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < KIE_R; ++r) acc[r] = a2[r].x + a2[r].y;
}

// The common full slot (KIE_R rows x KIE_KC_F16 columns) with compile-time
// bounds, so the loads of all iterations can be in flight together.
__device__ __forceinline__ void slot_f16_full(const uint8_t* slot, int k0, const float* act, int half, int lane,
                                              float* acc) {
    constexpr int NPC = KIE_KC_F16 / 8;
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
    float2 a2[KIE_R];
#pragma unroll
    for (int r = 0; r < KIE_R; ++r) a2[r] = make_float2(0.f, 0.f);
    constexpr int kUnroll = KIE_F16_UNROLL;
#pragma unroll kUnroll
    for (int it = 0; it < NPC / 32; ++it) {
        const int p = lane + it * 32;
        const float4 xl = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh = *reinterpret_cast<const float4*>(ahi + p * 4);
#pragma unroll
        for (int r = 0; r < KIE_R; ++r) {
            const uint4 w = *reinterpret_cast<const uint4*>(slot + size_t(r) * KIE_KC_F16 * 2 + size_t(p) * 16);
            a2[r] = piece_f16(w, xl, xh, a2[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < KIE_R; ++r) acc[r] = a2[r].x + a2[r].y;
}

// acc += w[0..7] * (xl, xh) for one 8-element piece of FP8 E4M3 codes.
__device__ __forceinline__ float2 piece_f8(const uint2& w, const float4& xl, const float4& xh, float2 s) {
    float f[8];
    e4m3x4_to_f32(w.x, f);
    e4m3x4_to_f32(w.y, f + 4);
#if KIE_FFMA2
    s = ffma2(make_float2(f[0], f[1]), make_float2(xl.x, xl.y), s);
    s = ffma2(make_float2(f[2], f[3]), make_float2(xl.z, xl.w), s);
    s = ffma2(make_float2(f[4], f[5]), make_float2(xh.x, xh.y), s);
    s = ffma2(make_float2(f[6], f[7]), make_float2(xh.z, xh.w), s);
#else
    float t = s.x;
    t = fmaf(f[0], xl.x, t); t = fmaf(f[1], xl.y, t); t = fmaf(f[2], xl.z, t); t = fmaf(f[3], xl.w, t);
    t = fmaf(f[4], xh.x, t); t = fmaf(f[5], xh.y, t); t = fmaf(f[6], xh.z, t); t = fmaf(f[7], xh.w, t);
    s.x = t;
#endif
    return s;
}

// FP8 E4M3 slot: codes [rows_g][kc], row-major, up to KIE_R8 rows; the rows'
// scales are applied in row_sum.  Each lane takes 8-element pieces, as for fp16.
__device__ __forceinline__ void slot_f8(const uint8_t* slot, int rows_g, int kc, int k0, const float* act,
                                        int half, int lane, float* acc) {
    const int npc = kc >> 3;
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
    float2 a2[KIE_R8];
#pragma unroll
    for (int r = 0; r < KIE_R8; ++r) a2[r] = make_float2(0.f, 0.f);
#pragma unroll 2
    for (int p = lane; p < npc; p += 32) {
        const float4 xl = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh = *reinterpret_cast<const float4*>(ahi + p * 4);
#pragma unroll
        for (int r = 0; r < KIE_R8; ++r) {
            if (r < rows_g) {
                const uint2 w = *reinterpret_cast<const uint2*>(slot + size_t(r) * kc + size_t(p) * 8);
                a2[r] = piece_f8(w, xl, xh, a2[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < KIE_R8; ++r) acc[r] = a2[r].x + a2[r].y;
}

// The common full FP8 slot (KIE_R8 rows x KIE_KC_F16 columns) with compile-time
// bounds, so that the loads of consecutive pieces can be in flight together.
__device__ __forceinline__ void slot_f8_full(const uint8_t* slot, int k0, const float* act, int half, int lane,
                                             float* acc) {
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
    float2 a2[KIE_R8];
#pragma unroll
    for (int r = 0; r < KIE_R8; ++r) a2[r] = make_float2(0.f, 0.f);
    constexpr int kUnroll = KIE_F8_UNROLL;
#pragma unroll kUnroll
    for (int it = 0; it < KIE_KC_F16 / 256; ++it) {
        const int p = lane + it * 32;
        const float4 xl = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh = *reinterpret_cast<const float4*>(ahi + p * 4);
#pragma unroll
        for (int r = 0; r < KIE_R8; ++r) {
            const uint2 w = *reinterpret_cast<const uint2*>(slot + size_t(r) * KIE_KC_F16 + size_t(p) * 8);
            a2[r] = piece_f8(w, xl, xh, a2[r]);
        }
    }
#pragma unroll
    for (int r = 0; r < KIE_R8; ++r) acc[r] = a2[r].x + a2[r].y;
}

// NVFP4 slot: E2M1 codes [rows_g][kc/2] (element 2b in the low nibble of byte
// b), then the E4M3 block scales [rows_g][kc/16]; the rows' fp32 scales are
// applied in row_sum.  Each lane takes one 16-column block (two 8-element
// pieces of the activation) per iteration: the block's 16 codes become exact
// fp16 pairs, are multiplied by the activation in fp32 and summed, and the
// sum is scaled by the block's E4M3 scale (exact in fp32).
__device__ __forceinline__ void slot_f4(const uint8_t* slot, int rows_g, int kc, int k0, const float* act, int half,
                                        int lane, float* acc) {
    const int nb = kc >> 4;
    const uint8_t* bsc = slot + size_t(rows_g) * (kc / 2);
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
#pragma unroll
    for (int r = 0; r < KIE_R4; ++r) acc[r] = 0.f;
    for (int b = lane; b < nb; b += 32) {
        const int p = 2 * b;   // first of the block's two pieces
        const float4 xl0 = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh0 = *reinterpret_cast<const float4*>(ahi + p * 4);
        const float4 xl1 = *reinterpret_cast<const float4*>(alo + p * 4 + 4);
        const float4 xh1 = *reinterpret_cast<const float4*>(ahi + p * 4 + 4);
#pragma unroll
        for (int r = 0; r < KIE_R4; ++r) {
            if (r < rows_g) {
                const uint2 w = *reinterpret_cast<const uint2*>(slot + size_t(r) * (kc / 2) + size_t(b) * 8);
                float f[4];
                e4m3x4_to_f32(uint32_t(bsc[r * (kc >> 4) + b]), f);
                // piece p: codes 0..7 = bytes 0..3 of w.x; piece p+1: bytes 0..3 of w.y
                float2 s = make_float2(0.f, 0.f);
                s = ffma2(h2_to_f2(e2m1x2_to_h2(w.x & 0xFFu)), make_float2(xl0.x, xl0.y), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2((w.x >> 8) & 0xFFu)), make_float2(xl0.z, xl0.w), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2((w.x >> 16) & 0xFFu)), make_float2(xh0.x, xh0.y), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2(w.x >> 24)), make_float2(xh0.z, xh0.w), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2(w.y & 0xFFu)), make_float2(xl1.x, xl1.y), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2((w.y >> 8) & 0xFFu)), make_float2(xl1.z, xl1.w), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2((w.y >> 16) & 0xFFu)), make_float2(xh1.x, xh1.y), s);
                s = ffma2(h2_to_f2(e2m1x2_to_h2(w.y >> 24)), make_float2(xh1.z, xh1.w), s);
                acc[r] = fmaf(f[0], s.x + s.y, acc[r]);
            }
        }
    }
}

// INT4 slot: codes [rows_g][kc/2] (element 2b in the low nibble of byte b, two's
// complement), then fp16 scales [rows_g][kc/128].  Each lane takes 8-element
// pieces; a piece lies inside one 128-column group.
__device__ __forceinline__ void slot_i4(const uint8_t* slot, int rows_g, int kc, int k0, const float* act,
                                        int half, int lane, float* acc) {
    const int npc = kc >> 3;
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + size_t(rows_g) * (kc / 2));
    const __half2 bias = __floats2half2_rn(1032.f, 1032.f);
    for (int p = lane; p < npc; p += 32) {
        const float4 xl = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh = *reinterpret_cast<const float4*>(ahi + p * 4);
        const float xlo[4] = {xl.x, xl.y, xl.z, xl.w};
        const float xhi[4] = {xh.x, xh.y, xh.z, xh.w};
        const int grp = p >> 4;
#pragma unroll
        for (int r = 0; r < KIE_R; ++r) {
            if (r < rows_g) {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(slot + size_t(r) * (kc / 2) + size_t(p) * 4);
                const uint32_t u = w ^ 0x88888888u;  // nibble q -> q + 8 in [0, 15]
                float t = 0.f;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    // (1024 + n) as fp16 for nibbles s and s+4, minus 1032 -> exact q
                    uint32_t hbits = ((u >> (4 * s)) & 0x000F000Fu) | 0x64006400u;
                    const __half2 q2 = __hsub2(*reinterpret_cast<__half2*>(&hbits), bias);
                    const float2 f = __half22float2(q2);
                    t = fmaf(f.x, xlo[s], t);
                    t = fmaf(f.y, xhi[s], t);
                }
                const float scale = __half2float(__ushort_as_half(sc[r * (kc >> 7) + grp]));
                acc[r] = fmaf(scale, t, acc[r]);
            }
        }
    }
}

// Row r's output: the sum of its chunks' partials (times its scale for FP8).
__device__ __forceinline__ float row_sum(const Smem& S, const Cursor& c, int r) {
    float y = 0.f;
    for (int ch = 0; ch < c.nK; ++ch) y += S.part[r * c.nK + ch];
    return (c.wfmt == WF_F8 || c.wfmt == WF_F4) ? y * S.wsc[r] : y;
}

// Scaled E5M2 cache: the scale of the slice holding position pos.  The first
// position of slice j >= 1 derives it from slice j-1 (its scale and largest
// stored magnitude, both final since the previous step); every other position
// reads the value written when its slice began (slice 0: set by the host).
__device__ __forceinline__ size_t slice_index(const KieParams& P, int layer, int kv, int j) {
    return (size_t(layer) * 2 + kv) * P.nslice + j;
}
__device__ __forceinline__ float slice_scale(const KieParams& P, int layer, int kv, int pos) {
    const int j = pos / KIE_KV_SLICE;
    if (j == 0 || pos % KIE_KV_SLICE != 0) return __ldcg(P.kv_sc + slice_index(P, layer, kv, j));
    const float sp = __ldcg(P.kv_sc + slice_index(P, layer, kv, j - 1));
    const float amax = __uint_as_float(__ldcg(P.kv_mx + slice_index(P, layer, kv, j - 1))) * sp;
    return (isfinite(amax) && amax > 0.f) ? amax / KIE_KV_SCALE_TARGET : sp;
}
// |value| of an E5M2 byte (NaN stays NaN: fmaxf then ignores it)
__device__ __forceinline__ float e5m2_mag(uint32_t b) {
    return fabsf(__half2float(__ushort_as_half((unsigned short)((b & 0xFFu) << 8))));
}

// store one element of the new K (kv=0) or V (kv=1) at position pos; returns
// the stored bits (fp16, or the E5M2 byte).  s: the slice's scale (scaled E5M2 cache).
__device__ __forceinline__ uint32_t kv_store(const KieParams& P, int layer, int kv, int h, int pos, int dim, float v,
                                             float s) {
    const __half hv = __float2half_rn(v);
    if (P.kv == KV_E5M2S) {   // E5M2 of fp16(v) / s
        uint8_t* base = kv ? P.vc : P.kc;
        const __half y = __float2half_rn(__half2float(hv) / s);
        const uint32_t b = f16x2_to_e5m2x2(y, y) & 0xFFu;
        base[kv_elem_index(P, layer, h, pos) + dim] = uint8_t(b);
        return b;
    }
    if (P.kv == KV_F16) {
        uint8_t* base = kv ? P.vc : P.kc;
        reinterpret_cast<__half*>(base)[kv_elem_index(P, layer, h, pos) + dim] = hv;
    } else if (P.kv == KV_E5M2) {
        uint8_t* base = kv ? P.vc : P.kc;
        const uint32_t b = f16x2_to_e5m2x2(hv, hv) & 0xFFu;
        base[kv_elem_index(P, layer, h, pos) + dim] = uint8_t(b);
        return b;
    } else {
        reinterpret_cast<__half*>(P.tail)[tail_index(P, layer, kv, h, pos % KIE_SEG) + dim] = hv;
    }
    return __half_as_ushort(hv);
}

// ---------------------------------------------------------------------------------------------
// phase epilogues
// ---------------------------------------------------------------------------------------------
// The epilogues of the QKV, O, GU and D phases run per row group, by the warp
// that completes the group's last column chunk, as soon as it is complete:
// the phase's outputs leave the CTA while its other warps are still in the
// GEMV, and the last one right after the CTA's last slot.
struct EpiArgs {
    int type;              // PH_QKV, PH_O, PH_GU, PH_D; PH_LM: no group epilogue
    int layer, pos;
    uint32_t n;            // write number of the layer (tags of q, K, V, a)
    float rinv;            // QKV, GU: 1 / sqrt(mean(x^2) + eps) of the staged x
    const uint16_t* erow;  // first layer's O: the embedding row is the old x
    uint32_t par_in, par_out;   // O, D: parity of the old and the new x
    bool have_xres;        // O, D: the old x of this CTA's rows is in S.xres
};

// Unit u (local) of the QKV phase: the RoPE pair (i, i + hd/2) of q or K of
// head h, or the same pair of V.  Writes the cache (for later steps) and the
// tagged q / current-position K, V (for this step's attention).
__device__ __forceinline__ void qkv_unit(const KieParams& P, const Smem& S, const Cursor& c, const EpiArgs& e,
                                         int u, float ya, float yb, float& mk, float& mv) {
    const int hh = P.hd / 2, lhh = P.hd == 128 ? 6 : 5;   // hd is 64 or 128
    const int per = P.H * hh;  // units per matrix
    const uint32_t par = tag_par(e.n), ep16 = tag_ep16(e.n);
    const int U = c.unit0 + u;
    const int which = (U >= per) + (U >= 2 * per), rem = U - which * per;
    const int h = rem >> lhh, i = rem & (hh - 1);
    const int e0 = h * P.hd + i;
    if (which == 2) {
        const float sv = S.red[KVS_SLOT + 1];
        const uint32_t b0 = kv_store(P, e.layer, 1, h, e.pos, i, ya, sv), b1 = kv_store(P, e.layer, 1, h, e.pos, i + hh, yb, sv);
        st_relaxed_u32(P.vcur + e0, (b0 << 16) | ep16);
        st_relaxed_u32(P.vcur + e0 + hh, (b1 << 16) | ep16);
        if (P.kv == KV_E5M2S) {
            mv = fmaxf(mv, fmaxf(e5m2_mag(b0), e5m2_mag(b1)));
            if (h == 0 && i == 0 && e.pos % KIE_KV_SLICE == 0)   // the slice's first position: publish its scale
                P.kv_sc[slice_index(P, e.layer, 1, e.pos / KIE_KV_SLICE)] = sv;
        }
        return;
    }
    const float cs = S.rope[i], sn = S.rope[hh + i];
    const float ra = ya * cs - yb * sn, rb = yb * cs + ya * sn;
    if (which == 0) {
        st_relaxed_f32(P.q + e0, tag_f32(ra, par));
        st_relaxed_f32(P.q + e0 + hh, tag_f32(rb, par));
    } else {
        const float sk = S.red[KVS_SLOT];
        const uint32_t b0 = kv_store(P, e.layer, 0, h, e.pos, i, ra, sk), b1 = kv_store(P, e.layer, 0, h, e.pos, i + hh, rb, sk);
        st_relaxed_u32(P.kcur + e0, (b0 << 16) | ep16);
        st_relaxed_u32(P.kcur + e0 + hh, (b1 << 16) | ep16);
        if (P.kv == KV_E5M2S) {
            mk = fmaxf(mk, fmaxf(e5m2_mag(b0), e5m2_mag(b1)));
            if (h == 0 && i == 0 && e.pos % KIE_KV_SLICE == 0)
                P.kv_sc[slice_index(P, e.layer, 0, e.pos / KIE_KV_SLICE)] = sk;
        }
    }
}

// Row r (local) of the O or D phase: x[row] += y.  The old x[row] comes from
// S.xres when this launch ran the staging that kept it (at most KIE_XRES
// rows), is the embedding row in the first layer's O phase, and is otherwise
// polled with parity par_in; the new x carries par_out.
__device__ __forceinline__ void residual_row(const KieParams& P, const KieLaunch& Lc, const Smem& S,
                                             const Cursor& c, const EpiArgs& e, int r, float y, int cta) {
    const int row = c.unit0 + r;
    const float xo = (e.have_xres && c.rows <= KIE_XRES) ? S.xres[r]
                     : e.erow ? __half2float(__ushort_as_half(e.erow[row]))
                              : wait_f32(P, Lc, S, P.x + row, e.par_in, cta);
    const float xn = tag_f32(xo + y, e.par_out);
#pragma unroll
    for (int k = 0; k < KIE_REPL; ++k) st_relaxed_f32(P.x + k * P.d + row, xn);
}

// The epilogue of row group g (rows_g rows from row g * R), one unit or row a lane.
__device__ __forceinline__ void epi_group(const KieParams& P, const KieLaunch& Lc, const Smem& S, const Cursor& c,
                                          const EpiArgs& e, int g, int rows_g, int lane, int cta) {
    const int r0 = g * c.R;
    if (e.type == PH_QKV || e.type == PH_GU) {   // units are row pairs
        float mk = 0.f, mv = 0.f;   // scaled E5M2 cache: largest stored K / V magnitudes of this lane
        if (2 * lane < rows_g) {
            const int u = (r0 >> 1) + lane;
            const float ya = row_sum(S, c, 2 * u) * e.rinv, yb = row_sum(S, c, 2 * u + 1) * e.rinv;
            if (e.type == PH_QKV) qkv_unit(P, S, c, e, u, ya, yb, mk, mv);
            else {
                const float av = tag_f32((ya / (1.f + expf(-ya))) * yb, tag_par(e.n));
#pragma unroll
                for (int k = 0; k < KIE_REPL; ++k) st_relaxed_f32(P.a + k * P.F + c.unit0 + u, av);
            }
        }
        if (P.kv == KV_E5M2S && e.type == PH_QKV) {   // the slice's running maxima (fp32 bits order as uints)
            mk = warp_max(mk);
            mv = warp_max(mv);
            const int j = e.pos / KIE_KV_SLICE;
            if (lane == 0 && mk > 0.f) atomicMax(P.kv_mx + slice_index(P, e.layer, 0, j), __float_as_uint(mk));
            if (lane == 0 && mv > 0.f) atomicMax(P.kv_mx + slice_index(P, e.layer, 1, j), __float_as_uint(mv));
        }
    } else if (lane < rows_g) {
        residual_row(P, Lc, S, c, e, r0 + lane, row_sum(S, c, r0 + lane), cta);
    }
}

// The common full INT4 slot (KIE_R rows x KIE_KC_I4 columns) with compile-time
// bounds: each iteration loads the codes of all rows, their group scales and
// the piece's activations first, so several iterations' loads are in flight.
// Same arithmetic and order as slot_i4.
__device__ __forceinline__ void slot_i4_full(const uint8_t* slot, int k0, const float* act, int half, int lane,
                                             float* acc) {
    constexpr int KC = KIE_KC_I4, NPC = KC / 8;
    const float* alo = act + (k0 >> 3) * 4;
    const float* ahi = alo + half;
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(slot + size_t(KIE_R) * (KC / 2));
    const __half2 bias = __floats2half2_rn(1032.f, 1032.f);
    constexpr int kUnroll = KIE_I4_UNROLL;
#pragma unroll kUnroll
    for (int it = 0; it < NPC / 32; ++it) {
        const int p = lane + it * 32;
        const float4 xl = *reinterpret_cast<const float4*>(alo + p * 4);
        const float4 xh = *reinterpret_cast<const float4*>(ahi + p * 4);
        const float xlo[4] = {xl.x, xl.y, xl.z, xl.w};
        const float xhi[4] = {xh.x, xh.y, xh.z, xh.w};
        const int grp = p >> 4;
        uint32_t w[KIE_R];
        float scale[KIE_R];
#pragma unroll
        for (int r = 0; r < KIE_R; ++r) {
            w[r] = *reinterpret_cast<const uint32_t*>(slot + size_t(r) * (KC / 2) + size_t(p) * 4);
            scale[r] = __half2float(__ushort_as_half(sc[r * (KC >> 7) + grp]));
        }
#pragma unroll
        for (int r = 0; r < KIE_R; ++r) {
            const uint32_t u = w[r] ^ 0x88888888u;  // nibble q -> q + 8 in [0, 15]
            float t = 0.f;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                // (1024 + n) as fp16 for nibbles s4 and s4+4, minus 1032 -> exact q
                uint32_t hbits = ((u >> (4 * s4)) & 0x000F000Fu) | 0x64006400u;
                const __half2 q2 = __hsub2(*reinterpret_cast<__half2*>(&hbits), bias);
                const float2 f = __half22float2(q2);
                t = fmaf(f.x, xlo[s4], t);
                t = fmaf(f.y, xhi[s4], t);
            }
            acc[r] = fmaf(scale[r], t, acc[r]);
        }
    }
}

// Consume this phase's slots (those with global index == warp mod NW), leave
// per-(row, chunk) partial sums in S.part, and run the epilogue of every row
// group this warp completes.  Returns false on abort.
__device__ bool run_gemv(const KieParams& P, const KieLaunch& Lc, const Smem& S, const Cursor& c, uint32_t& gc,
                         const EpiArgs& e, int warp, int lane, int cta) {
    const uint32_t nslot = uint32_t(P.nslot);
    const int half = P.act_floats / 2;
    bool ok = true;
    const uint32_t first = uint32_t(warp);   // slot j of a phase -> warp j % NW (mode independent)
    for (uint32_t j = first; j < c.nslots; j += NW) {
        const uint32_t gidx = gc + j;
        const uint32_t slot = gidx % nslot;
        if (!warp_wait_full(P, Lc, S, gidx, cta, lane)) { ok = false; break; }
        if (lane == 0) slot_stamp(Lc, cta, gidx, 1);
        int g, ch, rows_g, kc;
        slot_geom(c, j, g, ch, rows_g, kc);
        const uint8_t* sl = S.ring + size_t(slot) * KIE_SLOT_BYTES;
        if (c.wfmt == WF_F4) {
            float acc[KIE_R4];
            slot_f4(sl, rows_g, kc, ch * c.KC, S.act, half, lane, acc);
#pragma unroll
            for (int r = 0; r < KIE_R4; ++r) acc[r] = warp_sum(acc[r]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < KIE_R4; ++r)   // constant indices: acc stays in registers
                    if (r < rows_g) S.part[(g * c.R + r) * c.nK + ch] = acc[r];
            }
        } else if (c.wfmt == WF_F8) {
            float acc[KIE_R8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if (rows_g == KIE_R8 && kc == KIE_KC_F16) slot_f8_full(sl, ch * c.KC, S.act, half, lane, acc);
            else slot_f8(sl, rows_g, kc, ch * c.KC, S.act, half, lane, acc);
#pragma unroll
            for (int r = 0; r < KIE_R8; ++r) acc[r] = warp_sum(acc[r]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < KIE_R8; ++r)   // constant indices: acc stays in registers
                    if (r < rows_g) S.part[(g * c.R + r) * c.nK + ch] = acc[r];
            }
        } else {
            float acc[KIE_R] = {0.f, 0.f, 0.f, 0.f};
            if (c.wfmt == WF_F16) {
                if (rows_g == KIE_R && kc == KIE_KC_F16) slot_f16_full(sl, ch * c.KC, S.act, half, lane, acc);
                else slot_f16(sl, rows_g, kc, ch * c.KC, S.act, half, lane, acc);
            }
            else if (rows_g == KIE_R && kc == KIE_KC_I4) slot_i4_full(sl, ch * c.KC, S.act, half, lane, acc);
            else slot_i4(sl, rows_g, kc, ch * c.KC, S.act, half, lane, acc);
#pragma unroll
            for (int r = 0; r < KIE_R; ++r) acc[r] = warp_sum(acc[r]);
            if (lane == 0) {
#pragma unroll
                for (int r = 0; r < KIE_R; ++r)
                    if (r < rows_g) S.part[(g * c.R + r) * c.nK + ch] = acc[r];
            }
        }
        __syncwarp();
        if (lane == 0) {
            slot_stamp(Lc, cta, gidx, 2);
            mbar_arrive_cnt(&S.empty[slot], NW);
        }
        if (e.type != PH_LM) {
            // the group is complete when its last chunk is in (one chunk: now)
            int done = 1;
            if (c.nK > 1) {
                if (lane == 0) {
                    __threadfence_block();
                    done = atomicAdd(&S.cnt[g], 1) == c.nK - 1;
                    __threadfence_block();
                }
                __syncwarp();
                done = __shfl_sync(0xffffffffu, done, 0);
            }
            if (done) epi_group(P, Lc, S, c, e, g, rows_g, lane, cta);
        }
    }
    gc += c.nslots;
    if (!ok) S.flags[0] = 1;
    consumer_sync(NCT);
    return ld_volatile_i32(&S.flags[0]) == 0;
}

// LM head: logits, per-CTA argmax (lowest index on ties), last CTA reduces.
// Returns the reduced token through S.flags[2] on the reducing CTA only.
__device__ void epi_lm(const KieParams& P, const KieLaunch& Lc, const Smem& S, const Cursor& c, int cta, int tid,
                       int step, int pos) {
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    const float nr = norm_r(P, S);
    for (int r = tid; r < c.rows; r += NCT) {
        const float y = row_sum(S, c, r) / nr;
        const int row = c.unit0 + r;
        if (Lc.out_logits) Lc.out_logits[size_t(step - Lc.lm_from_step) * P.V + row] = y;
        if (y > best || (y == best && row < bidx)) { best = y; bidx = row; }
    }
    // block argmax
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (ov > best || (ov == best && oi < bidx)) { best = ov; bidx = oi; }
    }
    int* ridx = reinterpret_cast<int*>(S.red + 32);
    if ((tid & 31) == 0) { S.red[tid >> 5] = best; ridx[tid >> 5] = bidx; }
    consumer_sync(NCT);
    if (tid == 0) {
        for (int w = 1; w < NW; ++w) {
            if (S.red[w] > best || (S.red[w] == best && ridx[w] < bidx)) { best = S.red[w]; bidx = ridx[w]; }
        }
        P.amax_val[cta] = best;
        P.amax_idx[cta] = bidx;
        __threadfence();
        const uint32_t old = atomicAdd(&P.ctl->amax_cnt, 1u);
        S.flags[1] = (old == uint32_t(P.G) - 1u) ? 1 : 0;
    }
    consumer_sync(NCT);
    const int warp = tid >> 5, lane = tid & 31;
    if (S.flags[1] && warp == 0) {
        __threadfence();
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = lane; i < P.G; i += 32) {
            const float v = __ldcg(P.amax_val + i);
            const int ix = __ldcg(P.amax_idx + i);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) {
            if (bi < 0 || bi >= P.V) bi = 0;  // all logits NaN: keep a valid id
            P.ctl->amax_cnt = 0u;
            P.ctl->tok = bi;
            P.ctl->pos = pos + 1;
            if (Lc.out_tokens) Lc.out_tokens[step] = bi;
            __threadfence();
        }
    }
}

// ---------------------------------------------------------------------------------------------
// split-KV attention
// ---------------------------------------------------------------------------------------------
// One row's 16 dims [dim0, dim0+16) of K or V as raw storage (converted to fp32
// only when used, so several rows can be in flight per lane).
// mode: 0 = stored (fp16 / E5M2 / u8 codes with the segment's scale, zp),
//       1 = u8 open segment, read from the fp16 tail,
//       2 = u8 segment completed in this step (quantised now with fz's scale, zp).
struct RawRow {
    uint4 a, b;     // fp16: 32 bytes; 8-bit formats: a only
    float sc;       // u8 mode 0
    int zp;
    int mode;
};

template <int KVF>
__device__ __forceinline__ void load_raw(const KieParams& P, int layer, int kv, int h, int pos, int dim0, int mode,
                                         RawRow& r) {
    r.mode = mode;
    if (KVF == KV_F16 || (KVF == KV_U8 && mode != 0)) {
        const uint4* src;
        if (KVF == KV_F16) {
            const uint8_t* base = kv ? P.vc : P.kc;
            src = reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(base) +
                                                 kv_elem_index(P, layer, h, pos) + dim0);
        } else {
            src = reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(P.tail) +
                                                 tail_index(P, layer, kv, h, pos % KIE_SEG) + dim0);
        }
        r.a = __ldcg(src);
        r.b = __ldcg(src + 1);
    } else {
        const uint8_t* base = kv ? P.vc : P.kc;
        r.a = __ldcg(reinterpret_cast<const uint4*>(base + kv_elem_index(P, layer, h, pos) + dim0));
        if (KVF == KV_U8) {
            const size_t mi = meta_index(P, layer, kv, h, pos / KIE_SEG);
            r.sc = __ldcg(P.seg_scale + mi);
            r.zp = __ldcg(P.seg_zp + mi);
        }
    }
}

template <int KVF>
__device__ __forceinline__ void convert_row(const RawRow& r, const float* fz, float* f) {
    if (KVF == KV_F16 || (KVF == KV_U8 && r.mode != 0)) {
        const uint32_t w[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) { const float2 t = h2_to_f2(w[i]); f[2 * i] = t.x; f[2 * i + 1] = t.y; }
        if (KVF == KV_U8 && r.mode == 2) {
            const float sc = fz[0];
            const int zp = __float_as_int(fz[1]);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int qv = min(max(__float2int_rn(f[i] / sc) + zp, 0), 255);
                f[i] = float(qv - zp) * sc;
            }
        }
    } else if (KVF == KV_E5M2 || KVF == KV_E5M2S) {
        e5m2x4_to_f32(r.a.x, f); e5m2x4_to_f32(r.a.y, f + 4); e5m2x4_to_f32(r.a.z, f + 8); e5m2x4_to_f32(r.a.w, f + 12);
    } else {
        const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = float(int((w[i >> 2] >> (8 * (i & 3))) & 0xFFu) - r.zp) * r.sc;
    }
}

// The current position's 16 dims [dim0, dim0+16) of K (kv=0) or V, from the
// tagged copy written in this step's QKV epilogue, as a RawRow of the stored
// format (fp16 pairs; E5M2 bytes).  The uint8 cache keeps the open segment in
// fp16, so its current row is fp16 too.  cur_row_issue starts the loads (K's
// and V's together), cur_row_finish polls whatever has not arrived yet and
// packs the row.
__device__ __forceinline__ void cur_row_issue(const KieParams& P, int kv, int h, int dim0, uint4* w) {
    const uint32_t* src = (kv ? P.vcur : P.kcur) + h * P.hd + dim0;
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = ld_relaxed_u4(src + 4 * i);
}
template <int KVF>
__device__ __forceinline__ void cur_row_finish(const KieParams& P, const KieLaunch& Lc, const Smem& S, int kv, int h,
                                               int dim0, uint32_t ep16, int cta, uint4* w, RawRow& r) {
    const uint32_t* src = (kv ? P.vcur : P.kcur) + h * P.hd + dim0;
    uint32_t bad = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (!has_ep4(w[i], ep16)) bad |= 1u << i;
    if (bad) {
        TagWait tw;
        do {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                if ((bad >> i) & 1u) {
                    w[i] = ld_relaxed_u4(src + 4 * i);
                    if (has_ep4(w[i], ep16)) bad &= ~(1u << i);
                }
            }
        } while (bad && tw.again(P, Lc, S, cta));
    }
    r.sc = 0.f;
    r.zp = 0;
    if (KVF == KV_E5M2 || KVF == KV_E5M2S) {
        uint32_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            b[i] = ((w[i].x >> 16) & 0xFFu) | (((w[i].y >> 16) & 0xFFu) << 8) | (((w[i].z >> 16) & 0xFFu) << 16) |
                   (((w[i].w >> 16) & 0xFFu) << 24);
        r.a = make_uint4(b[0], b[1], b[2], b[3]);
        r.b = make_uint4(0, 0, 0, 0);
    } else {
        uint32_t hp[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            hp[2 * i] = (w[i].x >> 16) | (w[i].y & 0xFFFF0000u);
            hp[2 * i + 1] = (w[i].z >> 16) | (w[i].w & 0xFFFF0000u);
        }
        r.a = make_uint4(hp[0], hp[1], hp[2], hp[3]);
        r.b = make_uint4(hp[4], hp[5], hp[6], hp[7]);
    }
}

// Element i of a (layer, kv, head) open segment (row i / hd of the fp16 tail;
// row prow is the current position, read from its tagged copy).
__device__ __forceinline__ float seg_elem(const KieParams& P, const KieLaunch& Lc, const Smem& S, const __half* t,
                                          int kv, int h, int i, int prow, uint32_t ep16, int cta) {
    if (i / P.hd == prow) {
        const uint32_t* cur = (kv ? P.vcur : P.kcur) + h * P.hd + i % P.hd;
        return __half2float(__ushort_as_half((unsigned short)wait_cur(P, Lc, S, cur, ep16, cta)));
    }
    return __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short*>(t) + i)));
}

// scale/zp of one (layer, kv, head) open segment, from its 128 fp16 tail rows.
__device__ void u8_segment_params(const KieParams& P, const KieLaunch& Lc, const Smem& S, int layer, int kv, int h,
                                  int prow, uint32_t ep16, int tid, int cta, float* out /* [0]=scale, [1]=zp bits */) {
    const __half* t = reinterpret_cast<const __half*>(P.tail) + tail_index(P, layer, kv, h, 0);
    const int n = KIE_SEG * P.hd;
    float mn = INFINITY, mx = -INFINITY;
    for (int i = tid; i < n; i += NCT) {
        const float v = seg_elem(P, Lc, S, t, kv, h, i, prow, ep16, cta);
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    mx = block_max(mx, S.red, tid);
    mn = -block_max(-mn, S.red, tid);
    if (tid == 0) {
        float sc;
        int zp;
        if (mx == mn) { sc = 1.f; zp = __float2int_rn(-mn); }
        else { sc = (mx - mn) / 255.f; zp = __float2int_rn(-mn / sc); }
        out[0] = sc;
        out[1] = __int_as_float(zp);
    }
    consumer_sync(NCT);
}

// Write codes + meta of a segment completed in this step (its owner CTA only).
__device__ void u8_segment_commit(const KieParams& P, const KieLaunch& Lc, const Smem& S, int layer, int kv, int h,
                                  int seg, int prow, uint32_t ep16, const float* fz, int tid, int cta) {
    const __half* t = reinterpret_cast<const __half*>(P.tail) + tail_index(P, layer, kv, h, 0);
    uint8_t* dst = (kv ? P.vc : P.kc) + kv_elem_index(P, layer, h, seg * KIE_SEG);
    const float sc = fz[0];
    const int zp = __float_as_int(fz[1]);
    const int n = KIE_SEG * P.hd;
    for (int i = tid; i < n; i += NCT) {
        const float v = seg_elem(P, Lc, S, t, kv, h, i, prow, ep16, cta);
        dst[i] = uint8_t(min(max(__float2int_rn(v / sc) + zp, 0), 255));
    }
    if (tid == 0) {
        const size_t mi = meta_index(P, layer, kv, h, seg);
        P.seg_scale[mi] = sc;
        P.seg_zp[mi] = zp;
    }
}

// 16 dims of a row held in shared memory (ring slot) -> fp32.
template <int KVF>
__device__ __forceinline__ void smem_row16(const uint8_t* row, int dim0, float sc, int zp, float* f) {
    if (KVF == KV_F16) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + dim0 * 2);
        const uint4 b = *reinterpret_cast<const uint4*>(row + dim0 * 2 + 16);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) { const float2 t = h2_to_f2(w[i]); f[2 * i] = t.x; f[2 * i + 1] = t.y; }
    } else if (KVF == KV_E5M2 || KVF == KV_E5M2S) {
        const uint4 a = *reinterpret_cast<const uint4*>(row + dim0);
        e5m2x4_to_f32(a.x, f); e5m2x4_to_f32(a.y, f + 4); e5m2x4_to_f32(a.z, f + 8); e5m2x4_to_f32(a.w, f + 12);
    } else {
        const uint4 a = *reinterpret_cast<const uint4*>(row + dim0);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = float(int((w[i >> 2] >> (8 * (i & 3))) & 0xFFu) - zp) * sc;
    }
}

// The 16 uint8 codes [dim0, dim0 + 16) of a ring row as exact floats: each
// byte goes into the low mantissa of 2^23 (one byte permute) and 2^23 is
// subtracted, two instructions a code.  The segment's zero point and scale are
// applied outside, once per row: q.k = sc (sum q_i c_i - zp sum q_i), and
// sum_j p_j v_j = sum_j (p_j sc_j) c_j - sum_j (p_j sc_j) zp_j.
__device__ __forceinline__ void u8_codes16(const uint8_t* row, int dim0, float* c) {
    const uint4 a = *reinterpret_cast<const uint4*>(row + dim0);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        c[i] = __uint_as_float(__byte_perm(w[i >> 2], 0x4B000000u, 0x7650u + (i & 3))) - 8388608.f;
}

// Online-softmax state of one lane: running max m, sum l and weighted V sum of
// its 16 dims over the rows its row group has seen.
struct SoftState {
    float m, l, acc[16];
};
// Fold one row (score s, V dims v) into the state.
__device__ __forceinline__ void soft_row(SoftState& st, float s, const float* v) {
    const float mn = fmaxf(st.m, s);
    const float cf = expf(st.m - mn), p = expf(s - mn);   // st.m = -inf: cf = 0
    st.l = fmaf(st.l, cf, p);
#pragma unroll
    for (int i = 0; i < 16; ++i) st.acc[i] = fmaf(st.acc[i], cf, p * v[i]);
    st.m = mn;
}

// BAT (the batched kernel): the CTA's (request, head) pair comes from
// att_chunk_b for step t, and q, the current K/V and o are that request's.
template <int HD, int KVF, bool BAT = false>
__device__ bool attention(const KieParams& P, const KieLaunch& Lc, const Smem& S, int layer, int pos, uint32_t tn,
                          int cta, uint32_t& gc, int warp, int lane, int tid, int t = 0) {
    const uint32_t par = tag_par(tn), ep16 = tag_ep16(tn);   // tags of this layer's q, K, V (read) and o (written)
    constexpr int LPR = HD / 16;       // lanes per row (16 dims each)
    constexpr int RPI = 32 / LPR;      // row groups of a warp (rows per warp instruction)
    constexpr int NRG = NW * RPI;      // row groups per CTA (direct rows)
    constexpr int UR = 4;              // direct rows in flight per lane group
    constexpr int RB = HD * (KVF == KV_F16 ? 2 : 1);
    constexpr int RMAX = KIE_SLOT_BYTES / (2 * RB * RPI);   // rows of one row group in a slot
#ifndef KIE_ATT_RU
#define KIE_ATT_RU 4
#endif
    constexpr int RU = KIE_ATT_RU;     // ring rows in flight per row group
    const AttChunk a = BAT ? att_chunk_b(P, S.flags + 8, cta, t) : att_chunk(P, cta, pos);
    if (BAT) pos = a.pos;
    const int h = a.h, j0 = a.j0, j1 = a.j1, jt = a.jt;
    const int hb = BAT ? a.b * P.H + h : h;   // row of the pair's q, current K/V and o
    const int n = j1 - j0, nt = jt - j0;
    const int lg = lane % LPR, rw = lane / LPR;
    const int dim0 = lg * 16;
    const int rps = att_rows_per_slot(P, a);
    const uint32_t nsl = att_nslots(P, a), nslot = uint32_t(P.nslot);
    float* fz = S.red + NW * (KIE_MAX_HEAD_DIM + 2);   // [0..1] K scale/zp, [2..3] V scale/zp (fresh segment)
    float* segm = S.part;                              // uint8: per-segment scale/zp of this chunk [2][nseg][2]
    const bool u8_fresh = (KVF == KV_U8) && (pos % KIE_SEG == KIE_SEG - 1);
    const int open_seg = pos / KIE_SEG;
    const int seg0 = j0 / KIE_SEG, nsegc = (KVF == KV_U8 && nt > 0) ? (jt - 1) / KIE_SEG - seg0 + 1 : 0;
    if (KVF == KV_U8) {
        for (int i = tid; i < 2 * nsegc; i += NCT) {
            const int kv = i / nsegc, sg = seg0 + i % nsegc;
            const size_t mi = meta_index(P, layer, kv, h, sg);
            segm[2 * i] = __ldcg(P.seg_scale + mi);
            segm[2 * i + 1] = __int_as_float(__ldcg(P.seg_zp + mi));
        }
        if (u8_fresh && j1 > open_seg * KIE_SEG) {
            const int prow = pos % KIE_SEG;
            u8_segment_params(P, Lc, S, layer, 0, h, prow, ep16, tid, cta, fz);
            u8_segment_params(P, Lc, S, layer, 1, h, prow, ep16, tid, cta, fz + 2);
            if (j1 == pos + 1) {  // the CTA holding position pos stores the codes for later steps
                u8_segment_commit(P, Lc, S, layer, 0, h, open_seg, prow, ep16, fz, tid, cta);
                u8_segment_commit(P, Lc, S, layer, 1, h, open_seg, prow, ep16, fz + 2, tid, cta);
                fence_proxy_async_global();
            }
        }
        consumer_sync(NCT);
    }
    // scaled E5M2 cache: the scales of the slices the chunk's ring rows lie in, [K | V][slice]
    // (all final: ring rows precede pos, and a slice's scale is written at its first position)
    const int sl0 = j0 / KIE_KV_SLICE, nslc = (KVF == KV_E5M2S && nt > 0) ? (jt - 1) / KIE_KV_SLICE - sl0 + 1 : 0;
    if (KVF == KV_E5M2S) {
        for (int i = tid; i < 2 * nslc; i += NCT) segm[i] = __ldcg(P.kv_sc + slice_index(P, layer, i / nslc, sl0 + i % nslc));
        consumer_sync(NCT);
    }
    const bool has_pos = (j1 == pos + 1);
    const bool own_pos = has_pos && warp == 0 && rw == 0;
    float qv[16];
    {
        const float* qp = P.q + hb * HD + dim0;
        float4 v4[4];
        uint32_t bad = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v4[i] = ld_relaxed_f4(qp + 4 * i);
            if (!has_tag4(v4[i], par)) bad |= 1u << i;
        }
        if (bad) {
            TagWait tw;
            do {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if ((bad >> i) & 1u) {
                        v4[i] = ld_relaxed_f4(qp + 4 * i);
                        if (has_tag4(v4[i], par)) bad &= ~(1u << i);
                    }
                }
            } while (bad && tw.again(P, Lc, S, cta));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qv[4 * i] = v4[i].x * P.attn_scale; qv[4 * i + 1] = v4[i].y * P.attn_scale;
            qv[4 * i + 2] = v4[i].z * P.attn_scale; qv[4 * i + 3] = v4[i].w * P.attn_scale;
        }
    }
    if (tid == 0) stamp(P, Lc, BAT ? t : pos - (Lc.pos0 >= 0 ? Lc.pos0 : pos), 5 * layer + 1, 4, cta);
    // The current position is the last row of the head's last chunk; warp 0's
    // first row group fetches its tagged K and V together with q.  fp16 / E5M2
    // stream every other row through the ring; a uint8 cache reads the rest of
    // its open segment directly (mode 1: fp16 tail; mode 2: the segment
    // completes in this step and is quantised with its fresh scale / zp).
    const int dmode = (KVF == KV_U8) ? (u8_fresh ? 2 : 1) : 0;
    const int ndir = has_pos ? n - 1 : n;        // direct rows other than pos: [nt, ndir)
    RawRow kpos, vpos;
    kpos.a = kpos.b = vpos.a = vpos.b = make_uint4(0, 0, 0, 0);
    kpos.sc = vpos.sc = 0.f; kpos.zp = vpos.zp = 0; kpos.mode = vpos.mode = dmode;
    if (own_pos) {   // K and V loads travel together: one round trip
        uint4 wk[4], wv[4];
        cur_row_issue(P, 0, hb, dim0, wk);
        cur_row_issue(P, 1, hb, dim0, wv);
        cur_row_finish<KVF>(P, Lc, S, 0, hb, dim0, ep16, cta, wk, kpos);
        cur_row_finish<KVF>(P, Lc, S, 1, hb, dim0, ep16, cta, wv, vpos);
        kpos.mode = vpos.mode = dmode;
    }

    SoftState st;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) st.acc[i] = 0.f;
    // uint8 ring rows: sum of this lane's q dims, and the weighted V zero points
    float qsum = 0.f, vcorr = 0.f;
    if (KVF == KV_U8) {
#pragma unroll
        for (int i = 0; i < 16; ++i) qsum += qv[i];
    }

    // ---- ring slots: slot j holds rows [j*rps, j*rps + rs) of the chunk, K
    // then V.  The first nrr (whole rounds) go to warp j % NW, whose row groups
    // take rows rw, rw + RPI, ...; each slot of the last partial round is
    // shared by all warps (row group rw of warp w takes rows w*RPI + rw + k*NRG).
    // Each row group keeps its own online softmax.
    bool ok = true;
    const uint32_t nrr = (nsl / NW) * NW, nmine = nrr / NW + (nsl - nrr);
    for (uint32_t i = 0; i < nmine; ++i) {
        const bool shared = i >= nrr / NW;
        const uint32_t j = shared ? nrr + (i - nrr / NW) : uint32_t(warp) + i * NW;
        const int rbase = shared ? warp * RPI : 0, rstr = shared ? NRG : RPI;
        const uint32_t gidx = gc + j, slot = gidx % nslot;
        if (!warp_wait_full(P, Lc, S, gidx, cta, lane)) { ok = false; break; }
        if (lane == 0) slot_stamp(Lc, cta, gidx, 1);
        const uint8_t* ks = S.ring + size_t(slot) * KIE_SLOT_BYTES;
        const uint8_t* vs = ks + size_t(rps) * RB;
        const int r0 = int(j) * rps, rs = min(rps, nt - r0);
        float sc[RMAX];
        float mloc = -INFINITY;
#pragma unroll
        for (int k0 = 0; k0 < RMAX; k0 += RU) {
            if (rbase + k0 * rstr >= rs) break;         // uniform over the warp
            float dsum[RU];
#pragma unroll
            for (int u = 0; u < RU; ++u) {
                const int rl = rbase + rw + (k0 + u) * rstr;
                float kf[16];
                if (KVF == KV_U8) {
                    float scl = 0.f, zpf = 0.f;
                    if (rl < rs) {
                        const int sg = (j0 + r0 + rl) / KIE_SEG - seg0;
                        scl = segm[2 * sg];
                        zpf = float(__float_as_int(segm[2 * sg + 1]));
                    }
                    u8_codes16(ks + size_t(min(rl, rs - 1)) * RB, dim0, kf);
                    float d0 = 0.f, d1 = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; i += 2) { d0 = fmaf(qv[i], kf[i], d0); d1 = fmaf(qv[i + 1], kf[i + 1], d1); }
                    dsum[u] = scl * fmaf(-zpf, qsum, d0 + d1);
                } else {
                    smem_row16<KVF>(ks + size_t(min(rl, rs - 1)) * RB, dim0, 0.f, 0, kf);
                    float d0 = 0.f, d1 = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; i += 2) { d0 = fmaf(qv[i], kf[i], d0); d1 = fmaf(qv[i + 1], kf[i + 1], d1); }
                    dsum[u] = d0 + d1;
                    if (KVF == KV_E5M2S) dsum[u] *= segm[(j0 + r0 + min(rl, rs - 1)) / KIE_KV_SLICE - sl0];
                }
            }
#pragma unroll
            for (int o = 1; o < LPR; o <<= 1) {
#pragma unroll
                for (int u = 0; u < RU; ++u) dsum[u] += __shfl_xor_sync(0xffffffffu, dsum[u], o);
            }
#pragma unroll
            for (int u = 0; u < RU; ++u) {
                const int rl = rbase + rw + (k0 + u) * rstr;
                sc[k0 + u] = rl < rs ? dsum[u] : -INFINITY;
                mloc = fmaxf(mloc, sc[k0 + u]);
            }
        }
        // V rows of the same slot (no shuffles: row groups may diverge)
        const float mn = fmaxf(st.m, mloc);
        if (mn > -INFINITY) {
            const float cf = expf(st.m - mn);
            st.l *= cf;
            if (KVF == KV_U8) vcorr *= cf;
#pragma unroll
            for (int i = 0; i < 16; ++i) st.acc[i] *= cf;
#pragma unroll
            for (int k0 = 0; k0 < RMAX; k0 += RU) {
                if (rbase + k0 * rstr >= rs) break;
#pragma unroll
                for (int u = 0; u < RU; ++u) {
                    const int rl = rbase + rw + (k0 + u) * rstr;
                    if (rl < rs) {
                        float vf[16];
                        const float p = expf(sc[k0 + u] - mn);
                        st.l += p;
                        if (KVF == KV_U8) {
                            const int sg = (j0 + r0 + rl) / KIE_SEG - seg0;
                            const float wv = p * segm[2 * (nsegc + sg)];
                            vcorr = fmaf(wv, float(__float_as_int(segm[2 * (nsegc + sg) + 1])), vcorr);
                            u8_codes16(vs + size_t(rl) * RB, dim0, vf);
#pragma unroll
                            for (int i = 0; i < 16; ++i) st.acc[i] = fmaf(wv, vf[i], st.acc[i]);
                        } else {
                            smem_row16<KVF>(vs + size_t(rl) * RB, dim0, 0.f, 0, vf);
                            const float pw = (KVF == KV_E5M2S) ? p * segm[nslc + (j0 + r0 + rl) / KIE_KV_SLICE - sl0] : p;
#pragma unroll
                            for (int i = 0; i < 16; ++i) st.acc[i] = fmaf(pw, vf[i], st.acc[i]);
                        }
                    }
                }
            }
            st.m = mn;
        }
        __syncwarp();
        if (lane == 0) {
            slot_stamp(Lc, cta, gidx, 2);
            mbar_arrive_cnt(&S.empty[slot], shared ? 1u : uint32_t(NW));
        }
    }
    gc += nsl;
    if (KVF == KV_U8) {   // the zero points of the uint8 V rows folded in above
#pragma unroll
        for (int i = 0; i < 16; ++i) st.acc[i] -= vcorr;
    }
    if (!ok) S.flags[0] = 1;
    if (lane == 0 && warp == 0) stamp(P, Lc, BAT ? t : pos - (Lc.pos0 >= 0 ? Lc.pos0 : pos), 5 * layer + 1, 5, cta);

    // ---- direct rows [jt, j1)
    if (has_pos && warp == 0) {                         // uniform over warp 0
        float kf[16];
        convert_row<KVF>(kpos, fz, kf);
        float dsum = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) dsum = fmaf(qv[i], kf[i], dsum);
#pragma unroll
        for (int o = 1; o < LPR; o <<= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
        if (KVF == KV_E5M2S) dsum *= slice_scale(P, layer, 0, pos);
        if (rw == 0) {
            float vf[16];
            convert_row<KVF>(vpos, fz + 2, vf);
            if (KVF == KV_E5M2S) {
                const float sv = slice_scale(P, layer, 1, pos);
#pragma unroll
                for (int i = 0; i < 16; ++i) vf[i] *= sv;
            }
            soft_row(st, dsum, vf);
        }
    }
    if (KVF == KV_U8)
    for (int base = nt + warp * RPI; base < ndir; base += NRG * UR) {
        RawRow kr[UR], vr[UR];
#pragma unroll
        for (int u = 0; u < UR; ++u) {
            const int r = base + rw + u * NRG;
            kr[u].a = kr[u].b = vr[u].a = vr[u].b = make_uint4(0, 0, 0, 0);
            kr[u].sc = vr[u].sc = 0.f; kr[u].zp = vr[u].zp = 0; kr[u].mode = vr[u].mode = 0;
            if (r < ndir) {
                load_raw<KVF>(P, layer, 0, h, j0 + r, dim0, dmode, kr[u]);
                load_raw<KVF>(P, layer, 1, h, j0 + r, dim0, dmode, vr[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < UR; ++u) {
            const int r = base + rw + u * NRG;
            float kf[16];
            convert_row<KVF>(kr[u], fz, kf);
            float dsum = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) dsum = fmaf(qv[i], kf[i], dsum);
#pragma unroll
            for (int o = 1; o < LPR; o <<= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
            if (r < ndir) {
                float vf[16];
                convert_row<KVF>(vr[u], fz + 2, vf);
                soft_row(st, dsum, vf);
            }
        }
    }

    // ---- merge the row groups of this warp (lanes with equal lg), then the warps
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, st.m, o), lo = __shfl_xor_sync(0xffffffffu, st.l, o);
        const float mn = fmaxf(st.m, mo);
        const float c1 = (st.m == -INFINITY) ? 0.f : expf(st.m - mn);
        const float c2 = (mo == -INFINITY) ? 0.f : expf(mo - mn);
        st.l = st.l * c1 + lo * c2;
#pragma unroll
        for (int i = 0; i < 16; ++i) st.acc[i] = st.acc[i] * c1 + __shfl_xor_sync(0xffffffffu, st.acc[i], o) * c2;
        st.m = mn;
    }
    float* wp = S.red + warp * (KIE_MAX_HEAD_DIM + 2);
    if (lane < LPR) {
#pragma unroll
        for (int i = 0; i < 16; ++i) wp[2 + dim0 + i] = st.acc[i];
        if (lane == 0) { wp[0] = st.m; wp[1] = st.l; }
    }
    consumer_sync(NCT);
    if (ld_volatile_i32(&S.flags[0]) != 0) return false;
    // this CTA's partial (m, l, o[HD]), tagged with the layer's parity; an empty
    // chunk stores m = -FLT_MAX (finite, so the tag bit cannot make it a NaN)
    float* gp = P.att_part + size_t(cta) * (HD + 4);
    if (tid < HD) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, S.red[w * (KIE_MAX_HEAD_DIM + 2)]);
        float ov = 0.f, lv = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float* ww = S.red + w * (KIE_MAX_HEAD_DIM + 2);
            const float e = (ww[0] == -INFINITY) ? 0.f : expf(ww[0] - M);
            ov = fmaf(e, ww[2 + tid], ov);
            lv = fmaf(e, ww[1], lv);
        }
        st_relaxed_f32(gp + 4 + tid, tag_f32(ov, par));
        if (tid == 0) {
            st_relaxed_f32(gp, tag_f32(M == -INFINITY ? -FLT_MAX : M, par));
            st_relaxed_f32(gp + 1, tag_f32(lv, par));
        }
    }
    // The head's first CTA combines its CTAs' partials in CTA order (the same
    // in every mode) and publishes o_h with the layer's parity.
    if (cta == a.c0 && tid < HD) {
        constexpr int MAXC = 10;
        float M = -INFINITY, Ls = 0.f, Os = 0.f;
        for (int k0 = 0; k0 < a.nh; k0 += MAXC) {
            float mk[MAXC], lk[MAXC], ok[MAXC];
            uint32_t bad = 0;
#pragma unroll
            for (int k = 0; k < MAXC; ++k) {
                if (k0 + k < a.nh) {
                    const float* pp = P.att_part + size_t(a.c0 + k0 + k) * (HD + 4);
                    mk[k] = ld_relaxed_f32(pp);
                    lk[k] = ld_relaxed_f32(pp + 1);
                    ok[k] = ld_relaxed_f32(pp + 4 + tid);
                    if (((__float_as_uint(mk[k]) ^ par) | (__float_as_uint(lk[k]) ^ par) |
                         (__float_as_uint(ok[k]) ^ par)) & 1u) bad |= 1u << k;
                }
            }
            if (bad) {
                TagWait tw;
                do {
#pragma unroll
                    for (int k = 0; k < MAXC; ++k) {
                        if ((bad >> k) & 1u) {
                            const float* pp = P.att_part + size_t(a.c0 + k0 + k) * (HD + 4);
                            mk[k] = ld_relaxed_f32(pp);
                            lk[k] = ld_relaxed_f32(pp + 1);
                            ok[k] = ld_relaxed_f32(pp + 4 + tid);
                            if ((((__float_as_uint(mk[k]) ^ par) | (__float_as_uint(lk[k]) ^ par) |
                                  (__float_as_uint(ok[k]) ^ par)) & 1u) == 0u) bad &= ~(1u << k);
                        }
                    }
                } while (bad && tw.again(P, Lc, S, cta));
            }
            float Mb = M;
#pragma unroll
            for (int k = 0; k < MAXC; ++k) if (k0 + k < a.nh) Mb = fmaxf(Mb, mk[k]);
            const float cf = (M == -INFINITY) ? 0.f : expf(M - Mb);
            Ls *= cf;
            Os *= cf;
#pragma unroll
            for (int k = 0; k < MAXC; ++k) {
                if (k0 + k < a.nh) {
                    const float w = expf(mk[k] - Mb);          // -FLT_MAX (empty chunk): 0
                    Ls = fmaf(w, lk[k], Ls);
                    Os = fmaf(w, ok[k], Os);
                }
            }
            M = Mb;
        }
        const float ov = tag_f32(Os / Ls, par);
#pragma unroll
        for (int k = 0; k < KIE_REPL; ++k) st_relaxed_f32(P.o + k * (BAT ? P.nb : 1) * P.H * HD + hb * HD + tid, ov);
    }
    return true;
}

__device__ __forceinline__ bool grid_barrier(const KieParams& P, const KieLaunch& Lc, const Smem& S,
                                             uint32_t& nbar, int tid, int cta) {
    consumer_sync(NCT);
    if (tid == 0) {
        // red.release is cumulative: the block's writes ordered before it by the
        // consumer barrier above become visible to every acquirer of the count.
        // (A test can make one CTA skip its first arrival: the others' bounded
        // waits then run out and report a timeout.)
        if (!(nbar == 0u && cta == Lc.skip_arrival_cta)) red_release_gpu_add(&P.ctl->bar, 1u);
        const uint32_t target = (nbar + 1u) * uint32_t(P.G);
        const uint64_t t0 = globaltimer();
        int spins = 0;
        while (int32_t(ld_acquire_gpu(&P.ctl->bar) - target) < 0) {
            if ((++spins & 15) == 0) {
                if (ld_volatile_i32(&P.ctl->err) != 0) { S.flags[0] = 1; break; }
                if (globaltimer() - t0 > Lc.timeout_ns) {
                    set_error(P, KERR_TIMEOUT_GRID, cta);
                    S.flags[0] = 1;
                    break;
                }
            }
        }
    }
    ++nbar;
    consumer_sync(NCT);
    return ld_volatile_i32(&S.flags[0]) == 0;
}

}  // namespace
