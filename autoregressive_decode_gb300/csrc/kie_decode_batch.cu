// The batched decode program: nb <= 8 independent requests, each with its own
// KV cache, position and greedy chain, advance one token each per step while
// every weight byte streams from HBM once per step (low-batch decode: the Kog
// page runs batch 1 for its preview and names larger batches as the production
// case, TL;DR and section "What changes with autonomous agents").
//
// The structure is the single-request kernel's (kie_decode.cu): one CTA per
// SM, a producer warp streaming this CTA's weights into the shared-memory ring,
// tagged activations instead of phase barriers, one grid barrier per step, and
// the split-KV attention, now over the nb * H (request, head) pairs.  What
// changes is the GEMV: with nb activation vectors per weight row it is a
// skinny GEMM, done with warp-level tensor-core MMAs (mma.sync m16n8k16, fp16
// operands, fp32 accumulation):
//   A (16 x 16)  the activations: row m < 8 holds request m's hi = fp16(a),
//                row 8 + m its lo = fp16(a - hi) (the fp32 activation split in
//                two, as the tensor-core prefill does);
//   B (16 x 8)   8 weight rows;
//   D (16 x 8)   D[m][n] = sum_k A[m][k] W[n][k]; request b's output of row n
//                is D[b][n] + D[8 + b][n].
// The MMA work is small next to the HBM stream (2 x 8 x 16 multiply-adds per
// weight pair of bytes), so warp-level MMAs reading the ring directly suffice;
// tcgen05's 64-row minimum M would exceed the 14-row tiles the O and down
// projections give each CTA.
//
// Weight slots hold 16 rows x 512 fp16 columns, chunk-major: for each group of
// 8 columns, the slot's rows' 16 bytes one after the other, so that one
// ldmatrix.x4 loads the B fragments of both 8-row groups for 16 columns
// without bank conflicts.  A warp owns whole row tiles of a phase: all column
// chunks of a tile accumulate in its registers, and its epilogue runs in the
// same lanes that hold the results (a lane holds request lane/4's outputs of
// rows 2(lane%4), +1, +8, +9 of the tile: a RoPE pair, a gate/up pair).
// Because a warp's consecutive slots can then lie more than the ring apart,
// the warp first waits until the producer has issued the slot (S.flags[5]):
// once slot g is issued, generation g - 2*nslot of its ring slot has landed,
// which is what the full-barrier parity wait needs.
// Activations are staged per block of 2048 input columns (64 KB of MMA
// fragments for 8 requests); a phase with more columns (the down projection)
// streams its slots in the order (block, row tile, chunk) and restages
// between blocks.
#include "kie_decode_core.cuh"

using namespace kie;

namespace {

constexpr int NB = KIE_MAX_BATCH;
// S.red regions of the batched kernel (after attention's per-warp partials and
// its 64 floats of scratch)
constexpr int RED_NORM = NW * (KIE_MAX_HEAD_DIM + 2) + 64;   // [NB][NW] sums of squares of the staged x
constexpr int RED_AMV = RED_NORM + NB * NW;                  // [NW][NB] LM argmax values
constexpr int RED_AMI = RED_AMV + NB * NW;                   // [NW][NB] LM argmax indices

constexpr int KSTEP_WORDS = 128;                             // fragment words per 16 columns (32 lanes x 4)
constexpr int KSTEP_STRIDE = KSTEP_WORDS + 4;                // their stride in S.act (the pad spreads a warp's stores over the banks)

__device__ __forceinline__ void mma16816(float* d, const uint4& a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

// No memory clobber: the ring data it reads is ordered by the (volatile) full-barrier
// wait before and the release after, and the loads of several k-steps may overlap.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// The A-fragment layout of a staged block: per 16 columns (one MMA k-step) 32
// lanes x 4 words (k-steps KSTEP_STRIDE words apart); lane 4b + t holds {hi, lo} of columns 2t, 2t+1 (words 0, 1)
// and of columns 8 + 2t, 8 + 2t + 1 (words 2, 3) of request b.  Request b's hi
// is MMA row b, its lo row 8 + b.  One staging item is one lane's four words:
// the fp32 values (a0, a1) of columns 2t, 2t+1 and (c0, c1) of 8 + 2t, 8 + 2t + 1.
__device__ __forceinline__ uint4 frag_quad(float2 a, float2 c) {
    // packed conversions (two values an instruction); the same roundings as one at a time
    const __half2 ha = __float22half2_rn(a), hc = __float22half2_rn(c);
    const float2 fa = __half22float2(ha), fc = __half22float2(hc);
    const __half2 la = __float22half2_rn(make_float2(a.x - fa.x, a.y - fa.y));
    const __half2 lc = __float22half2_rn(make_float2(c.x - fc.x, c.y - fc.y));
    return make_uint4(*reinterpret_cast<const uint32_t*>(&ha), *reinterpret_cast<const uint32_t*>(&la),
                      *reinterpret_cast<const uint32_t*>(&hc), *reinterpret_cast<const uint32_t*>(&lc));
}

__device__ __forceinline__ float2 ld_relaxed_f2(const float* p) {
    float2 v;
    asm volatile("ld.relaxed.gpu.global.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ bool has_tag2(const float2& v, uint32_t par) {
    return (((__float_as_uint(v.x) ^ par) | (__float_as_uint(v.y) ^ par)) & 1u) == 0u;
}

// Stage columns [k0, k0 + kb) of every request's input vector into S.act as
// MMA fragments (kb a multiple of 64).  scaled: x (tagged with parity par, the
// copy at src, request stride n) or, for the first layer's QKV, the requests'
// embedding rows, times the RMSNorm gains g (staged in S.wsc); the sums of
// squares go to S.red[RED_NORM] (per request and warp: set by the first
// block, added by later ones) and the raw x of rows [cap0, cap0 + ncap) to S.xres (per
// request).  Otherwise: src (o or a, tagged with parity par) as is.
// Every CTA reads every request's vector, so the time goes into round trips
// to L2 under the weight stream's load: all of a block lands with one round of
// asynchronous 16-byte copies (global -> shared, L2 only, no registers held)
// into the fragment area itself, k-step by k-step (request b's 16 columns of
// k-step s in words b*16 .. b*16+15 of its slot).  Then each warp turns its
// k-steps into fragments in place: lane 4b + t reads columns 2t, 2t+1, 8+2t,
// 9+2t of request b (re-polling with relaxed loads if a tag is not there
// yet), and after a warp barrier writes its {hi, lo} words over the slot.
// Ends with a consumer barrier.
__device__ void stage_b(const KieParams& P, const KieLaunch& Lc, const Smem& S, const float* src, int n,
                        bool from_emb, const float* g, bool scaled, uint32_t par, int k0, int kb, bool first_blk,
                        int cap0, int ncap, int tid, int cta) {
    const int warp = tid >> 5, lane = tid & 31, nb = P.nb, nks = kb >> 4;
    uint32_t* act = reinterpret_cast<uint32_t*>(S.act);
    {
        const int q4 = kb >> 2, nq = from_emb ? 0 : nb * q4;   // 16-byte pieces: (request, 4 columns)
        for (int i = tid; i < nq; i += NCT) {
            const int b = i / q4, c4 = i - b * q4;
            cp_async16(act + (c4 >> 2) * KSTEP_STRIDE + b * 16 + (c4 & 3) * 4, src + size_t(b) * n + k0 + 4 * c4);
        }
        if (scaled)   // the block's gains travel in the same round, into S.wsc
            for (int i = tid; i < q4; i += NCT) cp_async16(S.wsc + 4 * i, g + k0 + 4 * i);
        cp_async_wait_all();
        consumer_sync(NCT);
    }
    const int b = lane >> 2, t2 = 2 * (lane & 3);
    const bool live = b < nb;
    float ss = 0.f;
    for (int s = warp; s < nks; s += NW) {
        const int k = k0 + 16 * s + t2;          // this lane's columns: k, k+1, k+8, k+9
        uint32_t* blk = act + s * KSTEP_STRIDE;
        float2 a = make_float2(0.f, 0.f), c = a;
        if (live) {
            if (from_emb) {
                const uint16_t* er = P.emb + size_t(S.clist[b]) * P.d + k;
                a = h2_to_f2(*reinterpret_cast<const uint32_t*>(er));
                c = h2_to_f2(*reinterpret_cast<const uint32_t*>(er + 8));
            } else {
                a = *reinterpret_cast<const float2*>(blk + b * 16 + t2);
                c = *reinterpret_cast<const float2*>(blk + b * 16 + 8 + t2);
                if (!has_tag2(a, par) || !has_tag2(c, par)) {   // not written yet when the copy read it
                    const float* gp = src + size_t(b) * n + k;
                    TagWait w;
                    do {
                        a = ld_relaxed_f2(gp);
                        c = ld_relaxed_f2(gp + 8);
                    } while (!(has_tag2(a, par) && has_tag2(c, par)) && w.again(P, Lc, S, cta));
                }
            }
            if (scaled) {
                ss += (a.x * a.x + a.y * a.y) + (c.x * c.x + c.y * c.y);
                if (ncap > 0) {
                    const float xv[4] = {a.x, a.y, c.x, c.y};
                    const int kk[4] = {k, k + 1, k + 8, k + 9};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (kk[e] >= cap0 && kk[e] < cap0 + ncap) S.xres[b * KIE_XRES + kk[e] - cap0] = xv[e];
                }
                const float2 ga = *reinterpret_cast<const float2*>(S.wsc + (k - k0));
                const float2 gc = *reinterpret_cast<const float2*>(S.wsc + (k - k0) + 8);
                a = make_float2(a.x * ga.x, a.y * ga.y);
                c = make_float2(c.x * gc.x, c.y * gc.y);
            }
        }
        const uint4 fq = frag_quad(a, c);
        __syncwarp();   // every lane has read the slot's fp32 values
        *reinterpret_cast<uint4*>(blk + lane * 4) = fq;
    }
    if (scaled) {   // lanes 4b .. 4b+3 hold request b
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if ((lane & 3) == 0 && live) {
            float* r = S.red + RED_NORM + b * NW + warp;
            *r = first_blk ? ss : *r + ss;
        }
    }
    consumer_sync(NCT);
}

// 1 / sqrt(mean(x_b^2) + eps) of request b's staged x (after the staging's barrier).
__device__ __forceinline__ float rinv_b(const KieParams& P, const Smem& S, int b) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += S.red[RED_NORM + b * NW + w];
    return 1.0f / sqrtf(s / float(P.d) + P.eps);
}

// Warp-uniform wait until the producer has issued global slot gidx (every lane
// acquires the issue count itself).  False on abort or timeout.
__device__ __forceinline__ bool wait_issued(const KieParams& P, const KieLaunch& Lc, const Smem& S, uint32_t gidx,
                                            int cta, int lane) {
    const uint64_t t0 = globaltimer();
    while (true) {
        const bool done = ld_acquire_cta_shared(&S.flags[5]) > int32_t(gidx);
        if (__all_sync(0xffffffffu, done)) return true;
        int bad = 0;
        if (lane == 0) {
            if (ld_volatile_i32(&S.flags[0]) != 0 || ld_volatile_i32(&P.ctl->err) != 0) bad = 1;
            else if (globaltimer() - t0 > Lc.timeout_ns) { set_error(P, KERR_TIMEOUT_FULL, cta); bad = 1; }
        }
        if (__shfl_sync(0xffffffffu, bad, 0)) return false;
    }
}

// One k-step: B fragments of both 8-row groups (ldmatrix.x4 at byte address
// wa), the A fragment of 16 columns, two MMAs into accumulator set d.
__device__ __forceinline__ void kstep(uint32_t wa, const uint4* af, float (*d)[4], int set) {
    uint32_t b00, b01, b10, b11;
    ldsm_x4(wa, b00, b01, b10, b11);
    const uint4 a = *af;
    mma16816(d[set], a, b00, b01);
    mma16816(d[2 + set], a, b10, b11);
}

// The slot's rows_g x kc weights (chunk-major) times the staged fragments of
// its columns (af: this lane's word quad of the slot's first k-step).
// acc[0..1]: row group 0 (even / odd k-steps), acc[2..3]: row group 1.
__device__ __forceinline__ void slot_mma(const uint8_t* slot, int rows_g, int kc, const uint4* af, int lane,
                                         float (*acc)[4]) {
    const int m = lane >> 3;                                   // ldmatrix matrix this lane addresses
    const int row = min(((m >> 1) << 3) + (lane & 7), rows_g - 1);
    const uint32_t base = smem_u32(slot) + uint32_t(((m & 1) * rows_g + row) * 16);
    const uint32_t kstr = uint32_t(rows_g) * 32u;              // bytes per k-step (two 8-column chunks)
    const int nks = kc >> 4;
    int s = 0;
#pragma unroll 4
    for (; s + 1 < nks; s += 2) {
        kstep(base + uint32_t(s) * kstr, af + s * (KSTEP_STRIDE / 4), acc, 0);
        kstep(base + uint32_t(s + 1) * kstr, af + (s + 1) * (KSTEP_STRIDE / 4), acc, 1);
    }
    if (s < nks) kstep(base + uint32_t(s) * kstr, af + s * (KSTEP_STRIDE / 4), acc, 0);
}

struct EpiB {
    int type, layer, t, phi;
    uint32_t n;                 // write number of the layer (tags)
    uint32_t par_in, par_out;   // O, D: parity of the old and the new x
};

// store one element of request b's new K (kv=0) or V (kv=1); returns the stored bits
__device__ __forceinline__ uint32_t kv_store_b(const KieParams& P, int b, int layer, int kv, int h, int pos, int dim,
                                               float v) {
    const __half hv = __float2half_rn(v);
    const size_t idx = size_t(b) * size_t(P.kv_req) + kv_elem_index(P, layer, h, pos) + dim;
    uint8_t* base = kv ? P.vc : P.kc;
    if (P.kv == KV_E5M2) {
        const uint32_t e = f16x2_to_e5m2x2(hv, hv) & 0xFFu;
        base[idx] = uint8_t(e);
        return e;
    }
    reinterpret_cast<__half*>(base)[idx] = hv;
    return __half_as_ushort(hv);
}

// Unit u (local) of the QKV phase for request b (see qkv_unit).
__device__ __forceinline__ void qkv_unit_b(const KieParams& P, const Smem& S, const Cursor& c, const EpiB& e, int b,
                                           int u, float ya, float yb) {
    const int hh = P.hd / 2, lhh = P.hd == 128 ? 6 : 5;
    const int per = P.H * hh;
    const uint32_t par = tag_par(e.n), ep16 = tag_ep16(e.n);
    const int U = c.unit0 + u;
    const int which = (U >= per) + (U >= 2 * per), rem = U - which * per;
    const int h = rem >> lhh, i = rem & (hh - 1);
    const int pos = S.flags[8 + b] + e.t;
    const int e0 = (b * P.H + h) * P.hd + i;
    if (which == 2) {
        const uint32_t b0 = kv_store_b(P, b, e.layer, 1, h, pos, i, ya), b1 = kv_store_b(P, b, e.layer, 1, h, pos, i + hh, yb);
        st_relaxed_u32(P.vcur + e0, (b0 << 16) | ep16);
        st_relaxed_u32(P.vcur + e0 + hh, (b1 << 16) | ep16);
        return;
    }
    const float* rope = S.rope + b * KIE_MAX_HEAD_DIM;
    const float cs = rope[i], sn = rope[hh + i];
    const float ra = ya * cs - yb * sn, rb = yb * cs + ya * sn;
    if (which == 0) {
        st_relaxed_f32(P.q + e0, tag_f32(ra, par));
        st_relaxed_f32(P.q + e0 + hh, tag_f32(rb, par));
    } else {
        const uint32_t b0 = kv_store_b(P, b, e.layer, 0, h, pos, i, ra), b1 = kv_store_b(P, b, e.layer, 0, h, pos, i + hh, rb);
        st_relaxed_u32(P.kcur + e0, (b0 << 16) | ep16);
        st_relaxed_u32(P.kcur + e0 + hh, (b1 << 16) | ep16);
    }
}

// Row r (local) of the O or D phase for request b: x_b[row] += y (see residual_row).
__device__ __forceinline__ void residual_b(const KieParams& P, const KieLaunch& Lc, const Smem& S, const Cursor& c,
                                           const EpiB& e, int b, int r, float y, int cta) {
    const int row = c.unit0 + r;
    float xo;
    if (c.rows <= KIE_XRES) xo = S.xres[b * KIE_XRES + r];
    else if (e.type == PH_O && e.layer == 0) xo = __half2float(__ushort_as_half(P.emb[size_t(S.clist[b]) * P.d + row]));
    else xo = wait_f32(P, Lc, S, P.x + size_t(b) * P.d + row, e.par_in, cta);
    const float xn = tag_f32(xo + y, e.par_out);
#pragma unroll
    for (int k = 0; k < KIE_REPL; ++k) st_relaxed_f32(P.x + (size_t(k) * P.nb + b) * P.d + row, xn);
}

// LM logits of one row for request b: written out, and folded into the lane's running argmax.
__device__ __forceinline__ void lm_row_b(const KieParams& P, const KieLaunch& Lc, const Cursor& c, int b, int r,
                                         float y, int step, float& bv, int& bi) {
    const int row = c.unit0 + r;
    if (Lc.out_logits) Lc.out_logits[(size_t(step - Lc.lm_from_step) * P.nb + b) * P.V + row] = y;
    if (y > bv || (y == bv && row < bi)) { bv = y; bi = row; }
}

// The epilogue of one lane's results for row tile `tile`: request gq's outputs
// y of rows 2tq, 2tq+1, 8+2tq, 8+2tq+1 of the tile.
__device__ __forceinline__ void epi_lane_b(const KieParams& P, const KieLaunch& Lc, const Smem& S, const Cursor& c,
                                           const EpiB& e, int tile, int lane, const float* y, float& bv, int& bi,
                                           int cta) {
    const int gq = lane >> 2, tq = lane & 3;
    if (gq >= P.nb) return;
    const int rA = tile * KIE_RB + 2 * tq, rB = rA + 8;   // first rows of this lane's two pairs
    if (e.type == PH_QKV || e.type == PH_GU) {
        const float ri = rinv_b(P, S, gq);
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int r = p ? rB : rA;
            if (r < c.rows) {
                const float ya = y[2 * p] * ri, yb = y[2 * p + 1] * ri;
                if (e.type == PH_QKV) qkv_unit_b(P, S, c, e, gq, r >> 1, ya, yb);
                else {
                    const float av = tag_f32((ya / (1.f + expf(-ya))) * yb, tag_par(e.n));
#pragma unroll
                    for (int k = 0; k < KIE_REPL; ++k)
                        st_relaxed_f32(P.a + (size_t(k) * P.nb + gq) * P.F + c.unit0 + (r >> 1), av);
                }
            }
        }
    } else if (e.type == PH_LM) {
        const float ri = rinv_b(P, S, gq);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = (i < 2 ? rA : rB) + (i & 1);
            if (r < c.rows) lm_row_b(P, Lc, c, gq, r, y[i] * ri, e.t, bv, bi);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = (i < 2 ? rA : rB) + (i & 1);
            if (r < c.rows) residual_b(P, Lc, S, c, e, gq, r, y[i], cta);
        }
    }
}

// request lane/4's sums of rows 2(lane%4), +1 (group 0) and 8+2(lane%4), +1
// (group 1) of a tile: hi + lo of the even and odd k-step accumulators
__device__ __forceinline__ void tile_sums(const float (*acc)[4], float* y) {
    y[0] = (acc[0][0] + acc[1][0]) + (acc[0][2] + acc[1][2]);
    y[1] = (acc[0][1] + acc[1][1]) + (acc[0][3] + acc[1][3]);
    y[2] = (acc[2][0] + acc[3][0]) + (acc[2][2] + acc[3][2]);
    y[3] = (acc[2][1] + acc[3][1]) + (acc[2][3] + acc[3][3]);
}

// One GEMV phase of the batched kernel: staging block by block, the row tiles
// on the tensor cores, the epilogue in the lanes holding the results.
// A phase with at least NW row tiles gives each warp whole tiles (all chunks
// of a tile accumulate in its registers).  One with fewer (the QKV, O and
// down projections' 1-3 tiles a CTA) spreads its (tile, chunk) slots over the
// warps in slot order; each slot's sums go to S.part and the tile's warp adds
// them up in chunk order after the block.  Running sums of a phase staged in
// several blocks stay in S.part as well.  Returns false on abort.
__device__ bool run_phase_b(const KieParams& P, const KieLaunch& Lc, const Smem& S, const Cursor& c, uint32_t& gc,
                            const EpiB& e, const float* src, int n, bool from_emb, const float* g, bool scaled,
                            uint32_t par_src, int cap0, int ncap, int warp, int lane, int tid, int cta) {
    const int nblk = (c.K + KIE_KBLK - 1) / KIE_KBLK, ntiles = (c.rows + KIE_RB - 1) / KIE_RB;
    const int cpb = KIE_KBLK / KIE_KCB;
    const bool split = ntiles < NW;
    const uint32_t nslot = uint32_t(P.nslot);
    const int tq = lane & 3;
    float* run = S.part;                             // [ntiles][128] running sums over blocks
    float* sp = S.part + (nblk > 1 ? ntiles : 0) * 128;   // split: [ntiles][cpb][128] per-slot sums
    float bv = -INFINITY;   // LM: this lane's argmax for request lane / 4
    int bi = 0x7fffffff;
    bool ok = true;
    uint32_t jbase = 0;
    (void)tq;
    for (int blk = 0; blk < nblk; ++blk) {
        const int k0 = blk * KIE_KBLK, kb = min(KIE_KBLK, c.K - k0);
        const int nch = (kb + c.KC - 1) / c.KC;
        const bool last = blk == nblk - 1;
        // Every warp runs every block's barriers, also after a failed wait (the
        // waits then return at once), so the barrier counts always match.
        if (blk > 0) consumer_sync(NCT);   // every warp is done with the previous block's fragments
        stage_b(P, Lc, S, src, n, from_emb, g, scaled, par_src, k0, kb, blk == 0, cap0, ncap, tid, cta);
        if (tid == 0 && blk == 0) stamp(P, Lc, e.t, e.phi, 1, cta);
        const int nsl = ntiles * nch;
        for (int j = split ? warp : warp * nch; ok && j < nsl; j += split ? NW : NW * nch) {
            const int tile = j / nch;
            const int rows_g = min(KIE_RB, c.rows - tile * KIE_RB);
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[a][q] = 0.f;
            for (int ch = j % nch; ch < (split ? j % nch + 1 : nch); ++ch) {
                const uint32_t gidx = gc + jbase + uint32_t(tile * nch + ch);
                if (!wait_issued(P, Lc, S, gidx, cta, lane) || !warp_wait_full(P, Lc, S, gidx, cta, lane)) {
                    ok = false;
                    S.flags[0] = 1;
                    break;
                }
                const uint32_t slot = gidx % nslot;
                if (lane == 0) slot_stamp(Lc, cta, gidx, 1);
                const int kc = min(c.KC, kb - ch * c.KC);
                const uint4* af = reinterpret_cast<const uint4*>(S.act) + (ch * (c.KC >> 4)) * (KSTEP_STRIDE / 4) + lane;
                slot_mma(S.ring + size_t(slot) * KIE_SLOT_BYTES, rows_g, kc, af, lane, acc);
                __syncwarp();
                if (lane == 0) {
                    slot_stamp(Lc, cta, gidx, 2);
                    mbar_arrive_cnt(&S.empty[slot], NW);
                }
            }
            if (!ok) break;
            float y[4];
            tile_sums(acc, y);
            if (split) {   // this slot's sums; the tile's warp adds the block up below
                float* pw = sp + ((tile * cpb) + j % nch) * 128 + lane * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i) pw[i] = y[i];
                continue;
            }
            if (nblk > 1) {   // blocks add up in this lane's own words
                float* pw = run + tile * 128 + lane * 4;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    y[i] = blk == 0 ? y[i] : pw[i] + y[i];
                    pw[i] = y[i];
                }
            }
            if (last) epi_lane_b(P, Lc, S, c, e, tile, lane, y, bv, bi, cta);
        }
        jbase += uint32_t(ntiles * nch);
        if (split) {
            consumer_sync(NCT);   // every slot's sums are in
            for (int tile = warp; tile < ntiles; tile += NW) {
                float y[4] = {0.f, 0.f, 0.f, 0.f};
                for (int ch = 0; ch < nch; ++ch) {
                    const float* pw = sp + ((tile * cpb) + ch) * 128 + lane * 4;
#pragma unroll
                    for (int i = 0; i < 4; ++i) y[i] += pw[i];
                }
                if (nblk > 1) {
                    float* pw = run + tile * 128 + lane * 4;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        y[i] = blk == 0 ? y[i] : pw[i] + y[i];
                        pw[i] = y[i];
                    }
                }
                if (last && ld_volatile_i32(&S.flags[0]) == 0) epi_lane_b(P, Lc, S, c, e, tile, lane, y, bv, bi, cta);
            }
        }
    }
    gc += c.nslots;
    if (!ok) S.flags[0] = 1;
    if (e.type == PH_LM) {   // the warp's argmax per request: lanes 4b..4b+3 hold request b
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if ((lane & 3) == 0) {
            S.red[RED_AMV + warp * NB + (lane >> 2)] = bv;
            reinterpret_cast<int*>(S.red)[RED_AMI + warp * NB + (lane >> 2)] = bi;
        }
    }
    consumer_sync(NCT);
    return ld_volatile_i32(&S.flags[0]) == 0;
}

// LM argmax over the grid, per request (lowest index on ties): this CTA's best
// per request into amax_val/idx [nb][G]; the last CTA to arrive reduces them,
// sets each request's next token and position and clears the arrival count.
__device__ void lm_reduce_b(const KieParams& P, const KieLaunch& Lc, const Smem& S, int cta, int tid, int step) {
    const int nb = P.nb, warp = tid >> 5, lane = tid & 31;
    const int* ridx = reinterpret_cast<const int*>(S.red);
    if (tid < nb) {
        float best = -INFINITY;
        int bidx = 0x7fffffff;
        for (int w = 0; w < NW; ++w) {
            const float v = S.red[RED_AMV + w * NB + tid];
            const int ix = ridx[RED_AMI + w * NB + tid];
            if (v > best || (v == best && ix < bidx)) { best = v; bidx = ix; }
        }
        P.amax_val[tid * P.G + cta] = best;
        P.amax_idx[tid * P.G + cta] = bidx;
        __threadfence();
    }
    consumer_sync(NCT);
    if (tid == 0) {
        const uint32_t old = atomicAdd(&P.ctl->amax_cnt, 1u);
        S.flags[1] = (old == uint32_t(P.G) - 1u) ? 1 : 0;
    }
    consumer_sync(NCT);
    if (!S.flags[1]) return;
    __threadfence();
    for (int b = warp; b < nb; b += NW) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = lane; i < P.G; i += 32) {
            const float v = __ldcg(P.amax_val + b * P.G + i);
            const int ix = __ldcg(P.amax_idx + b * P.G + i);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) {
            if (bi < 0 || bi >= P.V) bi = 0;   // all logits NaN: keep a valid id
            P.req_tok[b] = bi;
            P.req_pos[b] = S.flags[8 + b] + step + 1;
            if (Lc.out_tokens) Lc.out_tokens[size_t(step) * nb + b] = bi;
        }
    }
    consumer_sync(NCT);
    if (tid == 0) {
        P.ctl->amax_cnt = 0u;
        __threadfence();
    }
}

template <int HD, int KVF>
__device__ void consumer_b(const KieParams& P, const KieLaunch& Lc, const Smem& S, int cta, int warp, int lane) {
    const int tid = warp * 32 + lane, nb = P.nb;
    uint32_t gc = 0, nbar = 0;
    // fragments of requests >= nb stay zero
    for (int i = tid; i < P.act_floats; i += NCT) S.act[i] = 0.f;
    consumer_sync(NCT);
    for (int t = 0; t < Lc.n_steps; ++t) {
        for (int phi = Lc.phase_begin; phi < Lc.phase_end; ++phi) {
            int layer, sub;
            phase_of(phi, P.L, layer, sub);
            if (sub == 5 && t < Lc.lm_from_step) continue;
            if (Lc.use_grid_barrier && (t > 0 || phi > Lc.phase_begin) && layer == 0 && sub == 0) {
                fence_proxy_async_global();
                if (!grid_barrier(P, Lc, S, nbar, tid, cta)) return;
            }
            if (tid == 0) {
                st_release_cta_shared(&S.flags[4], t * (Lc.phase_end - Lc.phase_begin) + (phi - Lc.phase_begin));
                stamp(P, Lc, t, phi, 0, cta);
            }
            // writes are numbered by request 0's position (all requests advance together)
            const uint32_t tn = tag_seq(P, S.flags[8] + t, layer), par = tag_par(tn);
            if (sub == 1) {
                if (tid == 0) stamp(P, Lc, t, phi, 1, cta);
                if (!attention<HD, KVF, true>(P, Lc, S, layer, 0, tn, cta, gc, warp, lane, tid, t)) return;
                if (tid == 0) stamp(P, Lc, t, phi, 2, cta);
                if (tid == 0) stamp(P, Lc, t, phi, 3, cta);
                continue;
            }
            const int type = sub == 0 ? PH_QKV : sub == 2 ? PH_O : sub == 3 ? PH_GU : sub == 4 ? PH_D : PH_LM;
            const Cursor c = cursor(P, S, type);
            if (layer == 0 && type == PH_QKV) {   // the step's input tokens
                if (tid < nb) {
                    int tk = __ldcg(P.req_tok + tid);
                    if (tk < 0 || tk >= P.V) { set_error(P, KERR_BAD_TOKEN, tk); tk = 0; }
                    S.clist[tid] = tk;
                }
                consumer_sync(NCT);
            }
            if (type == PH_QKV) {   // cos / sin of every request's position
                const int hh = P.hd / 2;
                for (int i = tid; i < nb * hh; i += NCT) {
                    const int b = i / hh, k = i - b * hh;
                    float sn, cs;
                    sincosf(float(S.flags[8 + b] + t) * P.inv_freq[k], &sn, &cs);
                    S.rope[b * KIE_MAX_HEAD_DIM + k] = cs;
                    S.rope[b * KIE_MAX_HEAD_DIM + hh + k] = sn;
                }
            }
            EpiB e;
            e.type = type;
            e.layer = layer;
            e.t = t;
            e.phi = phi;
            e.n = tn;
            e.par_in = type == PH_O ? 0u : 1u;
            e.par_out = type == PH_O ? 1u : 0u;
            const int rep = cta % KIE_REPL;
            bool ok;
            if (type == PH_O || type == PH_D) {
                const int n = type == PH_O ? P.H * P.hd : P.F;
                const float* s = (type == PH_O ? P.o : P.a) + size_t(rep) * nb * n;
                ok = run_phase_b(P, Lc, S, c, gc, e, s, n, false, nullptr, false, par, 0, 0, warp, lane, tid, cta);
            } else {
                const bool from_emb = type == PH_QKV && layer == 0;
                const float* gains = type == PH_LM ? P.norms + size_t(P.L) * 2 * P.d
                                                   : P.norms + size_t(layer) * 2 * P.d + (type == PH_GU ? P.d : 0);
                int cap0 = 0, ncap = 0;
                if (type != PH_LM) {
                    const int rt = type == PH_QKV ? PH_O : PH_D;
                    cap0 = S.plan[rt * 4 + 0];
                    ncap = S.plan[rt * 4 + 1] <= KIE_XRES ? S.plan[rt * 4 + 1] : 0;
                }
                ok = run_phase_b(P, Lc, S, c, gc, e, P.x + size_t(rep) * nb * P.d, P.d, from_emb, gains, true,
                                 type == PH_GU ? 1u : 0u, cap0, ncap, warp, lane, tid, cta);
            }
            if (!ok) return;
            if (tid == 0) stamp(P, Lc, t, phi, 2, cta);
            if (type == PH_LM) lm_reduce_b(P, Lc, S, cta, tid, t);
            if (tid == 0) stamp(P, Lc, t, phi, 3, cta);
        }
    }
}

}  // namespace

template <int HD, int KVF>
__global__ void __launch_bounds__(KIE_THREADS, 1) kie_decode_batch_kernel(const KieParams P, const KieLaunch Lc) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    if (kie_smem_layout(P.part_floats, P.act_floats, P.nslot, P.nb).total > dynamic_smem_size() ||
        P.nslot < NW || P.nslot > KIE_MAX_SLOTS || P.G > KIE_MAX_GRID || P.nb < 1 || P.nb > KIE_MAX_BATCH ||
        P.nb * P.H > P.G || P.act_floats < (KIE_KBLK / 16) * KSTEP_STRIDE) {
        if (threadIdx.x == 0) set_error(P, KERR_SMEM, cta);
        return;
    }
    const Smem S = carve<true>(smem_raw, P);
    if (threadIdx.x == 0) {
        for (int i = 0; i < P.nslot; ++i) {
            mbar_init(&S.full[2 * i], 1);
            mbar_init(&S.full[2 * i + 1], 1);
            mbar_init(&S.empty[i], NW);
        }
        S.flags[0] = 0;
        S.flags[1] = 0;
        S.flags[4] = -1;
        S.flags[5] = 0;
        for (int b = 0; b < P.nb; ++b) S.flags[8 + b] = P.req_pos[b];
        for (int t = 0; t < PH_NTYPES; ++t) {
            S.plan[t * 4 + 0] = P.ph[t].unit_begin[cta];
            S.plan[t * 4 + 1] = P.ph[t].unit_begin[cta + 1] - P.ph[t].unit_begin[cta];
            S.plan[t * 4 + 2] = int32_t(P.ph[t].nslots[cta]);
            S.plan[t * 4 + 3] = int32_t(P.ph[t].bytes[cta]);
        }
        S.cbase[0] = P.cta_base[cta];
        S.cbase[1] = P.cta_layer[cta];
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == NW) {
        if (lane == 0) producer<true>(P, Lc, S, cta);
    } else {
        consumer_b<HD, KVF>(P, Lc, S, cta, warp, lane);
    }
}

// Rewrite every weight slot of the batched stream from row-major ([row][kc]
// fp16) to chunk-major ([kc/8][row][8] fp16).  table: per slot {byte offset
// (low, high 32 bits), rows, kc}; one CTA per slot.
__global__ void kie_slot_chunk_major_kernel(uint8_t* stream, const uint4* table, int nslots) {
    __shared__ uint4 buf[KIE_SLOT_BYTES / 16];
    const int i = blockIdx.x;
    if (i >= nslots) return;
    const uint4 d = table[i];
    uint4* p = reinterpret_cast<uint4*>(stream + ((uint64_t(d.y) << 32) | d.x));
    const int rows = int(d.z), nc = int(d.w) / 8, n = rows * nc;
    if (n * 16 > KIE_SLOT_BYTES) return;
    for (int k = threadIdx.x; k < n; k += blockDim.x) buf[k] = p[k];
    __syncthreads();
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        const int j = k / rows, r = k - j * rows;   // destination: chunk j, row r
        p[k] = buf[r * nc + j];
    }
}

#include <cuda_runtime.h>

extern "C" void* kie_decode_batch_kernel_ptr(int hd, int kv) {
    if (hd == 128) {
        if (kv == KV_F16) return (void*)&kie_decode_batch_kernel<128, KV_F16>;
        if (kv == KV_E5M2) return (void*)&kie_decode_batch_kernel<128, KV_E5M2>;
    }
    if (hd == 64) {
        if (kv == KV_F16) return (void*)&kie_decode_batch_kernel<64, KV_F16>;
        if (kv == KV_E5M2) return (void*)&kie_decode_batch_kernel<64, KV_E5M2>;
    }
    return nullptr;
}

extern "C" cudaError_t kie_launch_slot_chunk_major(uint8_t* stream, const uint4* table, int nslots, cudaStream_t st) {
    if (nslots <= 0) return cudaSuccess;
    kie_slot_chunk_major_kernel<<<nslots, 256, 0, st>>>(stream, table, nslots);
    return cudaGetLastError();
}
