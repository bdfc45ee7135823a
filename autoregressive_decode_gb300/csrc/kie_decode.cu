// The decode program: one kernel that runs a range of phases of one or more
// decode steps.  Persistent mode launches it once (cooperatively, one CTA per
// SM) for all steps, with grid-wide barriers between phases; graph mode
// launches it once per phase inside a CUDA graph.  Both run the same code with
// the same partitioning, so they produce bit-identical results.
//
// Design (Kog page, table "Where standard inference stacks lose microseconds"):
//  - row "kernel boundaries": one resident program for the whole decode path;
//  - row "CPU scheduling and sampling": LM head and argmax on the GPU, the next
//    token fed back without the host;
//  - row "grid synchronization": grid barriers are a single gpu-scope counter
//    with acquire/release, every wait bounded by %globaltimer;
//  - rows "weight reloading" and "non-GEMM work": each CTA's weights for the
//    whole step are one contiguous stream that a producer warp copies into a
//    shared-memory ring with bulk async copies, independently of the
//    activations, so HBM keeps streaming while consumers wait at barriers,
//    normalise, do attention or reduce (beta == 1: every weight byte is read
//    exactly once per token).
#include "kie_decode_core.cuh"

using namespace kie;

namespace {

template <int HD, int KVF>
__device__ void consumer(const KieParams& P, const KieLaunch& Lc, const Smem& S, int cta, int warp, int lane) {
    const int tid = warp * 32 + lane;
    uint32_t gc = 0, nbar = 0;
    const int pos0 = Lc.pos0 >= 0 ? Lc.pos0 : ld_volatile_i32(&P.ctl->pos);
    bool first_phase = true;
    int tok = 0;
    for (int t = 0; t < Lc.n_steps; ++t) {
        const int pos = pos0 + t;
        for (int phi = Lc.phase_begin; phi < Lc.phase_end; ++phi) {
            int layer, sub;
            phase_of(phi, P.L, layer, sub);
            if (sub == 5 && t < Lc.lm_from_step) continue;
            // One grid barrier per step, before its first phase: it publishes
            // the previous step's token and its K/V cache writes (read by this
            // step's bulk copies).  Inside a step the tags order everything.
            if (Lc.use_grid_barrier && !first_phase && layer == 0 && sub == 0) {
                // the K/V this thread wrote into the cache during the step are read
                // by the next steps' bulk copies (the async proxy): one proxy fence
                // per step, before the barrier that publishes them
                fence_proxy_async_global();
                if (!grid_barrier(P, Lc, S, nbar, tid, cta)) return;
            }
            first_phase = false;
            if (tid == 0) {
                st_release_cta_shared(&S.flags[4], t * (Lc.phase_end - Lc.phase_begin) + (phi - Lc.phase_begin));
                stamp(P, Lc, t, phi, 0, cta);
            }
            const uint32_t tn = tag_seq(P, pos, layer), par = tag_par(tn);
            const float* gains = P.norms + size_t(layer) * 2 * P.d;
            if (sub == 1) {
                if (tid == 0) stamp(P, Lc, t, phi, 1, cta);
                if (!attention<HD, KVF>(P, Lc, S, layer, pos, tn, cta, gc, warp, lane, tid)) return;
                if (tid == 0) stamp(P, Lc, t, phi, 2, cta);
            } else {
                // One call site each for the activation staging, the GEMV and
                // every epilogue: the phases share their instructions, which
                // keeps the per-layer instruction working set small.
                const int type = sub == 0 ? PH_QKV : sub == 2 ? PH_O : sub == 3 ? PH_GU : sub == 4 ? PH_D : PH_LM;
                const Cursor c = cursor(P, S, type);
                if (c.wfmt == WF_F8 || c.wfmt == WF_F4) {   // this CTA's row scales, visible after the staging's barrier
                    const KiePhasePlan& pp = P.ph[type];
                    const float* ws = pp.wscale + (type == PH_LM ? 0 : int64_t(layer) * pp.wscale_layer) +
                                      int64_t(c.unit0) * c.rpu;
                    for (int r = tid; r < c.rows; r += NCT) S.wsc[r] = __ldg(ws + r);
                }
                if (c.nK > 1) {   // chunk counters of the row groups, zero after the staging's barrier
                    for (int i = tid; i * c.R < c.rows; i += NCT) S.cnt[i] = 0;
                }
                // the step's input token: read by the first layer's QKV phase,
                // and again by its O phase when that phase starts a launch
                if (layer == 0 && (type == PH_QKV || (type == PH_O && phi == Lc.phase_begin))) {
                    if (tid == 0) {
                        int tk = (t == 0 && Lc.first_tok >= 0) ? Lc.first_tok
                                 : (Lc.forced ? Lc.forced[t] : __ldcg(&P.ctl->tok));
                        if (tk < 0 || tk >= P.V) { set_error(P, KERR_BAD_TOKEN, tk); tk = 0; }
                        S.flags[2] = tk;
                    }
                    consumer_sync(NCT);
                    tok = S.flags[2];
                }
                const uint16_t* erow = P.emb + size_t(tok) * P.d;   // the residual stream before layer 0
                if (type == PH_O || type == PH_D) {
                    // o and a carry this layer's parity
                    // every reader polls the copy its CTA index selects (copies spread the
                    // all-CTA polling of one vector over more L2 lines)
                    const int rep = cta % KIE_REPL;
                    act_copy(P, Lc, S, type == PH_O ? P.o + rep * P.H * P.hd : P.a + rep * P.F,
                             type == PH_O ? P.H * P.hd : P.F, par, tid, cta);
                } else {
                    // x: parity 0 after a D epilogue (QKV, LM), 1 after an O epilogue (GU)
                    const bool from_emb = type == PH_QKV && layer == 0;
                    const float* g = type == PH_QKV ? gains : type == PH_GU ? gains + P.d
                                                                             : P.norms + size_t(P.L) * 2 * P.d;
                    if (type == PH_QKV) rope_table(P, S, pos, tid);
                    // scaled E5M2 cache: the K and V scales this position is stored with
                    // (visible to the epilogues after the staging's barrier)
                    if (P.kv == KV_E5M2S && type == PH_QKV && tid < 2) S.red[KVS_SLOT + tid] = slice_scale(P, layer, tid, pos);
                    // keep the raw x of the rows the next residual epilogue (O after
                    // QKV, D after GU) updates
                    int cap0 = 0, ncap = 0;
                    if (type != PH_LM) {
                        const int rt = type == PH_QKV ? PH_O : PH_D;
                        cap0 = S.plan[rt * 4 + 0];
                        ncap = S.plan[rt * 4 + 1] <= KIE_XRES ? S.plan[rt * 4 + 1] : 0;
                    }
                    act_scaled(P, Lc, S, from_emb ? nullptr : P.x + (cta % KIE_REPL) * P.d, from_emb ? erow : nullptr, g,
                               type == PH_GU ? 1u : 0u, tid, cta, cap0, ncap);
                }
                if (tid == 0) stamp(P, Lc, t, phi, 1, cta);
                EpiArgs ea;
                ea.type = type;
                ea.layer = layer;
                ea.pos = pos;
                ea.n = tn;
                ea.rinv = (type == PH_QKV || type == PH_GU) ? 1.0f / norm_r(P, S) : 1.f;
                ea.erow = (type == PH_O && layer == 0) ? erow : nullptr;
                ea.par_in = type == PH_O ? 0u : 1u;    // x: 0 after a D epilogue, 1 after an O epilogue
                ea.par_out = type == PH_O ? 1u : 0u;
                // the staging that kept the old x (QKV for O, GU for D) ran in this launch
                ea.have_xres = type == PH_O ? phi - 2 >= Lc.phase_begin : phi - 1 >= Lc.phase_begin;
                if (!run_gemv(P, Lc, S, c, gc, ea, warp, lane, cta)) return;
                if (tid == 0) stamp(P, Lc, t, phi, 2, cta);
                if (type == PH_LM) epi_lm(P, Lc, S, c, cta, tid, t, pos);
            }
            if (tid == 0) stamp(P, Lc, t, phi, 3, cta);
        }
    }
}

}  // namespace

template <int HD, int KVF>
__global__ void __launch_bounds__(KIE_THREADS, 1) kie_decode_kernel(const KieParams P, const KieLaunch Lc) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    // Refuse to run if the launch gave less shared memory than the layout needs
    // (uniform across the block, before any shared-memory access).
    if (kie_smem_layout(P.part_floats, P.act_floats, P.nslot).total > dynamic_smem_size() ||
        P.nslot < 1 || P.nslot > KIE_MAX_SLOTS || P.G > KIE_MAX_GRID) {
        if (threadIdx.x == 0) set_error(P, KERR_SMEM, cta);
        return;
    }
    const Smem S = carve(smem_raw, P);
    if (threadIdx.x == 0) {
        for (int i = 0; i < P.nslot; ++i) {
            mbar_init(&S.full[2 * i], 1);
            mbar_init(&S.full[2 * i + 1], 1);
            mbar_init(&S.empty[i], NW);   // a slot's user arrives with NW, or each warp of a shared slot with 1
        }
        S.flags[0] = 0;
        S.flags[1] = 0;
        S.flags[4] = -1;
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
        if (lane == 0) producer<false>(P, Lc, S, cta);
    } else {
        consumer<HD, KVF>(P, Lc, S, cta, warp, lane);
    }
}

// Set the control block from launch parameters (no host staging buffer involved).
__global__ void kie_ctl_kernel(KieControl* c, int tok, int pos, int clear) {
    c->tok = tok;
    c->pos = pos;
    if (clear) {
        c->bar = 0u;
        c->err = 0;
        c->err_info = 0;
        c->amax_cnt = 0u;
    }
}

// Copy a device error recorded in one control block into another (first error wins).
__global__ void kie_err_merge_kernel(const KieControl* src, KieControl* dst) {
    if (src->err != 0 && dst->err == 0) {
        dst->err = src->err;
        dst->err_info = src->err_info;
    }
}

// host-visible launch helpers -----------------------------------------------------------------
#include <cuda_runtime.h>

extern "C" cudaError_t kie_launch_err_merge(const KieControl* src, KieControl* dst, cudaStream_t st) {
    kie_err_merge_kernel<<<1, 1, 0, st>>>(src, dst);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_ctl(KieControl* c, int tok, int pos, int clear, cudaStream_t st) {
    kie_ctl_kernel<<<1, 1, 0, st>>>(c, tok, pos, clear);
    return cudaGetLastError();
}

typedef void (*kie_kernel_t)(const KieParams, const KieLaunch);

extern "C" void* kie_decode_kernel_ptr(int hd, int kv) {
    if (hd == 128) {
        if (kv == KV_F16) return (void*)&kie_decode_kernel<128, KV_F16>;
        if (kv == KV_E5M2) return (void*)&kie_decode_kernel<128, KV_E5M2>;
        if (kv == KV_E5M2S) return (void*)&kie_decode_kernel<128, KV_E5M2S>;
        return (void*)&kie_decode_kernel<128, KV_U8>;
    }
    if (hd == 64) {
        if (kv == KV_F16) return (void*)&kie_decode_kernel<64, KV_F16>;
        if (kv == KV_E5M2) return (void*)&kie_decode_kernel<64, KV_E5M2>;
        if (kv == KV_E5M2S) return (void*)&kie_decode_kernel<64, KV_E5M2S>;
        return (void*)&kie_decode_kernel<64, KV_U8>;
    }
    return nullptr;
}
