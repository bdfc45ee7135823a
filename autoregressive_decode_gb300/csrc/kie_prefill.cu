// Prompt prefill on the tensor cores: the whole prompt goes
// through each layer as [T x K] GEMMs instead of T single-token decode steps.
//
//   per layer:  u = RMSNorm(x) g1             kie_pf_norm_split   (fp32 -> fp16 hi + lo tiles)
//               [q k v] = u Wqkv^T            kie_pf_gemm         (tcgen05, fp32 accumulate in TMEM)
//               RoPE q, k; store k, v         kie_pf_qkv_post     (cache in its storage format)
//               o = causal softmax(q k^T) v   kie_pf_attention    (tcgen05; reads the stored K/V, as decode does)
//               x += o Wo^T                   kie_pf_split, kie_pf_gemm, kie_pf_residual
//               u = RMSNorm(x) g2             kie_pf_norm_split
//               [g u] = u Wgu^T               kie_pf_gemm
//               x += (silu(g) u) Wd^T         kie_pf_swiglu_split, kie_pf_gemm, kie_pf_residual
//   last row:   logits = RMSNorm(x) gf Wlm^T  kie_pf_norm_split (one row), kie_pf_gemm
//
// Operands.  The MMA takes fp16; activations are fp32 in this path (as in the
// decode kernel), so every activation a is split into hi = fp16(a) and
// lo = fp16(a - hi) and each K step issues two MMAs, A_hi W^T + A_lo W^T, into
// the same fp32 accumulator: the product then carries a's full precision up to
// 2^-22 relative, well inside the fp32 reference's tolerance.  Weights are fp16
// as given; FP8 E4M3 weights enter the MMA as their exact fp16 values and
// their per-row scale multiplies the output column in the epilogue.
//
// Tile layout.  Both operands are stored in global memory already in the
// tensor cores' canonical no-swizzle K-major layout, tile by tile (tiles of
// 128 rows for activations, 256 rows for weights, 64 columns of K), so one
// plain bulk copy moves a tile into shared memory: element (r, k) of a tile
// sits at byte (r/8)*1024 + (k/8)*128 + (r%8)*16 + (k%8)*2, i.e. 8-row x
// 16-byte core matrices, 128 bytes apart along K and 1024 bytes apart along
// rows; tile (rb, kb) starts at element (rb * KB + kb) * rows * 64.
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "kie_device.cuh"
#include "kie_internal.h"

using namespace kie;

namespace {

// Output tiles of BM x BN.  Weights are packed in tiles of WT = 256 rows; a
// 128-column output tile reads one half of a weight tile (its rows 0-127 or
// 128-255 are 16 KB apart in the canonical layout).  BN = 256 (the default)
// runs one CTA per SM with 3 stages of 64 KB; BN = 128 two CTAs per SM with 2
// stages of 48 KB each, overlapping one CTA's epilogue with the other's MMAs,
// and measured slower.
constexpr int BM = 128, BN = KIE_PF_BN, BK = 64, WT = 256;
constexpr int STAGES = BN == 256 ? 3 : 2, GEMM_CTAS_PER_SM = BN == 256 ? 1 : 2;
static_assert(BN == 128 || BN == 256, "output tile width");
constexpr uint32_t A_BYTES = BM * BK * 2;                 // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;                 // 16 or 32 KB
constexpr uint32_t STAGE_BYTES = 2 * A_BYTES + B_BYTES;   // A hi, A lo, B
constexpr uint32_t GEMM_SMEM = STAGES * STAGE_BYTES + 256;

__device__ __forceinline__ size_t tile_idx(int r, int k, int rows, int KB) {
    return (size_t(r / rows) * KB + (k >> 6)) * size_t(rows) * 64 + size_t((r % rows) >> 3) * 512 +
           size_t((k & 63) >> 3) * 64 + size_t(r & 7) * 8 + size_t(k & 7);
}

__device__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, int* err) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (ld_volatile_i32(err) != 0) return false;
        if (globaltimer() - t0 > timeout_ns) { atomicExch(err, 1); return false; }
    }
    return true;
}

// C[m, n] = sum_k (Ahi + Alo)[m, k] W[n, k] for one 128 x 256 tile of C.
// Thread 0 streams the K tiles (3-stage ring), thread 32 issues the MMAs, all
// four warps then move their 32 TMEM lanes (rows) to C.  Rows >= m_valid are
// not stored.  Split K (gridDim.z = s > 1): CTA z takes the 64-column K tiles
// [z KB / s, (z+1) KB / s) and stores its partial sum at C + z * c_stride; the
// next kernel adds the s partials in order.  Every wait is bounded; a timeout
// sets *err.
__global__ void __launch_bounds__(128, GEMM_CTAS_PER_SM) kie_pf_gemm_kernel(const __half* __restrict__ Ahi,
                                                             const __half* __restrict__ Alo,
                                                             const __half* __restrict__ W, float* __restrict__ C,
                                                             int ldc, int KB, int m_valid,
                                                             const float* __restrict__ col_scale,
                                                             size_t c_stride, uint64_t timeout_ns, int* err) {
    extern __shared__ __align__(1024) uint8_t sm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* done = empty + STAGES;
    uint32_t* taddr = reinterpret_cast<uint32_t*>(done + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nb = blockIdx.x, mb = blockIdx.y, z = blockIdx.z, ns = gridDim.z;
    const int kb0 = int((int64_t(z) * KB) / ns), kb1 = int((int64_t(z + 1) * KB) / ns), nkb = kb1 - kb0;
    C += size_t(z) * c_stride;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(done, 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(taddr, BN);   // 128 lanes x BN fp32 columns
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tacc = *taddr;
    const size_t a_off = size_t(mb) * KB * (BM * BK);
    const size_t w_off = size_t(nb * BN / WT) * KB * (WT * BK) + size_t((nb * BN) % WT) * BK;
    if (threadIdx.x == 0) {
        for (int j = 0; j < nkb; ++j) {
            const int s = j % STAGES, kb = kb0 + j;
            if (j >= STAGES && !wait_bounded(&empty[s], uint32_t((j / STAGES) - 1) & 1u, timeout_ns, err)) break;
            uint8_t* dst = sm + s * STAGE_BYTES;
            mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
            bulk_g2s_keep(dst, Ahi + a_off + size_t(kb) * (BM * BK), A_BYTES, &full[s]);
            bulk_g2s_keep(dst + A_BYTES, Alo + a_off + size_t(kb) * (BM * BK), A_BYTES, &full[s]);
            bulk_g2s_keep(dst + 2 * A_BYTES, W + w_off + size_t(kb) * (WT * BK), B_BYTES, &full[s]);
        }
    } else if (threadIdx.x == 32) {
        // kind::f16 instruction descriptor: fp32 D (bit 4), fp16 A and B, both
        // K-major, N / 8 in bits 17..22, M / 16 in bits 24..28
        const uint32_t idesc = (1u << 4) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);
        bool ok = true;
        for (int j = 0; j < nkb; ++j) {
            const int s = j % STAGES;
            if (!wait_bounded(&full[s], uint32_t(j / STAGES) & 1u, timeout_ns, err)) { ok = false; break; }
            tc_fence_after();
            const uint8_t* st = sm + s * STAGE_BYTES;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {   // K = 16 per MMA: two core matrices, 256 bytes
                const uint64_t bd = smem_desc_noswz(st + 2 * A_BYTES + kk * 256, 128, 1024);
                tc_mma_f16(tacc, smem_desc_noswz(st + kk * 256, 128, 1024), bd, idesc, (j | kk) != 0 ? 1u : 0u);
                tc_mma_f16(tacc, smem_desc_noswz(st + A_BYTES + kk * 256, 128, 1024), bd, idesc, 1u);
            }
            tc_commit(&empty[s]);
        }
        if (ok) tc_commit(done);
    }
    __syncwarp();
    const bool ok = wait_bounded(done, 0u, timeout_ns, err);
    tc_fence_after();
    __syncwarp();
    if (ok) {
        const int row = mb * BM + warp * 32 + lane;
        float* crow = C + size_t(row) * ldc + size_t(nb) * BN;
        for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tacc + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
            if (row < m_valid) {
                const float* cs = col_scale ? col_scale + size_t(nb) * BN + c0 : nullptr;
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    float4 o = make_float4(__uint_as_float(v[i]), __uint_as_float(v[i + 1]), __uint_as_float(v[i + 2]),
                                           __uint_as_float(v[i + 3]));
                    if (cs) { o.x *= cs[i]; o.y *= cs[i + 1]; o.z *= cs[i + 2]; o.w *= cs[i + 3]; }
                    *reinterpret_cast<float4*>(crow + c0 + i) = o;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tacc, BN);
}

// Repack rows [0, n) of a row-major fp16 matrix [n x K] into rows [row0, row0 + n)
// of a weight tile array (256-row tiles).  One thread per 8-element group.
__global__ void kie_pf_pack_kernel(const __half* __restrict__ src, int n, int K, int row0, __half* __restrict__ dst) {
    const int KB = K / 64, g8 = K / 8;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < size_t(n) * g8; i += size_t(gridDim.x) * blockDim.x) {
        const int r = int(i / g8), k = int(i % g8) * 8;
        *reinterpret_cast<uint4*>(dst + tile_idx(row0 + r, k, WT, KB)) =
            *reinterpret_cast<const uint4*>(src + size_t(r) * K + k);
    }
}

// The same for E4M3 codes [n x K] (one byte each), written as their exact fp16 values.
__global__ void kie_pf_pack_e4m3_kernel(const uint8_t* __restrict__ src, int n, int K, int row0,
                                        __half* __restrict__ dst) {
    const int KB = K / 64, g8 = K / 8;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < size_t(n) * g8; i += size_t(gridDim.x) * blockDim.x) {
        const int r = int(i / g8), k = int(i % g8) * 8;
        const uint2 c = *reinterpret_cast<const uint2*>(src + size_t(r) * K + k);
        float f[8];
        e4m3x4_to_f32(c.x, f);
        e4m3x4_to_f32(c.y, f + 4);
        __align__(16) __half h[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) h[j] = __float2half_rn(f[j]);   // exact: E4M3 values are fp16 values
        *reinterpret_cast<uint4*>(dst + tile_idx(row0 + r, k, WT, KB)) = *reinterpret_cast<const uint4*>(h);
    }
}

// The same for NVFP4: packed E2M1 codes [n x K/2] (element 2j in the low
// nibble of byte j) and E4M3 block scales [n x K/16], written as the exact
// fp16 values code * block scale (at most 6 significant bits, magnitude in
// [2^-10, 2688]); the fp32 row scale is applied to the GEMM's output column.
__global__ void kie_pf_pack_fp4_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ bscales, int n,
                                       int K, int row0, __half* __restrict__ dst) {
    const int KB = K / 64, g8 = K / 8;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < size_t(n) * g8; i += size_t(gridDim.x) * blockDim.x) {
        const int r = int(i / g8), k = int(i % g8) * 8;
        const uint32_t c = *reinterpret_cast<const uint32_t*>(codes + size_t(r) * (K / 2) + k / 2);
        float bs[4];
        e4m3x4_to_f32(uint32_t(bscales[size_t(r) * (K / 16) + k / 16]), bs);
        __align__(16) __half h[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 v = h2_to_f2(e2m1x2_to_h2((c >> (8 * j)) & 0xFFu));
            h[2 * j] = __float2half_rn(v.x * bs[0]);       // exact (see above)
            h[2 * j + 1] = __float2half_rn(v.y * bs[0]);
        }
        *reinterpret_cast<uint4*>(dst + tile_idx(row0 + r, k, WT, KB)) = *reinterpret_cast<const uint4*>(h);
    }
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// 8 fp32 values as fp16 hi (into *hi) and lo = fp16(v - hi) (into *lo)
__device__ __forceinline__ void split8(const float* v, uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2 hh = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        const float2 f = __half22float2(hh);
        h[i] = *reinterpret_cast<const uint32_t*>(&hh);
        l[i] = pack_half2(v[2 * i] - f.x, v[2 * i + 1] - f.y);
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}
// Columns [k8, k8 + 8) of row t (8-aligned: 16 contiguous bytes of a tile) as hi / lo.
__device__ __forceinline__ void put_split8(__half* hi, __half* lo, size_t idx, const float* v) {
    uint4 h, l;
    split8(v, h, l);
    *reinterpret_cast<uint4*>(hi + idx) = h;
    *reinterpret_cast<uint4*>(lo + idx) = l;
}
__device__ __forceinline__ void load8(const float* p, float* v) {
    const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ float block_sum256(float v, float* red) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += red[w];
    __syncthreads();
    return s;
}

// x[t] = fp32(E[tokens[t]])
__global__ void kie_pf_embed_kernel(const int32_t* __restrict__ tokens, const uint16_t* __restrict__ emb, int d,
                                    float* __restrict__ x) {
    const int t = blockIdx.x;
    const uint16_t* row = emb + size_t(tokens[t]) * d;
    for (int k = threadIdx.x; k < d; k += blockDim.x) x[size_t(t) * d + k] = __half2float(__ushort_as_half(row[k]));
}

// Rows [0, T) of x (row stride ld): u = x / sqrt(mean(x^2) + eps) * g split into
// hi / lo tiles of 128 rows; rows [T, T_pad) are written as zeros.  256 threads
// per row, 8 consecutive columns a thread at a time (16-byte tile stores).
__global__ void kie_pf_norm_split_kernel(const float* __restrict__ x, int ld, const float* __restrict__ g, float eps,
                                         int T, int d, __half* __restrict__ hi, __half* __restrict__ lo) {
    __shared__ float red[8];
    const int t = blockIdx.x, KB = d / 64;
    if (t >= T) {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k8 = 8 * threadIdx.x; k8 < d; k8 += 8 * blockDim.x) put_split8(hi, lo, tile_idx(t, k8, BM, KB), z);
        return;
    }
    const float* xr = x + size_t(t) * ld;
    float ss = 0.f;
    for (int k8 = 8 * threadIdx.x; k8 < d; k8 += 8 * blockDim.x) {
        float v[8];
        load8(xr + k8, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
    }
    ss = block_sum256(ss, red);
    const float r = sqrtf(ss / float(d) + eps);
    for (int k8 = 8 * threadIdx.x; k8 < d; k8 += 8 * blockDim.x) {
        float v[8], gv[8];
        load8(xr + k8, v);
        load8(g + k8, gv);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = v[e] / r * gv[e];
        put_split8(hi, lo, tile_idx(t, k8, BM, KB), v);
    }
}

// Rows [0, T) of src (row stride ld, K columns) split into hi / lo tiles; rows [T, T_pad) zero.
__global__ void kie_pf_split_kernel(const float* __restrict__ src, int ld, int T, int K, __half* __restrict__ hi,
                                    __half* __restrict__ lo) {
    const int t = blockIdx.x, KB = K / 64;
    for (int k8 = 8 * threadIdx.x; k8 < K; k8 += 8 * blockDim.x) {
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t < T) load8(src + size_t(t) * ld + k8, v);
        put_split8(hi, lo, tile_idx(t, k8, BM, KB), v);
    }
}

// a = silu(C[:, i]) * C[:, F + i], split into hi / lo tiles; rows [T, T_pad) zero.
__global__ void kie_pf_swiglu_split_kernel(const float* __restrict__ C, int ldc, int T, int F, __half* __restrict__ hi,
                                           __half* __restrict__ lo) {
    const int t = blockIdx.x, KB = F / 64;
    for (int i8 = 8 * threadIdx.x; i8 < F; i8 += 8 * blockDim.x) {
        float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (t < T) {
            float gt[8], up[8];
            load8(C + size_t(t) * ldc + i8, gt);
            load8(C + size_t(t) * ldc + F + i8, up);
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] = (gt[e] / (1.f + expf(-gt[e]))) * up[e];
        }
        put_split8(hi, lo, tile_idx(t, i8, BM, KB), a);
    }
}

// Element (t, k) of a GEMM output stored as ns split-K partials c_stride apart,
// added in partial order.
__device__ __forceinline__ float c_sum(const float* C, size_t at, int ns, size_t c_stride) {
    float v = C[at];
    for (int z = 1; z < ns; ++z) v += C[size_t(z) * c_stride + at];
    return v;
}

// x[t, :] += C[t, :d]
__global__ void kie_pf_residual_kernel(float* __restrict__ x, const float* __restrict__ C, int ldc, int d, int ns,
                                       size_t c_stride) {
    const int t = blockIdx.x;
    for (int k4 = 4 * threadIdx.x; k4 < d; k4 += 4 * blockDim.x) {
        float4 v = *reinterpret_cast<const float4*>(C + size_t(t) * ldc + k4);
        for (int z = 1; z < ns; ++z) {
            const float4 w = *reinterpret_cast<const float4*>(C + size_t(z) * c_stride + size_t(t) * ldc + k4);
            v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
        }
        float4* xp = reinterpret_cast<float4*>(x + size_t(t) * d + k4);
        const float4 o = *xp;
        *xp = make_float4(o.x + v.x, o.y + v.y, o.z + v.z, o.w + v.w);
    }
}

// Rotate q and k of row t (position pos0 + t) by RoPE (half-split pairs), store
// k and v into the cache in its storage format (fp16 round to nearest even;
// E5M2 from that fp16), and q (fp32) into Q[t][H*hd].  A thread takes 4
// consecutive pair indices i (hd / 2 is a multiple of 4): 16-byte loads of the
// GEMM's partials and of q, 8- or 4-byte cache stores.
__device__ __forceinline__ float4 c_sum4(const float* C, size_t at, int ns, size_t c_stride) {
    float4 v = *reinterpret_cast<const float4*>(C + at);
    for (int z = 1; z < ns; ++z) {
        const float4 w = *reinterpret_cast<const float4*>(C + size_t(z) * c_stride + at);
        v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
    }
    return v;
}
__device__ __forceinline__ void store4(uint8_t* cache, size_t at, int kvfmt, const float* v) {
    __half h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __float2half_rn(v[e]);
    if (kvfmt == KV_F16) {
        uint2 w;
        w.x = uint32_t(__half_as_ushort(h[0])) | (uint32_t(__half_as_ushort(h[1])) << 16);
        w.y = uint32_t(__half_as_ushort(h[2])) | (uint32_t(__half_as_ushort(h[3])) << 16);
        *reinterpret_cast<uint2*>(reinterpret_cast<__half*>(cache) + at) = w;
    } else {
        uint32_t w = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) w |= (uint32_t(f16x2_to_e5m2x2(h[e], h[e])) & 0xFFu) << (8 * e);
        *reinterpret_cast<uint32_t*>(cache + at) = w;
    }
}
__global__ void kie_pf_qkv_post_kernel(const float* __restrict__ C, int ldc, int pos0, int H, int hd,
                                       const float* __restrict__ inv_freq, int kvfmt, uint8_t* __restrict__ kc,
                                       uint8_t* __restrict__ vc, int layer, int max_ctx, float* __restrict__ Q, int ns,
                                       size_t c_stride) {
    const int t = blockIdx.x, pos = pos0 + t, hh = hd / 2, HD = H * hd;
    const size_t row = size_t(t) * ldc;
    for (int u4 = threadIdx.x; u4 < H * hh / 4; u4 += blockDim.x) {
        const int u = 4 * u4, h = u / hh, i = u % hh;
        float sn[4], cs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) sincosf(float(pos) * inv_freq[i + e], &sn[e], &cs[e]);
        const int e0 = h * hd + i;
        const float4 qa4 = c_sum4(C, row + e0, ns, c_stride), qb4 = c_sum4(C, row + e0 + hh, ns, c_stride);
        const float4 ka4 = c_sum4(C, row + HD + e0, ns, c_stride), kb4 = c_sum4(C, row + HD + e0 + hh, ns, c_stride);
        const float4 va4 = c_sum4(C, row + 2 * HD + e0, ns, c_stride);
        const float4 vb4 = c_sum4(C, row + 2 * HD + e0 + hh, ns, c_stride);
        const float qa[4] = {qa4.x, qa4.y, qa4.z, qa4.w}, qb[4] = {qb4.x, qb4.y, qb4.z, qb4.w};
        const float ka[4] = {ka4.x, ka4.y, ka4.z, ka4.w}, kb[4] = {kb4.x, kb4.y, kb4.z, kb4.w};
        float q0[4], q1[4], k0[4], k1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            q0[e] = qa[e] * cs[e] - qb[e] * sn[e];
            q1[e] = qb[e] * cs[e] + qa[e] * sn[e];
            k0[e] = ka[e] * cs[e] - kb[e] * sn[e];
            k1[e] = kb[e] * cs[e] + ka[e] * sn[e];
        }
        *reinterpret_cast<float4*>(Q + size_t(t) * HD + e0) = make_float4(q0[0], q0[1], q0[2], q0[3]);
        *reinterpret_cast<float4*>(Q + size_t(t) * HD + e0 + hh) = make_float4(q1[0], q1[1], q1[2], q1[3]);
        const size_t base = ((size_t(layer) * H + h) * max_ctx + pos) * hd + i;
        const float v0[4] = {va4.x, va4.y, va4.z, va4.w}, v1[4] = {vb4.x, vb4.y, vb4.z, vb4.w};
        store4(kc, base, kvfmt, k0);
        store4(kc, base + hh, kvfmt, k1);
        store4(vc, base, kvfmt, v0);
        store4(vc, base + hh, kvfmt, v1);
    }
}

// ---- causal attention on the tensor cores ---------------------------------------------------
// One CTA of 128 threads takes 128 query rows of one head; thread t owns query
// row t (TMEM lane t) and its online softmax.  Per 128-key tile of the stored
// cache (the values decode reads; E5M2 bytes become exact fp16):
//   S = Q K^T     tcgen05.mma kind::f16, M 128 x N 128 keys, K = head_dim, into
//                 TMEM columns [0, 128); Q (scaled by 1/sqrt(hd)) enters as
//                 fp16 hi + lo, as in the GEMMs;
//   softmax       each thread reads its row of S, masks keys after its position,
//                 updates its running max m and sum l, rescales its row of O by
//                 exp(m_old - m_new) (TMEM load / store), and writes
//                 P = exp(S - m) as fp16 hi + lo into shared memory;
//   O += P V      tcgen05.mma, M 128 x N head_dim, K = 128 keys, into TMEM columns
//                 [128, 128 + head_dim), B = V^T (K-major: for each dim, the 128
//                 keys), transposed 8 x 8 at a time while the tile is staged.
// All operand tiles use the canonical no-swizzle K-major layout: element
// (row, k) at (row/8)*SBO + (k/8)*128 + (row%8)*16 + (k%8)*2.
// V tile layout: 0 (default) = V^T K-major, transposed 8 x 8 through registers
// while staged; 1 = V as stored (keys x dims, dims contiguous) in the MN-major
// canonical layout, fp16 copied asynchronously like K, the MMA's B operand
// marked MN-major.  For the MN-major operand the descriptor keeps the roles of
// its two byte offsets: the leading one steps along K (here the keys: 8 keys,
// SBO_D bytes), the stride one along N (the dims: 8 dims, 128 bytes); read the
// other way round the prefill parity tests fail.  Both are parity-green; 1 was
// not faster (1.8B 2,048-token prompt 22.9 ms either way).
#ifndef KIE_PF_VMN
#define KIE_PF_VMN 0
#endif
template <int HD>
struct AttnTc {
    static constexpr uint32_t SBO_D = (HD / 8) * 128;   // Q and K tiles: K = head_dim
    static constexpr uint32_t SBO_K = (128 / 8) * 128;  // P and V^T tiles: K = 128 keys
    static constexpr uint32_t Q_BYTES = 128 * HD * 2, K_BYTES = 128 * HD * 2, V_BYTES = HD * 128 * 2,
                              P_BYTES = 128 * 128 * 2;
    static constexpr uint32_t SMEM = 2 * Q_BYTES + K_BYTES + V_BYTES + 2 * P_BYTES + 64;
};

// MN-major V tile: element (key, dim) in 8-key x 8-dim core matrices of 128 bytes,
// 128 bytes apart along the dims and sbo_k apart along the keys.
__device__ __forceinline__ uint32_t vmn(int key, int dim, uint32_t sbo_k) {
    return uint32_t(dim >> 3) * 128u + uint32_t(key >> 3) * sbo_k + uint32_t(key & 7) * 16u + uint32_t(dim & 7) * 2u;
}
__device__ __forceinline__ uint32_t kmaj(int row, int k, uint32_t sbo) {
    return uint32_t(row >> 3) * sbo + uint32_t(k >> 3) * 128u + uint32_t(row & 7) * 16u + uint32_t(k & 7) * 2u;
}
// 8 stored K or V values (fp16, or E5M2 bytes) of one position as fp16
template <int KVF>
__device__ __forceinline__ uint4 load8_f16(const uint8_t* base, size_t elem) {
    if (KVF == KV_F16) return __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const __half*>(base) + elem));
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(base + elem));   // E5M2 byte = fp16 top byte
    return make_uint4(__byte_perm(b.x, 0u, 0x1404), __byte_perm(b.x, 0u, 0x3424), __byte_perm(b.y, 0u, 0x1404),
                      __byte_perm(b.y, 0u, 0x3424));
}

template <int HD, int KVF>
__global__ void __launch_bounds__(128, 1) kie_pf_attn_tc_kernel(const float* __restrict__ Q, const uint8_t* __restrict__ kc,
                                                                const uint8_t* __restrict__ vc, int layer, int H,
                                                                int max_ctx, int pos0, int T, float scale,
                                                                float* __restrict__ O, uint64_t timeout_ns, int* err) {
    using C = AttnTc<HD>;
    extern __shared__ __align__(1024) uint8_t sm[];
    uint8_t* Qh = sm;
    uint8_t* Ql = Qh + C::Q_BYTES;
    uint8_t* Ks = Ql + C::Q_BYTES;
    uint8_t* Vt = Ks + C::K_BYTES;
    uint8_t* Ph = Vt + C::V_BYTES;
    uint8_t* Pl = Ph + C::P_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(Pl + C::P_BYTES);   // [0] S ready, [1] O += P V done
    uint32_t* taddr = reinterpret_cast<uint32_t*>(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, q0 = blockIdx.x * 128;
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_fence_init();
    }
    if (warp == 0) tmem_alloc(taddr, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = *taddr, tO = *taddr + 128u;
    const int HDall = H * HD;
    // Q block, scaled, as fp16 hi + lo tiles
    for (int i = tid; i < 128 * (HD / 8); i += 128) {
        const int r = i / (HD / 8), c8 = (i % (HD / 8)) * 8;
        float v[8];
        if (q0 + r < T) {
            const float* src = Q + size_t(q0 + r) * HDall + size_t(h) * HD + c8;
            const float4 a = *reinterpret_cast<const float4*>(src), b = *reinterpret_cast<const float4*>(src + 4);
            v[0] = a.x * scale; v[1] = a.y * scale; v[2] = a.z * scale; v[3] = a.w * scale;
            v[4] = b.x * scale; v[5] = b.y * scale; v[6] = b.z * scale; v[7] = b.w * scale;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
        uint4 hi, lo;
        split8(v, hi, lo);
        *reinterpret_cast<uint4*>(Qh + kmaj(r, c8, C::SBO_D)) = hi;
        *reinterpret_cast<uint4*>(Ql + kmaj(r, c8, C::SBO_D)) = lo;
    }
    const int row = warp * 32 + lane;                      // query row and TMEM lane of this thread
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const int qpos = pos0 + q0 + row;
    const int last = pos0 + min(T, q0 + 128) - 1;          // the block's largest query position
    const int ntile = last / 128 + 1;
    const size_t head_base = (size_t(layer) * H + h) * max_ctx;
    const uint32_t idesc_s = (1u << 4) | (uint32_t(128 >> 3) << 17) | (uint32_t(128 >> 4) << 24);
    // B = V: K-major V^T, or (KIE_PF_VMN) MN-major V (transpose-B bit 16)
    const uint32_t idesc_o = (1u << 4) | (KIE_PF_VMN ? (1u << 16) : 0u) | (uint32_t(HD >> 3) << 17) |
                             (uint32_t(128 >> 4) << 24);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    int committed = 0;                                     // O commits issued (bar[1] phases to retire)
    // fp16 cache: K tiles land by asynchronous copies straight into Ks, the next
    // one issued as soon as the tile's S = Q K^T has read Ks, so its latency
    // passes during the softmax and O += P V (E5M2 goes through registers)
    auto k_async = [&](int k0) {
        for (int i = tid; i < 128 * (HD / 8); i += 128) {
            const int key = i / (HD / 8), db = i % (HD / 8), j = k0 + key;
            const bool valid = j <= last && j < max_ctx;
            const uint8_t* src = kc + ((head_base + (valid ? j : 0)) * HD + db * 8) * 2;
            cp_async16_zfill(Ks + kmaj(key, db * 8, C::SBO_D), src, valid);
        }
    };
    auto v_async = [&](int k0) {   // MN-major V tile (KIE_PF_VMN), fp16 cache
        for (int i = tid; i < 128 * (HD / 8); i += 128) {
            const int key = i / (HD / 8), db = i % (HD / 8), j = k0 + key;
            const bool valid = j <= last && j < max_ctx;
            const uint8_t* src = vc + ((head_base + (valid ? j : 0)) * HD + db * 8) * 2;
            cp_async16_zfill(Vt + vmn(key, db * 8, C::SBO_D), src, valid);
        }
    };
    if (KVF == KV_F16) { k_async(0); cp_async_commit(); }
    for (int kt = 0; kt < ntile && ok; ++kt) {
        const int k0 = kt * 128;
        // the previous tile's O += P V has read Vt, Ph, Pl (every decision below is
        // CTA-uniform: the TMEM loads and stores are warp-collective)
        if (kt > 0 && !__syncthreads_and(wait_bounded(&bar[1], uint32_t(kt - 1) & 1u, timeout_ns, err))) {
            ok = false;
            break;
        }
        if (KIE_PF_VMN) {
            if (KVF == KV_F16) {   // V lands during S = Q K^T and the softmax
                v_async(k0);
                cp_async_commit();
            } else {   // E5M2: K and V expanded to fp16 through registers, no transposition
                for (int i = tid; i < 128 * (HD / 8); i += 128) {
                    const int key = i / (HD / 8), db = i % (HD / 8), j = k0 + key;
                    uint4 kr = make_uint4(0u, 0u, 0u, 0u), vr = kr;
                    if (j <= last && j < max_ctx) {
                        const size_t at = (head_base + j) * HD + db * 8;
                        kr = load8_f16<KVF>(kc, at);
                        vr = load8_f16<KVF>(vc, at);
                    }
                    *reinterpret_cast<uint4*>(Ks + kmaj(key, db * 8, C::SBO_D)) = kr;
                    *reinterpret_cast<uint4*>(Vt + vmn(key, db * 8, C::SBO_D)) = vr;
                }
            }
        } else {
            // K tile (rows = keys) and V^T tile (rows = dims): 8 keys x 8 dims an item, dims fastest
            for (int i = tid; i < 16 * (HD / 8); i += 128) {
                const int db = i % (HD / 8), kb = i / (HD / 8);
                uint4 kr[8], vr[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = k0 + kb * 8 + u;
                    if (j <= last && j < max_ctx) {
                        const size_t at = (head_base + j) * HD + db * 8;
                        if (KVF != KV_F16) kr[u] = load8_f16<KVF>(kc, at);
                        vr[u] = load8_f16<KVF>(vc, at);
                    } else {
                        kr[u] = vr[u] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (KVF != KV_F16) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(Ks + kmaj(kb * 8 + u, db * 8, C::SBO_D)) = kr[u];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {   // dim db*8 + e over the 8 keys
                    const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
                    const int wi = e >> 1;
                    const uint32_t w0 = __byte_perm((&vr[0].x)[wi], (&vr[1].x)[wi], sel);
                    const uint32_t w1 = __byte_perm((&vr[2].x)[wi], (&vr[3].x)[wi], sel);
                    const uint32_t w2 = __byte_perm((&vr[4].x)[wi], (&vr[5].x)[wi], sel);
                    const uint32_t w3 = __byte_perm((&vr[6].x)[wi], (&vr[7].x)[wi], sel);
                    *reinterpret_cast<uint4*>(Vt + kmaj(db * 8 + e, kb * 8, C::SBO_K)) = make_uint4(w0, w1, w2, w3);
                }
            }
        }
        // this thread's copies of the K tile have landed (V's may still be in flight)
        if (KVF == KV_F16) { if (KIE_PF_VMN) cp_async_wait_group<1>(); else cp_async_wait_group<0>(); }
        fence_proxy_async_shared();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < HD / 16; ++kk) {
                const uint64_t bd = smem_desc_noswz(Ks + kk * 256, 128, C::SBO_D);
                tc_mma_f16(tS, smem_desc_noswz(Qh + kk * 256, 128, C::SBO_D), bd, idesc_s, kk != 0 ? 1u : 0u);
                tc_mma_f16(tS, smem_desc_noswz(Ql + kk * 256, 128, C::SBO_D), bd, idesc_s, 1u);
            }
            tc_commit(&bar[0]);
        }
        __syncwarp();
        if (!__syncthreads_and(wait_bounded(&bar[0], uint32_t(kt) & 1u, timeout_ns, err))) {
            ok = false;
            break;
        }
        tc_fence_after();
        if (KVF == KV_F16 && kt + 1 < ntile) { k_async(k0 + 128); cp_async_commit(); }   // S has read Ks
        // this row's scores: the tile's maximum, then P = exp(S - m) as fp16 hi + lo
        float mt = -INFINITY;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t sv[32];
            tmem_ld_32x32b_x32(tS + lane_off + uint32_t(c0), sv);
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (k0 + c0 + e <= qpos) mt = fmaxf(mt, __uint_as_float(sv[e]));
        }
        const float mn = fmaxf(m, mt);
        const float cf = (m == -INFINITY) ? 0.f : expf(m - mn);
        float ps = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t sv[32];
            tmem_ld_32x32b_x32(tS + lane_off + uint32_t(c0), sv);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                float p[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = k0 + c0 + 8 * g + e;
                    p[e] = (j <= qpos && mn > -INFINITY) ? expf(__uint_as_float(sv[8 * g + e]) - mn) : 0.f;
                    ps += p[e];
                }
                uint4 hi, lo;
                split8(p, hi, lo);
                *reinterpret_cast<uint4*>(Ph + kmaj(row, c0 + 8 * g, C::SBO_K)) = hi;
                *reinterpret_cast<uint4*>(Pl + kmaj(row, c0 + 8 * g, C::SBO_K)) = lo;
            }
        }
        l = l * cf + ps;
        m = mn;
        // O row *= exp(m_old - m_new) before this tile's P V is added; a warp whose
        // rows all kept their maximum (factor exactly 1) skips the TMEM round trip
        if (kt > 0 && __any_sync(0xffffffffu, cf != 1.f)) {
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t ov[32];
                tmem_ld_32x32b_x32(tO + lane_off + uint32_t(c0), ov);
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * cf);
                tmem_st_32x32b_x32(tO + lane_off + uint32_t(c0), ov);
            }
        }
        if (KIE_PF_VMN && KVF == KV_F16) {   // this thread's copies of the V tile have landed
            if (kt + 1 < ntile) cp_async_wait_group<1>(); else cp_async_wait_group<0>();
        }
        tc_fence_before();
        fence_proxy_async_shared();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk) {
                const uint64_t bd = KIE_PF_VMN ? smem_desc_noswz(Vt + kk * 2 * C::SBO_D, C::SBO_D, 128)
                                               : smem_desc_noswz(Vt + kk * 256, 128, C::SBO_K);
                tc_mma_f16(tO, smem_desc_noswz(Ph + kk * 256, 128, C::SBO_K), bd, idesc_o,
                           (kt > 0 || kk > 0) ? 1u : 0u);
                tc_mma_f16(tO, smem_desc_noswz(Pl + kk * 256, 128, C::SBO_K), bd, idesc_o, 1u);
            }
            tc_commit(&bar[1]);
        }
        __syncwarp();
        committed = kt + 1;
    }
    if (KVF == KV_F16) cp_async_wait_group<0>();   // no copy of a K or V tile is left in flight (error paths)
    // every issued O update has landed (also on the error path, bounded), then O / l
    const bool done = __syncthreads_and(committed > 0 &&
                                        wait_bounded(&bar[1], uint32_t(committed - 1) & 1u, timeout_ns, err));
    tc_fence_after();
    if (ok && done) {   // CTA-uniform; rows past T load with their warp but store nothing
        float* orow = O + size_t(q0 + row) * HDall + size_t(h) * HD;
        const float il = 1.f / l;
#pragma unroll
        for (int c0 = 0; c0 < HD; c0 += 32) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(tO + lane_off + uint32_t(c0), ov);
            if (q0 + row < T) {
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4*>(orow + c0 + e) =
                        make_float4(__uint_as_float(ov[e]) * il, __uint_as_float(ov[e + 1]) * il,
                                    __uint_as_float(ov[e + 2]) * il, __uint_as_float(ov[e + 3]) * il);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(*taddr, 256);
}

template <int HD, int KVF>
cudaError_t launch_attention(const float* Q, const uint8_t* kc, const uint8_t* vc, int layer, int H, int max_ctx,
                             int pos0, int T, float scale, float* O, uint64_t timeout_ns, int* err, cudaStream_t st) {
    const size_t smem = AttnTc<HD>::SMEM;
    cudaError_t r = cudaFuncSetAttribute(kie_pf_attn_tc_kernel<HD, KVF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (r != cudaSuccess) return r;
    kie_pf_attn_tc_kernel<HD, KVF><<<dim3((T + 127) / 128, H), 128, smem, st>>>(Q, kc, vc, layer, H, max_ctx, pos0,
                                                                                  T, scale, O, timeout_ns, err);
    return cudaGetLastError();
}

}  // namespace

// ---- launch wrappers (host code in kie_api.cu) -----------------------------------------------
extern "C" size_t kie_pf_tile_elems(int rows_pad, int K) { return size_t(rows_pad) * K; }

extern "C" cudaError_t kie_pf_gemm(const __half* Ahi, const __half* Alo, const __half* W, float* C, int ldc,
                                   int M_pad, int N_pad, int K, int m_valid, const float* col_scale, int ksplit,
                                   size_t c_stride, uint64_t timeout_ns, int* err, cudaStream_t st) {
    if (ksplit < 1 || ksplit > K / BK) return cudaErrorInvalidValue;
    cudaError_t r = cudaFuncSetAttribute(kie_pf_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(GEMM_SMEM));
    if (r != cudaSuccess) return r;
    kie_pf_gemm_kernel<<<dim3(N_pad / BN, M_pad / BM, ksplit), 128, GEMM_SMEM, st>>>(
        Ahi, Alo, W, C, ldc, K / BK, m_valid, col_scale, c_stride, timeout_ns, err);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_pack_fp4(const uint8_t* codes, const uint8_t* bscales, int n, int K, int row0, __half* dst,
                                       cudaStream_t st) {
    const size_t work = size_t(n) * (K / 8);
    const unsigned blocks = unsigned(std::min<size_t>((work + 255) / 256, 65535));
    kie_pf_pack_fp4_kernel<<<blocks, 256, 0, st>>>(codes, bscales, n, K, row0, dst);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_pack_e4m3(const uint8_t* codes, int n, int K, int row0, __half* dst, cudaStream_t st) {
    const size_t work = size_t(n) * (K / 8);
    const int blocks = int(std::min<size_t>((work + 255) / 256, 65535));
    kie_pf_pack_e4m3_kernel<<<blocks, 256, 0, st>>>(codes, n, K, row0, dst);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_pack(const __half* src, int n, int K, int row0, __half* dst, cudaStream_t st) {
    const size_t work = size_t(n) * (K / 8);
    const int blocks = int(std::min<size_t>((work + 255) / 256, 65535));
    kie_pf_pack_kernel<<<blocks, 256, 0, st>>>(src, n, K, row0, dst);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_embed(const int32_t* tokens, int T, const uint16_t* emb, int d, float* x,
                                    cudaStream_t st) {
    kie_pf_embed_kernel<<<T, 256, 0, st>>>(tokens, emb, d, x);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_norm_split(const float* x, int ld, const float* g, float eps, int T, int T_pad, int d,
                                         __half* hi, __half* lo, cudaStream_t st) {
    kie_pf_norm_split_kernel<<<T_pad, 256, 0, st>>>(x, ld, g, eps, T, d, hi, lo);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_split(const float* src, int ld, int T, int T_pad, int K, __half* hi, __half* lo,
                                    cudaStream_t st) {
    kie_pf_split_kernel<<<T_pad, 256, 0, st>>>(src, ld, T, K, hi, lo);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_swiglu_split(const float* C, int ldc, int T, int T_pad, int F, __half* hi, __half* lo,
                                           cudaStream_t st) {
    kie_pf_swiglu_split_kernel<<<T_pad, 256, 0, st>>>(C, ldc, T, F, hi, lo);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_residual(float* x, const float* C, int ldc, int T, int d, int ns, size_t c_stride,
                                       cudaStream_t st) {
    kie_pf_residual_kernel<<<T, 256, 0, st>>>(x, C, ldc, d, ns, c_stride);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_qkv_post(const float* C, int ldc, int T, int pos0, int H, int hd, const float* inv_freq,
                                       int kvfmt, uint8_t* kc, uint8_t* vc, int layer, int max_ctx, float* Q, int ns,
                                       size_t c_stride, cudaStream_t st) {
    kie_pf_qkv_post_kernel<<<T, 256, 0, st>>>(C, ldc, pos0, H, hd, inv_freq, kvfmt, kc, vc, layer, max_ctx, Q, ns,
                                              c_stride);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_pf_attention(const float* Q, const uint8_t* kc, const uint8_t* vc, int layer, int H,
                                        int hd, int kvfmt, int max_ctx, int pos0, int T, float scale, float* O,
                                        uint64_t timeout_ns, int* err, cudaStream_t st) {
    if (hd == 128) {
        return kvfmt == KV_F16
                   ? launch_attention<128, KV_F16>(Q, kc, vc, layer, H, max_ctx, pos0, T, scale, O, timeout_ns, err, st)
                   : launch_attention<128, KV_E5M2>(Q, kc, vc, layer, H, max_ctx, pos0, T, scale, O, timeout_ns, err, st);
    }
    return kvfmt == KV_F16
               ? launch_attention<64, KV_F16>(Q, kc, vc, layer, H, max_ctx, pos0, T, scale, O, timeout_ns, err, st)
               : launch_attention<64, KV_E5M2>(Q, kc, vc, layer, H, max_ctx, pos0, T, scale, O, timeout_ns, err, st);
}
