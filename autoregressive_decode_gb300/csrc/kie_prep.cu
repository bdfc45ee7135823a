// One-off preparation kernels: weight repacking into per-CTA streams, INT4
// quantisation, adaptive-range uint8 segment quantisation, fp16 -> E5M2, and
// writing a supplied context into the KV cache.  None of these is on the
// per-token path.
#include <cuda_fp16.h>
#include <stdint.h>

#include "kie_device.cuh"
#include "kie_internal.h"

using namespace kie;

// ---- repack: byte copies described by (dst offset, src offset, length) ----------------------
struct CopyDesc {
    uint64_t dst;
    uint64_t src;
    uint32_t len;
    uint32_t pad;
};

__global__ void kie_copy_desc_kernel(uint8_t* dst_base, const uint8_t* src_base, const CopyDesc* desc, int n) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int i = warp; i < n; i += nwarps) {
        const CopyDesc d = desc[i];
        uint8_t* dp = dst_base + d.dst;
        const uint8_t* sp = src_base + d.src;
        if (((d.dst | d.src | d.len) & 15u) == 0) {
            const uint32_t nv = d.len >> 4;
            for (uint32_t k = lane; k < nv; k += 32)
                reinterpret_cast<uint4*>(dp)[k] = reinterpret_cast<const uint4*>(sp)[k];
        } else {
            for (uint32_t k = lane; k < d.len; k += 32) dp[k] = sp[k];
        }
    }
}

// ---- INT4 g128 symmetric quantisation -------------------------------------------------------
// One warp per (row, group of 128 columns).  s = fp16_rne(absmax / 7) with the
// division in fp32; q = clamp(rint_half_even(w / fp32(s)), -8, 7); q = 0 when s == 0.
// packed: element 2b in the low nibble of byte b (two's complement); or, when
// codes_i8 != null, one int8 per element.
__global__ void kie_quant_int4_kernel(const uint16_t* w, int rows, int cols, uint8_t* packed, int8_t* codes_i8,
                                      uint16_t* scales) {
    const int ngrp = cols / 128;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows * ngrp) return;
    const int r = warp / ngrp, g = warp % ngrp;
    const uint16_t* src = w + size_t(r) * cols + size_t(g) * 128;
    float v[4];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = __half2float(__ushort_as_half(src[lane * 4 + i]));
        am = fmaxf(am, fabsf(v[i]));
    }
    am = warp_max(am);
    const __half s16 = __float2half_rn(am / 7.0f);
    const float s = __half2float(s16);
    int q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = (s > 0.f) ? min(max(__float2int_rn(v[i] / s), -8), 7) : 0;
    if (codes_i8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) codes_i8[size_t(r) * cols + size_t(g) * 128 + lane * 4 + i] = int8_t(q[i]);
    }
    if (packed) {
        uint8_t* dst = packed + size_t(r) * (cols / 2) + size_t(g) * 64 + lane * 2;
        dst[0] = uint8_t((q[0] & 0xF) | ((q[1] & 0xF) << 4));
        dst[1] = uint8_t((q[2] & 0xF) | ((q[3] & 0xF) << 4));
    }
    if (lane == 0) scales[size_t(r) * ngrp + g] = __half_as_ushort(s16);
}

// ---- FP8 E4M3 weights, one scale per output row ----------------------------------------------
// One warp per row: s = absmax / 448 in fp32 (IEEE division); code = E4M3 of
// w / s (IEEE division; cvt round to nearest even, satfinite); s == 0 -> 0.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));   // first source -> upper byte
    return r;
}
__global__ void kie_quant_fp8_kernel(const uint16_t* w, int rows, int cols, uint8_t* codes, float* scales) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const uint16_t* src = w + size_t(warp) * cols;
    float am = 0.f;
    for (int k = lane; k < cols; k += 32) am = fmaxf(am, fabsf(__half2float(__ushort_as_half(src[k]))));
    am = warp_max(am);
    const float s = am / 448.0f;
    uint8_t* dst = codes + size_t(warp) * cols;
    for (int k = 2 * lane; k < cols; k += 64) {   // cols is even
        const float a = __half2float(__ushort_as_half(src[k])), b = __half2float(__ushort_as_half(src[k + 1]));
        const uint32_t c = s > 0.f ? f32x2_to_e4m3x2(a / s, b / s) : 0u;
        dst[k] = uint8_t(c & 0xFFu);
        dst[k + 1] = uint8_t(c >> 8);
    }
    if (lane == 0) scales[warp] = s;
}

// ---- NVFP4 weights: E2M1 codes, an E4M3 scale per 16 columns, an fp32 scale per row --------
// One warp per row, one lane per 16-column block at a time, every step in fp32
// with IEEE division and products rounded once:
//   rs = absmax(row) / 2688                       (2688 = 6 * 448)
//   bs = e4m3(absmax(block) / (6 * rs))           (round to nearest even, saturating)
//   code = e2m1(w / (float(bs) * rs))             (round to nearest even, saturating at +-6)
// rs == 0 gives bs = 0 and codes 0; a block scale of 0 gives codes 0.
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(x));   // x -> the low byte
    return r & 0xFFu;
}
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {          // lo -> low nibble
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_to_f32_exact(uint32_t b) {
    float f[4];
    e4m3x4_to_f32(b & 0xFFu, f);
    return f[0];
}
// packed: [rows][cols/2] (element 2j in the low nibble of byte j) or null;
// codes: [rows][cols] one code (0..15) per byte, or null; bscales [rows][cols/16]; rscales [rows].
__global__ void kie_quant_fp4_kernel(const uint16_t* w, int rows, int cols, uint8_t* packed, uint8_t* codes,
                                     uint8_t* bscales, float* rscales) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= rows) return;
    const uint16_t* src = w + size_t(warp) * cols;
    float am = 0.f;
    for (int k = lane; k < cols; k += 32) am = fmaxf(am, fabsf(__half2float(__ushort_as_half(src[k]))));
    am = warp_max(am);
    const float rs = am / 2688.0f;
    const float six_rs = 6.0f * rs;
    const int nb = cols / 16;
    for (int b = lane; b < nb; b += 32) {
        float v[16];
        float bm = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            v[j] = __half2float(__ushort_as_half(src[b * 16 + j]));
            bm = fmaxf(bm, fabsf(v[j]));
        }
        const uint32_t bsc = rs > 0.f ? f32_to_e4m3(bm / six_rs) : 0u;
        const float denom = e4m3_to_f32_exact(bsc) * rs;
        uint32_t pk[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            const uint32_t c2 = denom > 0.f ? f32x2_to_e2m1x2(v[j] / denom, v[j + 1] / denom) : 0u;
            pk[j >> 3] |= c2 << (4 * (j & 7));
            if (codes) {
                codes[size_t(warp) * cols + b * 16 + j] = uint8_t(c2 & 0xFu);
                codes[size_t(warp) * cols + b * 16 + j + 1] = uint8_t(c2 >> 4);
            }
        }
        if (packed) *reinterpret_cast<uint2*>(packed + size_t(warp) * (cols / 2) + b * 8) = make_uint2(pk[0], pk[1]);
        bscales[size_t(warp) * nb + b] = uint8_t(bsc);
    }
    if (lane == 0) rscales[warp] = rs;
}

// ---- adaptive-range uint8 quantisation ------------------------------------------------------
// One CTA per segment.  A segment is `rows` rows of `row_elems` fp16 values;
// element (r, k) of segment s is at src[s*src_seg + r*src_row + k] and its code
// goes to codes[s*dst_seg + r*dst_row + k].  scale = (max-min)/255 and
// zp = rint_half_even(-min/scale) in fp32 (IEEE division); constant segment:
// scale 1, zp = rint(-min); code = clamp(rint(x/scale) + zp, 0, 255).
__global__ void kie_quant_u8_kernel(const uint16_t* src, int64_t src_seg, int64_t src_row, int rows, int row_elems,
                                    uint8_t* codes, int64_t dst_seg, int64_t dst_row, float* scale_out,
                                    int32_t* zp_out, int64_t meta_stride) {
    const int s = blockIdx.x;
    const int n = rows * row_elems;
    const uint16_t* sp = src + s * src_seg;
    float mn = INFINITY, mx = -INFINITY;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int r = i / row_elems, k = i % row_elems;
        const float v = __half2float(__ushort_as_half(sp[r * src_row + k]));
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    __shared__ float smn[32], smx[32];
    mn = -warp_max(-mn);
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) { smn[threadIdx.x >> 5] = mn; smx[threadIdx.x >> 5] = mx; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < int(blockDim.x >> 5); ++w) { mn = fminf(mn, smn[w]); mx = fmaxf(mx, smx[w]); }
        smn[0] = mn;
        smx[0] = mx;
    }
    __syncthreads();
    mn = smn[0];
    mx = smx[0];
    float sc;
    int zp;
    if (mx == mn) { sc = 1.f; zp = __float2int_rn(-mn); }
    else { sc = (mx - mn) / 255.f; zp = __float2int_rn(-mn / sc); }
    uint8_t* dp = codes + s * dst_seg;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int r = i / row_elems, k = i % row_elems;
        const float v = __half2float(__ushort_as_half(sp[r * src_row + k]));
        dp[r * dst_row + k] = uint8_t(min(max(__float2int_rn(v / sc) + zp, 0), 255));
    }
    if (threadIdx.x == 0) {
        scale_out[s * meta_stride] = sc;
        zp_out[s * meta_stride] = zp;
    }
}

// ---- fp16 -> E5M2 ----------------------------------------------------------------------------
__global__ void kie_e5m2_kernel(const uint16_t* x, size_t n, uint8_t* out) {
    for (size_t i = (size_t(blockIdx.x) * blockDim.x + threadIdx.x) * 2; i < n;
         i += size_t(gridDim.x) * blockDim.x * 2) {
        const __half a = __ushort_as_half(x[i]);
        const __half b = (i + 1 < n) ? __ushort_as_half(x[i + 1]) : __ushort_as_half(0);
        const uint16_t r = f16x2_to_e5m2x2(a, b);
        out[i] = uint8_t(r & 0xFF);
        if (i + 1 < n) out[i + 1] = uint8_t(r >> 8);
    }
}

// ---- context loading: [n][H][hd] fp16 -> cache layout [H][max_ctx][hd] ----------------------
// fmt 0: fp16 copy; 1: E5M2; 2: fp16 into the open-segment tail (positions >= first_tail).
__global__ void kie_set_kv_kernel(const uint16_t* src, int n, int H, int hd, int max_ctx, int fmt, uint8_t* dst,
                                  uint16_t* tail, int first_tail) {
    const size_t total = size_t(n) * H * hd;
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += size_t(gridDim.x) * blockDim.x) {
        const int k = int(i % hd);
        const int h = int((i / hd) % H);
        const int p = int(i / (size_t(hd) * H));
        const uint16_t v = src[i];
        const size_t di = (size_t(h) * max_ctx + p) * hd + k;
        if (fmt == 0) {
            reinterpret_cast<uint16_t*>(dst)[di] = v;
        } else if (fmt == 1) {
            const __half hv = __ushort_as_half(v);
            dst[di] = uint8_t(f16x2_to_e5m2x2(hv, hv) & 0xFF);
        } else if (p >= first_tail) {
            tail[(size_t(h) * KIE_SEG + (p - first_tail)) * hd + k] = v;
        }
    }
}

// ---- launch wrappers (host) --------------------------------------------------------------------
// ---- scaled E5M2 cache (context loading and rewinds) ---------------------------------------------
__device__ __forceinline__ float e5m2_mag_prep(uint32_t b) {
    return fabsf(__half2float(__ushort_as_half((unsigned short)((b & 0xFFu) << 8))));
}

// Slice j of one (layer, K or V) begins: for j >= 1 its scale from slice j-1
// (largest stored magnitude m, scale s: m * s / 127, or s when that is zero or
// not finite); its running maximum starts at zero.  sc, mx: that entry's [nslice].
__global__ void kie_kv_slice_start_kernel(float* sc, uint32_t* mx, int j) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    if (j > 0) {
        const float sp = sc[j - 1];
        const float amax = __uint_as_float(mx[j - 1]) * sp;
        sc[j] = (isfinite(amax) && amax > 0.f) ? amax / KIE_KV_SCALE_TARGET : sp;
    }
    mx[j] = 0u;
}

// Positions [p0, p1) of one layer's K or V (fp16 source [n][H][hd]) as E5M2
// codes of x / sc[0] into dst ([H][max_ctx][hd] of that layer), folding their
// magnitudes into *mx by atomic max (fp32 bits of non-negative values order as
// unsigned integers).
__global__ void kie_kv_slice_quant_kernel(const uint16_t* src, int p0, int p1, int H, int hd, int max_ctx,
                                          const float* sc, uint8_t* dst, uint32_t* mx) {
    const int per = H * hd;
    const int64_t n = int64_t(p1 - p0) * per;
    const float s = *sc;
    float m = 0.f;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += int64_t(gridDim.x) * blockDim.x) {
        const int p = p0 + int(i / per), r = int(i % per), h = r / hd, d = r - h * hd;
        const __half x = __ushort_as_half(src[size_t(p) * per + r]);
        const __half y = __float2half_rn(__half2float(x) / s);
        const uint32_t b = f16x2_to_e5m2x2(y, y) & 0xFFu;
        dst[(size_t(h) * max_ctx + p) * hd + d] = uint8_t(b);
        m = fmaxf(m, e5m2_mag_prep(b));
    }
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(mx, __float_as_uint(m));
}

// After a move of the position to pos: the running maximum of pos's slice over
// the positions [slice start, pos) still in the cache, and zero for every later
// slice.  One block per (layer, K or V).
__global__ void kie_kv_rescan_kernel(const uint8_t* kc, const uint8_t* vc, uint32_t* mx, int H, int hd, int max_ctx,
                                     int nslice, int pos) {
    __shared__ float red[32];
    const int lk = blockIdx.x, layer = lk >> 1, kv = lk & 1;
    const uint8_t* base = (kv ? vc : kc) + size_t(layer) * H * max_ctx * hd;
    const int j = pos / KIE_KV_SLICE, q0 = j * KIE_KV_SLICE, per_h = (pos - q0) * hd;
    float m = 0.f;
    for (int h = 0; h < H; ++h)
        for (int i = threadIdx.x; i < per_h; i += blockDim.x)
            m = fmaxf(m, e5m2_mag_prep(base[(size_t(h) * max_ctx + q0) * hd + i]));
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < int(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
        if (j < nslice) mx[size_t(lk) * nslice + j] = __float_as_uint(m);
    }
    for (int s = j + 1 + int(threadIdx.x); s < nslice; s += blockDim.x) mx[size_t(lk) * nslice + s] = 0u;
}

#include <cuda_runtime.h>

extern "C" cudaError_t kie_launch_kv_slice(const uint16_t* src, int p0, int p1, int H, int hd, int max_ctx, float* sc,
                                           uint32_t* mx, int j, uint8_t* dst, cudaStream_t st) {
    kie_kv_slice_start_kernel<<<1, 32, 0, st>>>(sc, mx, j);
    if (p1 <= p0) return cudaGetLastError();
    size_t blocks = (size_t(p1 - p0) * H * hd + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    kie_kv_slice_quant_kernel<<<unsigned(blocks), 256, 0, st>>>(src, p0, p1, H, hd, max_ctx, sc + j, dst, mx + j);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_kv_rescan(const uint8_t* kc, const uint8_t* vc, uint32_t* mx, int L, int H, int hd,
                                            int max_ctx, int nslice, int pos, cudaStream_t st) {
    kie_kv_rescan_kernel<<<2 * L, 256, 0, st>>>(kc, vc, mx, H, hd, max_ctx, nslice, pos);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_copy_desc(uint8_t* dst, const uint8_t* src, const void* desc, int n,
                                            cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const int threads = 256;
    int blocks = (n + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    kie_copy_desc_kernel<<<blocks, threads, 0, st>>>(dst, src, reinterpret_cast<const CopyDesc*>(desc), n);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_quant_int4(const uint16_t* w, int rows, int cols, uint8_t* packed,
                                             int8_t* codes_i8, uint16_t* scales, cudaStream_t st) {
    const long warps = long(rows) * (cols / 128);
    const int threads = 256;
    const long blocks = (warps * 32 + threads - 1) / threads;
    kie_quant_int4_kernel<<<unsigned(blocks), threads, 0, st>>>(w, rows, cols, packed, codes_i8, scales);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_quant_fp8(const uint16_t* w, int rows, int cols, uint8_t* codes, float* scales,
                                            cudaStream_t st) {
    const int threads = 256;
    const long blocks = (long(rows) * 32 + threads - 1) / threads;
    kie_quant_fp8_kernel<<<unsigned(blocks), threads, 0, st>>>(w, rows, cols, codes, scales);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_quant_fp4(const uint16_t* w, int rows, int cols, uint8_t* packed, uint8_t* codes,
                                            uint8_t* bscales, float* rscales, cudaStream_t st) {
    const int threads = 256;
    const long blocks = (long(rows) * 32 + threads - 1) / threads;
    kie_quant_fp4_kernel<<<unsigned(blocks), threads, 0, st>>>(w, rows, cols, packed, codes, bscales, rscales);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_quant_u8(const uint16_t* src, int n_seg, int64_t src_seg, int64_t src_row,
                                           int rows, int row_elems, uint8_t* codes, int64_t dst_seg,
                                           int64_t dst_row, float* scale, int32_t* zp, int64_t meta_stride,
                                           cudaStream_t st) {
    if (n_seg <= 0) return cudaSuccess;
    kie_quant_u8_kernel<<<n_seg, 256, 0, st>>>(src, src_seg, src_row, rows, row_elems, codes, dst_seg, dst_row,
                                               scale, zp, meta_stride);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_e5m2(const uint16_t* x, size_t n, uint8_t* out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n / 2 + 255) / 256 + 1;
    if (blocks > 8192) blocks = 8192;
    kie_e5m2_kernel<<<unsigned(blocks), 256, 0, st>>>(x, n, out);
    return cudaGetLastError();
}

extern "C" cudaError_t kie_launch_set_kv(const uint16_t* src, int n, int H, int hd, int max_ctx, int fmt,
                                         uint8_t* dst, uint16_t* tail, int first_tail, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    size_t total = size_t(n) * H * hd;
    size_t blocks = (total + 255) / 256;
    if (blocks > 16384) blocks = 16384;
    kie_set_kv_kernel<<<unsigned(blocks), 256, 0, st>>>(src, n, H, hd, max_ctx, fmt, dst, tail, first_tail);
    return cudaGetLastError();
}
