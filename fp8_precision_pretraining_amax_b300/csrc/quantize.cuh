// Fused amax + scale + E4M3 cast kernels (HBM-bound).
//
// Rule implemented (fine-grained block quantization that the Puro-2B report,
// section 2 "FP8", adopts from DeepSeek-V3 for its main linear layers):
// per tile, amax = max |x|; s = amax / 448 rounded to FP32 (s = 1 when
// amax == 0); code = E4M3(x / s) where x / s is the correctly rounded FP32
// quotient and E4M3() rounds half to even with saturation to +-448.
//
// Every kernel reads its input exactly once with 128-bit (or 32-bit
// column-pair) coalesced loads, reduces amax in registers and warp shuffles,
// and writes codes and scales once.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace fp8bq {

// ------------------------------------------------------------ element math

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// s = amax / 448 (IEEE, round to nearest even), 1 for an all-zero tile.
__device__ __forceinline__ float tile_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Two quotients -> two E4M3 codes packed low byte first (element a first).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b, float s) {
    float2 v = make_float2(__fdiv_rn(a, s), __fdiv_rn(b, s));
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// Eight values -> eight codes in two 32-bit words (memory order).
__device__ __forceinline__ uint2 e4m3x8(const float (&v)[8], float s) {
    uint2 o;
    o.x = e4m3x2(v[0], v[1], s) | (e4m3x2(v[2], v[3], s) << 16);
    o.y = e4m3x2(v[4], v[5], s) | (e4m3x2(v[6], v[7], s) << 16);
    return o;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& w, float (&v)[8]) {
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x);
    v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    v[4] = bf16lo(w.z); v[5] = bf16hi(w.z);
    v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// ------------------------------------------------------------------ row-wise
//
// One 1x128 tile per group of 8 lanes (4 tiles per warp).  Lane j of a group
// owns elements [8j, 8j+8) and [64+8j, 64+8j+8) of its tile (16 values), so
// each warp-wide 16-byte load reads 4 fully used 128-byte segments.  Tiles are
// numbered row-major (tile = r * C/128 + t) so consecutive warps stream
// consecutive memory.

template <bool kF32>
__global__ void __launch_bounds__(256) quantize_rowwise_kernel(const void* __restrict__ x, int64_t R, int64_t C,
                                                               int64_t ldx, uint8_t* __restrict__ q,
                                                               float* __restrict__ s) {
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;
    const int64_t T = C >> 7;
    const int64_t ntiles = R * T;
    const int64_t tile = ((static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) << 2) + (lane >> 3);
    const bool valid = tile < ntiles;
    const int64_t r = valid ? tile / T : 0;
    const int64_t t = valid ? tile - r * T : 0;

    float v[16];
    if (!kF32) {
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(x) + r * ldx + t * 128;
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = make_uint4(0, 0, 0, 0);
        if (valid) {
            w0 = ldg_nc_v4(src + 8 * j);
            w1 = ldg_nc_v4(src + 64 + 8 * j);
        }
        float a[8], b[8];
        unpack_bf16x8(w0, a);
        unpack_bf16x8(w1, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
    } else {
        // lane j owns elements [4j + 32p, 4j + 32p + 4), p = 0..3
        const float* src = static_cast<const float*>(x) + r * ldx + t * 128;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (valid) w = ldg_nc_v4(src + 32 * p + 4 * j);
            v[4 * p + 0] = __uint_as_float(w.x);
            v[4 * p + 1] = __uint_as_float(w.y);
            v[4 * p + 2] = __uint_as_float(w.z);
            v[4 * p + 3] = __uint_as_float(w.w);
        }
    }

    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    const float sc = tile_scale(amax);

    if (!valid) return;
    uint8_t* dst = q + r * C + t * 128;
    if (!kF32) {
        float a[8], b[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) { a[i] = v[i]; b[i] = v[8 + i]; }
        *reinterpret_cast<uint2*>(dst + 8 * j) = e4m3x8(a, sc);
        *reinterpret_cast<uint2*>(dst + 64 + 8 * j) = e4m3x8(b, sc);
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint32_t w = e4m3x2(v[4 * p], v[4 * p + 1], sc) | (e4m3x2(v[4 * p + 2], v[4 * p + 3], sc) << 16);
            *reinterpret_cast<uint32_t*>(dst + 32 * p + 4 * j) = w;
        }
    }
    if (j == 0) s[t * R + r] = sc;
}

// --------------------------------------------------------------- column-wise
//
// CTA = 256 threads over a slab of 128 tokens x (64 * VEC) columns, VEC = 2
// for BF16 (a thread owns a column pair, 4-byte loads) and 1 for FP32.
// Thread (g = tid % 64, quarter = tid / 64) loads tokens [32*quarter, +32) of
// its column(s): each warp-wide load covers 128 contiguous bytes of one row.
// The per-column amax is combined across the four quarters in shared memory,
// and each thread writes its 32 codes per column as 32 contiguous bytes of
// the transposed output row qT[c][m].

template <bool kF32>
__global__ void __launch_bounds__(256) quantize_colwise_kernel(const void* __restrict__ x, int64_t M, int64_t C,
                                                               int64_t ldx, uint8_t* __restrict__ qT,
                                                               float* __restrict__ s) {
    constexpr int VEC = kF32 ? 1 : 2;
    constexpr int CW = 64 * VEC;  // columns per CTA
    __shared__ float red[4][CW];

    const int tid = threadIdx.x;
    const int g = tid & 63;
    const int quarter = tid >> 6;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c = static_cast<int64_t>(blockIdx.x) * CW + g * VEC;  // first column of this thread
    const bool valid = c < C;

    float v[VEC][32];
    if (!kF32) {
        const uint16_t* src = static_cast<const uint16_t*>(x) + (m0 + quarter * 32) * ldx + c;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            uint32_t w = valid ? ldg_nc_u32(src + i * ldx) : 0u;
            v[0][i] = bf16lo(w);
            v[1 % VEC][i] = bf16hi(w);
        }
    } else {
        const float* src = static_cast<const float*>(x) + (m0 + quarter * 32) * ldx + c;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[0][i] = valid ? __uint_as_float(ldg_nc_u32(src + i * ldx)) : 0.0f;
    }

    float amax[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[e][i]));
        red[quarter][g * VEC + e] = a;
    }
    __syncthreads();
    float sc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const int col = g * VEC + e;
        amax[e] = fmaxf(fmaxf(red[0][col], red[1][col]), fmaxf(red[2][col], red[3][col]));
        sc[e] = tile_scale(amax[e]);
    }
    if (!valid) return;

#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = e4m3x2(v[e][4 * i], v[e][4 * i + 1], sc[e]) | (e4m3x2(v[e][4 * i + 2], v[e][4 * i + 3], sc[e]) << 16);
        uint8_t* dst = qT + (c + e) * M + m0 + quarter * 32;
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (quarter == 0) s[blockIdx.y * C + c + e] = sc[e];
    }
}

// ------------------------------------------------------------- weight block
//
// One CTA (256 threads) per 128x128 block.  Thread t owns the 8x8 sub-block
// rows [8a, 8a+8), columns [8b, 8b+8) with a = t / 16, b = t % 16: a warp's
// loads of one sub-block row cover two full 256-byte block rows.  The block
// amax goes through warp shuffles and shared memory.  Codes are written
// row-major (q) and, from the same quotients paired down the columns,
// transposed (qT), so q and qT hold bit-identical codes.

template <bool kF32>
__global__ void __launch_bounds__(256) quantize_weight_block_kernel(const void* __restrict__ w, int64_t N,
                                                                    int64_t K, int64_t ldw, uint8_t* __restrict__ q,
                                                                    uint8_t* __restrict__ qT,
                                                                    float* __restrict__ s) {
    __shared__ float red[8];
    const int tid = threadIdx.x;
    const int a = tid >> 4, b = tid & 15;
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * 128 + 8 * a;  // first row of the sub-block
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 128 + 8 * b;  // first column

    float v[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (!kF32) {
            const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(w) + (n0 + i) * ldw + k0;
            unpack_bf16x8(ldg_nc_v4(src), v[i]);
        } else {
            const float* src = static_cast<const float*>(w) + (n0 + i) * ldw + k0;
            uint4 lo = ldg_nc_v4(src), hi = ldg_nc_v4(src + 4);
            v[i][0] = __uint_as_float(lo.x); v[i][1] = __uint_as_float(lo.y);
            v[i][2] = __uint_as_float(lo.z); v[i][3] = __uint_as_float(lo.w);
            v[i][4] = __uint_as_float(hi.x); v[i][5] = __uint_as_float(hi.y);
            v[i][6] = __uint_as_float(hi.z); v[i][7] = __uint_as_float(hi.w);
        }
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) amax = fmaxf(amax, fabsf(v[i][jj]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
    if ((tid & 31) == 0) red[tid >> 5] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
    const float sc = tile_scale(amax);

    // quotients once, then two pairings
    float y[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) y[i][jj] = __fdiv_rn(v[i][jj], sc);

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            lo |= static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(y[i][2 * p], y[i][2 * p + 1]),
                                                                 __NV_SATFINITE, __NV_E4M3)) << (16 * p);
            hi |= static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(y[i][4 + 2 * p], y[i][5 + 2 * p]),
                                                                 __NV_SATFINITE, __NV_E4M3)) << (16 * p);
        }
        *reinterpret_cast<uint2*>(q + (n0 + i) * K + k0) = make_uint2(lo, hi);
    }
    if (qT != nullptr) {
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                lo |= static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(y[2 * p][jj], y[2 * p + 1][jj]),
                                                                     __NV_SATFINITE, __NV_E4M3)) << (16 * p);
                hi |= static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(y[4 + 2 * p][jj], y[5 + 2 * p][jj]),
                                                                     __NV_SATFINITE, __NV_E4M3)) << (16 * p);
            }
            *reinterpret_cast<uint2*>(qT + (k0 + jj) * N + n0) = make_uint2(lo, hi);
        }
    }
    if (tid == 0) s[blockIdx.y * (K >> 7) + blockIdx.x] = sc;
}

}  // namespace fp8bq
