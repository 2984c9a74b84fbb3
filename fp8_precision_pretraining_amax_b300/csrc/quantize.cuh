// Fused amax + scale + E4M3 cast kernels (HBM-bound).
//
// Rule implemented (fine-grained block quantization that the Puro-2B report,
// section 2 "FP8", adopts from DeepSeek-V3 for its main linear layers):
// per tile, amax = max |x|; s = amax / 448 rounded to FP32 (s = 1 when
// amax == 0); code = E4M3(x / s) where x / s is the correctly rounded FP32
// quotient and E4M3() rounds half to even with saturation to +-448.
//
// Two kernel families, both reading their input exactly once:
//   quantize_rowwise_kernel  streams 1x128 tiles straight from HBM with
//                            128-bit coalesced loads (no shared memory).
//   quantize_tile_kernel     stages a 128x128 slab in shared memory with
//                            16-byte cp.async copies and serves every layout
//                            that needs columns: column-wise 128x1 tiles
//                            emitted transposed, the fused row-wise +
//                            column-wise pass over one slab, and 128x128
//                            weight blocks (row-major and transposed codes).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ptx.cuh"

namespace fp8bq {

// ------------------------------------------------------------ element math

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// s = amax / 448 (IEEE, round to nearest even), 1 for an all-zero tile.
__device__ __forceinline__ float tile_scale(float amax) {
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Below this tile amax the reciprocal-based quotient is not guaranteed to be
// the correctly rounded one (the residual x - q0 s can fall into the FP32
// subnormal range and lose bits), so such tiles use IEEE division.  Checked
// exhaustively over every pair of BF16 values (x, amax), |x| <= amax.
constexpr float kRecipMinAmax = 0x1p-80f;

// Per-tile divisor: the scale, its correctly rounded reciprocal, and whether
// the one-step reciprocal quotient applies.
struct TileDiv {
    float s, ns, r;
    bool fast;
};

__device__ __forceinline__ TileDiv tile_div(float amax) {
    TileDiv d;
    d.s = tile_scale(amax);
    d.ns = -d.s;
    d.r = __frcp_rn(d.s);
    d.fast = amax >= kRecipMinAmax;
    return d;
}

// Sign of x copied onto q: x / s carries the sign of x (s > 0), which the
// correction step below loses for x = -0 only.
__device__ __forceinline__ float with_sign_of(float q, float x) {
    return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

// Two correctly rounded quotients a / s, b / s.  Fast path (Markstein's
// division theorem, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with r = RN(1/s),
// q0 = RN(x r) lies within one ulp of x / s, the residual x - q0 s is exact
// under FMA, and q0 + r (x - q0 s) rounded once is RN(x / s).  Packed f32x2
// arithmetic, two quotients per instruction.
__device__ __forceinline__ float2 quot2(float a, float b, const TileDiv& d) {
    if (!d.fast) return make_float2(__fdiv_rn(a, d.s), __fdiv_rn(b, d.s));
    float q0a, q0b;
    fmul2(q0a, q0b, a, b, d.r, d.r);
    float ea = a, eb = b;
    ffma2(ea, eb, q0a, q0b, d.ns, d.ns);  // e = x - q0 s (exact)
    ffma2(q0a, q0b, ea, eb, d.r, d.r);    // q = q0 + e r
    return make_float2(with_sign_of(q0a, a), with_sign_of(q0b, b));
}

// Two values -> two E4M3 codes packed low byte first (element a first).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b, const TileDiv& d) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(quot2(a, b, d), __NV_SATFINITE, __NV_E4M3));
}

// Four values -> four codes in one 32-bit word (memory order).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float e, const TileDiv& d) {
    return e4m3x2(a, b, d) | (e4m3x2(c, e, d) << 16);
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

// 16-byte global -> shared copy that bypasses L1; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
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
    const TileDiv d = tile_div(amax);

    if (!valid) return;
    uint8_t* dst = q + r * C + t * 128;
    if (!kF32) {
        *reinterpret_cast<uint2*>(dst + 8 * j) =
            make_uint2(e4m3x4(v[0], v[1], v[2], v[3], d), e4m3x4(v[4], v[5], v[6], v[7], d));
        *reinterpret_cast<uint2*>(dst + 64 + 8 * j) =
            make_uint2(e4m3x4(v[8], v[9], v[10], v[11], d), e4m3x4(v[12], v[13], v[14], v[15], d));
    } else {
#pragma unroll
        for (int p = 0; p < 4; ++p)
            *reinterpret_cast<uint32_t*>(dst + 32 * p + 4 * j) =
                e4m3x4(v[4 * p], v[4 * p + 1], v[4 * p + 2], v[4 * p + 3], d);
    }
    if (j == 0) s[t * R + r] = d.s;
}

// ------------------------------------------------------------- 128x128 slabs
//
// CTA = 256 threads, one slab of 128 rows x 128 columns (rows r0.., columns
// c0..; all 128 rows exist, trailing columns past C read as zero and are not
// written).  The slab is copied to shared memory with 16-byte cp.async
// (row pitch 128 * element size), then read in two ways, both free of bank
// conflicts because every warp access covers contiguous bytes of one row:
//   column view  thread = (4-byte unit u of a row, group g of rows): BF16 has
//                64 units (column pairs) x 4 groups of 32 rows, FP32 128
//                units (columns) x 2 groups of 64 rows.  Per-column amax over
//                the group, combined over groups in shared memory; codes of
//                a column's rows are contiguous in the transposed output.
//   row view     8 lanes per row, 16 values per lane (the row-wise kernel's
//                mapping), 32 rows per pass, 4 passes.
// Modes:
//   kTileCol     column-wise 128x1 tiles: qT [C][R], s_col [R/128][C]
//   kTileDual    row-wise 1x128 and column-wise 128x1 tiles of the same
//                slab: q [R][C], s_row [C/128][R], qT, s_col (one read of x)
//   kTileWeight  one 128x128 block: q [R][C], qT [C][R] (optional),
//                s_row = block scales [R/128][C/128]

enum TileMode : int { kTileCol = 0, kTileDual = 1, kTileWeight = 2 };

template <bool kF32>
constexpr int tile_smem_bytes() { return 128 * 128 * (kF32 ? 4 : 2); }

template <bool kF32, int kMode>
__global__ void __launch_bounds__(256) quantize_tile_kernel(const void* __restrict__ x, int64_t R, int64_t C,
                                                            int64_t ldx, uint8_t* __restrict__ q,
                                                            float* __restrict__ s_row, uint8_t* __restrict__ qT,
                                                            float* __restrict__ s_col) {
    constexpr int E = kF32 ? 4 : 2;
    constexpr int RB = 128 * E;       // slab row pitch in shared memory (bytes)
    constexpr int CPR = RB / 16;      // 16-byte chunks per row
    constexpr int UPR = RB / 4;       // 4-byte units per row (column view)
    constexpr int VEC = 4 / E;        // columns per unit
    constexpr int G = 256 / UPR;      // row groups (column view)
    constexpr int RPG = 128 / G;      // rows per group
    extern __shared__ __align__(16) uint8_t slab[];
    __shared__ float red[G][128];
    __shared__ float wred[8];

    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
    const uint8_t* xb = static_cast<const uint8_t*>(x);

    // ---- stage the slab
    const uint32_t sbase = smem_addr(slab);
#pragma unroll
    for (int k = 0; k < (128 * CPR) / 256; ++k) {
        const int i = tid + 256 * k;
        const int row = i / CPR, ch = i % CPR;
        const int64_t col = c0 + ch * (16 / E);
        const bool ok = col < C;
        const uint8_t* src = xb + ((r0 + row) * ldx + (ok ? col : c0)) * E;
        cp_async_16(sbase + row * RB + ch * 16, src, ok ? 16u : 0u);
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- column view: amax of this thread's column(s) over its row group
    const int u = tid % UPR, g = tid / UPR;
    const uint8_t* colp = slab + g * RPG * RB + u * 4;
    float cmax[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) cmax[e] = 0.0f;
#pragma unroll 8
    for (int i = 0; i < RPG; ++i) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(colp + i * RB);
        if (!kF32) {
            cmax[0] = fmaxf(cmax[0], fabsf(bf16lo(w)));
            cmax[VEC - 1] = fmaxf(cmax[VEC - 1], fabsf(bf16hi(w)));
        } else {
            cmax[0] = fmaxf(cmax[0], fabsf(__uint_as_float(w)));
        }
    }
    TileDiv cd[VEC];
    if (kMode != kTileWeight) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) red[g][u * VEC + e] = cmax[e];
        __syncthreads();
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            float a = red[0][u * VEC + e];
#pragma unroll
            for (int gg = 1; gg < G; ++gg) a = fmaxf(a, red[gg][u * VEC + e]);
            cd[e] = tile_div(a);
        }
    } else {
        float a = cmax[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) a = fmaxf(a, cmax[e]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
        if ((tid & 31) == 0) wred[tid >> 5] = a;
        __syncthreads();
        a = wred[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) a = fmaxf(a, wred[w]);
#pragma unroll
        for (int e = 0; e < VEC; ++e) cd[e] = tile_div(a);
        if (tid == 0) s_row[(r0 >> 7) * (C >> 7) + (c0 >> 7)] = cd[0].s;
    }

    // ---- column view: codes, transposed (qT[c][r0 + g*RPG ...], 16 rows per store)
    if (kMode != kTileWeight || qT != nullptr) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int64_t c = c0 + u * VEC + e;
            if (c < C) {
                uint8_t* dst = qT + c * R + r0 + g * RPG;
#pragma unroll
                for (int h = 0; h < RPG / 16; ++h) {
                    uint32_t wv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float f[4];
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            const uint32_t w =
                                *reinterpret_cast<const uint32_t*>(colp + (h * 16 + k * 4 + m) * RB);
                            f[m] = kF32 ? __uint_as_float(w) : (e == 0 ? bf16lo(w) : bf16hi(w));
                        }
                        wv[k] = e4m3x4(f[0], f[1], f[2], f[3], cd[e]);
                    }
                    *reinterpret_cast<uint4*>(dst + h * 16) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                if (kMode != kTileWeight && g == 0) s_col[(r0 >> 7) * C + c] = cd[e].s;
            }
        }
    }

    // ---- row view: row-wise tiles (dual) or the block's row-major codes (weight)
    if (kMode == kTileCol) return;
    const int j = tid & 7;
#pragma unroll 1
    for (int p = 0; p < 4; ++p) {
        const int row = p * 32 + (tid >> 3);
        const uint8_t* rp = slab + row * RB;
        float v[16];
        if (!kF32) {
            float a[8], b[8];
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rp + 16 * j), a);
            unpack_bf16x8(*reinterpret_cast<const uint4*>(rp + 16 * (j + 8)), b);
#pragma unroll
            for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 w = *reinterpret_cast<const uint4*>(rp + 16 * (j + 8 * k));
                v[4 * k + 0] = __uint_as_float(w.x);
                v[4 * k + 1] = __uint_as_float(w.y);
                v[4 * k + 2] = __uint_as_float(w.z);
                v[4 * k + 3] = __uint_as_float(w.w);
            }
        }
        TileDiv d;
        if (kMode == kTileDual) {
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
            d = tile_div(amax);
            if (j == 0) s_row[(c0 >> 7) * R + r0 + row] = d.s;
        } else {
            d = cd[0];
        }
        uint8_t* dst = q + (r0 + row) * C + c0;
        if (!kF32) {
            *reinterpret_cast<uint2*>(dst + 8 * j) =
                make_uint2(e4m3x4(v[0], v[1], v[2], v[3], d), e4m3x4(v[4], v[5], v[6], v[7], d));
            *reinterpret_cast<uint2*>(dst + 64 + 8 * j) =
                make_uint2(e4m3x4(v[8], v[9], v[10], v[11], d), e4m3x4(v[12], v[13], v[14], v[15], d));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint32_t*>(dst + 32 * k + 4 * j) =
                    e4m3x4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3], d);
        }
    }
}

}  // namespace fp8bq
