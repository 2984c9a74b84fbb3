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

// Per-tile divisor: the scale, its negation and the negated correctly
// rounded reciprocal -RN(1/s).  nr == 0 marks a tile that needs IEEE division
// (amax < 2^-80); this lets the divisor travel through shared memory as two
// floats (s, nr).
struct TileDiv {
    float s, ns, nr;
};

__device__ __forceinline__ TileDiv tile_div(float amax) {
    TileDiv d;
    d.s = tile_scale(amax);
    d.ns = -d.s;
    d.nr = amax >= kRecipMinAmax ? -__frcp_rn(d.s) : 0.0f;
    return d;
}

__device__ __forceinline__ TileDiv tile_div_from(float s, float nr) {
    TileDiv d;
    d.s = s;
    d.ns = -s;
    d.nr = nr;
    return d;
}

__device__ __forceinline__ bool tile_fast(const TileDiv& d) { return d.nr != 0.0f; }

// Two NEGATED correctly rounded quotients -RN(a / s), -RN(b / s).  Fast path
// (Markstein's division theorem, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// r = RN(1/s), q0 = RN(x r) lies within one ulp of x / s, the residual
// x - q0 s is exact under FMA, and q0 + r (x - q0 s) rounded once is
// RN(x / s).  It runs on the negated quantities q0' = RN(x (-r)) = -q0 and
// e = x + q0' s, giving RN(q0' - e r) = -RN(x / s); rounding to nearest is
// symmetric, so only signed zeros could differ, and those come out negated
// too (x = -0 gives +0, x = +0 gives -0), so the sign flip after the E4M3
// conversion restores every code.  Packed f32x2 arithmetic, two quotients per
// instruction.  The slow path (tiny tiles) is IEEE division by -s.  Callers
// choose the path once per tile.
template <bool kFast>
__device__ __forceinline__ float2 neg_quot2(float a, float b, const TileDiv& d) {
    if (!kFast) return make_float2(__fdiv_rn(a, d.ns), __fdiv_rn(b, d.ns));
    float q0a, q0b;
    fmul2(q0a, q0b, a, b, d.nr, d.nr);    // q0' = -RN(x r)
    float ea = a, eb = b;
    ffma2(ea, eb, q0a, q0b, d.s, d.s);    // e = x - RN(x r) s (exact)
    ffma2(q0a, q0b, ea, eb, d.nr, d.nr);  // q0' - e r = -(q0 + e r)
    return make_float2(q0a, q0b);
}

// Two values -> the E4M3 codes of their negated quotients, packed low byte
// first (element a first).  E4M3 with saturation is symmetric in the sign.
template <bool kFast>
__device__ __forceinline__ uint32_t neg_e4m3x2(float a, float b, const TileDiv& d) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(neg_quot2<kFast>(a, b, d), __NV_SATFINITE, __NV_E4M3));
}

// Four values -> four codes of x / s in one 32-bit word (memory order): the
// codes of -x / s with every sign bit flipped.
template <bool kFast>
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float e, const TileDiv& d) {
    return (neg_e4m3x2<kFast>(a, b, d) | (neg_e4m3x2<kFast>(c, e, d) << 16)) ^ 0x80808080u;
}

// Eight values -> eight codes (memory order), path chosen per tile.
__device__ __forceinline__ uint2 e4m3x8(const float* v, const TileDiv& d) {
    if (tile_fast(d))
        return make_uint2(e4m3x4<true>(v[0], v[1], v[2], v[3], d), e4m3x4<true>(v[4], v[5], v[6], v[7], d));
    return make_uint2(e4m3x4<false>(v[0], v[1], v[2], v[3], d), e4m3x4<false>(v[4], v[5], v[6], v[7], d));
}

// Lane-wise max of |a| and |b| for two packed BF16 pairs (sign bits cleared,
// then one bf16x2 max).  Inputs are finite (NaN is outside the contract).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a & 0x7FFF7FFFu), "r"(b & 0x7FFF7FFFu));
    return d;
}

// max(|lo|, |hi|) of a packed pair whose sign bits are already clear, as FP32.
__device__ __forceinline__ float bf16x2_max_halves(uint32_t m) { return fmaxf(bf16lo(m), bf16hi(m)); }

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
// Helpers for a 1x128 row tile held by 4 lanes (32 values each, lane j owning
// the 16-byte chunks j, j+4, j+8, j+12), used by the slab kernel's row view.

// amax of a tile spread over 4 lanes (lanes 4t..4t+3 of the warp).
template <bool kF32>
__device__ __forceinline__ float quarter_amax(const float (&v)[32], uint32_t pm) {
    float a = 0.0f;
    if (!kF32) {
        a = bf16x2_max_halves(pm);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) a = fmaxf(a, fabsf(v[i]));
    }
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    return fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
}

// Writes the lane's 32 codes of a row tile to `dst` (its 128-byte row).
// Register group k holds input chunk j + 4 (k ^ flip) (flip: 0 or 1 for BF16,
// whose groups are 8 values; FP32 groups are 4 values and use flip 0).
template <bool kF32>
__device__ __forceinline__ void store_row_quarter(uint8_t* dst, int j, const float (&v)[32], const TileDiv& d,
                                                  int flip = 0) {
    if (!kF32) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<uint2*>(dst + 8 * (j + 4 * (k ^ flip))) = e4m3x8(v + 8 * k, d);
    } else {
        // FP32 chunks hold 4 values: lane j owns chunks j + 4k, k = 0..7
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
            const uint2 c = e4m3x8(v + 4 * k, d);  // chunks j+4k and j+4k+4
            *reinterpret_cast<uint32_t*>(dst + 4 * (j + 4 * k)) = c.x;
            *reinterpret_cast<uint32_t*>(dst + 4 * (j + 4 * k + 4)) = c.y;
        }
    }
}

// Streaming kernel: one 1x128 tile per group of 8 lanes (4 tiles per warp),
// lane j owning elements [8j, 8j+8) and [64+8j, 64+8j+8) (BF16) or
// [4j + 32p, 4j + 32p + 4), p = 0..3 (FP32), so each warp-wide 16-byte load
// reads whole 128-byte lines.
template <bool kF32>
__global__ void __launch_bounds__(256) quantize_rowwise_kernel(const void* __restrict__ x, int64_t R, int64_t C,
                                                               int64_t ldx, uint8_t* __restrict__ q,
                                                               float* __restrict__ s) {
    const int lane = threadIdx.x & 31;
    const int j = lane & 7;
    const uint32_t T = static_cast<uint32_t>(C >> 7);
    const uint32_t ntiles = static_cast<uint32_t>(R) * T;  // < 2^31 (checked on the host)
    const uint32_t tile = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 4u + (lane >> 3);
    const bool valid = tile < ntiles;
    const uint32_t r = valid ? tile / T : 0;
    const uint32_t t = valid ? tile - r * T : 0;

    float v[16];
    float amax = 0.0f;
    if (!kF32) {
        const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(x) + static_cast<int64_t>(r) * ldx + t * 128;
        uint4 wa = make_uint4(0, 0, 0, 0), wb = make_uint4(0, 0, 0, 0);
        if (valid) {
            wa = ldg_nc_v4(src + 8 * j);
            wb = ldg_nc_v4(src + 64 + 8 * j);
        }
        amax = bf16x2_max_halves(absmax_bf16x2(absmax_bf16x2(absmax_bf16x2(wa.x, wa.y), absmax_bf16x2(wa.z, wa.w)),
                                               absmax_bf16x2(absmax_bf16x2(wb.x, wb.y), absmax_bf16x2(wb.z, wb.w))));
        float a[8], b[8];
        unpack_bf16x8(wa, a);
        unpack_bf16x8(wb, b);
#pragma unroll
        for (int i = 0; i < 8; ++i) { v[i] = a[i]; v[8 + i] = b[i]; }
    } else {
        const float* src = static_cast<const float*>(x) + static_cast<int64_t>(r) * ldx + t * 128;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (valid) w = ldg_nc_v4(src + 32 * p + 4 * j);
            v[4 * p + 0] = __uint_as_float(w.x);
            v[4 * p + 1] = __uint_as_float(w.y);
            v[4 * p + 2] = __uint_as_float(w.z);
            v[4 * p + 3] = __uint_as_float(w.w);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    const TileDiv d = tile_div(amax);

    if (!valid) return;
    uint8_t* dst = q + static_cast<int64_t>(r) * C + t * 128;
    if (!kF32) {
        *reinterpret_cast<uint2*>(dst + 8 * j) = e4m3x8(v, d);
        *reinterpret_cast<uint2*>(dst + 64 + 8 * j) = e4m3x8(v + 8, d);
    } else {
        const uint2 c0 = e4m3x8(v, d), c1 = e4m3x8(v + 8, d);
        *reinterpret_cast<uint32_t*>(dst + 4 * j) = c0.x;
        *reinterpret_cast<uint32_t*>(dst + 32 + 4 * j) = c0.y;
        *reinterpret_cast<uint32_t*>(dst + 64 + 4 * j) = c1.x;
        *reinterpret_cast<uint32_t*>(dst + 96 + 4 * j) = c1.y;
    }
    if (j == 0) s[static_cast<int64_t>(t) * R + r] = d.s;
}

// ------------------------------------------------------------- 128x128 slabs
//
// CTA = 256 threads, one slab of 128 rows x 128 columns (rows r0.., columns
// c0..; all 128 rows exist, trailing columns past C read as zero and are not
// written).  The slab is copied to shared memory with 16-byte cp.async
// (row pitch 128 * element size), then read in two ways:
//   column view  thread = (4-byte unit u of a row, group g of rows): BF16 has
//                64 units (column pairs) x 4 groups of 32 rows, FP32 128
//                units (columns) x 2 groups of 64 rows.  A warp reads 128
//                contiguous bytes of one row (no bank conflicts).  Partial
//                column amaxes meet in shared memory; one thread per column
//                forms its divisor, which every group then reads; codes of a
//                column's rows are contiguous in the transposed output.
//   row view     4 lanes per row, 32 values per lane (chunks j + 4k), 64 rows
//                per pass, 2 passes; odd rows take their chunks in the order
//                k ^ 1 so the two rows a quarter-warp reads hit different
//                banks.
// Modes:
//   kTileCol     column-wise 128x1 tiles: qT [C][R], s_col [R/128][C]
//   kTileDual    row-wise 1x128 and column-wise 128x1 tiles of the same
//                slab: q [R][C], s_row [C/128][R], qT, s_col (one read of x)
//   kTileWeight  one 128x128 block: q [R][C], qT [C][R] (optional),
//                s_row = block scales [R/128][C/128]
//   kTileSwiglu  BF16 only: x holds g in columns [0, C) and u in columns
//                [uoff, uoff + C); the slab becomes H = BF16(silu(g) * u)
//                (optionally written to h), then as kTileDual on H

enum TileMode : int { kTileCol = 0, kTileDual = 1, kTileWeight = 2, kTileSwiglu = 3 };

template <bool kF32, int kMode = kTileDual>
__host__ __device__ constexpr int tile_smem_bytes() { return 128 * 128 * (kF32 ? 4 : 2) * (kMode == kTileSwiglu ? 2 : 1); }

// h = silu(g) * u = g u / (1 + exp(-g)) in FP32, rounded to BF16 once.  The
// exponential is the hardware approximation (__expf, relative error below
// 2e-5 for |g| <= 88) and the division a correctly rounded reciprocal times
// g: together far inside half a BF16 ulp (2^-9), so the BF16 h is within one
// ulp of the exact value.  exp(-g) beyond the FP32 range is +inf and gives
// h = +-0; the reciprocal keeps the FP32-subnormal range of 1 + exp(-g)
// (g between about -88.7 and -87.3) exact enough.
__device__ __forceinline__ float swiglu_f32(float g, float u) {
    return __fmul_rn(__fmul_rn(g, __frcp_rn(__fadd_rn(1.0f, __expf(-g)))), u);
}

// swiglu_f32 with the hardware reciprocal approximation (relative error about
// 2^-23) in place of the correctly rounded one: the same bound holds, but the
// approximation flushes results below 2^-126 to zero, so it is only used
// when g > -87 (1 + exp(-g) < 2^126).
__device__ __forceinline__ float swiglu_f32_fast(float g, float u) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.0f, __expf(-g))));
    return __fmul_rn(__fmul_rn(g, r), u);
}

// Shared-memory scratch of one slab's processing (besides the slab itself).
template <bool kF32>
struct SlabScratch {
    static constexpr int G = 256 / ((128 * (kF32 ? 4 : 2)) / 4);   // row groups of the column view
    float red[G][128];
    float cdiv[2][128];    // per column (or [.][0] for the block): s, nr
    float wred[8];
};

// Issues the 16-byte cp.async copies of the slab at (r0, c0) into shared
// memory at `sbase` (row pitch 128 elements; the u slab of the SwiGLU mode
// right after the g slab).  Columns past C read as zero.
template <bool kF32, int kMode>
__device__ __forceinline__ void slab_load(uint32_t sbase, const uint8_t* xb, int64_t r0, int64_t c0, int64_t C,
                                          int64_t ldx, int64_t uoff, int tid) {
    constexpr int E = kF32 ? 4 : 2;
    constexpr int RB = 128 * E;
    constexpr int CPR = RB / 16;
#pragma unroll
    for (int k = 0; k < (128 * CPR) / 256; ++k) {
        const int i = tid + 256 * k;
        const int row = i / CPR, ch = i % CPR;
        const int64_t col = c0 + ch * (16 / E);
        const bool ok = col < C;
        const uint8_t* src = xb + ((r0 + row) * ldx + (ok ? col : c0)) * E;
        cp_async_16(sbase + row * RB + ch * 16, src, ok ? 16u : 0u);
        if (kMode == kTileSwiglu)  // u slab right after the g slab
            cp_async_16(sbase + 128 * RB + row * RB + ch * 16, src + uoff * E, ok ? 16u : 0u);
    }
}

// Quantizes the slab at (r0, c0), already in shared memory at `slab`, into
// the outputs of mode kMode (see the list above).  Every thread of the
// 256-thread CTA takes part; the slab may be overwritten once it returns and
// the CTA has synchronized.
template <bool kF32, int kMode>
__device__ __forceinline__ void slab_process(uint8_t* __restrict__ slab, SlabScratch<kF32>& sc, int64_t r0, int64_t c0,
                                             int64_t R, int64_t C, uint8_t* __restrict__ q, float* __restrict__ s_row,
                                             uint8_t* __restrict__ qT, float* __restrict__ s_col,
                                             uint16_t* __restrict__ h, int tid) {
    constexpr int E = kF32 ? 4 : 2;
    constexpr int RB = 128 * E;       // slab row pitch in shared memory (bytes)
    constexpr int CPR = RB / 16;      // 16-byte chunks per row
    constexpr int UPR = RB / 4;       // 4-byte units per row (column view)
    constexpr int VEC = 4 / E;        // columns per unit
    constexpr int G = 256 / UPR;      // row groups (column view)
    constexpr int RPG = 128 / G;      // rows per group
    float (&red)[G][128] = sc.red;
    float (&cdiv)[2][128] = sc.cdiv;
    float (&wred)[8] = sc.wred;

    if (kMode == kTileSwiglu) {
        // H = BF16(silu(g) * u), in place over the g slab (and to h)
#pragma unroll
        for (int k = 0; k < (128 * CPR) / 256; ++k) {
            const int i = tid + 256 * k;
            const int row = i / CPR, ch = i % CPR;
            uint4* gp = reinterpret_cast<uint4*>(slab + row * RB + ch * 16);
            const uint4 gw = *gp;
            const uint4 uw = *reinterpret_cast<const uint4*>(slab + 128 * RB + row * RB + ch * 16);
            const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w}, uv[4] = {uw.x, uw.y, uw.z, uw.w};
            uint32_t hv[4];
            bool fast = true;
#pragma unroll
            for (int m = 0; m < 4; ++m) fast = fast && bf16lo(gv[m]) > -87.0f && bf16hi(gv[m]) > -87.0f;
            if (__all_sync(0xFFFFFFFFu, fast)) {   // the whole warp takes the fast form
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    __nv_bfloat162 hb = __floats2bfloat162_rn(swiglu_f32_fast(bf16lo(gv[m]), bf16lo(uv[m])),
                                                              swiglu_f32_fast(bf16hi(gv[m]), bf16hi(uv[m])));
                    hv[m] = *reinterpret_cast<uint32_t*>(&hb);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    __nv_bfloat162 hb = __floats2bfloat162_rn(swiglu_f32(bf16lo(gv[m]), bf16lo(uv[m])),
                                                              swiglu_f32(bf16hi(gv[m]), bf16hi(uv[m])));
                    hv[m] = *reinterpret_cast<uint32_t*>(&hb);
                }
            }
            const uint4 hw = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *gp = hw;
            const int64_t col = c0 + ch * 8;
            if (h != nullptr && col < C) *reinterpret_cast<uint4*>(h + (r0 + row) * C + col) = hw;
        }
        __syncthreads();
    }

    // ---- column view: this thread's column(s) over its row group (BF16:
    //      kept in registers for the code pass; FP32 re-reads shared memory)
    const int u = tid % UPR, g = tid / UPR;
    const uint8_t* colp = slab + g * RPG * RB + u * 4;
    constexpr int NCW = kF32 ? 1 : RPG;
    uint32_t cw[NCW] = {};
    auto colword = [&](int i) -> uint32_t {
        return kF32 ? *reinterpret_cast<const uint32_t*>(colp + i * RB) : cw[kF32 ? 0 : i];
    };
    float cmax[VEC];
    if (!kF32) {
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < NCW; ++i) {
            cw[i] = *reinterpret_cast<const uint32_t*>(colp + i * RB);
            m = absmax_bf16x2(m, cw[i]);
        }
        cmax[0] = bf16lo(m);
        cmax[VEC - 1] = bf16hi(m);
    } else {
        cmax[0] = 0.0f;
#pragma unroll 8
        for (int i = 0; i < RPG; ++i) cmax[0] = fmaxf(cmax[0], fabsf(__uint_as_float(colword(i))));
    }
    if (kMode != kTileWeight) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) red[g][u * VEC + e] = cmax[e];
        __syncthreads();
        if (tid < 128) {  // one thread per column forms the divisor
            float a = red[0][tid];
#pragma unroll
            for (int gg = 1; gg < G; ++gg) a = fmaxf(a, red[gg][tid]);
            const TileDiv d = tile_div(a);
            cdiv[0][tid] = d.s;
            cdiv[1][tid] = d.nr;
            if (c0 + tid < C) s_col[(r0 >> 7) * C + c0 + tid] = d.s;
        }
    } else {
        float a = cmax[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) a = fmaxf(a, cmax[e]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, off));
        if ((tid & 31) == 0) wred[tid >> 5] = a;
        __syncthreads();
        if (tid == 0) {
            a = wred[0];
#pragma unroll
            for (int w = 1; w < 8; ++w) a = fmaxf(a, wred[w]);
            const TileDiv d = tile_div(a);
            cdiv[0][0] = d.s;
            cdiv[1][0] = d.nr;
            s_row[(r0 >> 7) * (C >> 7) + (c0 >> 7)] = d.s;
        }
    }
    __syncthreads();

    // ---- column view: codes, transposed (qT[c][r0 + g*RPG ...], 16 rows per store)
    if (kMode != kTileWeight || qT != nullptr) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int cc = u * VEC + e;
            const int64_t c = c0 + cc;
            if (c < C) {
                const int di = kMode == kTileWeight ? 0 : cc;
                const TileDiv d = tile_div_from(cdiv[0][di], cdiv[1][di]);
                uint8_t* dst = qT + c * R + r0 + g * RPG;
#pragma unroll
                for (int h = 0; h < RPG / 16; ++h) {
                    float f[16];
#pragma unroll
                    for (int m = 0; m < 16; ++m) {
                        const uint32_t w = colword(h * 16 + m);
                        f[m] = kF32 ? __uint_as_float(w) : (e == 0 ? bf16lo(w) : bf16hi(w));
                    }
                    const uint2 lo = e4m3x8(f, d), hi = e4m3x8(f + 8, d);
                    *reinterpret_cast<uint4*>(dst + h * 16) = make_uint4(lo.x, lo.y, hi.x, hi.y);
                }
            }
        }
    }

    // ---- row view: row-wise tiles (dual) or the block's row-major codes (weight)
    if (kMode == kTileCol) return;
    const int j = tid & 3;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int row = pass * 64 + (tid >> 2);
        const uint8_t* rp = slab + row * RB;
        // BF16: odd rows take chunk j + 4 (k ^ 1) into register group k, so
        // the two rows a quarter-warp reads hit different banks (FP32 rows
        // are 512 bytes, one row per quarter-warp: no conflict to avoid).
        const int flip = kF32 ? 0 : (row & 1);
        float v[32];
        uint32_t pm = 0;
        if (!kF32) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 w = *reinterpret_cast<const uint4*>(rp + 16 * (j + 4 * (k ^ flip)));
                    if (kMode == kTileDual || kMode == kTileSwiglu)
                    pm = absmax_bf16x2(pm, absmax_bf16x2(absmax_bf16x2(w.x, w.y), absmax_bf16x2(w.z, w.w)));
                float t[8];
                unpack_bf16x8(w, t);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[8 * k + i] = t[i];
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 w = *reinterpret_cast<const uint4*>(rp + 16 * (j + 4 * k));
                v[4 * k + 0] = __uint_as_float(w.x);
                v[4 * k + 1] = __uint_as_float(w.y);
                v[4 * k + 2] = __uint_as_float(w.z);
                v[4 * k + 3] = __uint_as_float(w.w);
            }
        }
        TileDiv d;
        if (kMode == kTileDual || kMode == kTileSwiglu) {
            d = tile_div(quarter_amax<kF32>(v, pm));
            if (j == 0) s_row[(c0 >> 7) * R + r0 + row] = d.s;
        } else {
            d = tile_div_from(cdiv[0][0], cdiv[1][0]);
        }
        store_row_quarter<kF32>(q + (r0 + row) * C + c0, j, v, d, flip);
    }
}

template <bool kF32, int kMode>
__global__ void __launch_bounds__(256, 4) quantize_tile_kernel(const void* __restrict__ x, int64_t R, int64_t C,
                                                            int64_t ldx, uint8_t* __restrict__ q,
                                                            float* __restrict__ s_row, uint8_t* __restrict__ qT,
                                                            float* __restrict__ s_col, int64_t uoff = 0,
                                                            uint16_t* __restrict__ h = nullptr) {
    static_assert(kMode != kTileSwiglu || !kF32, "the SwiGLU mode takes BF16 input");
    extern __shared__ __align__(16) uint8_t slab[];
    __shared__ SlabScratch<kF32> sc;
    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
    slab_load<kF32, kMode>(smem_addr(slab), static_cast<const uint8_t*>(x), r0, c0, C, ldx, uoff, tid);
    cp_async_wait_all();
    __syncthreads();
    slab_process<kF32, kMode>(slab, sc, r0, c0, R, C, q, s_row, qT, s_col, h, tid);
}

// Several weights' 128x128 block quantization in one launch: block b of the
// grid is block b - first_block[i] (row-major over that weight's blocks) of
// weight i, first_block[i] <= b < first_block[i + 1].  One launch replaces a
// launch per weight, whose short grids end in a partly idle wave each.
constexpr int kMaxWeightGroup = 16;

struct WeightGroup {
    int n;
    int first_block[kMaxWeightGroup + 1];
    int nbx[kMaxWeightGroup];   // blocks per row of blocks (K / 128)
    const void* w[kMaxWeightGroup];
    int64_t N[kMaxWeightGroup], K[kMaxWeightGroup], ldw[kMaxWeightGroup];
    uint8_t* q[kMaxWeightGroup];
    uint8_t* qT[kMaxWeightGroup];
    float* s[kMaxWeightGroup];
};

template <bool kF32>
__global__ void __launch_bounds__(256, 4) quantize_weight_group_kernel(const __grid_constant__ WeightGroup g) {
    extern __shared__ __align__(16) uint8_t slab[];
    __shared__ SlabScratch<kF32> sc;
    const int tid = threadIdx.x;
    const int b = static_cast<int>(blockIdx.x);
    int i = 0;
    while (i + 1 < g.n && b >= g.first_block[i + 1]) ++i;
    const int lb = b - g.first_block[i];
    const int64_t r0 = static_cast<int64_t>(lb / g.nbx[i]) * 128;
    const int64_t c0 = static_cast<int64_t>(lb % g.nbx[i]) * 128;
    slab_load<kF32, kTileWeight>(smem_addr(slab), static_cast<const uint8_t*>(g.w[i]), r0, c0, g.K[i], g.ldw[i], 0,
                                 tid);
    cp_async_wait_all();
    __syncthreads();
    slab_process<kF32, kTileWeight>(slab, sc, r0, c0, g.N[i], g.K[i], g.q[i], g.s[i], g.qT[i], nullptr, nullptr, tid);
}

}  // namespace fp8bq
