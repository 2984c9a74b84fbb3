// MX variant of the layer: E4M3 codes with one power-of-two scale 2^E per
// 1x32 block along the reduction dimension (the block shape and 8-bit
// exponent scale, "E8M0", of the OCP Microscaling formats specification), so
// that the tensor cores apply the scales inside the MMA
// (tcgen05.mma.kind::mxf8f6f4.block_scale) and no per-chunk promotion is
// needed.  The exponent rule keeps the layer's amax/448 scale, rounded up to
// a power of two: E is the smallest integer >= -127 with amax <= 448 * 2^E,
// so nothing saturates and the largest element of a block lands in
// (224, 448]; code = E4M3(x * 2^-E), round half to even.
//
// Storage (all K-major like the block-scaled path):
//   codes      row-wise [R][C], or column-wise emitted transposed [C][M]
//   exponents  bytes E + 127, "chunk-major": e[C/128][R][4] (row-wise) or
//              e[M/128][C][4] (column-wise); byte t of row r in chunk c
//              covers elements 128c + 32t .. 128c + 32t + 31 of that row, so
//              one 32-bit word holds the four blocks of a 128-element chunk.
//
// Kernels:
//   mx_quantize_rowwise_kernel   streams 1x32 blocks with 16-byte loads
//   mx_quantize_slab_kernel      stages a 128x128 slab in shared memory for
//                                the column-wise layout, optionally also the
//                                row-wise one from the same read
//   mx_gemm_kernel               persistent, one CTA per SM, 128 x 192
//                                output tiles, TMA ring, block-scaled MMA
//                                accumulating the whole reduction in TMEM
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "gemm.cuh"
#include "ptx.cuh"
#include "quantize.cuh"

namespace fp8bq {

// Shared exponent of a block from the bits of its (non-negative) amax:
// amax = f * 2^k with f in [1, 2) and 448 = 1.75 * 2^8, so amax <= 448 * 2^E
// first holds at E = k - 8 when f <= 1.75 (mantissa field <= 0x600000) and at
// k - 7 otherwise.  Zero and FP32 subnormals (and everything below 448 *
// 2^-127) take the smallest scale, 2^-127.
__device__ __forceinline__ int mx_exponent(float amax) {
    const uint32_t u = __float_as_uint(amax);
    const int bexp = static_cast<int>(u >> 23);
    const int e = bexp - 135 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return bexp == 0 ? -127 : max(e, -127);
}

// 2^-E as FP32 (E in [-127, 121], so 127 - E in [6, 254]: always normal).
__device__ __forceinline__ float mx_inv_scale(int e) { return __uint_as_float(static_cast<uint32_t>(127 - e) << 23); }

// Two values times 2^-E -> two codes.  The product is exact unless it falls
// below 2^-126, where the code is a signed zero either way.
__device__ __forceinline__ uint32_t mx_e4m3x2(float a, float b, float inv) {
    return static_cast<uint32_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(a * inv, b * inv), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ uint32_t mx_e4m3x4(float a, float b, float c, float d, float inv) {
    return mx_e4m3x2(a, b, inv) | (mx_e4m3x2(c, d, inv) << 16);
}

// ------------------------------------------------------------------ row-wise
//
// One 1x32 block per group of L lanes (L = 4 for BF16: 8 values per lane;
// L = 8 for FP32: 4 values per lane), so one warp-wide 16-byte load reads 512
// contiguous bytes.  Each warp takes kMxRowSteps such steps with all loads in
// flight before any math.  Blocks are numbered row by row; a step starts at a
// multiple of 4 blocks and C is a multiple of 128, so each aligned group of 4
// blocks is one chunk of one row, whose four exponent bytes form one word.
constexpr int kMxRowSteps = 4;

template <bool kF32>
__global__ void __launch_bounds__(256) mx_quantize_rowwise_kernel(const void* __restrict__ x, int64_t R, int64_t C,
                                                                  int64_t ldx, uint8_t* __restrict__ q,
                                                                  uint32_t* __restrict__ ew) {
    constexpr int L = kF32 ? 8 : 4;      // lanes per block
    constexpr int BPS = 32 / L;          // blocks per warp step
    constexpr int VPL = kF32 ? 4 : 8;    // values per lane
    const int lane = threadIdx.x & 31;
    const int j = lane % L, g = lane / L;
    const uint32_t nbc = static_cast<uint32_t>(C >> 5);       // blocks per row
    const uint32_t nb = static_cast<uint32_t>(R) * nbc;       // < 2^31 (checked on the host)
    const uint32_t warp_id = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);

    uint4 w[kMxRowSteps];
#pragma unroll
    for (int u = 0; u < kMxRowSteps; ++u) {
        const uint32_t blk = (warp_id * kMxRowSteps + u) * BPS + g;
        w[u] = make_uint4(0, 0, 0, 0);
        if (blk < nb) {
            const uint32_t r = blk / nbc, t = blk - r * nbc;
            const size_t off = static_cast<size_t>(r) * ldx + t * 32 + j * VPL;
            w[u] = kF32 ? ldg_nc_v4(static_cast<const float*>(x) + off)
                        : ldg_nc_v4(static_cast<const __nv_bfloat16*>(x) + off);
        }
    }
#pragma unroll
    for (int u = 0; u < kMxRowSteps; ++u) {
        const uint32_t blk = (warp_id * kMxRowSteps + u) * BPS + g;
        const bool valid = blk < nb;
        float v[VPL];
        float amax;
        if (!kF32) {
            amax = bf16x2_max_halves(absmax_bf16x2(absmax_bf16x2(w[u].x, w[u].y), absmax_bf16x2(w[u].z, w[u].w)));
            float t8[8];
            unpack_bf16x8(w[u], t8);
#pragma unroll
            for (int i = 0; i < VPL; ++i) v[i] = t8[i];
        } else {
            v[0] = __uint_as_float(w[u].x);
            v[1] = __uint_as_float(w[u].y);
            v[2] = __uint_as_float(w[u].z);
            v[3] = __uint_as_float(w[u].w);
            amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
        }
#pragma unroll
        for (int m = 1; m < L; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
        const int e = mx_exponent(amax);
        const float inv = mx_inv_scale(e);
        // the four exponent bytes of an aligned group of 4 blocks, gathered
        // on the group's first lane (all lanes take part in the shuffles)
        const uint32_t byte = static_cast<uint32_t>(e + 127);
        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, byte, L);
        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, byte, 2 * L);
        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, byte, 3 * L);
        if (!valid) continue;
        const uint32_t r = blk / nbc, t = blk - r * nbc;
        uint8_t* dst = q + static_cast<size_t>(r) * C + t * 32 + j * VPL;
        if (!kF32)
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(mx_e4m3x4(v[0], v[1], v[2], v[3], inv), mx_e4m3x4(v[4], v[5], v[6], v[7], inv));
        else
            *reinterpret_cast<uint32_t*>(dst) = mx_e4m3x4(v[0], v[1], v[2], v[3], inv);
        if (j == 0 && (g & 3) == 0)
            ew[static_cast<size_t>(t >> 2) * R + r] = byte | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
}

// ------------------------------------------------- column-wise (and row-wise)
//
// CTA = 256 threads, slab of 128 rows (m0..) x 128 columns (c0..), copied to
// shared memory with 16-byte cp.async (row pitch 128 elements), then read in
// up to two ways:
//   column view  thread t owns column t & 127 and the 32-row blocks 2h, 2h + 1
//                (h = t >> 7): it reads its 64 values down the column (a warp
//                reads one contiguous row segment per step: no bank
//                conflicts), writes each block's 32 codes as two 16-byte
//                stores into the transposed output qT [C][M] and its two
//                exponent bytes as one 16-bit store.
//   row view     (kRows) thread t owns row t >> 1 and the 64 columns of half
//                t & 1 (two 1x32 blocks); it reads them as 16-byte chunks in
//                the rotated order (i + lane) mod n, so the 8 lanes of a
//                quarter-warp hit 8 different bank groups, keeps a per-block
//                amax with predicated maxima and writes each chunk's codes to
//                q [M][C] at the chunk's own position.
// One read of x then serves both layouts: X (Fprop row-wise, Wgrad
// column-wise), W (Fprop row-wise, Dgrad column-wise) and dY (Dgrad row-wise,
// Wgrad column-wise).
template <bool kF32>
constexpr int mx_col_smem_bytes() { return 128 * 128 * (kF32 ? 4 : 2); }

template <bool kF32, bool kRows>
__global__ void __launch_bounds__(256) mx_quantize_slab_kernel(const void* __restrict__ x, int64_t M, int64_t C,
                                                               int64_t ldx, uint8_t* __restrict__ qT,
                                                               uint16_t* __restrict__ ehT, uint8_t* __restrict__ q,
                                                               uint16_t* __restrict__ eh) {
    extern __shared__ __align__(16) uint8_t slab[];
    constexpr int ES = kF32 ? 4 : 2;
    constexpr int CPR = 128 * ES / 16;  // 16-byte chunks per slab row
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * 128;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 128;
    const uint8_t* src = static_cast<const uint8_t*>(x) + (m0 * ldx + c0) * ES;
    const uint32_t sbase = smem_addr(slab);
#pragma unroll
    for (int i = threadIdx.x; i < 128 * CPR; i += 256) {
        const int row = i / CPR, ch = i - row * CPR;
        cp_async_16(sbase + i * 16, src + static_cast<int64_t>(row) * ldx * ES + ch * 16, 16);
    }
    cp_async_wait_all();
    __syncthreads();

    {
        const int c = threadIdx.x & 127;
        const int h = threadIdx.x >> 7;
        uint32_t bytes = 0;
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
            const int b = 2 * h + bb;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int row = 32 * b + i;
                if (kF32)
                    v[i] = reinterpret_cast<const float*>(slab)[row * 128 + c];
                else
                    v[i] = __uint_as_float(
                        static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(slab)[row * 128 + c]) << 16);
            }
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
            const int e = mx_exponent(amax);
            const float inv = mx_inv_scale(e);
            uint8_t* dst = qT + (c0 + c) * M + m0 + 32 * b;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float* p = v + 16 * k;
                *reinterpret_cast<uint4*>(dst + 16 * k) =
                    make_uint4(mx_e4m3x4(p[0], p[1], p[2], p[3], inv), mx_e4m3x4(p[4], p[5], p[6], p[7], inv),
                               mx_e4m3x4(p[8], p[9], p[10], p[11], inv), mx_e4m3x4(p[12], p[13], p[14], p[15], inv));
            }
            bytes |= static_cast<uint32_t>(e + 127) << (8 * bb);
        }
        // bytes 2h, 2h + 1 of word (m0 / 128) * C + c0 + c
        ehT[((m0 >> 7) * C + c0 + c) * 2 + h] = static_cast<uint16_t>(bytes);
    }

    if (kRows) {
        constexpr int NCH = 64 * ES / 16;     // 16-byte chunks in the thread's 64 columns (8 or 16)
        constexpr int CPB = NCH / 2;          // chunks per 32-element block
        const int lane = threadIdx.x & 31;
        const int r = threadIdx.x >> 1, hf = threadIdx.x & 1;
        const uint8_t* rowp = slab + r * (128 * ES) + hf * (64 * ES);
        uint4 w[NCH];
#pragma unroll
        for (int i = 0; i < NCH; ++i) w[i] = *reinterpret_cast<const uint4*>(rowp + 16 * ((i + lane) & (NCH - 1)));
        float m[2] = {0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            float a;
            if (!kF32)
                a = bf16x2_max_halves(absmax_bf16x2(absmax_bf16x2(w[i].x, w[i].y), absmax_bf16x2(w[i].z, w[i].w)));
            else
                a = fmaxf(fmaxf(fabsf(__uint_as_float(w[i].x)), fabsf(__uint_as_float(w[i].y))),
                          fmaxf(fabsf(__uint_as_float(w[i].z)), fabsf(__uint_as_float(w[i].w))));
            const bool second = ((i + lane) & (NCH - 1)) >= CPB;
            m[0] = second ? m[0] : fmaxf(m[0], a);
            m[1] = second ? fmaxf(m[1], a) : m[1];
        }
        const int e0 = mx_exponent(m[0]), e1 = mx_exponent(m[1]);
        const float inv0 = mx_inv_scale(e0), inv1 = mx_inv_scale(e1);
        uint8_t* dst = q + (m0 + r) * C + c0 + hf * 64;
#pragma unroll
        for (int i = 0; i < NCH; ++i) {
            const int ch = (i + lane) & (NCH - 1);
            const float inv = ch >= CPB ? inv1 : inv0;
            if (!kF32) {
                float f[8];
                unpack_bf16x8(w[i], f);
                *reinterpret_cast<uint2*>(dst + 8 * ch) =
                    make_uint2(mx_e4m3x4(f[0], f[1], f[2], f[3], inv), mx_e4m3x4(f[4], f[5], f[6], f[7], inv));
            } else {
                *reinterpret_cast<uint32_t*>(dst + 4 * ch) =
                    mx_e4m3x4(__uint_as_float(w[i].x), __uint_as_float(w[i].y), __uint_as_float(w[i].z),
                              __uint_as_float(w[i].w), inv);
            }
        }
        // bytes 2hf, 2hf + 1 of word (c0 / 128) * M + m0 + r
        eh[((c0 >> 7) * M + m0 + r) * 2 + hf] = static_cast<uint16_t>((e0 + 127) | ((e1 + 127) << 8));
    }
}

// ---------------------------------------------------------------------- GEMM
//
// D[i][j] = sum_k (2^ea(i,k) A[i][k]) (2^eb(j,k) B[j][k]) for K-major E4M3
// operands A [I][K], B [J][K] and exponent words ea [K/128][I], eb [K/128][J]
// (byte t = the 32-element block 4c + t), BF16 output [I][J].  Fprop, Dgrad
// and Wgrad are all this product of the MX quantizers' outputs.
//
// Persistent, one CTA per SM, 128 x 192 output tiles (192 keeps two FP32
// accumulators, 2 x 192 columns, plus the scale-factor slots inside the 512
// TMEM columns; all 3.8B-layer widths are multiples of 192 or waste < 2 %),
// 128-deep K chunks:
//   warp 0     TMA loads of A (128 x 128 B) and B (192 x 128 B) into a
//              5-stage ring (128-byte swizzle).
//   warp 2     bulk copies of each chunk's exponent words (128 for A, up to
//              192 for B) into a 4-slot shared-memory ring.
//   warps 4-7  (one per TMEM lane quarter) copy each slot's words into a TMEM
//              scale-factor slot with tcgen05.st: word of row m in lane
//              m % 32 (every quarter holds the same copy) and column m / 32,
//              the four bytes being the chunk's four K blocks.
//   warp 1     allocates TMEM; one thread issues per chunk four
//              tcgen05.mma.kind::mxf8f6f4.block_scale (128 x 192 x 32, scale
//              byte k for step k) accumulating into one of two TMEM
//              accumulators for the whole reduction, and commits the stage,
//              the scale slot and, after a tile's last chunk, the
//              accumulator.
//   warps 8-11 (one per lane quarter) read the finished accumulator
//              (tcgen05.ld), hand it back, round to BF16 and store with TMA
//              while the next tile accumulates into the other buffer.
// Every wait is bounded; a timeout records FP8BQ_ERR_TIMEOUT in the status
// word, raises the CTA's abort flag and the CTA unwinds (in-flight copies and
// MMAs drained before TMEM is freed).
constexpr int kMxBM = 128;
constexpr int kMxBN = 192;
constexpr int kMxBK = 128;
constexpr int kMxStages = 5;
constexpr int kMxSfSlots = 4;
constexpr int kMxThreads = 384;
constexpr uint32_t kMxStageA = kMxBM * kMxBK;
constexpr uint32_t kMxStageB = kMxBN * kMxBK;
constexpr uint32_t kMxAccStride = 256;    // accumulator b at TMEM columns [256 b, 256 b + 192)
constexpr uint32_t kMxSfCol = kMxBN;      // scale slot s at columns 192 + 16 s: A +0..3, B +8..15
constexpr uint32_t kMxTmemCols = 512;
constexpr uint32_t kMxEpiWarpBytes = 2 * 2048;  // two 32 x 64-byte staging boxes per epilogue warp

struct alignas(16) MxSfSlot {
    uint32_t a[kMxBM];
    uint32_t b[kMxBN];
};

struct alignas(16) MxCtl {
    uint64_t full[kMxStages];
    uint64_t empty[kMxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t sfull[kMxSfSlots];   // the slot's exponent words landed in shared memory
    uint64_t sempty[kMxSfSlots];  // the four writer warps copied them to TMEM
    uint64_t tsfull[kMxSfSlots];  // the TMEM scale slot is written
    uint64_t tsempty[kMxSfSlots]; // the MMAs that read the TMEM slot completed
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    uint32_t issued;              // operand stages the producer issued
    uint32_t sf_issued;           // exponent slots the scale producer issued
    MxSfSlot sf[kMxSfSlots];
};

constexpr size_t kMxSmemBytes = 1024 + kMxStages * (kMxStageA + kMxStageB) + 4 * kMxEpiWarpBytes + sizeof(MxCtl);
static_assert(kMxSmemBytes <= 232448, "more dynamic shared memory than one sm_103 CTA can have");
static_assert(kMxSfCol + 16 * kMxSfSlots <= kMxAccStride, "scale slots overlap the second accumulator");
static_assert(kMxAccStride + kMxBN <= kMxTmemCols, "accumulators exceed the TMEM allocation");

struct MxParams {
    const uint32_t* ea;   // [K/128][I]
    const uint32_t* eb;   // [K/128][J]
    int I, J, KC;
    int tiles_n;          // ceil(J / 192)
    int num_tiles;        // (I / 128) * tiles_n
    uint64_t timeout_ns;
};

__device__ __forceinline__ void mx_raise_abort(MxCtl* ctl, unsigned int* status) {
    if ((threadIdx.x & 31) == 0) {
        ctl->abort = 1;
        atomicOr(status, 1u);
    }
}

__global__ void __launch_bounds__(kMxThreads, 1)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const MxParams p, unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = base;
    uint8_t* smB = base + kMxStages * kMxStageA;
    uint8_t* smEpi = smB + kMxStages * kMxStageB;
    MxCtl* ctl = reinterpret_cast<MxCtl*>(smEpi + 4 * kMxEpiWarpBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], 4);
        }
        for (int q = 0; q < kMxSfSlots; ++q) {
            mbar_init(&ctl->sfull[q], 1);
            mbar_init(&ctl->sempty[q], 4);
            mbar_init(&ctl->tsfull[q], 4);
            mbar_init(&ctl->tsempty[q], 1);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->sf_issued = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), kMxTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort;
    const uint64_t lim = p.timeout_ns;

    if (warp == 0) {
        // ----------------------------------------------------- operand producer
        uint32_t s = 0, ph = 0, issued = 0;
        bool ok = true;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++it) {
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            for (int i = 0; i < p.KC; ++i) {
                const int c = chunk_of(i, it, p.KC);  // odd tiles walk the reduction backwards
                if (!warp_wait(&ctl->empty[s], ph ^ 1, abort_flag, lim)) { ok = false; break; }
                if (lane == 0) {
                    const uint32_t fb = smem_addr(&ctl->full[s]);
                    mbar_arrive_expect_tx(&ctl->full[s], kMxStageA + kMxStageB);
                    tma_load_2d(smem_addr(smA + s * kMxStageA), &tmA, fb, c * kMxBK, tm * kMxBM);
                    tma_load_2d(smem_addr(smB + s * kMxStageB), &tmB, fb, c * kMxBK, tn * kMxBN);
                }
                ++issued;
                if (++s == kMxStages) { s = 0; ph ^= 1; }
            }
        }
        if (!ok) mx_raise_abort(ctl, status);
        if (lane == 0) ctl->issued = issued;
    } else if (warp == 2) {
        // -------------------------------------------------- exponent producer
        uint32_t q = 0, qph = 0, issued = 0;
        bool ok = true;
        int it = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++it) {
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            const int j0 = tn * kMxBN;
            const uint32_t b_bytes = static_cast<uint32_t>(min(p.J - j0, kMxBN)) * 4u;
            for (int i = 0; i < p.KC; ++i) {
                const int c = chunk_of(i, it, p.KC);  // the operand producer's order
                if (!warp_wait_backoff(&ctl->sempty[q], qph ^ 1, abort_flag, lim)) { ok = false; break; }
                if (lane == 0) {
                    MxSfSlot& sl = ctl->sf[q];
                    const uint32_t bar = smem_addr(&ctl->sfull[q]);
                    mbar_arrive_expect_tx(&ctl->sfull[q], kMxBM * 4u + b_bytes);
                    bulk_load(smem_addr(sl.a), p.ea + static_cast<int64_t>(c) * p.I + tm * kMxBM, kMxBM * 4u, bar);
                    bulk_load(smem_addr(sl.b), p.eb + static_cast<int64_t>(c) * p.J + j0, b_bytes, bar);
                }
                ++issued;
                if (++q == kMxSfSlots) { q = 0; qph ^= 1; }
            }
        }
        if (!ok) mx_raise_abort(ctl, status);
        if (lane == 0) ctl->sf_issued = issued;
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA
        bool ok = true;
        if (lane == 0) {
            uint32_t s = 0, ph = 0, q = 0, qph = 0, buf = 0, tph = 0;
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
                if (!bounded_wait(&ctl->tempty[buf], tph ^ 1, abort_flag, lim)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + buf * kMxAccStride;
                for (int c = 0; c < p.KC; ++c) {
                    if (!bounded_wait(&ctl->full[s], ph, abort_flag, lim)) { ok = false; break; }
                    if (!bounded_wait(&ctl->tsfull[q], qph, abort_flag, lim)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(smA + s * kMxStageA);
                    const uint32_t b0 = smem_addr(smB + s * kMxStageB);
                    const uint32_t sfa = tmem + kMxSfCol + 16 * q;
#pragma unroll
                    for (int k = 0; k < kMxBK / 32; ++k)
                        mma_mx_e4m3(d, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k),
                                    idesc_mx_e4m3(kMxBM, kMxBN, k), sfa, sfa + 8, (c | k) != 0);
                    mma_commit(smem_addr(&ctl->empty[s]));
                    mma_commit(smem_addr(&ctl->tsempty[q]));
                    if (++s == kMxStages) { s = 0; ph ^= 1; }
                    if (++q == kMxSfSlots) { q = 0; qph ^= 1; }
                }
                if (!ok) break;
                mma_commit(smem_addr(&ctl->tfull[buf]));
                buf ^= 1;
                if (buf == 0) tph ^= 1;
            }
        }
        __syncwarp();
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!ok) mx_raise_abort(ctl, status);
    } else if (warp >= 4 && warp < 8) {
        // -------------------------------------------- scale factors into TMEM
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        uint32_t q = 0, qph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            const int tn = tile % p.tiles_n;
            const int j0 = tn * kMxBN;
            for (int c = 0; c < p.KC; ++c) {
                if (!warp_wait(&ctl->sfull[q], qph, abort_flag, lim)) { ok = false; break; }
                if (!warp_wait(&ctl->tsempty[q], qph ^ 1, abort_flag, lim)) { ok = false; break; }
                tc_fence_after();
                const MxSfSlot& sl = ctl->sf[q];
                uint32_t bw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int n = lane + 32 * i;  // row of the B tile
                    // rows past J (and the two unused cells) get scale 1
                    bw[i] = (n < kMxBN && j0 + n < p.J) ? sl.b[n] : 0x7F7F7F7Fu;
                }
                const uint32_t col = tmem + lane_off + kMxSfCol + 16 * q;
                tmem_st_32x32b_x4(col, sl.a[lane], sl.a[lane + 32], sl.a[lane + 64], sl.a[lane + 96]);
                tmem_st_32x32b_x8(col + 8, bw);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctl->tsfull[q]);
                    mbar_arrive(&ctl->sempty[q]);
                }
                if (++q == kMxSfSlots) { q = 0; qph ^= 1; }
            }
        }
        if (!ok) mx_raise_abort(ctl, status);
    } else if (warp >= 8) {
        // ----------------------------------------------------------- epilogue
        const int quarter = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint8_t* stg0 = smEpi + (warp - 8) * kMxEpiWarpBytes;
        uint32_t buf = 0, tph = 0, nstore = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            if (!warp_wait(&ctl->tfull[buf], tph, abort_flag, lim)) { ok = false; break; }
            tc_fence_after();
            uint32_t pk[kMxBN / 2];
            const uint32_t t0 = tmem + lane_off + buf * kMxAccStride;
#pragma unroll
            for (int g = 0; g < kMxBN / 32; ++g) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(t0 + 32 * g, r);
                tmem_wait_ld();
                reg_fence32(r);
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[16 * g + i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
            buf ^= 1;
            if (buf == 0) tph ^= 1;
            // six boxes of 32 rows x 32 columns through two staging buffers
            const int y0 = tm * kMxBM + quarter * 32;
#pragma unroll
            for (int g = 0; g < kMxBN / 32; ++g) {
                uint8_t* stg = stg0 + (nstore & 1) * 2048;
                if (lane == 0) bulk_wait_group_read<1>();
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t* w = pk + 16 * g + 4 * k;
                    // 64-byte swizzle: 16-byte chunk k of row r sits at chunk k ^ ((r >> 1) & 3)
                    *reinterpret_cast<uint4*>(stg + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async_smem();
                __syncwarp();
                const int x0 = tn * kMxBN + 32 * g;
                if (lane == 0) {
                    if (x0 < p.J) tma_store_2d(&tmD, smem_addr(stg), x0, y0);
                    bulk_commit_group();
                }
                ++nstore;
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        if (!ok) mx_raise_abort(ctl, status);
    }

    // Teardown: every role has stopped (all waits are bounded).  After an
    // abort, wait (bounded) for the copies the producers issued and for the
    // MMAs in flight before TMEM is freed.
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t n = ctl->issued;
            const uint32_t f0 = n > static_cast<uint32_t>(kMxStages) ? n - kMxStages : 0;
            for (uint32_t f = f0; f < n; ++f)
                bounded_wait(&ctl->full[f % kMxStages], (f / kMxStages) & 1, nullptr, lim);
        }
        if (warp == 2 && lane == 0) {
            const uint32_t n = ctl->sf_issued;
            const uint32_t f0 = n > static_cast<uint32_t>(kMxSfSlots) ? n - kMxSfSlots : 0;
            for (uint32_t f = f0; f < n; ++f)
                bounded_wait(&ctl->sfull[f % kMxSfSlots], (f / kMxSfSlots) & 1, nullptr, lim);
        }
        if (warp == 1 && lane == 0) {
            mma_commit(smem_addr(&ctl->drain));
            bounded_wait(&ctl->drain, 0, nullptr, lim);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kMxTmemCols);
}

}  // namespace fp8bq
