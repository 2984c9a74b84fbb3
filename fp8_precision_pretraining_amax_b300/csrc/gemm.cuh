// Block-scaled FP8 GEMM on the sm_103a tensor cores (tcgen05, TMEM, TMA).
//
// One kernel serves Fprop, Dgrad and Wgrad.  In all three the operands are
// K-major E4M3 codes (the reduction dimension is contiguous):
//   A [I][Kr] with per-row, per-chunk scales sA[c][i]         (row tiles)
//   B [J][Kr] with per-chunk scales that depend on the mode:
//     Fprop  sB(c, j) = sw[j/128][c]     (weight blocks, B = Wq)
//     Dgrad  sB(c, j) = sw[c][j/128]     (weight blocks, B = Wq^T)
//     Wgrad  sB(c, j) = sxT[c][j]        (column tiles of X, B = Xq^T)
//   D[i][j] = sum_c sA(c,i) * sB(c,j) * sum_{k in chunk c} A[i][k] B[j][k]
// which is the per-128-chunk scale promotion with FP32 accumulation that the
// Puro-2B report's FP8 recipe (section 2, after DeepSeek-V3) relies on.
//
// Design (one persistent CTA per SM, 384 threads = 3 warpgroups):
//   warp 0      TMA producer: 128x128 A tile + 256x128 B tile per chunk into a
//               4-stage shared-memory ring (128-byte swizzle), mbarrier tx.
//   warp 1      MMA issuer (one thread): four tcgen05.mma kind::f8f6f4
//               (128x256x32) per chunk into one of two TMEM partial buffers
//               of 256 FP32 columns, started fresh every chunk, then
//               tcgen05.commit to release the smem stage and publish the
//               partial.
//   warps 2, 3  idle (the first warpgroup gives up registers: 40 per thread)
//   warps 4..11 promotion (two warpgroups at 232 registers per thread): each
//               thread owns one output row and 128 columns;
//               it reads the chunk partial from TMEM (tcgen05.ld), multiplies
//               by the chunk's scale product and adds it into FP32 registers.
//               While it does so the tensor core is already computing the
//               next chunk into the other TMEM buffer.  After the last chunk
//               the accumulators are rounded to BF16 and stored.
// Every wait is bounded: a stalled pipeline records FP8BQ_ERR_TIMEOUT in the
// device status word and the CTA unwinds (draining its own in-flight copies
// and MMAs, then freeing TMEM) instead of hanging.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"

namespace fp8bq {

enum GemmMode : int { kModeFprop = 0, kModeDgrad = 1, kModeWgrad = 2 };

constexpr int kBM = 128;          // tile rows (TMEM lanes)
constexpr int kBN = 256;          // tile columns (MMA N)
constexpr int kBK = 128;          // one scale chunk of the reduction
constexpr int kStages = 3;
constexpr int kGemmThreads = 384;
constexpr int kFirstPromoWarp = 4;
constexpr int kPromoWarps = 8;
constexpr uint32_t kStageBytesA = kBM * kBK;
constexpr uint32_t kStageBytesB = kBN * kBK;
constexpr uint32_t kTmemCols = 2 * kBN;
// Epilogue staging: per promotion warp 32 rows x 128 BF16 columns as two
// 32 x 64 boxes of 128-byte rows, 128-byte swizzled for the TMA store.
constexpr uint32_t kEpiBoxBytes = 32 * 128;
constexpr uint32_t kEpiWarpBytes = 2 * kEpiBoxBytes;

struct GemmParams {
    const float* sA;
    const float* sB;
    uint16_t* D;          // [I][J] BF16 bit patterns
    int I, J, KC;         // output rows, output columns, reduction chunks
    int tiles_n;          // ceil(J / kBN)
    int num_tiles;
    uint64_t timeout_ns;
};

struct alignas(16) GemmCtl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    float sbw[kPromoWarps][2][128];  // Wgrad column scales: [warp][chunk parity][column]
};

constexpr size_t kGemmSmemBytes =
    1024 + kStages * (kStageBytesA + kStageBytesB) + kPromoWarps * kEpiWarpBytes + sizeof(GemmCtl);

// One lane waits, the verdict is broadcast so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = bounded_wait(bar, parity, abort_flag, limit_ns) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

__device__ __forceinline__ void raise_abort(GemmCtl* ctl, unsigned int* status) {
    if ((threadIdx.x & 31) == 0) {
        ctl->abort = 1;
        atomicOr(status, 1u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int MODE>
__device__ __forceinline__ float chunk_scale_b(const GemmParams& p, int c, int jh) {
    if (MODE == kModeFprop) return __ldg(p.sB + static_cast<int64_t>(jh >> 7) * p.KC + c);
    return __ldg(p.sB + static_cast<int64_t>(c) * (p.J >> 7) + (jh >> 7));
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_block_scaled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmD, const GemmParams p,
                             unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = base;
    uint8_t* smB = base + kStages * kStageBytesA;
    uint8_t* smEpi = smB + kStages * kStageBytesB;
    GemmCtl* ctl = reinterpret_cast<GemmCtl*>(smEpi + kPromoWarps * kEpiWarpBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], kPromoWarps);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort;
    const uint64_t lim = p.timeout_ns;
    uint32_t producer_issued = 0;

    // Register split (launch: 384 x 168): warpgroup 0 keeps 40, the two
    // promotion warpgroups take 232 each; 128*40 + 256*232 == 384*168.
    if (warp < kFirstPromoWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
    if (warp == 0) {
        // ---------------------------------------------------------- producer
        uint32_t s = 0, ph = 0, issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            for (int c = 0; c < p.KC; ++c) {
                if (!warp_wait(&ctl->empty[s], ph ^ 1, abort_flag, lim)) { ok = false; break; }
                if (lane == 0) {
                    const uint32_t fb = smem_addr(&ctl->full[s]);
                    mbar_arrive_expect_tx(&ctl->full[s], kStageBytesA + kStageBytesB);
                    tma_load_2d(smem_addr(smA + s * kStageBytesA), &tmA, fb, c * kBK, tm * kBM);
                    tma_load_2d(smem_addr(smB + s * kStageBytesB), &tmB, fb, c * kBK, tn * kBN);
                }
                ++issued;
                if (++s == kStages) { s = 0; ph ^= 1; }
            }
        }
        if (!ok) raise_abort(ctl, status);
        producer_issued = issued;
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        constexpr uint32_t idesc = idesc_e4m3_f32(kBM, kBN);
        uint32_t s = 0, ph = 0, buf = 0, tph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            for (int c = 0; c < p.KC; ++c) {
                if (!warp_wait(&ctl->tempty[buf], tph ^ 1, abort_flag, lim)) { ok = false; break; }
                if (!warp_wait(&ctl->full[s], ph, abort_flag, lim)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a0 = smem_addr(smA + s * kStageBytesA);
                    const uint32_t b0 = smem_addr(smB + s * kStageBytesB);
                    const uint32_t d = tmem + buf * kBN;
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_e4m3(d, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k), idesc, k > 0);
                    mma_commit(smem_addr(&ctl->empty[s]));
                    mma_commit(smem_addr(&ctl->tfull[buf]));
                }
                __syncwarp();
                if (++s == kStages) { s = 0; ph ^= 1; }
                buf ^= 1;
                if (buf == 0) tph ^= 1;
            }
        }
        if (!ok) raise_abort(ctl, status);
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;" ::: "memory");
        // --------------------------------------------------------- promotion
        const int pw = warp - kFirstPromoWarp;
        const int quarter = warp & 3;          // TMEM lanes this warp may access
        const int half = pw >> 2;              // which 128 columns of the tile
        const int row = quarter * 32 + lane;   // tile row == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        uint32_t buf = 0, tph = 0, it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            const int gi = tm * kBM + row;
            const int jh = tn * kBN + half * 128;
            const bool hv = jh < p.J;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;

            for (int c = 0; c < p.KC; ++c, ++it) {
                const float sa = __ldg(p.sA + static_cast<int64_t>(c) * p.I + gi);
                float sb = 0.0f;
                if (MODE != kModeWgrad) {
                    sb = hv ? chunk_scale_b<MODE>(p, c, jh) : 0.0f;
                } else {
                    // each warp stages its own copy of the 128 column scales
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (hv) v = __ldg(reinterpret_cast<const float4*>(p.sB + static_cast<int64_t>(c) * p.J + jh) + lane);
                    reinterpret_cast<float4*>(ctl->sbw[pw][it & 1])[lane] = v;
                    __syncwarp();
                }
                if (!warp_wait(&ctl->tfull[buf], tph, abort_flag, lim)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tbase = tmem + lane_off + buf * kBN + half * 128;
                if (MODE != kModeWgrad) {
                    // acc += (sA * sB) * partial, two columns per packed FMA
                    const float sab = sa * sb;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        uint32_t r0[32], r1[32];
                        tmem_ld_32x32b_x32(tbase + g * 64, r0);
                        tmem_ld_32x32b_x32(tbase + g * 64 + 32, r1);
                        tmem_wait_ld();
                        reg_fence32(r0);
                        reg_fence32(r1);
                        float* a = acc + g * 64;
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            ffma2(a[i], a[i + 1], sab, sab, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
                            ffma2(a[32 + i], a[33 + i], sab, sab, __uint_as_float(r1[i]), __uint_as_float(r1[i + 1]));
                        }
                    }
                } else {
                    // per-column scales: acc += sA * (sB[j] * partial)
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        uint32_t r0[32];
                        tmem_ld_32x32b_x32(tbase + g * 32, r0);
                        tmem_wait_ld();
                        reg_fence32(r0);
                        const float* sbv = &ctl->sbw[pw][it & 1][g * 32];
                        float* a = acc + g * 32;
#pragma unroll
                        for (int i = 0; i < 32; i += 4) {
                            const float4 b = *reinterpret_cast<const float4*>(sbv + i);
                            float t0, t1, t2, t3;
                            fmul2(t0, t1, __uint_as_float(r0[i]), __uint_as_float(r0[i + 1]), b.x, b.y);
                            fmul2(t2, t3, __uint_as_float(r0[i + 2]), __uint_as_float(r0[i + 3]), b.z, b.w);
                            ffma2(a[i], a[i + 1], t0, t1, sa, sa);
                            ffma2(a[i + 2], a[i + 3], t2, t3, sa, sa);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
                buf ^= 1;
                if (buf == 0) tph ^= 1;
            }
            if (!ok) break;
            // Epilogue: round to BF16 into this warp's swizzled staging boxes,
            // then one lane issues the TMA stores (asynchronous: they drain
            // while the next tile's chunks are promoted).
            uint8_t* stg = smEpi + pw * kEpiWarpBytes;
            if (lane == 0) bulk_wait_group_read<0>();  // the previous tile's stores left the buffer
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float* a = acc + h * 64 + j * 8;
                    uint4 o;
                    o.x = pack_bf16x2(a[0], a[1]);
                    o.y = pack_bf16x2(a[2], a[3]);
                    o.z = pack_bf16x2(a[4], a[5]);
                    o.w = pack_bf16x2(a[6], a[7]);
                    *reinterpret_cast<uint4*>(stg + h * kEpiBoxBytes + lane * 128 + ((j ^ (lane & 7)) << 4)) = o;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && hv) {
                const int y0 = tm * kBM + quarter * 32;
                tma_store_2d(&tmD, smem_addr(stg), jh, y0);
                tma_store_2d(&tmD, smem_addr(stg + kEpiBoxBytes), jh + 64, y0);
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // all output writes complete before exit
        if (!ok) raise_abort(ctl, status);
    }

    // Teardown.  Every role has stopped (all waits are bounded).  After an
    // abort, let this CTA's own in-flight copies land and its MMAs finish
    // before shared memory and TMEM are released.
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t n = producer_issued < kStages ? producer_issued : kStages;
            for (uint32_t i = 0; i < n; ++i) {
                const uint32_t f = producer_issued - 1 - i;
                bounded_wait(&ctl->full[f % kStages], (f / kStages) & 1, nullptr, lim);
            }
        }
        if (warp == 1 && lane == 0) {
            mma_commit(smem_addr(&ctl->drain));
            bounded_wait(&ctl->drain, 0, nullptr, lim);
        }
        __syncthreads();
    }
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Self-test of the bounded wait: one CTA waits on a barrier that nothing will
// complete, gives up after `limit_ns` and records the timeout.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, unsigned int* __restrict__ status) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (!bounded_wait(&bar, 0, &abort_flag, limit_ns)) atomicOr(status, 1u);
    }
}

}  // namespace fp8bq
