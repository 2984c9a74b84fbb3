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
// Design: persistent clusters of two CTAs (the two SMs of a TPC), 384
// threads each, one 256 x 256 output tile per cluster at a time, K chunk of
// 128 (one scale chunk).  CTA rank r of the pair owns output rows
// [128 r, 128 r + 128) of the tile and all 256 columns.
//   warp 0      operand producer (both CTAs): TMA loads of this CTA's 128
//               rows of A and its half (128 rows) of B per chunk into a
//               5-stage shared-memory ring (128-byte swizzle), completion
//               bytes counted on the even CTA's full barrier, which the even
//               producer arms for both CTAs' bytes.
//   warp 2      scale producer (both CTAs): bulk and cp.async copies of each
//               chunk's scales (this CTA's 128 row scales and the tile's
//               column scales) into a 6-slot ring, so no promotion warp ever
//               waits on a global-memory load.
//   warp 1      allocates the pair's TMEM (both CTAs); in the even CTA one
//               thread issues four tcgen05.mma.cta_group::2.kind::f8f6f4
//               (256x256x32) per chunk into one of two TMEM partial buffers
//               of 256 FP32 columns, started fresh every chunk, then commits
//               with a multicast to both CTAs' stage-empty barriers (the
//               producers may refill the stage) and partial-full barriers.
//   warp 3      idle (the first warpgroup gives up registers: 40 per thread)
//   warps 4..11 promotion (two warpgroups at 232 registers per thread, both
//               CTAs): each warp owns the 32 TMEM lanes (rows) of its SM
//               sub-partition and 128 of the tile's columns, 128 FP32
//               accumulators per thread (Fprop/Dgrad: one row and 128
//               columns; Wgrad: four rows and 32 columns, see load_group).
//               It reads the chunk partial from its CTA's TMEM (tcgen05.ld),
//               hands the buffer back to the MMA (the even CTA's
//               partial-empty barrier, 16 arrivals: 8 warps per CTA) as soon
//               as the partial is in registers, and multiplies it by the
//               chunk's scale product into the accumulators.  While it does
//               so the tensor cores already compute the next chunk into the
//               other buffer.  After the last chunk the accumulators are
//               rounded to BF16 (or kept in FP32 and optionally added into
//               the output with a TMA reduce) and stored with TMA.
// Odd-numbered tiles of a cluster walk the reduction backwards (chunk_of).
// Per SM and chunk this moves 32 KB through TMA and shared memory (a single
// CTA with a 128 x 256 tile needs 48 KB) for the same tensor-core work.
// Every wait is bounded: a stalled pipeline records FP8BQ_ERR_TIMEOUT in the
// device status word, raises the abort flag of both CTAs and the pair
// unwinds (draining in-flight copies and MMAs, then freeing TMEM) instead of
// hanging.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "ptx.cuh"
#include "quantize.cuh"

namespace fp8bq {

enum GemmMode : int { kModeFprop = 0, kModeDgrad = 1, kModeWgrad = 2 };

constexpr int kBM = 128;          // tile rows per CTA (TMEM lanes)
constexpr int kPairM = 256;       // tile rows per CTA pair
constexpr int kBN = 256;          // tile columns (MMA N)
constexpr int kBNHalf = 128;      // B rows each CTA loads
constexpr int kBRows = kBNHalf;   // B box height of the tensor map (rows per CTA)
constexpr int kBK = 128;          // one scale chunk of the reduction
constexpr int kStages = 5;
constexpr int kScaleSlots = 6;
constexpr int kGemmThreads = 384;
constexpr int kFirstPromoWarp = 4;
constexpr int kPromoWarps = 8;
constexpr uint32_t kStageBytesA = kBM * kBK;
constexpr uint32_t kStageBytesB = kBNHalf * kBK;
constexpr uint32_t kTmemCols = 2 * kBN;
// Balanced order: one promotion warp's accumulators (32 threads x 128 floats)
// in a split slot; the slots of one cluster (2 remainder segments x 2 CTA
// ranks x 8 warps) and the counters of one remaining tile (2 ranks x 8 warps).
constexpr int64_t kSplitSliceFloats = 32 * 128;
constexpr int64_t kSplitClusterBytes = 2 * 2 * kPromoWarps * kSplitSliceFloats * 4;
constexpr int64_t kSplitTileCounters = 2 * kPromoWarps;
// Epilogue staging: a promotion warp writes its 32 rows x 128 BF16 columns
// as four 32 x 32 boxes (64-byte rows, 64-byte swizzle) through three 2 KB
// staging boxes used in rotation, so a box is written while the TMA stores
// of the two before it are still reading theirs.  (A sixth operand stage
// measured slower than the second and third staging box on GEMMs with a
// short reduction, and no faster on long ones.)
constexpr uint32_t kEpiBoxBytes = 32 * 64;
constexpr uint32_t kEpiWarpBytes = 3 * kEpiBoxBytes;   // three staging boxes per warp

struct GemmParams {
    const float* sA;
    const float* sB;
    int I, J, KC;         // output rows, output columns, reduction chunks
    int tiles_n;          // ceil(J / kBN)
    int num_tiles;        // ceil(I / kPairM) * tiles_n
    int out_f32;          // D is FP32 (else BF16)
    int accumulate;       // FP32 D: add into it (TMA reduce-add) instead of overwriting
    int out_bf16;         // BF16 D is written (may be 0 when only codes are wanted)
    int out_q;            // also quantize the BF16-rounded output per 1x128 row tile
    float* sq;            // out_q: output scales [J/128][I]
    float* split_ws;      // balanced order: partial accumulators of split tiles
    unsigned int* split_cnt;  // balanced order: arrival counters (remaining tile, CTA rank, warp)
    uint64_t timeout_ns;
};

// One chunk's scales for one CTA: its 128 row scales and the tile's column
// scales (Wgrad: 256 per-column values; Fprop/Dgrad: one per 128-column
// block, b[0] and b[1]).
struct alignas(16) ScaleSlot {
    float a[128];
    float b[256];
};

struct alignas(16) GemmCtl {
    uint64_t full[kStages];    // even CTA: both CTAs' bytes of the stage landed
    uint64_t empty[kStages];   // both CTAs: the pair MMA has read the stage
    uint64_t tfull[2];         // both CTAs: the chunk partial is in TMEM
    uint64_t tempty[2];        // even CTA: both CTAs' promotion warps read it
    uint64_t sfull[kScaleSlots];   // the slot's scale copies landed
    uint64_t sempty[kScaleSlots];  // the promotion warps are done with the slot (8 warps)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
    uint32_t issued;           // stages this CTA's producer filled
    uint32_t peer_issued;      // even CTA: stages the odd CTA's producer filled
    uint32_t scl_issued;       // scale slots this CTA's scale producer filled
    ScaleSlot scl[kScaleSlots];
};
static_assert(offsetof(GemmCtl, scl) % 16 == 0, "scale slots are read with 16-byte vector loads");

constexpr size_t kGemmSmemBytes =
    1024 + kStages * (kStageBytesA + kStageBytesB) + kPromoWarps * kEpiWarpBytes + sizeof(GemmCtl);
static_assert(kGemmSmemBytes <= 232448, "more dynamic shared memory than one sm_103 CTA can have");

// One lane waits, the result is broadcast so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = bounded_wait(bar, parity, abort_flag, limit_ns) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// warp_wait for the scale producer, which runs far ahead: lane 0 backs off
// between polls so the promotion warps of its SM sub-partition keep their
// issue slots.
__device__ __forceinline__ bool warp_wait_backoff(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  uint64_t limit_ns) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = bounded_wait_backoff(bar, parity, abort_flag, limit_ns, 128) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// The reduction chunk a cluster's producers load i-th for the it-th tile the
// cluster takes: odd tiles walk the reduction backwards.  The clusters take
// their tiles in step, so a new tile starts on the chunks the previous wave
// of tiles read last, which are still in L2, and the operands it shares with
// that wave (the B column blocks of a row-major wave) come from L2 instead of
// HBM.  Chunk partials are summed in that order; the result stays within
// the same bound (any order of the FP32 sum over chunks is a valid reading).
__host__ __device__ __forceinline__ int chunk_of(int i, int it, int KC) { return (it & 1) ? KC - 1 - i : i; }

// Balanced order (the kBal kernels, Wgrad with scratch).  Whole-tile rounds
// leave the grid partly idle in the last round when num_tiles is not a
// multiple of the n clusters, and a Wgrad tile reduces over all tokens, so
// that round costs a whole tile's time.  Here the R = num_tiles / n full
// rounds run in tile order (cluster cid: tiles cid, cid + n, ..., walking
// odd rounds backwards, so concurrent tiles share operand chunks in L2), and
// the chunks of the rem = num_tiles - R n remaining tiles, U_r = rem * KC in
// tile-major order, are shared out equally: cluster c takes [b_c, b_{c+1}),
// b_c = U_r c / n.  A share is no longer than a tile, so it lies in at most
// two remaining tiles (the cluster's remainder segments 0 and 1), and a
// remaining tile is covered by every cluster whose share meets it: its parts.
// The host guarantees U_r * n < 2^31.
__host__ __device__ __forceinline__ int rem_bound(const GemmParams& p, int ncl, int c) {
    const int rem = p.num_tiles - (p.num_tiles / ncl) * ncl;
    return rem * p.KC * c / ncl;
}

// Segment k of cluster cid: chunks [c_lo, c_hi) of tile; rt = the remaining
// tile's index (-1 in the full rounds).  False when there is no segment k.
__host__ __device__ __forceinline__ bool hyb_segment(const GemmParams& p, int cid, int ncl, int k, int& tile,
                                                     int& c_lo, int& c_hi, int& rt) {
    const int R = p.num_tiles / ncl;
    if (k < R) {
        tile = cid + k * ncl;
        c_lo = 0;
        c_hi = p.KC;
        rt = -1;
        return true;
    }
    const int b0 = rem_bound(p, ncl, cid), b1 = rem_bound(p, ncl, cid + 1);
    const int t = b0 / p.KC + (k - R);
    const int lo = max(b0, t * p.KC), hi = min(b1, (t + 1) * p.KC);
    if (lo >= hi) return false;
    rt = t;
    tile = R * ncl + t;
    c_lo = lo - t * p.KC;
    c_hi = hi - t * p.KC;
    return true;
}

// All chunks cluster cid works through in the balanced order.
__host__ __device__ __forceinline__ int hyb_chunk_count(const GemmParams& p, int cid, int ncl) {
    return (p.num_tiles / ncl) * p.KC + rem_bound(p, ncl, cid + 1) - rem_bound(p, ncl, cid);
}

// Does cluster c's share meet remaining tile rt?
__host__ __device__ __forceinline__ bool hyb_meets(const GemmParams& p, int ncl, int c, int rt) {
    return max(rem_bound(p, ncl, c), rt * p.KC) < min(rem_bound(p, ncl, c + 1), (rt + 1) * p.KC);
}

// The clusters that can hold a part of remaining tile rt: [first, last], the
// clusters whose shares start at or before its first and last chunks (an
// empty share in between meets no tile: check each with hyb_meets).
__host__ __device__ __forceinline__ void hyb_part_range(const GemmParams& p, int ncl, int rt, int& first, int& last) {
    const int64_t ur = static_cast<int64_t>(p.num_tiles - (p.num_tiles / ncl) * ncl) * p.KC;
    first = min(ncl - 1, static_cast<int>(((static_cast<int64_t>(rt) * p.KC + 1) * ncl - 1) / ur));
    last = min(ncl - 1, static_cast<int>((static_cast<int64_t>(rt + 1) * p.KC * ncl - 1) / ur));
}

// Which of cluster c's remainder segments (0 or 1) covers remaining tile rt:
// its split slot.
__host__ __device__ __forceinline__ int hyb_slot_segment(const GemmParams& p, int ncl, int c, int rt) {
    return rem_bound(p, ncl, c) / p.KC == rt ? 0 : 1;
}

// Stop both CTAs of the pair and record the timeout.
__device__ __forceinline__ void raise_abort(GemmCtl* ctl, uint32_t peer_abort, unsigned int* status) {
    if ((threadIdx.x & 31) == 0) {
        ctl->abort = 1;
        st_cluster_u32(peer_abort, 1u);
        atomicOr(status, 1u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_16g(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once this thread's prior cp.async copies have landed
// (counts against the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_drain() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Launched as clusters of two CTAs (grid = 2 x clusters).
template <int MODE, bool kBal = false>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_block_scaled_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmQ,
                             const GemmParams p, unsigned int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = base;
    uint8_t* smB = base + kStages * kStageBytesA;
    uint8_t* smEpi = smB + kStages * kStageBytesB;
    GemmCtl* ctl = reinterpret_cast<GemmCtl*>(smEpi + kPromoWarps * kEpiWarpBytes);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int first_tile = static_cast<int>(cluster_id_x());
    const int tile_step = static_cast<int>(cluster_count_x());

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ctl->tfull[b], 1);
            mbar_init(&ctl->tempty[b], 2 * kPromoWarps);
        }
        for (int q = 0; q < kScaleSlots; ++q) {
            // one expect_tx arrival for the bulk copies, plus the two cp.async
            // arrivals of the weight-block scales in Fprop/Dgrad
            mbar_init(&ctl->sfull[q], MODE == kModeWgrad ? 1 : 3);
            mbar_init(&ctl->sempty[q], kPromoWarps);
        }
        mbar_init(&ctl->drain, 1);
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->peer_issued = 0;
        ctl->scl_issued = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmD);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&ctl->tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    // Both CTAs' barriers are initialised and the pair's TMEM is allocated
    // before any copy, MMA or remote arrive targets them.
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();

    const uint32_t tmem = ctl->tmem_base;
    volatile int* abort_flag = &ctl->abort;
    const uint32_t peer_abort = mapa_shared(smem_addr(&ctl->abort), rank ^ 1u);
    const uint64_t lim = p.timeout_ns;

    // Register split (launch: 384 x 168): warpgroup 0 keeps 40, the two
    // promotion warpgroups take 232 each; 128*40 + 256*232 == 384*168.
    if (warp < kFirstPromoWarp) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 40;" ::: "memory");
    if (warp == 0) {
        // ------------------------------------------------- operand producer
        const uint32_t full0 = mapa_shared(smem_addr(&ctl->full[0]), 0);
        uint32_t s = 0, ph = 0, issued = 0;
        bool ok = true;
        int it = -1, tile = first_tile - tile_step, c_lo = 0, c_hi = p.KC, rt = -1;
        while (ok) {
            if constexpr (kBal) {
                if (!hyb_segment(p, first_tile, tile_step, it + 1, tile, c_lo, c_hi, rt)) break;
            } else {
                tile += tile_step;
                if (tile >= p.num_tiles) break;
            }
            ++it;
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            const int r0 = tm * kPairM + static_cast<int>(rank) * kBM;  // this CTA's first row
            const int b0 = tn * kBN + static_cast<int>(rank) * kBNHalf;  // this CTA's first B row
            for (int i = c_lo; i < c_hi; ++i) {
                const int c = rt >= 0 ? i : chunk_of(i, it, p.KC);
                if (!warp_wait(&ctl->empty[s], ph ^ 1, abort_flag, lim)) { ok = false; break; }
                if (lane == 0) {
                    if (leader) mbar_arrive_expect_tx(&ctl->full[s], 2 * (kStageBytesA + kStageBytesB));
                    const uint32_t fb = full0 + s * 8;
                    tma_load_2d_pair(smem_addr(smA + s * kStageBytesA), &tmA, fb, c * kBK, r0);
                    tma_load_2d_pair(smem_addr(smB + s * kStageBytesB), &tmB, fb, c * kBK, b0);
                }
                ++issued;
                if (++s == kStages) { s = 0; ph ^= 1; }
            }
        }
        if (!ok) raise_abort(ctl, peer_abort, status);
        if (lane == 0) ctl->issued = issued;
    } else if (warp == 2) {
        // --------------------------------------------------- scale producer
        // Copies each chunk's scales into the next ring slot: this CTA's 128
        // row scales and Wgrad's column scales with bulk copies (one lane,
        // completion in bytes), Fprop/Dgrad's weight-block scale of each
        // 128-column half with two 4-byte cp.async.  Rows and columns past
        // the problem are skipped.
        uint32_t q = 0, qph = 0, issued = 0;
        bool ok = true;
        int it = -1, tile = first_tile - tile_step, c_lo = 0, c_hi = p.KC, rt = -1;
        while (ok) {
            if constexpr (kBal) {
                if (!hyb_segment(p, first_tile, tile_step, it + 1, tile, c_lo, c_hi, rt)) break;
            } else {
                tile += tile_step;
                if (tile >= p.num_tiles) break;
            }
            ++it;
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            const int r0 = tm * kPairM + static_cast<int>(rank) * kBM;
            const int j0 = tn * kBN;
            const uint32_t a_bytes = r0 < p.I ? 128u * 4u : 0u;
            const uint32_t b_bytes = MODE == kModeWgrad ? static_cast<uint32_t>(min(p.J - j0, kBN)) * 4u : 0u;
            for (int i = c_lo; i < c_hi; ++i) {
                const int c = rt >= 0 ? i : chunk_of(i, it, p.KC);
                if (!warp_wait_backoff(&ctl->sempty[q], qph ^ 1, abort_flag, lim)) { ok = false; break; }
                ScaleSlot& sl = ctl->scl[q];
                if (lane == 0) {
                    const uint32_t bar = smem_addr(&ctl->sfull[q]);
                    mbar_arrive_expect_tx(&ctl->sfull[q], a_bytes + b_bytes);
                    if (a_bytes) bulk_load(smem_addr(sl.a), p.sA + static_cast<int64_t>(c) * p.I + r0, a_bytes, bar);
                    if (b_bytes) bulk_load(smem_addr(sl.b), p.sB + static_cast<int64_t>(c) * p.J + j0, b_bytes, bar);
                }
                if (MODE != kModeWgrad && lane < 2) {
                    const int jb = (j0 >> 7) + lane;  // 128-column block of the weight
                    if (jb * 128 < p.J) {
                        const float* src = MODE == kModeFprop ? p.sB + static_cast<int64_t>(jb) * p.KC + c
                                                              : p.sB + static_cast<int64_t>(c) * (p.J >> 7) + jb;
                        cp_async_4(smem_addr(&sl.b[lane]), src);
                    }
                    cp_async_arrive(&ctl->sfull[q]);
                }
                ++issued;
                if (++q == kScaleSlots) { q = 0; qph ^= 1; }
            }
        }
        cp_async_drain();
        if (!ok) raise_abort(ctl, peer_abort, status);
        if (lane == 0) ctl->scl_issued = issued;
    } else if (warp == 1 && leader) {
        // --------------------------------------------------------------- MMA
        // One thread runs the whole loop (no per-wait warp broadcast).
        bool ok = true;
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(kPairM, kBN);
            uint32_t s = 0, ph = 0, buf = 0, tph = 0;
            // balanced: the MMAs need no tile boundaries, one flat loop
            const int n_outer = kBal ? 1 : p.num_tiles;
            const int n_inner = kBal ? hyb_chunk_count(p, first_tile, tile_step) : p.KC;
            for (int tile = kBal ? 0 : first_tile; tile < n_outer && ok; tile += kBal ? 1 : tile_step) {
                for (int c = 0; c < n_inner; ++c) {
                    // Both waits suspend (try_wait): this thread shares its SM
                    // sub-partition with two promotion warps (TMEM lanes 32-63),
                    // the last to hand the partial buffer back, so it must not
                    // take their issue slots by spinning.
                    if (!bounded_wait(&ctl->tempty[buf], tph ^ 1, abort_flag, lim)) { ok = false; break; }
                    if (!bounded_wait(&ctl->full[s], ph, abort_flag, lim)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = smem_addr(smA + s * kStageBytesA);
                    const uint32_t b0 = smem_addr(smB + s * kStageBytesB);
                    const uint32_t d = tmem + buf * kBN;
#pragma unroll
                    for (int k = 0; k < kBK / 32; ++k)
                        mma_e4m3_pair(d, sw128_kmajor_desc(a0 + 32 * k), sw128_kmajor_desc(b0 + 32 * k), idesc,
                                      k > 0);
                    // the stage is free once these MMAs have read it; the
                    // partial is ready once they have completed
                    mma_commit_pair_mc(smem_addr(&ctl->empty[s]), 0x3);
                    mma_commit_pair_mc(smem_addr(&ctl->tfull[buf]), 0x3);
                    if (++s == kStages) { s = 0; ph ^= 1; }
                    buf ^= 1;
                    if (buf == 0) tph ^= 1;
                }
            }
        }
        __syncwarp();
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        if (!ok) raise_abort(ctl, peer_abort, status);
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 232;" ::: "memory");
        // --------------------------------------------------------- promotion
        const int pw = warp - kFirstPromoWarp;
        const int quarter = warp & 3;          // TMEM lanes this warp may access
        const int half = pw >> 2;              // which 128 columns of the tile
        const int row = quarter * 32 + lane;   // tile row == TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tempty0 = mapa_shared(smem_addr(&ctl->tempty[0]), 0);
        uint32_t buf = 0, tph = 0, q = 0, qph = 0;
        int nbox = 0;   // staging box of the next BF16 output box
        bool ok = true;
        int tile = first_tile - tile_step, c_lo = 0, c_hi = p.KC, rt = -1;
        for (int seg = 0; ok; ++seg) {
            if constexpr (kBal) {
                if (!hyb_segment(p, first_tile, tile_step, seg, tile, c_lo, c_hi, rt)) break;
            } else {
                tile += tile_step;
                if (tile >= p.num_tiles) break;
            }
            const int tm = tile / p.tiles_n, tn = tile - tm * p.tiles_n;
            const int r0 = tm * kPairM + static_cast<int>(rank) * kBM;  // first row of this CTA's half
            const bool rv = r0 < p.I;
            const int jh = tn * kBN + half * 128;
            const bool hv = jh < p.J;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;

            for (int c = c_lo; c < c_hi; ++c) {
                if (!warp_wait(&ctl->sfull[q], qph, abort_flag, lim)) { ok = false; break; }
                const ScaleSlot& sl = ctl->scl[q];
                const float sab = MODE == kModeWgrad ? 0.0f : sl.a[row] * sl.b[half];
                // Wgrad: this thread's row scales (see load_group) and the
                // column scales of this half, by shared-window address
                const uint32_t sas = smem_addr(&sl.a[quarter * 32 + (lane >> 2)]);
                const uint32_t sbs = smem_addr(&sl.b[half * 128 + 2 * (lane & 3)]);
                if (!warp_wait(&ctl->tfull[buf], tph, abort_flag, lim)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tbase = tmem + lane_off + buf * kBN + half * 128;
                // The partial in four groups of 32 values per thread.
                // Fprop/Dgrad (32x32b shape): the thread's row (its TMEM lane),
                // columns 32g .. 32g + 31.  Wgrad (16x256b shape): lanes
                // 16(g & 1) + lane/4 and + 8 of this warp's quarter, columns
                // 64(g >> 1) + 8k + 2(lane % 4) + {0, 1} for k < 8, so that a
                // thread needs 32 of the chunk's column scales instead of 128
                // (the scales reach every lane through shared-memory
                // broadcasts, one 128-byte wavefront per 128 bytes that the
                // warp receives).
                auto load_group = [&](int g, uint32_t (&v)[32]) {
                    if (MODE != kModeWgrad)
                        tmem_ld_32x32b_x32(tbase + 32 * g, v);
                    else
                        tmem_ld_16x256b_x8(tbase + (static_cast<uint32_t>((g & 1) * 16) << 16) + (g >> 1) * 64, v);
                };
                // Wgrad: the column scales of groups 2h and 2h + 1 (the same
                // columns of the two 16-lane halves), loaded once for both
                float2 sbv[8];
                auto load_col_scales = [&](int h) {
                    if (MODE == kModeWgrad) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) sbv[k] = lds_f32x2(sbs + h * 256 + 32 * k);
                    }
                };
                // acc += (sA * sB) * partial (Fprop, Dgrad), or
                // acc += sA * (sB[j] * partial) (Wgrad).
                auto promote = [&](const uint32_t (&v)[32], int g) {
                    float* a = acc + g * 32;
                    if (MODE != kModeWgrad) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) a[i] = __fmaf_rn(sab, __uint_as_float(v[i]), a[i]);
                    } else {
                        const float s0 = lds_f32(sas + (g & 1) * 64), s1 = lds_f32(sas + (g & 1) * 64 + 32);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const float2 b = sbv[k];
                            float t0, t1, t2, t3;
                            fmul2(t0, t1, __uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]), b.x, b.y);
                            fmul2(t2, t3, __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]), b.x, b.y);
                            ffma2(a[4 * k], a[4 * k + 1], t0, t1, s0, s0);
                            ffma2(a[4 * k + 2], a[4 * k + 3], t2, t3, s1, s1);
                        }
                    }
                };
                // Two 32-value staging buffers: groups 0 and 1 load together,
                // group 2 loads while group 0 is multiplied in, group 3 while
                // group 1 is; the TMEM buffer goes back to the MMA as soon as
                // group 3 is in registers.
                uint32_t ra[32], rb[32];
                load_group(0, ra);
                load_group(1, rb);
                tmem_wait_ld();
                reg_fence32(ra);
                reg_fence32(rb);
                load_col_scales(0);
                promote(ra, 0);
                load_group(2, ra);
                promote(rb, 1);
                load_group(3, rb);
                tmem_wait_ld();
                reg_fence32(ra);
                reg_fence32(rb);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty0 + buf * 8);
                load_col_scales(1);
                promote(ra, 2);
                promote(rb, 3);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->sempty[q]);
                if (++q == kScaleSlots) { q = 0; qph ^= 1; }
                buf ^= 1;
                if (buf == 0) tph ^= 1;
            }
            if (!ok) break;
            if constexpr (kBal) {
                if (rt >= 0) {
                    // A remaining tile, shared by the clusters whose shares meet
                    // it (see hyb_segment).  Each part leaves its partial
                    // accumulators in its own slot (cluster, segment) and counts
                    // itself in; the last to arrive sums every part's slot in
                    // cluster order (the same sum whichever part arrives last)
                    // and writes the tile.  Warp-sized slices: warp pw of every
                    // part holds the same rows and columns.
                    const int ncl = tile_step;
                    int cf, cl;
                    hyb_part_range(p, ncl, rt, cf, cl);
                    auto slot = [&](int c) -> float* {
                        const int j = hyb_slot_segment(p, ncl, c, rt);
                        return p.split_ws +
                               ((static_cast<int64_t>(c) * 2 + j) * 2 + rank) * kSplitSliceFloats * kPromoWarps +
                               static_cast<int64_t>(pw) * kSplitSliceFloats;
                    };
                    float* mine = slot(first_tile);
#pragma unroll
                    for (int i4 = 0; i4 < 32; ++i4)
                        *reinterpret_cast<float4*>(mine + (i4 * 32 + lane) * 4) =
                            make_float4(acc[4 * i4], acc[4 * i4 + 1], acc[4 * i4 + 2], acc[4 * i4 + 3]);
                    __threadfence();
                    __syncwarp();
                    unsigned int nparts = 0;
                    for (int c = cf; c <= cl; ++c) nparts += hyb_meets(p, ncl, c, rt) ? 1u : 0u;
                    unsigned int* cnt = p.split_cnt + (rt * 2 + static_cast<int>(rank)) * kPromoWarps + pw;
                    unsigned int arrived = 0;
                    if (lane == 0) arrived = atomicAdd(cnt, 1u);
                    arrived = __shfl_sync(0xFFFFFFFFu, arrived, 0);
                    if (arrived + 1 != nparts) continue;   // another part completes the tile
                    __threadfence();
#pragma unroll
                    for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
                    for (int c = cf; c <= cl; ++c) {
                        if (!hyb_meets(p, ncl, c, rt)) continue;
                        const float* part = slot(c);
#pragma unroll
                        for (int i4 = 0; i4 < 32; ++i4) {
                            const float4 o = __ldcg(reinterpret_cast<const float4*>(part + (i4 * 32 + lane) * 4));
                            acc[4 * i4] = __fadd_rn(acc[4 * i4], o.x);
                            acc[4 * i4 + 1] = __fadd_rn(acc[4 * i4 + 1], o.y);
                            acc[4 * i4 + 2] = __fadd_rn(acc[4 * i4 + 2], o.z);
                            acc[4 * i4 + 3] = __fadd_rn(acc[4 * i4 + 3], o.w);
                        }
                    }
                    if (lane == 0) *cnt = 0u;   // zero again for the next launch
                }
            }
            // Epilogue: round to BF16 (or keep FP32) into this warp's swizzled
            // staging box, then one lane issues the TMA store or reduce-add
            // (asynchronous: the last one drains while the next tile's chunks
            // are promoted).
            uint8_t* stg = smEpi + pw * kEpiWarpBytes;
            const int y0 = r0 + quarter * 32;
            const bool store = hv && rv;
            if (!p.out_f32) {
                if (p.out_bf16 && !p.out_q) {
                    // BF16 only: round while staging, four boxes of 32 x 32
#pragma unroll
                    for (int bx = 0; bx < 4; ++bx) {
                        // three staging boxes in rotation: the store that last
                        // read this one is at least the third most recent
                        uint8_t* stg = smEpi + pw * kEpiWarpBytes + nbox * kEpiBoxBytes;
                        if (++nbox == 3) nbox = 0;
                        if (lane == 0) bulk_wait_group_read<2>();
                        __syncwarp();
                        if (MODE != kModeWgrad) {
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float* a = acc + bx * 32 + j * 8;
                                *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                                    make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                               pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
                            }
                        } else {
                            // Wgrad layout: box bx holds repetitions 4(bx & 1) ..
                            // + 3 of groups 2(bx >> 1) and + 1, two rows each
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int lh = e >> 3, kk = (e >> 1) & 3, rs = e & 1;
                                const float* a = acc + (lh + 2 * (bx >> 1)) * 32 + 4 * (4 * (bx & 1) + kk) + 2 * rs;
                                const int R = lh * 16 + rs * 8 + (lane >> 2);
                                *reinterpret_cast<uint32_t*>(stg + R * 64 + ((kk ^ ((R >> 1) & 3)) << 4) + 4 * (lane & 3)) =
                                    pack_bf16x2(a[0], a[1]);
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (store) tma_store_2d(&tmD, smem_addr(stg), jh + bx * 32, y0);
                            bulk_commit_group();
                        }
                    }
                } else {
                // round to BF16 once: pk[i] holds columns 2i, 2i+1
                uint32_t pk[64];
#pragma unroll
                for (int i = 0; i < 64; ++i) pk[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
                if (p.out_bf16) {
                    // BF16: four boxes of 32 rows x 32 columns
#pragma unroll
                    for (int bx = 0; bx < 4; ++bx) {
                        // the previous box's store has finished reading the buffer
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t* w = pk + bx * 16 + j * 4;
                            // 64-byte swizzle: 16-byte chunk j of row r sits at chunk j ^ ((r >> 1) & 3)
                            *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (store) tma_store_2d(&tmD, smem_addr(stg), jh + bx * 32, y0);
                            bulk_commit_group();
                        }
                    }
                }
                if (p.out_q) {
                    // The thread's 128 BF16 outputs are one 1x128 row tile of
                    // the next linear's input: quantize them exactly as the
                    // row-wise quantizer would (codes in two 32 x 64 boxes).
                    uint32_t m = 0;
#pragma unroll
                    for (int i = 0; i < 64; ++i) m = absmax_bf16x2(m, pk[i]);
                    const TileDiv d = tile_div(bf16x2_max_halves(m));
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx) {
                        if (lane == 0) bulk_wait_group_read<0>();
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float f[16];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                f[2 * i] = bf16lo(pk[bx * 32 + j * 8 + i]);
                                f[2 * i + 1] = bf16hi(pk[bx * 32 + j * 8 + i]);
                            }
                            const uint2 lo = e4m3x8(f, d), hi = e4m3x8(f + 8, d);
                            *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(lo.x, lo.y, hi.x, hi.y);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (store) tma_store_2d(&tmQ, smem_addr(stg), jh + bx * 64, y0);
                            bulk_commit_group();
                        }
                    }
                    if (store) p.sq[static_cast<int64_t>(jh >> 7) * p.I + r0 + row] = d.s;
                }
                }
            } else {
                // FP32: eight boxes of 32 rows x 16 columns, stored or added
#pragma unroll
                for (int bx = 0; bx < 8; ++bx) {
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
                    if (MODE != kModeWgrad) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float* a = acc + bx * 16 + j * 4;
                            *reinterpret_cast<float4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                                make_float4(a[0], a[1], a[2], a[3]);
                        }
                    } else {
                        // Wgrad layout: box bx holds repetitions 2(bx & 3) and
                        // + 1 of groups 2(bx >> 2) and + 1, two rows each
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int lh = e >> 2, kk = (e >> 1) & 1, rs = e & 1;
                            const float* a = acc + (lh + 2 * (bx >> 2)) * 32 + 4 * (2 * (bx & 3) + kk) + 2 * rs;
                            const int R = lh * 16 + rs * 8 + (lane >> 2);
                            const int C = 8 * kk + 2 * (lane & 3);   // column within the box
                            *reinterpret_cast<float2*>(stg + R * 64 + (((C >> 2) ^ ((R >> 1) & 3)) << 4) + (C & 3) * 4) =
                                make_float2(a[0], a[1]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (store) {
                            if (p.accumulate)
                                tma_reduce_add_2d(&tmD, smem_addr(stg), jh + bx * 16, y0);
                            else
                                tma_store_2d(&tmD, smem_addr(stg), jh + bx * 16, y0);
                        }
                        bulk_commit_group();
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // all output writes complete before exit
        if (!ok) raise_abort(ctl, peer_abort, status);
    }

    // Teardown.  Every role has stopped (all waits are bounded).  The odd CTA
    // reports how many stages its producer filled; after an abort each CTA
    // waits (bounded) for the scale copies it issued, and the even CTA for
    // every operand copy either producer issued and for its own in-flight
    // MMAs, which read both CTAs' shared memory and write both CTAs' TMEM,
    // before either CTA frees TMEM or exits.  A stage that only one producer
    // filled is first made completable: the bytes of the half that was never
    // loaded are counted as done (and, if the even producer stopped first,
    // the stage is armed for both halves).  The producers are at most a ring
    // apart (the odd one refills a stage only after the MMA consumed it, which
    // needed the even one's arming), and only the last ring-depth stages can
    // still be in flight: a stage is refilled only after its previous contents
    // were consumed.
    tc_fence_before();
    __syncthreads();
    if (!leader && threadIdx.x == 0) st_cluster_u32(mapa_shared(smem_addr(&ctl->peer_issued), 0), ctl->issued);
    cluster_sync_all();
    if (*abort_flag && warp == 2 && lane == 0) {
        const uint32_t n = ctl->scl_issued;
        const uint32_t f0 = n > static_cast<uint32_t>(kScaleSlots) ? n - kScaleSlots : 0;
        for (uint32_t f = f0; f < n; ++f)
            bounded_wait(&ctl->sfull[f % kScaleSlots], (f / kScaleSlots) & 1, nullptr, lim);
    }
    if (leader && *abort_flag) {
        if (warp == 0 && lane == 0) {
            const uint32_t a = ctl->issued, b = ctl->peer_issued;
            for (uint32_t f = b; f < a; ++f)   // the odd half never loaded
                mbar_complete_tx(&ctl->full[f % kStages], kStageBytesA + kStageBytesB);
            for (uint32_t f = a; f < b; ++f) {  // only the odd half loaded
                mbar_arrive_expect_tx(&ctl->full[f % kStages], 2 * (kStageBytesA + kStageBytesB));
                mbar_complete_tx(&ctl->full[f % kStages], kStageBytesA + kStageBytesB);
            }
            const uint32_t n = a > b ? a : b;
            const uint32_t f0 = n > static_cast<uint32_t>(kStages) ? n - kStages : 0;
            for (uint32_t f = f0; f < n; ++f)
                bounded_wait(&ctl->full[f % kStages], (f / kStages) & 1, nullptr, lim);
        }
        if (warp == 1 && lane == 0) {
            mma_commit_pair(smem_addr(&ctl->drain));
            bounded_wait(&ctl->drain, 0, nullptr, lim);
        }
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
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
