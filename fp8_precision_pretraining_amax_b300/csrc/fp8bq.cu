// Host side of libfp8bq: argument validation, TMA descriptor encoding and
// kernel launches behind the C ABI declared in include/fp8bq.h.
//
// The whole device code is one translation unit (kernels from quantize.cuh
// and gemm.cuh), compiled for sm_103a only.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "fp8bq.h"
#include "gemm.cuh"
#include "mx.cuh"
#include "quantize.cuh"

namespace {

// Bit 0: a kernel gave up on a bounded wait.
__device__ unsigned int g_status_word;
// Where fp8bq_check's exchange kernel leaves the word it took.
__device__ unsigned int g_status_taken;

// Scratch of fp8bq_gemm_wgrad_balanced_static, in the module's own device
// memory (no allocation call): the balanced Wgrad's counters and split slots
// for up to 74 clusters, the CTA pairs of a 148-SM B300 (devices that run
// more are refused).  Zero at module load; every completed call leaves the
// counters zero again.
constexpr int kStaticScratchPairs = 74;
constexpr int64_t kStaticScratchBytes =
    ((static_cast<int64_t>(kStaticScratchPairs - 1) * fp8bq::kSplitTileCounters * 4 + 255) / 256) * 256 +
    static_cast<int64_t>(kStaticScratchPairs) * fp8bq::kSplitClusterBytes;
static __device__ __align__(256) uint8_t g_wgrad_scratch[kStaticScratchBytes];

// Reads the status word and clears it in one atomic step, so a timeout that
// a kernel on another stream records meanwhile is either taken now or stays
// for the next check.
__global__ void status_take_kernel(unsigned int* status, unsigned int* taken) {
    *taken = atomicExch(status, 0u);
}

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxDevices = 64;

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    int max_pairs = 0;               // co-resident GEMM clusters (CTA pairs)
    unsigned int* status = nullptr;  // device address of g_status_word
    unsigned int* taken = nullptr;   // device address of g_status_taken
    uint8_t* wgrad_scratch = nullptr;  // device address of g_wgrad_scratch
    std::mutex check_mu;             // one fp8bq_check at a time uses `taken`
};

// Launch configuration of the GEMM: `pairs` clusters of two CTAs.
void gemm_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, cudaStream_t stream) {
    cfg->gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
    cfg->blockDim = dim3(fp8bq::kGemmThreads, 1, 1);
    cfg->dynamicSmemBytes = fp8bq::kGemmSmemBytes;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
}

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// The FP32 slab (64 KB) exceeds the default 48 KB of dynamic shared memory.
template <bool kF32>
cudaError_t set_tile_smem() {
    const int bytes = fp8bq::tile_smem_bytes<kF32>();
    cudaError_t e = cudaFuncSetAttribute(fp8bq::quantize_tile_kernel<kF32, fp8bq::kTileCol>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fp8bq::quantize_tile_kernel<kF32, fp8bq::kTileDual>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fp8bq::quantize_tile_kernel<kF32, fp8bq::kTileWeight>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fp8bq::quantize_weight_group_kernel<kF32>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && !kF32)
        e = cudaFuncSetAttribute(fp8bq::quantize_tile_kernel<false, fp8bq::kTileSwiglu>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 fp8bq::tile_smem_bytes<false, fp8bq::kTileSwiglu>());
    return e;
}

fp8bq_status probe_device(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FP8BQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FP8BQ_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return FP8BQ_ERR_CUDA;
        d.supported = (major == 10 && minor == 3);
        d.sms = sms;
        if (d.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return FP8BQ_ERR_CUDA;
            d.status = static_cast<unsigned int*>(p);
            if (cudaGetSymbolAddress(&p, g_status_taken) != cudaSuccess) return FP8BQ_ERR_CUDA;
            d.taken = static_cast<unsigned int*>(p);
            if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess) return FP8BQ_ERR_CUDA;
            d.wgrad_scratch = static_cast<uint8_t*>(p);
            const int smem = static_cast<int>(fp8bq::kGemmSmemBytes);
            if (cudaFuncSetAttribute(fp8bq::gemm_block_scaled_kernel<fp8bq::kModeFprop>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                cudaFuncSetAttribute(fp8bq::gemm_block_scaled_kernel<fp8bq::kModeDgrad>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                cudaFuncSetAttribute(fp8bq::gemm_block_scaled_kernel<fp8bq::kModeWgrad>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
                cudaFuncSetAttribute(fp8bq::gemm_block_scaled_kernel<fp8bq::kModeWgrad, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
                return FP8BQ_ERR_CUDA;
            if (set_tile_smem<false>() != cudaSuccess || set_tile_smem<true>() != cudaSuccess) return FP8BQ_ERR_CUDA;
            if (cudaFuncSetAttribute(fp8bq::mx_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(fp8bq::kMxSmemBytes)) != cudaSuccess ||
                cudaFuncSetAttribute(fp8bq::mx_quantize_slab_kernel<true, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     fp8bq::mx_col_smem_bytes<true>()) != cudaSuccess ||
                cudaFuncSetAttribute(fp8bq::mx_quantize_slab_kernel<true, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     fp8bq::mx_col_smem_bytes<true>()) != cudaSuccess)
                return FP8BQ_ERR_CUDA;
            {
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute attr[1];
                gemm_launch_config(&cfg, attr, sms / 2, nullptr);
                int clusters = 0;
                if (cudaOccupancyMaxActiveClusters(&clusters, fp8bq::gemm_block_scaled_kernel<fp8bq::kModeFprop>,
                                                   &cfg) != cudaSuccess ||
                    clusters < 1)
                    return FP8BQ_ERR_CUDA;
                d.max_pairs = clusters;
            }
            if (g_encode == nullptr) {
                void* fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                        cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || fn == nullptr)
                    return FP8BQ_ERR_CUDA;
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
        }
        d.probed = true;
    }
    if (!d.supported) return FP8BQ_ERR_DEVICE;
    *out = &d;
    return FP8BQ_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Encoded TMA descriptors of recent calls.  A descriptor depends only on the
// arguments of the encode call (address, extents, box, element type,
// swizzle), which together form the key, so a hit is exactly the descriptor
// the encode would produce; repeated calls on the same buffers (every step of
// a training loop) skip the driver's encode.  Round-robin replacement.
struct MapKey {
    const void* ptr;
    uint64_t inner, outer;
    uint32_t box_inner, box_outer;
    int kind;
    bool operator==(const MapKey& o) const {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && box_inner == o.box_inner &&
               box_outer == o.box_outer && kind == o.kind;
    }
};

class MapCache {
   public:
    template <typename Encode>
    fp8bq_status get(const MapKey& k, CUtensorMap* out, Encode encode) {
        {
            std::lock_guard<std::mutex> lock(mu_);
            for (int i = 0; i < n_; ++i)
                if (keys_[i] == k) {
                    *out = maps_[i];
                    return FP8BQ_OK;
                }
        }
        const fp8bq_status st = encode(out);
        if (st != FP8BQ_OK) return st;
        std::lock_guard<std::mutex> lock(mu_);
        const int i = n_ < kSize ? n_++ : next_;
        next_ = (i + 1) % kSize;
        keys_[i] = k;
        maps_[i] = *out;
        return FP8BQ_OK;
    }

   private:
    static constexpr int kSize = 64;
    std::mutex mu_;
    MapKey keys_[kSize];
    CUtensorMap maps_[kSize];
    int n_ = 0, next_ = 0;
};

MapCache g_maps;

inline int elem_size(int dtype) { return dtype == FP8BQ_BF16 ? 2 : 4; }

inline fp8bq_status launch_status() { return cudaGetLastError() == cudaSuccess ? FP8BQ_OK : FP8BQ_ERR_CUDA; }

// 2-D uint8 tensor [outer][inner] (inner contiguous, pitch == inner), tiles of
// box_outer x 128 bytes with 128-byte swizzle.  Rows past `outer` read as 0.
fp8bq_status encode_u8_map_uncached(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {128, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BQ_OK : FP8BQ_ERR_CUDA;
}

fp8bq_status encode_u8_map(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer) {
    return g_maps.get(MapKey{ptr, inner, outer, 128, box_outer, 0}, map, [&](CUtensorMap* m) {
        return encode_u8_map_uncached(m, ptr, inner, outer, box_outer);
    });
}

// 2-D output [rows][cols] (dense), BF16 or FP32, store boxes of 32 rows x
// 64 bytes (32 BF16 or 16 FP32 columns) with 64-byte swizzle, matching the
// epilogue staging.
fp8bq_status encode_out_map_uncached(CUtensorMap* map, void* ptr, uint64_t cols, uint64_t rows, bool f32) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (f32 ? 4 : 2)};
    const cuuint32_t box[2] = {f32 ? 16u : 32u, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr,
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BQ_OK : FP8BQ_ERR_CUDA;
}

fp8bq_status encode_out_map(CUtensorMap* map, void* ptr, uint64_t cols, uint64_t rows, bool f32) {
    return g_maps.get(MapKey{ptr, cols, rows, f32 ? 16u : 32u, 32, f32 ? 2 : 1}, map, [&](CUtensorMap* m) {
        return encode_out_map_uncached(m, ptr, cols, rows, f32);
    });
}

// One 128x128 slab per CTA: grid (ceil(C/128), R/128).
template <int kMode>
fp8bq_status launch_tile(const DeviceState* dev, const void* x, int dtype, int64_t R, int64_t C, int64_t ldx,
                         uint8_t* q, float* s_row, uint8_t* qT, float* s_col, cudaStream_t cs) {
    (void)dev;
    dim3 grid(static_cast<unsigned>((C + 127) / 128), static_cast<unsigned>(R / 128));
    if (dtype == FP8BQ_BF16)
        fp8bq::quantize_tile_kernel<false, kMode>
            <<<grid, 256, fp8bq::tile_smem_bytes<false>(), cs>>>(x, R, C, ldx, q, s_row, qT, s_col);
    else
        fp8bq::quantize_tile_kernel<true, kMode>
            <<<grid, 256, fp8bq::tile_smem_bytes<true>(), cs>>>(x, R, C, ldx, q, s_row, qT, s_col);
    return launch_status();
}

// Outputs of one GEMM launch.  d: the product, BF16 (f32 = false) or FP32,
// may be null when only codes are wanted; accumulate (FP32 only) adds into d.
// q / sq: row-wise 1x128 E4M3 codes [I][J] and scales [J/128][I] of the
// BF16-rounded product (both or neither).
struct GemmOut {
    void* d = nullptr;
    bool f32 = false;
    bool accumulate = false;
    uint8_t* q = nullptr;
    float* sq = nullptr;
    uint8_t* scratch = nullptr;   // balanced order's split slots and counters (null: tile order)
    int64_t scratch_bytes = 0;
};

// Scratch of the balanced order for `pairs` clusters: one arrival counter per
// remaining tile (at most pairs - 1 of them), CTA rank and promotion warp
// (rounded up to 256 bytes), then each cluster's two split slots.
int64_t split_counter_bytes(int pairs) {
    return ((static_cast<int64_t>(pairs - 1) * fp8bq::kSplitTileCounters * 4 + 255) / 256) * 256;
}
int64_t split_scratch_bytes(int pairs) {
    return pairs < 2 ? 0 : split_counter_bytes(pairs) + static_cast<int64_t>(pairs) * fp8bq::kSplitClusterBytes;
}

// n FP32 values set to v (scales of all-zero tiles).
__global__ void fill_f32_kernel(float* p, int64_t n, float v) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i < n) p[i] = v;
}

// 2-D uint8 output [rows][cols] (dense), store boxes of 32 rows x 64 bytes
// with 64-byte swizzle (the quantized-output epilogue's staging).
fp8bq_status encode_u8_out_map_uncached(CUtensorMap* map, void* ptr, uint64_t cols, uint64_t rows) {
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BQ_OK : FP8BQ_ERR_CUDA;
}

fp8bq_status encode_u8_out_map(CUtensorMap* map, void* ptr, uint64_t cols, uint64_t rows) {
    return g_maps.get(MapKey{ptr, cols, rows, 64, 32, 3}, map, [&](CUtensorMap* m) {
        return encode_u8_out_map_uncached(m, ptr, cols, rows);
    });
}

// One 128x128 slab per CTA: grid (C/128, M/128).  Column-wise codes always,
// row-wise codes too when kRows.
template <bool kRows>
fp8bq_status launch_mx_slab(const void* x, int dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* qT, uint8_t* e8T,
                   uint8_t* q, uint8_t* e8, cudaStream_t cs) {
    dim3 grid(static_cast<unsigned>(C / 128), static_cast<unsigned>(M / 128));
    uint16_t* ehT = reinterpret_cast<uint16_t*>(e8T);
    uint16_t* eh = reinterpret_cast<uint16_t*>(e8);
    if (dtype == FP8BQ_BF16)
        fp8bq::mx_quantize_slab_kernel<false, kRows>
            <<<grid, 256, fp8bq::mx_col_smem_bytes<false>(), cs>>>(x, M, C, ldx, qT, ehT, q, eh);
    else
        fp8bq::mx_quantize_slab_kernel<true, kRows>
            <<<grid, 256, fp8bq::mx_col_smem_bytes<true>(), cs>>>(x, M, C, ldx, qT, ehT, q, eh);
    return launch_status();
}

template <int MODE>
fp8bq_status run_gemm(const uint8_t* A, const float* sA, const uint8_t* B, const float* sB, const GemmOut& o, int64_t I,
             int64_t J, int64_t Kr, cudaStream_t stream) {
    if (I < 0 || J < 0 || Kr < 0) return FP8BQ_ERR_SHAPE;
    if ((I % 128) || (J % 128) || (Kr % 128)) return FP8BQ_ERR_SHAPE;
    if (I >= (int64_t(1) << 31) || J >= (int64_t(1) << 31) || Kr >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    if (I == 0 || J == 0) return FP8BQ_OK;
    if (o.d == nullptr && o.q == nullptr) return FP8BQ_ERR_NULL;
    if ((o.q == nullptr) != (o.sq == nullptr)) return FP8BQ_ERR_NULL;
    if (Kr > 0 && (!A || !sA || !B || !sB)) return FP8BQ_ERR_NULL;
    if ((o.d && !aligned16(o.d)) || (o.q && (!aligned16(o.q) || !aligned16(o.sq)))) return FP8BQ_ERR_ALIGN;
    if (Kr > 0 && (!aligned16(A) || !aligned16(B) || !aligned16(sA) || !aligned16(sB))) return FP8BQ_ERR_ALIGN;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    if (o.scratch != nullptr && o.scratch_bytes < split_scratch_bytes(dev->max_pairs)) return FP8BQ_ERR_SHAPE;
    if (Kr == 0) {
        // empty reduction: the product is exactly zero (adding it changes
        // nothing); its tiles quantize to +0 codes with scale 1
        if (o.d && !o.accumulate &&
            cudaMemsetAsync(o.d, 0, static_cast<size_t>(I) * J * (o.f32 ? 4 : 2), stream) != cudaSuccess)
            return FP8BQ_ERR_CUDA;
        if (o.q) {
            if (cudaMemsetAsync(o.q, 0, static_cast<size_t>(I) * J, stream) != cudaSuccess) return FP8BQ_ERR_CUDA;
            const int64_t n = I * (J / 128);
            fill_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(o.sq, n, 1.0f);
            return launch_status();
        }
        return FP8BQ_OK;
    }

    CUtensorMap ta, tb, td, tq;
    if (encode_u8_map(&ta, A, Kr, I, fp8bq::kBM) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    if (encode_u8_map(&tb, B, Kr, J, fp8bq::kBRows) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    if (o.d && encode_out_map(&td, o.d, J, I, o.f32) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    if (o.q && encode_u8_out_map(&tq, o.q, J, I) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    if (!o.d) td = tq;  // unused by the kernel
    if (!o.q) tq = td;

    fp8bq::GemmParams p;
    p.sA = sA;
    p.sB = sB;
    p.I = static_cast<int>(I);
    p.J = static_cast<int>(J);
    p.KC = static_cast<int>(Kr / 128);
    p.tiles_n = static_cast<int>((J + fp8bq::kBN - 1) / fp8bq::kBN);
    const int64_t tiles = ((I + fp8bq::kPairM - 1) / fp8bq::kPairM) * p.tiles_n;
    if (tiles >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    p.num_tiles = static_cast<int>(tiles);
    p.out_f32 = o.f32 ? 1 : 0;
    p.accumulate = o.accumulate ? 1 : 0;
    p.out_bf16 = (o.d && !o.f32) ? 1 : 0;
    p.out_q = o.q ? 1 : 0;
    p.sq = o.sq;
    p.timeout_ns = kDefaultTimeoutNs;
    // persistent: one CTA pair per TPC that can hold one, never more pairs than tiles
    const int pairs = static_cast<int>(tiles < dev->max_pairs ? tiles : dev->max_pairs);
    // balanced order (with scratch, Wgrad only): the whole-tile rounds run in
    // tile order and the chunks of the tiles left over for a last, partly
    // filled round are shared out equally between all clusters.  Used where
    // that round would leave at least 10 % of the clusters idle; its
    // remainder chunk arithmetic is 32-bit.
    p.split_ws = nullptr;
    p.split_cnt = nullptr;
    const int64_t rem = tiles % pairs;
    const bool balanced = MODE == fp8bq::kModeWgrad && o.scratch != nullptr && pairs >= 2 && rem > 0 &&
                          10 * rem <= 9 * static_cast<int64_t>(pairs) && rem * p.KC * pairs < (int64_t(1) << 31);
    if (balanced) {
        p.split_cnt = reinterpret_cast<unsigned int*>(o.scratch);
        p.split_ws = reinterpret_cast<float*>(o.scratch + split_counter_bytes(pairs));
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    gemm_launch_config(&cfg, attr, pairs, stream);
    cudaError_t e;
    if constexpr (MODE == fp8bq::kModeWgrad) {
        if (balanced)
            e = cudaLaunchKernelEx(&cfg, fp8bq::gemm_block_scaled_kernel<MODE, true>, ta, tb, td, tq, p, dev->status);
        else
            e = cudaLaunchKernelEx(&cfg, fp8bq::gemm_block_scaled_kernel<MODE>, ta, tb, td, tq, p, dev->status);
    } else {
        e = cudaLaunchKernelEx(&cfg, fp8bq::gemm_block_scaled_kernel<MODE>, ta, tb, td, tq, p, dev->status);
    }
    if (e != cudaSuccess) return FP8BQ_ERR_CUDA;
    return launch_status();
}

}  // namespace

extern "C" {

fp8bq_status fp8bq_quantize_rowwise(const void* x, fp8bq_dtype dtype, int64_t R, int64_t C, int64_t ldx, uint8_t* q, float* s,
                                    fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (R < 0 || C < 0 || ldx < C || (C % 128)) return FP8BQ_ERR_SHAPE;
    if (R == 0 || C == 0) return FP8BQ_OK;
    if (!x || !q || !s) return FP8BQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s) || ((ldx * elem_size(dtype)) % 16)) return FP8BQ_ERR_ALIGN;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    const int64_t tiles = R * (C / 128);
    if (tiles >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;  // the kernel indexes tiles in 32 bits
    const int64_t blocks = (tiles + 31) / 32;                    // 8 warps x 4 tiles
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == FP8BQ_BF16)
        fp8bq::quantize_rowwise_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, cs>>>(x, R, C, ldx, q, s);
    else
        fp8bq::quantize_rowwise_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, cs>>>(x, R, C, ldx, q, s);
    return launch_status();
}

fp8bq_status fp8bq_quantize_colwise(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* qT, float* s,
                                    fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (M < 0 || C < 0 || ldx < C || (M % 128) || (C % 8)) return FP8BQ_ERR_SHAPE;
    if (M == 0 || C == 0) return FP8BQ_OK;
    if (!x || !qT || !s) return FP8BQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(qT) || !aligned16(s) || ((ldx * elem_size(dtype)) % 16)) return FP8BQ_ERR_ALIGN;
    if (M / 128 > 65535 || (C + 127) / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    return launch_tile<fp8bq::kTileCol>(dev, x, dtype, M, C, ldx, nullptr, nullptr, qT, s,
                                        reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_quantize_rowcol(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* q, float* s_row,
                                   uint8_t* qT, float* s_col, fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (M < 0 || C < 0 || ldx < C || (M % 128) || (C % 128)) return FP8BQ_ERR_SHAPE;
    if (M == 0 || C == 0) return FP8BQ_OK;
    if (!x || !q || !s_row || !qT || !s_col) return FP8BQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s_row) || !aligned16(qT) || !aligned16(s_col) ||
        ((ldx * elem_size(dtype)) % 16))
        return FP8BQ_ERR_ALIGN;
    if (M / 128 > 65535 || C / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    return launch_tile<fp8bq::kTileDual>(dev, x, dtype, M, C, ldx, q, s_row, qT, s_col,
                                         reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_swiglu_quantize(const void* gu, int64_t M, int64_t F, int64_t ldgu, uint16_t* h, uint8_t* q,
                                   float* s_row, uint8_t* qT, float* s_col, fp8bq_stream_t stream) {
    if (M < 0 || F < 0 || (M % 128) || (F % 128) || ldgu < 2 * F) return FP8BQ_ERR_SHAPE;
    if (M == 0 || F == 0) return FP8BQ_OK;
    if (!gu || !q || !s_row || !qT || !s_col) return FP8BQ_ERR_NULL;
    if (!aligned16(gu) || !aligned16(q) || !aligned16(s_row) || !aligned16(qT) || !aligned16(s_col) ||
        (h && !aligned16(h)) || ((ldgu * 2) % 16))
        return FP8BQ_ERR_ALIGN;
    if (M / 128 > 65535 || F / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    dim3 grid(static_cast<unsigned>(F / 128), static_cast<unsigned>(M / 128));
    fp8bq::quantize_tile_kernel<false, fp8bq::kTileSwiglu>
        <<<grid, 256, fp8bq::tile_smem_bytes<false, fp8bq::kTileSwiglu>(), reinterpret_cast<cudaStream_t>(stream)>>>(
            gu, M, F, ldgu, q, s_row, qT, s_col, F, h);
    return launch_status();
}

fp8bq_status fp8bq_quantize_weight_block(const void* w, fp8bq_dtype dtype, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                         uint8_t* qT, float* s, fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (N < 0 || K < 0 || ldw < K || (N % 128) || (K % 128)) return FP8BQ_ERR_SHAPE;
    if (N == 0 || K == 0) return FP8BQ_OK;
    if (!w || !q || !s) return FP8BQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (qT && !aligned16(qT)) ||
        ((ldw * elem_size(dtype)) % 16))
        return FP8BQ_ERR_ALIGN;
    if (N / 128 > 65535 || K / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    return launch_tile<fp8bq::kTileWeight>(dev, w, dtype, N, K, ldw, q, s, qT, nullptr,
                                           reinterpret_cast<cudaStream_t>(stream));
}

// Host-side checks of one weight block quantization (those of
// fp8bq_quantize_weight_block).
fp8bq_status check_weight_args(const void* w, int64_t N, int64_t K, int64_t ldw, const uint8_t* q, const uint8_t* qT,
                               const float* s, int dtype) {
    if (N < 0 || K < 0 || ldw < K || (N % 128) || (K % 128)) return FP8BQ_ERR_SHAPE;
    if (N == 0 || K == 0) return FP8BQ_OK;
    if (!w || !q || !s) return FP8BQ_ERR_NULL;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s) || (qT && !aligned16(qT)) ||
        ((ldw * elem_size(dtype)) % 16))
        return FP8BQ_ERR_ALIGN;
    if (N / 128 > 65535 || K / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    if ((N / 128) * (K / 128) >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;  // blocks are numbered in 32 bits
    return FP8BQ_OK;
}

fp8bq_status fp8bq_quantize_weight_blocks(const fp8bq_weight* weights, int count, fp8bq_dtype dtype,
                                          fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (count < 0) return FP8BQ_ERR_SHAPE;
    if (count == 0) return FP8BQ_OK;
    if (!weights) return FP8BQ_ERR_NULL;
    bool any = false;
    for (int i = 0; i < count; ++i) {
        const fp8bq_weight& e = weights[i];
        const fp8bq_status st = check_weight_args(e.w, e.N, e.K, e.ldw, e.q, e.qT, e.s, dtype);
        if (st != FP8BQ_OK) return st;
        any = any || (e.N > 0 && e.K > 0);
    }
    if (!any) return FP8BQ_OK;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    int i = 0;
    while (i < count) {
        fp8bq::WeightGroup g = {};
        int64_t blocks = 0;
        for (; i < count && g.n < fp8bq::kMaxWeightGroup; ++i) {
            const fp8bq_weight& e = weights[i];
            if (e.N == 0 || e.K == 0) continue;
            const int64_t nb = (e.N / 128) * (e.K / 128);
            if (blocks + nb >= (int64_t(1) << 31)) break;
            const int k = g.n++;
            g.first_block[k] = static_cast<int>(blocks);
            g.nbx[k] = static_cast<int>(e.K / 128);
            g.w[k] = e.w;
            g.N[k] = e.N;
            g.K[k] = e.K;
            g.ldw[k] = e.ldw;
            g.q[k] = e.q;
            g.qT[k] = e.qT;
            g.s[k] = e.s;
            blocks += nb;
        }
        if (g.n == 0) continue;
        g.first_block[g.n] = static_cast<int>(blocks);
        if (dtype == FP8BQ_BF16)
            fp8bq::quantize_weight_group_kernel<false>
                <<<static_cast<unsigned>(blocks), 256, fp8bq::tile_smem_bytes<false>(), cs>>>(g);
        else
            fp8bq::quantize_weight_group_kernel<true>
                <<<static_cast<unsigned>(blocks), 256, fp8bq::tile_smem_bytes<true>(), cs>>>(g);
        st = launch_status();
        if (st != FP8BQ_OK) return st;
    }
    return FP8BQ_OK;
}

fp8bq_status fp8bq_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, uint16_t* y, int64_t M,
                              int64_t N, int64_t K, fp8bq_stream_t stream) {
    if (y == nullptr && M > 0 && N > 0) return FP8BQ_ERR_NULL;
    GemmOut o;
    o.d = y;
    return run_gemm<fp8bq::kModeFprop>(xq, sx, wq, sw, o, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_gemm_fprop_q(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw, uint16_t* y,
                                uint8_t* yq, float* sy, int64_t M, int64_t N, int64_t K, fp8bq_stream_t stream) {
    if ((yq == nullptr || sy == nullptr) && M > 0 && N > 0) return FP8BQ_ERR_NULL;
    GemmOut o;
    o.d = y;
    o.q = yq;
    o.sq = sy;
    return run_gemm<fp8bq::kModeFprop>(xq, sx, wq, sw, o, M, N, K, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wqT, const float* sw, uint16_t* dx,
                              int64_t M, int64_t N, int64_t K, fp8bq_stream_t stream) {
    if (dx == nullptr && M > 0 && K > 0) return FP8BQ_ERR_NULL;
    GemmOut o;
    o.d = dx;
    return run_gemm<fp8bq::kModeDgrad>(dyq, sdy, wqT, sw, o, M, K, N, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_gemm_wgrad(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT, const float* sxT, uint16_t* dw,
                              int64_t M, int64_t N, int64_t K, fp8bq_stream_t stream) {
    if (dw == nullptr && N > 0 && K > 0) return FP8BQ_ERR_NULL;
    GemmOut o;
    o.d = dw;
    return run_gemm<fp8bq::kModeWgrad>(dyqT, sdyT, xqT, sxT, o, N, K, M, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_gemm_wgrad_scratch_bytes(int64_t* bytes) {
    if (bytes == nullptr) return FP8BQ_ERR_NULL;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    *bytes = split_scratch_bytes(dev->max_pairs);
    return FP8BQ_OK;
}

fp8bq_status fp8bq_gemm_wgrad_balanced(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT, const float* sxT,
                                       uint16_t* dw, int64_t M, int64_t N, int64_t K, void* scratch,
                                       int64_t scratch_bytes, fp8bq_stream_t stream) {
    if (dw == nullptr && N > 0 && K > 0) return FP8BQ_ERR_NULL;
    if (scratch == nullptr) return FP8BQ_ERR_NULL;
    if (!aligned16(scratch)) return FP8BQ_ERR_ALIGN;
    if (scratch_bytes < 0) return FP8BQ_ERR_SHAPE;
    GemmOut o;
    o.d = dw;
    o.scratch = static_cast<uint8_t*>(scratch);
    o.scratch_bytes = scratch_bytes;
    return run_gemm<fp8bq::kModeWgrad>(dyqT, sdyT, xqT, sxT, o, N, K, M, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_gemm_wgrad_balanced_static(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT,
                                              const float* sxT, uint16_t* dw, int64_t M, int64_t N, int64_t K,
                                              fp8bq_stream_t stream) {
    if (dw == nullptr && N > 0 && K > 0) return FP8BQ_ERR_NULL;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    if (split_scratch_bytes(dev->max_pairs) > kStaticScratchBytes) return FP8BQ_ERR_SHAPE;  // more clusters than it holds
    GemmOut o;
    o.d = dw;
    o.scratch = dev->wgrad_scratch;
    o.scratch_bytes = kStaticScratchBytes;
    return run_gemm<fp8bq::kModeWgrad>(dyqT, sdyT, xqT, sxT, o, N, K, M, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_gemm_wgrad_f32(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT, const float* sxT, float* dw,
                                  int64_t M, int64_t N, int64_t K, int accumulate, fp8bq_stream_t stream) {
    if (accumulate != 0 && accumulate != 1) return FP8BQ_ERR_SHAPE;
    if (dw == nullptr && N > 0 && K > 0) return FP8BQ_ERR_NULL;
    GemmOut o;
    o.d = dw;
    o.f32 = true;
    o.accumulate = accumulate == 1;
    return run_gemm<fp8bq::kModeWgrad>(dyqT, sdyT, xqT, sxT, o, N, K, M, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_mx_quantize_rowwise(const void* x, fp8bq_dtype dtype, int64_t R, int64_t C, int64_t ldx, uint8_t* q,
                                       uint8_t* e8, fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (R < 0 || C < 0 || ldx < C || (C % 128)) return FP8BQ_ERR_SHAPE;
    if (R == 0 || C == 0) return FP8BQ_OK;
    if (!x || !q || !e8) return FP8BQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(e8) || ((ldx * elem_size(dtype)) % 16)) return FP8BQ_ERR_ALIGN;
    const int64_t nb = R * (C / 32);
    if (nb >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;  // the kernel numbers blocks in 32 bits
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    const int64_t per_warp = (dtype == FP8BQ_BF16 ? 8 : 4) * fp8bq::kMxRowSteps;
    const int64_t blocks = ((nb + per_warp - 1) / per_warp + 7) / 8;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    uint32_t* ew = reinterpret_cast<uint32_t*>(e8);
    if (dtype == FP8BQ_BF16)
        fp8bq::mx_quantize_rowwise_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, cs>>>(x, R, C, ldx, q, ew);
    else
        fp8bq::mx_quantize_rowwise_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, cs>>>(x, R, C, ldx, q, ew);
    return launch_status();
}

fp8bq_status fp8bq_mx_quantize_colwise(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* qT,
                                       uint8_t* e8, fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (M < 0 || C < 0 || ldx < C || (M % 128) || (C % 128)) return FP8BQ_ERR_SHAPE;
    if (M == 0 || C == 0) return FP8BQ_OK;
    if (!x || !qT || !e8) return FP8BQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(qT) || !aligned16(e8) || ((ldx * elem_size(dtype)) % 16)) return FP8BQ_ERR_ALIGN;
    if (M / 128 > 65535 || C / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    return launch_mx_slab<false>(x, dtype, M, C, ldx, qT, e8, nullptr, nullptr,
                                 reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_mx_quantize_rowcol(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* q,
                                      uint8_t* e8, uint8_t* qT, uint8_t* e8T, fp8bq_stream_t stream) {
    if (dtype != FP8BQ_BF16 && dtype != FP8BQ_F32) return FP8BQ_ERR_DTYPE;
    if (M < 0 || C < 0 || ldx < C || (M % 128) || (C % 128)) return FP8BQ_ERR_SHAPE;
    if (M == 0 || C == 0) return FP8BQ_OK;
    if (!x || !q || !e8 || !qT || !e8T) return FP8BQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(q) || !aligned16(e8) || !aligned16(qT) || !aligned16(e8T) ||
        ((ldx * elem_size(dtype)) % 16))
        return FP8BQ_ERR_ALIGN;
    if (M / 128 > 65535 || C / 128 >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    return launch_mx_slab<true>(x, dtype, M, C, ldx, qT, e8T, q, e8, reinterpret_cast<cudaStream_t>(stream));
}

fp8bq_status fp8bq_mx_gemm(const uint8_t* a, const uint8_t* ea, const uint8_t* b, const uint8_t* eb, uint16_t* d, int64_t I,
                           int64_t J, int64_t K, fp8bq_stream_t stream) {
    if (I < 0 || J < 0 || K < 0 || (I % 128) || (J % 128) || (K % 128)) return FP8BQ_ERR_SHAPE;
    if (I >= (int64_t(1) << 31) || J >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    if (I == 0 || J == 0) return FP8BQ_OK;
    if (!d) return FP8BQ_ERR_NULL;
    if (K > 0 && (!a || !ea || !b || !eb)) return FP8BQ_ERR_NULL;
    if (!aligned16(d)) return FP8BQ_ERR_ALIGN;
    if (K > 0 && (!aligned16(a) || !aligned16(ea) || !aligned16(b) || !aligned16(eb))) return FP8BQ_ERR_ALIGN;
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {  // empty reduction: exact zeros
        return cudaMemsetAsync(d, 0, static_cast<size_t>(I) * J * 2, cs) == cudaSuccess ? FP8BQ_OK : FP8BQ_ERR_CUDA;
    }
    CUtensorMap ta, tb, td;
    if (encode_u8_map(&ta, a, K, I, fp8bq::kMxBM) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    if (encode_u8_map(&tb, b, K, J, fp8bq::kMxBN) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    if (encode_out_map(&td, d, J, I, false) != FP8BQ_OK) return FP8BQ_ERR_CUDA;
    fp8bq::MxParams p;
    p.ea = reinterpret_cast<const uint32_t*>(ea);
    p.eb = reinterpret_cast<const uint32_t*>(eb);
    p.I = static_cast<int>(I);
    p.J = static_cast<int>(J);
    p.KC = static_cast<int>(K / 128);
    p.tiles_n = static_cast<int>((J + fp8bq::kMxBN - 1) / fp8bq::kMxBN);
    const int64_t tiles = (I / fp8bq::kMxBM) * p.tiles_n;
    if (tiles >= (int64_t(1) << 31)) return FP8BQ_ERR_SHAPE;
    p.num_tiles = static_cast<int>(tiles);
    p.timeout_ns = kDefaultTimeoutNs;
    const int grid = static_cast<int>(tiles < dev->sms ? tiles : dev->sms);  // persistent, one CTA per SM
    fp8bq::mx_gemm_kernel<<<grid, fp8bq::kMxThreads, fp8bq::kMxSmemBytes, cs>>>(ta, tb, td, p, dev->status);
    return launch_status();
}

fp8bq_status fp8bq_check(fp8bq_stream_t stream) {
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    unsigned int word = 0;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return FP8BQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(dev->check_mu);
    status_take_kernel<<<1, 1, 0, cs>>>(dev->status, dev->taken);
    if (cudaGetLastError() != cudaSuccess) return FP8BQ_ERR_CUDA;
    if (cudaMemcpyAsync(&word, dev->taken, sizeof(word), cudaMemcpyDeviceToHost, cs) != cudaSuccess)
        return FP8BQ_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return FP8BQ_ERR_CUDA;
    return (word & 1u) ? FP8BQ_ERR_TIMEOUT : FP8BQ_OK;
}

const char* fp8bq_status_string(fp8bq_status status) {
    switch (status) {
        case FP8BQ_OK: return "ok";
        case FP8BQ_ERR_NULL: return "null pointer argument";
        case FP8BQ_ERR_SHAPE: return "invalid shape (negative, not a multiple of 128, or pitch < width)";
        case FP8BQ_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
        case FP8BQ_ERR_DTYPE: return "unknown input dtype";
        case FP8BQ_ERR_DEVICE: return "current device is not an sm_103 GPU";
        case FP8BQ_ERR_CUDA: return "CUDA call or kernel launch failed";
        case FP8BQ_ERR_TIMEOUT: return "a kernel gave up waiting on its pipeline (outputs undefined)";
        default: return "unknown status";
    }
}

fp8bq_status fp8bq_selftest_wait_timeout(int64_t limit_ns, fp8bq_stream_t stream) {
    DeviceState* dev = nullptr;
    fp8bq_status st = probe_device(&dev);
    if (st != FP8BQ_OK) return st;
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 2000000000ll) limit_ns = 2000000000ll;
    fp8bq::wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<uint64_t>(limit_ns), dev->status);
    return launch_status();
}

}  // extern "C"
