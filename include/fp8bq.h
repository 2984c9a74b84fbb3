/*
 * fp8bq.h — C ABI of the block-scaled FP8 linear layer for B300 (sm_103a).
 *
 * What the library computes.  The Puro-2B technical report (section 2, "FP8")
 * moves the matrix multiplications of the main linear layers onto an FP8
 * path using DeepSeek-V3's fine-grained block quantization, and keeps
 * numerically sensitive work in BF16/FP32.  This library is that path for one
 * nn.Linear with input X [M, K], weight W [N, K] and output gradient dY [M, N]:
 *
 *   quantize   activations and gradients per 1x128 tile, weights per 128x128
 *              block, to E4M3 (OCP FP8) with an FP32 scale per tile:
 *              s = amax / 448 (s = 1 when amax == 0), code = E4M3 of the
 *              correctly rounded FP32 quotient x / s, round half to even,
 *              saturating at +-448.
 *   GEMM       Fprop  Y  = X  W^T  (reduce over K),
 *              Dgrad  dX = dY W    (reduce over N),
 *              Wgrad  dW = dY^T X  (reduce over the M tokens);
 *              FP8 x FP8 products accumulate in FP32 per 128-wide reduction
 *              chunk, each chunk is multiplied by the product of its two
 *              scales and added into an FP32 accumulator, and the result is
 *              written as BF16 (round half to even).
 *
 * Conventions shared by every entry point
 *   - All pointers except `stream` are DEVICE pointers to memory the caller
 *     owns.  The library never allocates, frees or retains caller buffers.
 *   - Matrices are row-major with unit inner stride.  `ld*` arguments are row
 *     pitches in ELEMENTS of the input type; outputs are dense (pitch = width).
 *   - Scale arrays are FP32 and chunk-major: the scale of the tile that covers
 *     row r in reduction chunk c is at s[c * rows + r].  Weight scales are
 *     sw[N/128][K/128].
 *   - Every dimension that is quantized or reduced over must be a multiple of
 *     128; partial tiles are rejected (FP8BQ_ERR_SHAPE).  A zero dimension is
 *     a no-op that returns FP8BQ_OK (a GEMM with an empty reduction writes
 *     zeros).
 *   - Pointers must be 16-byte aligned and row pitches a multiple of 16 bytes
 *     (TMA and 128-bit vector access), else FP8BQ_ERR_ALIGN.  Inputs and
 *     outputs must not overlap.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and on the calling thread's current device, which must
 *     be an sm_103 GPU (else FP8BQ_ERR_DEVICE).  Argument errors are detected
 *     on the host before anything is launched and leave every buffer
 *     untouched.  A failed launch returns FP8BQ_ERR_CUDA.  Device-side faults
 *     the kernels detect themselves (a pipeline wait that ran out of time)
 *     are recorded in a per-device status word and reported by fp8bq_check.
 *   - The library is thread-safe; it keeps only a per-device status word, a
 *     cache of device properties and a mutex-guarded cache of the TMA
 *     descriptors it encoded (keyed by every argument of the encoding, so a
 *     buffer reused with the same shape is not encoded again), all created on
 *     first use.
 */
#ifndef FP8BQ_H
#define FP8BQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same representation as cudaStream_t, without requiring CUDA headers. */
typedef struct CUstream_st* fp8bq_stream_t;

typedef enum {
    FP8BQ_OK = 0,
    FP8BQ_ERR_NULL = 1,     /* a required pointer is NULL                        */
    FP8BQ_ERR_SHAPE = 2,    /* negative size, non-multiple of 128, pitch < width */
    FP8BQ_ERR_ALIGN = 3,    /* pointer or pitch not 16-byte aligned              */
    FP8BQ_ERR_DTYPE = 4,    /* unknown fp8bq_dtype                               */
    FP8BQ_ERR_DEVICE = 5,   /* current device is not sm_103                      */
    FP8BQ_ERR_CUDA = 6,     /* a CUDA runtime/driver call or launch failed       */
    FP8BQ_ERR_TIMEOUT = 7   /* a kernel gave up waiting (reported by fp8bq_check)*/
} fp8bq_status;

typedef enum {
    FP8BQ_BF16 = 0,         /* 16-bit bfloat16 input */
    FP8BQ_F32 = 1           /* 32-bit IEEE float input */
} fp8bq_dtype;

/*
 * Row-wise 1x128 quantization (Fprop activations X, Dgrad output gradients dY).
 *   x      [R][C] input of `dtype`, row pitch ldx elements (ldx >= C)
 *   q      [R][C] E4M3 codes, dense
 *   s      [C/128][R] FP32 scales: s[t*R + r] belongs to x[r][128t .. 128t+127]
 * Requires C % 128 == 0.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8": the
 *   main linear layers' matmuls in FP8 with DeepSeek-V3's fine-grained block
 *   quantization; 1x128 tiles, E4M3, amax/448 and RNE are this library's
 *   reading of it (the report prints no formula).
 */
fp8bq_status fp8bq_quantize_rowwise(const void* x, fp8bq_dtype dtype, int64_t R, int64_t C, int64_t ldx,
                                    uint8_t* q, float* s, fp8bq_stream_t stream);

/*
 * Column-wise 128x1 quantization emitted transposed (Wgrad operands: dY and
 * X quantized along the token dimension that Wgrad reduces over).
 *   x      [M][C] input of `dtype`, row pitch ldx elements (ldx >= C)
 *   qT     [C][M] E4M3 codes: qT[c*M + m] is the code of x[m][c], dense
 *   s      [M/128][C] FP32 scales: s[b*C + c] belongs to x[128b .. 128b+127][c]
 * Requires M % 128 == 0 and C % 8 == 0 (16-byte rows of BF16).
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8" (as
 *   fp8bq_quantize_rowwise), tiles along the token dimension that Wgrad
 *   reduces over.
 */
fp8bq_status fp8bq_quantize_colwise(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx,
                                    uint8_t* qT, float* s, fp8bq_stream_t stream);

/*
 * Row-wise 1x128 and column-wise 128x1 quantization of the same tensor in one
 * pass over it (the output gradient dY feeds Dgrad row-wise and Wgrad
 * column-wise; an activation X feeds Fprop row-wise and Wgrad column-wise).
 * Writes exactly what fp8bq_quantize_rowwise(x -> q, s_row) followed by
 * fp8bq_quantize_colwise(x -> qT, s_col) would, bit for bit, while reading x
 * from memory once instead of twice.
 *   x      [M][C] input of `dtype`, row pitch ldx elements (ldx >= C)
 *   q      [M][C] row-wise codes,      s_row [C/128][M]
 *   qT     [C][M] column-wise codes,   s_col [M/128][C]
 * Requires M % 128 == 0 and C % 128 == 0.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8" (as
 *   the two quantizers it fuses).
 */
fp8bq_status fp8bq_quantize_rowcol(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx,
                                   uint8_t* q, float* s_row, uint8_t* qT, float* s_col, fp8bq_stream_t stream);

/*
 * SwiGLU gate fused into the quantizer of the down projection's input.  From
 * the gate/up projection's output, h = silu(g) * u = g u / (1 + exp(-g)) is
 * computed in FP32 and rounded to BF16 once, and that BF16 H is quantized
 * row-wise (down projection Fprop) and column-wise (its Wgrad) exactly as
 * fp8bq_quantize_rowcol(H) would, reading g and u once and never writing
 * or re-reading H unless asked to (the SwiGLU MLP of the 3.8B architecture
 * on the n1n.ai page; the report's FP8 recipe, section 2, for the down
 * projection's input).
 *   gu     [M][ldgu] BF16: g in columns [0, F), u in columns [F, 2F)
 *   h      [M][F] BF16 output of H, or NULL to skip
 *   q      [M][F] row-wise codes,     s_row [F/128][M]
 *   qT     [F][M] column-wise codes,  s_col [M/128][F]
 * Requires M % 128 == 0, F % 128 == 0, ldgu >= 2F, 16-byte aligned pointers
 * and row pitch.  H is formed in FP32 with a hardware exponential and a
 * correctly rounded reciprocal (relative error far below half a BF16 ulp),
 * so it may differ from a correctly rounded silu(g) u by one BF16 ulp; the
 * codes and scales are always exactly those of the H the kernel formed.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8" for
 *   the quantization; the SwiGLU MLP of the 3.8B architecture in the n1n.ai
 *   "$998 3.8B" article, model-architecture list, for the gate.
 */
fp8bq_status fp8bq_swiglu_quantize(const void* gu, int64_t M, int64_t F, int64_t ldgu, uint16_t* h, uint8_t* q,
                                   float* s_row, uint8_t* qT, float* s_col, fp8bq_stream_t stream);

/*
 * Weight quantization per 128x128 block.
 *   w      [N][K] weight of `dtype` (nn.Linear layout), row pitch ldw elements
 *   q      [N][K] E4M3 codes (Fprop operand), dense
 *   qT     [K][N] the same codes transposed (Dgrad operand), or NULL to skip
 *   s      [N/128][K/128] FP32 block scales
 * Requires N % 128 == 0 and K % 128 == 0.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8":
 *   fine-grained block quantization of the weights; 128x128 blocks are this
 *   library's reading.
 */
fp8bq_status fp8bq_quantize_weight_block(const void* w, fp8bq_dtype dtype, int64_t N, int64_t K, int64_t ldw,
                                         uint8_t* q, uint8_t* qT, float* s, fp8bq_stream_t stream);

/* One weight of fp8bq_quantize_weight_blocks: the arguments of
 * fp8bq_quantize_weight_block for that weight. */
typedef struct {
    const void* w;      /* [N][K] weight, row pitch ldw elements             */
    int64_t N, K, ldw;
    uint8_t* q;         /* [N][K] E4M3 codes                                 */
    uint8_t* qT;        /* [K][N] the same codes transposed, or NULL to skip */
    float* s;           /* [N/128][K/128] FP32 block scales                  */
} fp8bq_weight;

/*
 * Weight quantization per 128x128 block for several weights in one launch
 * (a training step quantizes every weight once after the optimizer update).
 * Writes, for each entry, exactly what fp8bq_quantize_weight_block would,
 * bit for bit.  All weights have element type `dtype`; the same requirements
 * apply to each entry (entries with N or K == 0 are skipped); any entry that
 * fails them fails the whole call before anything is launched.  count may be
 * 0; lists longer than 16 are processed 16 entries per launch.  `weights`
 * is a HOST array, read during the call only.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8" (as
 *   fp8bq_quantize_weight_block).
 */
fp8bq_status fp8bq_quantize_weight_blocks(const fp8bq_weight* weights, int count, fp8bq_dtype dtype,
                                          fp8bq_stream_t stream);

/*
 * Fprop: Y[m][n] = sum_c sx[c][m] * sw[n/128][c] * sum_{k in chunk c} D(xq[m][k]) D(wq[n][k])
 *   xq [M][K] codes, sx [K/128][M]    (from fp8bq_quantize_rowwise of X)
 *   wq [N][K] codes, sw [N/128][K/128] (from fp8bq_quantize_weight_block of W)
 *   y  [M][N] BF16 output (16-bit patterns), dense
 * Requires M, N, K % 128 == 0.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8": FP8
 *   matmul of the main linear layers, per-chunk FP32 promotion and BF16 output
 *   as this library reads the recipe.
 */
fp8bq_status fp8bq_gemm_fprop(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                              uint16_t* y, int64_t M, int64_t N, int64_t K, fp8bq_stream_t stream);

/*
 * Fprop whose epilogue also quantizes its output for a following linear
 * layer: the product is rounded to BF16 (as fp8bq_gemm_fprop writes it) and
 * each 1x128 row tile of that BF16 output is quantized exactly as
 * fp8bq_quantize_rowwise would (the report's FP8 recipe, section 2, applied
 * to the next layer's input, fused into the producer so the BF16 output
 * need not be written and read back).
 *   y   [M][N] BF16 output, or NULL to skip writing it
 *   yq  [M][N] E4M3 codes of the BF16 output, row-wise 1x128 tiles
 *   sy  [N/128][M] their FP32 scales
 * Other arguments as fp8bq_gemm_fprop.  With K == 0 the output is zero:
 * codes +0, scales 1.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8"
 *   (Fprop, with the next layer's quantization fused).
 */
fp8bq_status fp8bq_gemm_fprop_q(const uint8_t* xq, const float* sx, const uint8_t* wq, const float* sw,
                                uint16_t* y, uint8_t* yq, float* sy, int64_t M, int64_t N, int64_t K,
                                fp8bq_stream_t stream);

/*
 * Dgrad: dX[m][k] = sum_c sdy[c][m] * sw[c][k/128] * sum_{n in chunk c} D(dyq[m][n]) D(wq[n][k])
 *   dyq [M][N] codes, sdy [N/128][M]   (from fp8bq_quantize_rowwise of dY)
 *   wqT [K][N] codes (the qT output of fp8bq_quantize_weight_block),
 *   sw  [N/128][K/128] the weight's block scales
 *   dx  [M][K] BF16 output, dense
 * Requires M, N, K % 128 == 0.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8": the
 *   backward matmul of the same linear layers.
 */
fp8bq_status fp8bq_gemm_dgrad(const uint8_t* dyq, const float* sdy, const uint8_t* wqT, const float* sw,
                              uint16_t* dx, int64_t M, int64_t N, int64_t K, fp8bq_stream_t stream);

/*
 * Wgrad: dW[n][k] = sum_c sdyT[c][n] * sxT[c][k] * sum_{m in chunk c} D(dyqT[n][m]) D(xqT[k][m])
 *   dyqT [N][M] codes, sdyT [M/128][N] (from fp8bq_quantize_colwise of dY)
 *   xqT  [K][M] codes, sxT  [M/128][K] (from fp8bq_quantize_colwise of X)
 *   dw   [N][K] BF16 output, dense
 * Requires M, N, K % 128 == 0.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8": the
 *   weight-gradient matmul of the same linear layers.
 */
fp8bq_status fp8bq_gemm_wgrad(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT, const float* sxT,
                              uint16_t* dw, int64_t M, int64_t N, int64_t K, fp8bq_stream_t stream);

/*
 * Wgrad, balanced work split: the same product as fp8bq_gemm_wgrad.  The
 * persistent grid's whole-tile rounds run in fp8bq_gemm_wgrad's tile order;
 * the reduction chunks of the tiles left over for a last, partly filled
 * round are shared out equally between all clusters, so no cluster idles
 * through that round (each Wgrad tile reduces over all M tokens, so it costs
 * a whole tile's time).  The split is used where that round would leave at
 * least 10 % of the clusters idle; otherwise the call runs fp8bq_gemm_wgrad's
 * tile order (scratch untouched).  Each cluster leaves its FP32 partial of a
 * shared tile in `scratch`; the last to finish adds all the parts in cluster
 * order and writes the tile, so the result does not depend on which finishes
 * last and is the same on every call.  It differs from fp8bq_gemm_wgrad's
 * only in the grouping of the FP32 sum over chunks on the shared tiles:
 * within the same acceptance bound.
 *   scratch        device buffer of at least scratch_bytes bytes, 16-byte
 *                  aligned, all zero before its first use; every completed
 *                  call leaves it ready for the next (the arrival counters at
 *                  its start back at zero; the rest holds no state between
 *                  calls).  Calls that share a scratch buffer must not
 *                  overlap in time (order them on one stream).  After
 *                  FP8BQ_ERR_TIMEOUT, zero it again.
 *   scratch_bytes  at least fp8bq_gemm_wgrad_scratch_bytes() for the
 *                  current device (else FP8BQ_ERR_SHAPE)
 * Other arguments and requirements as fp8bq_gemm_wgrad.
 * Source: none in the pages; a scheduling form of the Wgrad GEMM of the
 *   Puro-2B technical report (lkr-homepage blog), section 2 "FP8".
 */
fp8bq_status fp8bq_gemm_wgrad_balanced(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT, const float* sxT,
                                       uint16_t* dw, int64_t M, int64_t N, int64_t K, void* scratch,
                                       int64_t scratch_bytes, fp8bq_stream_t stream);

/* Bytes of scratch fp8bq_gemm_wgrad_balanced needs on the current device
 * (the same for every shape; 0 when the device runs a single cluster). */
fp8bq_status fp8bq_gemm_wgrad_scratch_bytes(int64_t* bytes);

/*
 * fp8bq_gemm_wgrad_balanced without a caller buffer: its scratch is a
 * fixed array in the library's own device memory (allocated with the module,
 * no allocation call), sized for up to 74 clusters (a 148-SM B300); a device
 * that runs more clusters gets FP8BQ_ERR_SHAPE.  The same result, bit for
 * bit, as fp8bq_gemm_wgrad_balanced.  Calls on one device must not overlap in
 * time (they share the array: order them on one stream).  After
 * FP8BQ_ERR_TIMEOUT the array's counters may be left non-zero; reload the
 * library.  Other arguments as fp8bq_gemm_wgrad.
 * Source: the pages have no counterpart (an allocation-free form of the
 *   balanced Wgrad above).
 */
fp8bq_status fp8bq_gemm_wgrad_balanced_static(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT,
                                              const float* sxT, uint16_t* dw, int64_t M, int64_t N, int64_t K,
                                              fp8bq_stream_t stream);

/*
 * Wgrad with an FP32 output, for keeping weight gradients in FP32 across
 * micro-batches and data-parallel ranks (the Puro-2B report keeps training
 * state in FP32, section 2 "FP8").  Same operands and product as
 * fp8bq_gemm_wgrad; the result is not rounded to BF16.
 *   dw          [N][K] FP32, dense
 *   accumulate  0: dw = dY^T X;  1: dw += dY^T X (each element is added once,
 *               in FP32, in L2; dw must hold the running sum on entry)
 * Requires M, N, K % 128 == 0 and accumulate in {0, 1} (else FP8BQ_ERR_SHAPE).
 * The adds of accumulate = 1 are atomic per element: calls that overlap in
 * time on the same dw still sum correctly, in an unspecified order.
 * Source: Puro-2B technical report (lkr-homepage blog), section 2 "FP8":
 *   training state kept in FP32.
 */
fp8bq_status fp8bq_gemm_wgrad_f32(const uint8_t* dyqT, const float* sdyT, const uint8_t* xqT, const float* sxT,
                                  float* dw, int64_t M, int64_t N, int64_t K, int accumulate, fp8bq_stream_t stream);

/* ------------------------------------------------------------------------
 * MX variant: one power-of-two scale per 1x32 block
 *
 * A variant of the layer whose scales the tensor cores apply inside the MMA
 * (tcgen05.mma.kind::mxf8f6f4.block_scale), so no per-chunk promotion runs on
 * the CUDA cores.  Block shape and scale type are those of the OCP
 * Microscaling (MX) formats specification: 32 consecutive elements along the
 * reduction dimension share a scale 2^E stored as the byte E + 127 ("E8M0").
 * E is the layer's amax/448 scale rounded up to a power of two: the smallest
 * integer >= -127 with amax <= 448 * 2^E (so nothing saturates; an all-zero
 * block gets E = -127).  code = E4M3 of x * 2^-E, round half to even.  This
 * is a different numerical contract from the FP32-scale entry points above;
 * its codes and exponents are not interchangeable with theirs.
 *
 * Exponent arrays are uint8 and chunk-major: byte t of the 32-bit word for
 * row r and 128-element reduction chunk c, e[(c * rows + r) * 4 + t], is the
 * exponent of elements 128c + 32t .. 128c + 32t + 31 of that row.
 * ------------------------------------------------------------------------ */

/*
 * Row-wise MX quantization (1x32 blocks along C).
 *   x   [R][C] BF16 or FP32, row pitch ldx elements (ldx >= C)
 *   q   [R][C] uint8 E4M3 codes, dense
 *   e8  [C/128][R][4] uint8 exponents (E + 127)
 * Requires C % 128 == 0 and R * C / 32 < 2^31.  One read of x.
 * Fprop operands: X [M][K] and W [N][K]; Dgrad's left operand dY [M][N].
 * Source: no passage of the pages: the MX variant follows the OCP
 *   Microscaling formats specification (block of 32, E8M0 scale) for
 *   comparison with the report's recipe.
 */
fp8bq_status fp8bq_mx_quantize_rowwise(const void* x, fp8bq_dtype dtype, int64_t R, int64_t C, int64_t ldx, uint8_t* q,
                                       uint8_t* e8, fp8bq_stream_t stream);

/*
 * Column-wise MX quantization (32x1 blocks along M), emitted transposed.
 *   x   [M][C] BF16 or FP32, row pitch ldx elements (ldx >= C)
 *   qT  [C][M] uint8 codes, qT[c][m] the code of x[m][c]
 *   e8  [M/128][C][4] uint8 exponents
 * Requires M % 128 == 0, C % 128 == 0, M / 128 <= 65535.
 * Dgrad's right operand (W [N][K] -> [K][N]) and both Wgrad operands
 * (dY [M][N] -> [N][M], X [M][K] -> [K][M]).
 * Source: as fp8bq_mx_quantize_rowwise.
 */
fp8bq_status fp8bq_mx_quantize_colwise(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* qT,
                                       uint8_t* e8, fp8bq_stream_t stream);

/*
 * Row-wise and column-wise MX quantization from one read of x: the outputs
 * of fp8bq_mx_quantize_rowwise (q, e8) and fp8bq_mx_quantize_colwise
 * (qT, e8T), bit for bit.
 *   x    [M][C] BF16 or FP32, row pitch ldx elements (ldx >= C)
 *   q    [M][C] codes,   e8  [C/128][M][4] exponents (1x32 blocks along C)
 *   qT   [C][M] codes,   e8T [M/128][C][4] exponents (32x1 blocks along M)
 * Requires M % 128 == 0, C % 128 == 0, M / 128 <= 65535.  One pass serves
 * X (Fprop and Wgrad), W (Fprop and Dgrad) and dY (Dgrad and Wgrad).
 * Source: as fp8bq_mx_quantize_rowwise.
 */
fp8bq_status fp8bq_mx_quantize_rowcol(const void* x, fp8bq_dtype dtype, int64_t M, int64_t C, int64_t ldx, uint8_t* q,
                                      uint8_t* e8, uint8_t* qT, uint8_t* e8T, fp8bq_stream_t stream);

/*
 * MX GEMM: d[i][j] = BF16( sum_k 2^(ea(i,k)-127) D(a[i][k]) * 2^(eb(j,k)-127) D(b[j][k]) )
 * for two K-major operands as the MX quantizers emit them:
 *   a   [I][K] codes, ea [K/128][I][4] exponents
 *   b   [J][K] codes, eb [K/128][J][4] exponents
 *   d   [I][J] BF16 output, dense
 * Fprop: (a, b) = (rowwise X, rowwise W), I = M, J = N, K = K.
 * Dgrad: (rowwise dY, colwise W), I = M, J = K, reduction N.
 * Wgrad: (colwise dY, colwise X), I = N, J = K, reduction M.
 * The products accumulate in FP32 in tensor memory; the acceptance bound of
 * the FP32-scale GEMMs applies.  Requires I, J, K % 128 == 0 and each < 2^31.
 * Source: as fp8bq_mx_quantize_rowwise (the block-scaled MMA applies the
 *   scales).
 */
fp8bq_status fp8bq_mx_gemm(const uint8_t* a, const uint8_t* ea, const uint8_t* b, const uint8_t* eb, uint16_t* d,
                           int64_t I, int64_t J, int64_t K, fp8bq_stream_t stream);

/*
 * Synchronize `stream`, then read and clear the current device's status word.
 * Returns FP8BQ_OK, FP8BQ_ERR_TIMEOUT if a kernel launched since the last
 * check gave up on a pipeline wait (its outputs are then undefined), or
 * FP8BQ_ERR_CUDA if the synchronization itself failed.
 * Source: no passage of the pages (failure detection of the library itself).
 */
fp8bq_status fp8bq_check(fp8bq_stream_t stream);

/* Static, human-readable name of a status code. */
const char* fp8bq_status_string(fp8bq_status status);

/*
 * Self-test of the bounded-wait path: launches one CTA that waits on a
 * shared-memory barrier nothing will ever complete, gives up after
 * `limit_ns` nanoseconds (clamped to [1000, 2e9]) and records
 * FP8BQ_ERR_TIMEOUT in the status word, exactly as a stalled GEMM pipeline
 * would.  Lets a caller verify, without faulting or hanging the GPU, that
 * fp8bq_check reports device-side timeouts.  Returns the launch status.
 * Source: no passage of the pages (failure detection of the library itself).
 */
fp8bq_status fp8bq_selftest_wait_timeout(int64_t limit_ns, fp8bq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BQ_H */
