/*
 * tg_gemm.h - C ABI of the tiled bf16 -> fp32 GEMM for GB300 (sm_103a).
 *
 * The operation (all entry points below compute it):
 *
 *     for every b < batch:   C_b[i][j] = sum_{k < K} A_b[i][k] * B_b[k][j]
 *
 * with A_b = A + b*strideA, B_b = B + b*strideB, C_b = C + b*strideC and
 * row-major addressing A_b[i][k] = A_b[i*lda + k], B_b[k][j] = B_b[k*ldb + j],
 * C_b[i][j] = C_b[i*ldc + j] (all strides in ELEMENTS).  A and B are bf16,
 * C is fp32; products are accumulated in fp32 and C is OVERWRITTEN.
 *
 * Sources for the operation and its schedule:
 *   - LuisaCompute "Pipelines and stage boundaries", section "Stage boundaries
 *     are lexical": the k-tile pipeline "load" stage (A and B tiles read with
 *     zero bounds) feeding the "compute" stage acc = mma(a, b, acc).
 *   - LuisaCompute "Execution Nests and coordinates", section "Dimensions and
 *     spaces": A(m, reduction), B(reduction, n), C(m, n).
 *   - OCANNL "Module Ir.Schedule": Split (tile loops), Pad-to-tile (arbitrary
 *     extents through zero-filled fringes and masks), Stage (shared-memory
 *     tiles), pipeline_depth, Tensorize, Partition (guard-free interior tiles
 *     plus masked fringe tiles) and the deterministic two-pass split reduction
 *     (split-K with a fixed combine order).
 *
 * Conventions shared by every entry point:
 *   - Operand storage: by default A is row-major M x K (lda >= K) and B
 *     row-major K x N (ldb >= N); tg_options.a_col_major / b_col_major select
 *     the transposed storage (A as K x M with lda >= M, B as N x K with
 *     ldb >= K).  C (D) is always row-major M x N.
 *   - Pointers are DEVICE pointers unless the name says _host.  The caller
 *     owns A, B, C and the stream; the library never frees caller memory.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *     and return once the work is enqueued.  Device-side failures (a watchdog
 *     expiry) are reported later by tg_device_error().
 *   - Arguments are validated before anything is enqueued:
 *       TG_ERR_INVALID_ARG  for a NULL pointer with a nonzero extent, M, N or
 *                           K < 0, batch < 1, a leading dimension shorter
 *                           than its stored row (lda < K, or < M when A is
 *                           column-major; ldb < N, or < K; ldc < N), a
 *                           negative batch stride, batch strides that make
 *                           two problems share an element of C, C
 *                           overlapping A or B, or an extent > 2^31 - 1.
 *   - M == 0 or N == 0: returns TG_OK and enqueues nothing.
 *     K == 0: C is filled with zeros (the empty sum).
 *   - Any alignment is accepted.  Operands whose base address or row/batch
 *     stride is not a multiple of 16 bytes are first copied by the library
 *     into an aligned scratch copy (the "pack" pass) - except in a small
 *     problem's direct-load kernel, which reads them in place; an fp32 C
 *     whose rows are not 16-byte aligned is written with plain masked stores
 *     instead of tensor-memory-accelerator stores.
 *   - Rounding: fp32 accumulation in an order fixed by the plan (tile shape
 *     and split-K factor).  Results are bitwise reproducible run to run for
 *     a fixed plan; different plans may differ in the last bits.
 *   - Thread safety: calls on different streams may run concurrently; each
 *     stream has its own scratch workspace.
 *   - CUDA graphs: the first call on a stream may allocate that stream's
 *     workspace and set kernel attributes; a later call of the same or a
 *     smaller plan on the stream enqueues only kernel launches, so it can be
 *     captured into a CUDA graph and replayed (each replay reads the
 *     operands' current contents).  tg_gemm_host and tg_tune synchronise
 *     and cannot be captured.
 */
#ifndef TG_GEMM_H
#define TG_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *tg_stream_t;

typedef enum tg_status {
    TG_OK = 0,
    TG_ERR_INVALID_ARG = 1, /* rejected before any work was enqueued       */
    TG_ERR_UNSUPPORTED = 2, /* valid request this build cannot run          */
    TG_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed            */
    TG_ERR_OOM = 4,         /* workspace allocation failed                  */
    TG_ERR_TIMEOUT = 5,     /* a device-side wait exceeded its limit        */
    TG_ERR_DEVICE_CHECK = 6 /* a device-side consistency check failed (only */
                            /* in a library built with TG_DEBUG_CHECKS)     */
} tg_status;

/* Plan overrides for tests and tuning (zero-initialise, then set fields).
 * A zero field means "let the planner choose". */
typedef struct tg_options {
    int32_t block_n;     /* output tile width: 64, 128, 192 or 256            */
    int32_t stages;      /* shared-memory ring depth, 2 .. the tile's maximum */
                         /* (outputs of at most 64 rows: 8 at width 128 and  */
                         /* 6 at width 192 select rings of 64-row A slots,   */
                         /* the planner's own choice there)                  */
    int32_t split_k;     /* K splits per output tile (1 = none)               */
    int32_t force_pack;  /* nonzero: copy A and B through the pack pass       */
    int32_t epilogue;    /* 1 = tensor-memory-accelerator stores, 2 = plain   */
                         /* masked stores (1 needs a 16-byte aligned C)       */
    int32_t max_ctas;    /* cap on the persistent grid (0 = one CTA per SM)   */
    uint64_t timeout_ns; /* watchdog limit of every device-side wait          */
                         /* (0 = 2 s)                                         */
    int32_t debug_stall; /* nonzero: the epilogue first waits on a barrier    */
                         /* nothing completes, so the watchdog must fire and  */
                         /* tg_device_error() must return TG_ERR_TIMEOUT;     */
                         /* 2 in a library built with TG_DEBUG_CHECKS: a      */
                         /* planted failed check instead (TG_ERR_DEVICE_CHECK)*/
    int32_t cta_pair;    /* 1 = one CTA per output tile; 2 = two-SM tiles:    */
                         /* a cluster of two CTAs computes 256 x block_n with */
                         /* one tcgen05 cta_group::2 MMA (block_n 128 or 256) */
    int32_t stream_k;    /* 1 = off; 2 = on when the last wave of tiles is    */
                         /* partial: each worker takes its full waves of      */
                         /* tiles, then an equal share of the remaining       */
                         /* tiles' k-blocks; split tiles are combined in a    */
                         /* fixed k order (cannot be combined with split_k)   */
    int32_t operands;    /* tg_plan only: the operand family to plan for - 0  */
                         /* bf16 (tg_gemm_ex), 1 8-bit (tg_gemm_fp8 layout:   */
                         /* ldb is the pitch of B stored N x K), 2 block-     */
                         /* scaled 8-bit (tg_gemm_mxfp8), 3 block-scaled      */
                         /* packed 4-bit (tg_gemm_mxfp4: K and pitches in     */
                         /* elements); the compute calls ignore it            */
    uint64_t trace_buffer; /* device address of grid x 8 uint64 (0 = off): per */
                         /* CTA %globaltimer stamps in ns: [0] entry, [1] set- */
                         /* up done, [2] first k-block ready, [3] last MMA    */
                         /* issued, [4] first epilogue start, [5] last store  */
                         /* issued, [6] stores complete, [7] exit             */
    int32_t a_col_major; /* nonzero: A is stored K x M (element A_b[i][k] at   */
                         /* A[b*strideA + k*lda + i], lda >= M)               */
    int32_t b_col_major; /* nonzero: B is stored N x K (element B_b[k][j] at   */
                         /* B[b*strideB + j*ldb + k], ldb >= K)               */
    int32_t direct;      /* direct-load kernel for small problems: 0 = the    */
                         /* planner decides, 1 = off, 2 = on (bf16 calls;    */
                         /* other overrides only at the kernel's own values  */
                         /* - block_n 64, split_k 1, cta_pair 1, stream_k 1, */
                         /* epilogue 2 - else TG_ERR_INVALID_ARG).  One CTA  */
                         /* per 128 x 64 tile of C copies its operand tiles  */
                         /* into shared memory with plain loads (any pitch   */
                         /* and alignment, so no pack pass), up to 4         */
                         /* k-blocks at a time, and multiplies them with     */
                         /* tcgen05.mma (OCANNL "Module Ir.Schedule", Stage  */
                         /* with a cooperative copy, and Pad-to-tile)        */
} tg_options;

/* What the planner chose (tg_plan output). */
typedef struct tg_plan_info {
    int32_t block_m, block_n, block_k, stages;  /* block_m: rows of A a tile     */
                         /* loads - 128, 256 for two-SM tiles, 64 for rings  */
                         /* of 64-row A slots (outputs of at most 64 rows)   */
    int32_t tiles_m, tiles_n, k_blocks, split_k;
    int64_t num_units;   /* batch * tiles_m * tiles_n * split_k                */
    int32_t grid;        /* persistent CTAs launched                          */
    int32_t pack_a;      /* 1 when A goes through the pack pass                */
    int32_t pack_b;      /* 1 when B goes through the pack pass                */
    int32_t epilogue;    /* 1 = tensor-memory-accelerator stores, 2 = plain    */
    int32_t smem_bytes;  /* dynamic shared memory per CTA                     */
    int32_t tmem_cols;   /* tensor-memory columns allocated per CTA           */
    int64_t workspace_bytes; /* scratch this call needs (pack copies, split-K  */
                             /* partial tiles, tile counters)                  */
    int32_t cta_pair;    /* 1 = one CTA per tile, 2 = two-SM tiles (block_m  */
                         /* is then 256 and grid counts CTAs, 2 per cluster) */
    int32_t stream_k;    /* 1 = off, 2 = on                                  */
    int32_t sk_tiles;    /* tiles whose k-blocks are shared between workers  */
    int32_t direct;      /* 1 = persistent kernel, 2 = direct-load kernel    */
                         /* (block 128 x 64, stages = k-blocks staged at     */
                         /* once, grid = one CTA per tile)                   */
    int32_t reserved[2];
} tg_plan_info;

/* The GEMM (see the header comment for the operation and conventions). */
tg_status tg_gemm(const void *A, const void *B, float *C,
                  int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc,
                  int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                  tg_stream_t stream);

/* Same as tg_gemm with plan overrides (opt may be NULL).  Returns
 * TG_ERR_INVALID_ARG for an override outside its documented range. */
tg_status tg_gemm_ex(const void *A, const void *B, float *C,
                     int64_t M, int64_t N, int64_t K,
                     int64_t lda, int64_t ldb, int64_t ldc,
                     int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                     tg_stream_t stream, const tg_options *opt);

/* Fused epilogue (OCANNL "Module Ir.Schedule", Epilogue fusion: the
 * elementwise tail of a reduction - bias add, activation, residual - folded
 * into the accumulator's store-back instead of a separate memory pass).
 *
 *     D_b[i][j] = act(alpha * (A_b B_b)[i][j] + bias_b[j]) + beta * R_b[i][j]
 *
 * applied once to the final fp32 value of every element (after any split-K
 * or stream-K combine), each product and sum rounded separately in fp32 (no
 * fused multiply-add).  With activation NONE or RELU the result therefore
 * equals, bit for bit, the same formula applied in fp32 to tg_gemm's output;
 * a bf16 D is that fp32 value rounded to nearest even. */
typedef enum tg_activation {
    TG_ACT_NONE = 0,
    TG_ACT_RELU = 1,      /* max(x, 0)                                        */
    TG_ACT_GELU_TANH = 2, /* x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))    */
    TG_ACT_SILU = 3       /* x / (1 + exp(-x))                                */
} tg_activation;

typedef enum tg_dtype { TG_F32 = 0, TG_BF16 = 1 } tg_dtype;

typedef struct tg_epilogue {
    float alpha;           /* scales A B                                       */
    float beta;            /* scales the residual (ignored without residual)   */
    const float *bias;     /* device, fp32: bias_b[j] = bias[b*bias_stride + j] */
                           /* (j < N), or NULL for none                        */
    int64_t bias_stride;   /* elements between problems' bias vectors (0: one  */
                           /* vector for all problems)                         */
    const void *residual;  /* device, same type as D: R_b[i][j] =              */
                           /* residual[b*strideR + i*ldr + j], or NULL. It may */
                           /* be D itself (same pointer and strides); any      */
                           /* other overlap with D is rejected                 */
    int64_t ldr, strideR;
    int32_t activation;    /* tg_activation                                    */
    int32_t out_type;      /* tg_dtype of D (and of the residual)              */
    int32_t reserved[6];
} tg_epilogue;

/* The GEMM with a fused epilogue writing D (fp32 or bf16, ep->out_type),
 * row-major with ldd / strideD in elements of D's type.  ep must not be
 * NULL.  Same conventions, checks and options as tg_gemm_ex; K == 0 gives
 * D = act(bias) + beta * R.  TG_ERR_INVALID_ARG also for an unknown
 * activation or out_type, or a residual with ldr < N. */
tg_status tg_gemm_fused(const void *A, const void *B, void *D,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldd,
                        int64_t batch, int64_t strideA, int64_t strideB, int64_t strideD,
                        const tg_epilogue *ep, tg_stream_t stream, const tg_options *opt);

/* 8-bit floating-point operand formats (OCP FP8: E4M3 with no infinities,
 * E5M2 with IEEE-style infinities and NaNs). */
typedef enum { TG_FP8_E4M3 = 0, TG_FP8_E5M2 = 1 } tg_fp8_format;

/* The GEMM with 8-bit floating-point A and B (a_format, b_format), fp32
 * accumulation and the fused epilogue of tg_gemm_fused (ep may be NULL:
 * D = A B in fp32).  Per-tensor scales of the operands go into ep->alpha.
 * Layout: A row-major M x K (element (i,k) at A[i*lda + k], lda >= K); B
 * column-major K x N, i.e. stored N x K (element (k,j) at B[j*ldb + k],
 * ldb >= K) - both operands contiguous along K, the layout the tensor cores
 * read for 8-bit types.  Strides count elements (bytes).  Requirements:
 * A and B 16-byte aligned, lda, ldb and the batch strides multiples of 16
 * (else TG_ERR_UNSUPPORTED); a_col_major, b_col_major and force_pack in opt
 * must be 0 (TG_ERR_INVALID_ARG).  Otherwise as tg_gemm_fused.  (The pages
 * define the contraction over any element type; 8-bit operands are the
 * block-scaled family's element types without the per-block scales.) */
tg_status tg_gemm_fp8(const void *A, const void *B, void *D,
                      int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldd,
                      int64_t batch, int64_t strideA, int64_t strideB, int64_t strideD,
                      int32_t a_format, int32_t b_format,
                      const tg_epilogue *ep, tg_stream_t stream, const tg_options *opt);

/* Block-scaled 8-bit GEMM (MXFP8: TVM "Tensor Layout", Case study: Blackwell
 * tensor memory, the per-block scale factors SFA / SFB of a block-scaled
 * MMA):
 *     D[b][i][j] = sum_k  2^(SFA[b][i][k/32] - 127) * A[b][i][k]
 *                       * 2^(SFB[b][j][k/32] - 127) * B[b][k][j]
 * then the fused epilogue of tg_gemm_fused (ep may be NULL: D in fp32).
 * Every run of 32 consecutive elements along K of a row of A (of a column of
 * B) shares one E8M0 scale: an unsigned byte e meaning 2^(e - 127) (e = 255
 * is NaN; the last run of a row may be shorter when K is not a multiple of
 * 32).  A, B, their formats, layouts and requirements as tg_gemm_fp8.
 * SFA (device bytes): the scale of row i, run r of problem b at
 * SFA[b*stride_sfa + i*ld_sfa + r], ld_sfa >= ceil(K/32); SFB likewise per
 * column j of B (SFB[b*stride_sfb + j*ld_sfb + r], ld_sfb >= ceil(K/32)).
 * A scale stride of 0 shares one scale matrix across the batch; where A (B)
 * is shared (strideA == 0 with batch > 1) its scales must be too.  Scales
 * are read, never written, and may alias anything but D.  The library
 * re-arranges them into device scratch it owns (512-byte blocks per 128
 * rows or columns of a tile and 128 elements of K) on `stream` before the
 * GEMM.
 * Tiles are 128 rows x 128, 192 or 224 columns (the planner's choice), one
 * CTA each: tensor memory holds two accumulators of up to 224 columns and
 * the scales of every ring slot.  opt->block_n must be 0, 128, 192 or 224,
 * opt->cta_pair 0 or 1, opt->stages 0, 2 or 4 (else TG_ERR_INVALID_ARG).
 * TG_ERR_INVALID_ARG also for a NULL scale pointer with K > 0, ld_sfa or
 * ld_sfb < ceil(K/32), or a negative scale stride. */
tg_status tg_gemm_mxfp8(const void *A, const void *B, void *D,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldd,
                        int64_t batch, int64_t strideA, int64_t strideB, int64_t strideD,
                        int32_t a_format, int32_t b_format,
                        const uint8_t *SFA, int64_t ld_sfa, int64_t stride_sfa,
                        const uint8_t *SFB, int64_t ld_sfb, int64_t stride_sfb,
                        const tg_epilogue *ep, tg_stream_t stream, const tg_options *opt);

/* Block-scaled 4-bit GEMM (MXFP4: the block-scaled family of TVM "Tensor
 * Layout", Case study: Blackwell tensor memory, on 4-bit elements):
 *     D[b][i][j] = sum_k  2^(SFA[b][i][k/32] - 127) * A[b][i][k]
 *                       * 2^(SFB[b][j][k/32] - 127) * B[b][k][j]
 * then the fused epilogue of tg_gemm_fused (ep may be NULL: D in fp32).
 * Elements are E2M1 codes (OCP MX: sign bit 3, exponent bits 2-1 with bias
 * 1, mantissa bit 0; values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives),
 * two to a byte: element k of a stored row is in byte k/2, in the low nibble
 * when k is even and in the high nibble when k is odd.  A row-major M x K
 * (element (i,k) in byte A[(i*lda + k)/2]); B column-major, i.e. stored
 * N x K (element (k,j) in byte B[(j*ldb + k)/2]).  K, lda, ldb, strideA and
 * strideB count ELEMENTS and must be even (else TG_ERR_INVALID_ARG);
 * A and B 16-byte aligned, lda, ldb and the batch strides multiples of 32
 * elements (16 bytes), else TG_ERR_UNSUPPORTED.  Scales SFA, SFB: E8M0
 * bytes, one per 32 elements of K, laid out and checked as in
 * tg_gemm_mxfp8.  D (ldd, strideD in elements of D's type) and ep as
 * tg_gemm_fused.  The library re-arranges the scales into device scratch it
 * owns (two 512-byte blocks per 128 rows or columns of a tile and 256
 * elements of K) on `stream` before the GEMM (tcgen05 kind::mxf4, 64
 * elements of K per instruction).  Tiles: 128 rows x 128, 192 or 224
 * columns, one CTA each; opt->block_n 0, 128, 192 or 224, opt->cta_pair 0
 * or 1, opt->stages 0, 2 or 4 (224-wide tiles: 0 or 2), else
 * TG_ERR_INVALID_ARG. */
tg_status tg_gemm_mxfp4(const void *A, const void *B, void *D,
                        int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldd,
                        int64_t batch, int64_t strideA, int64_t strideB, int64_t strideD,
                        const uint8_t *SFA, int64_t ld_sfa, int64_t stride_sfa,
                        const uint8_t *SFB, int64_t ld_sfb, int64_t stride_sfb,
                        const tg_epilogue *ep, tg_stream_t stream, const tg_options *opt);

/* The GEMM on HOST buffers: copies the spans of A and B that the strides
 * reach to device scratch owned by the library, runs tg_gemm_ex there into
 * a device C with 16-byte rows, and copies the M x N block of every problem
 * back.  The copies and the GEMM are pipelined over pieces that are
 * contiguous in host memory (problems of a stacked batch, rows of a
 * row-major A, columns of a column-major B; at most 8): copies in, GEMMs and
 * copies out run on three streams and overlap.  An operand copied whole
 * whose rows are not 16-byte aligned is realigned once on the device.
 * Synchronous: returns after C is on the host (pinned host memory makes the
 * copies faster; pageable also works).  Elements of C between rows
 * (ldc > N) or between problems are preserved.  Results equal tg_gemm_ex's
 * on the same data except where the pieces change the plan's split-K or
 * stream-K partition (then within the usual rounding of a split sum). */
tg_status tg_gemm_host(const void *A_host, const void *B_host, float *C_host,
                       int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc,
                       int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                       tg_stream_t stream, const tg_options *opt);

/* Run-time plan search (a tuner): times candidate plans for these arguments
 * on the caller's buffers and stream - every instantiated tile width, one
 * CTA or two-SM tiles, the two deepest ring depths (for outputs of at most
 * 64 rows also the rings of 64-row A slots), stream-K on and off,
 * and split-K factors where there are fewer tiles than SMs - each `reps`
 * times (1..100) with CUDA events, and returns the fastest (median) as
 * options in *best (the layout fields and other fields of `base` kept; base
 * may be NULL) and its time in microseconds in *best_us (may be NULL).
 * C is written with the product.  Synchronous.  (The pages call for a
 * search dimension over tile and depth choices; OCANNL "Module
 * Ir.Schedule", pipeline_depth.) */
tg_status tg_tune(const void *A, const void *B, float *C,
                  int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc,
                  int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                  tg_stream_t stream, const tg_options *base, int32_t reps,
                  tg_options *best, float *best_us);

/* The plan tg_gemm_ex would use for these arguments, without touching the
 * pointers' memory (opt->operands = 1 or 2: the plan of tg_gemm_fp8 or
 * tg_gemm_mxfp8 instead, with B stored N x K; TG_ERR_UNSUPPORTED where those
 * calls would refuse the alignment).  sm_count > 0 plans for that many SMs
 * and makes no CUDA call at all (host-only); sm_count == 0 queries the
 * current device. */
tg_status tg_plan(const void *A, const void *B, const float *C,
                  int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc,
                  int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                  int32_t sm_count, const tg_options *opt, tg_plan_info *out);

/* The split-K GEMM for callers that cannot allocate device memory.  (No page
 * of the method has a counterpart: this is a deployment variant of the
 * split-K path above.)
 *
 * Who needs it: code that runs as a plugin inside a host framework whose
 * memory pool owns the device (a cudaMalloc there bypasses the pool's
 * accounting or fails under its memory cap), and services that must not
 * allocate after start-up because cudaMalloc/cudaFree may synchronise the
 * device and have unbounded latency.  tg_gemm_ex allocates its split-K
 * scratch (partial tiles, tile counters, error word) on first use; this
 * entry point instead uses one static device array compiled into the
 * library and calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Same operation, arguments and argument checks as tg_gemm_ex, with the K
 * dimension split into `split_k` parts (1 <= split_k <= ceil(K/64)).
 * Limits of the static scratch (TG_ERR_UNSUPPORTED beyond them):
 *   - split-K partial tiles: at most 16 MiB, i.e.
 *     output tiles x split_k x 128 x block_n x 4 bytes <= 16 MiB;
 *   - at most 4096 output tiles (batch x ceil(M/128) x ceil(N/block_n));
 *   - A and B must be addressable by TMA: 16-byte aligned base, and row
 *     and batch strides that are multiples of 8 elements (this path has no
 *     pack copy).
 * The array (16 MiB + 16 KiB + 256 B) lives on every GPU that loads the
 * library until the process exits.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) once; make that first call
 * before any stream capture.  Every call shares the one array, which keeps
 * the previous call's contents; each call clears the tile counters it uses
 * before its kernel.  Calls whose kernels overlap on the GPU (different
 * streams, or graph branches) race on the array: serialise them.
 * A watchdog expiry in this entry point's kernel is recorded in the array's
 * own error word (one per device, shared by all calls of this entry point),
 * which keeps the first expiry until tg_device_error() - on any stream of
 * that device - reads and clears it; synchronise the stream the call ran on
 * (or pass it to tg_device_error) first.  Self-test: with the environment
 * variable TG_DEBUG_STALL_NS set to a positive number of nanoseconds, the
 * kernel first waits on a barrier that nothing completes, with that limit,
 * so the call leaves C unwritten and tg_device_error() returns
 * TG_ERR_TIMEOUT. */
tg_status tg_gemm_splitk_static(const void *A, const void *B, float *C,
                                int64_t M, int64_t N, int64_t K,
                                int64_t lda, int64_t ldb, int64_t ldc,
                                int64_t batch, int64_t strideA, int64_t strideB,
                                int64_t strideC, int32_t split_k, tg_stream_t stream);

/* Synchronises `stream`, then reads and clears the device error words that
 * the kernels' watchdog writes: the one of `stream`'s workspace, and the one
 * of tg_gemm_splitk_static on the current device.  TG_ERR_TIMEOUT if a wait
 * expired since the last call (the split-K tile counters of the stream's
 * workspace are then reset too), TG_ERR_DEVICE_CHECK if a consistency check
 * of a TG_DEBUG_CHECKS build failed, TG_ERR_CUDA if the stream reports a
 * CUDA error, else TG_OK.  Allocates nothing. */
tg_status tg_device_error(tg_stream_t stream);

/* Static English name of a status code. */
const char *tg_status_string(tg_status s);

/* Frees every cached workspace on every device.  Call only when no work
 * enqueued by this library is still running. */
void tg_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* TG_GEMM_H */
