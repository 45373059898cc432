// Internal interface between the host library (tg_host.cu) and the kernel
// translation units (tg_kernel_bn*.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only; the driver is reached through cudart)
#include <cuda_runtime.h>

namespace tg {

// Fixed tile geometry.  BM = 128 rows = the 128 tensor-memory lanes of one
// SM; BK = 64 bf16 = 128 bytes = one 128B swizzle atom row.
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int EPI_CHUNK = 32;      // columns per tensor-memory load / store box
constexpr int NUM_THREADS = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int EPI_BUFS = 2;        // staging buffers per epilogue warp
constexpr int SMEM_LIMIT = 232448; // max dynamic shared memory per CTA (227 KB)

// Watchdog codes written to the device error word (first writer wins).
enum : uint32_t {
    ERR_NONE = 0,
    ERR_TIMEOUT_PRODUCER = 1,
    ERR_TIMEOUT_MMA = 2,
    ERR_TIMEOUT_EPILOGUE = 3,
    ERR_TIMEOUT_DRAIN = 4,
    // Builds with TG_DEBUG_CHECKS: a device-side consistency check failed
    // (the word after the code says which; see tg_kernel.cuh).
    ERR_DEBUG_CHECK = 5,
};

struct KernelParams {
    int32_t M, N, K, batch;
    int32_t tiles_m, tiles_n;
    int32_t splits;       // K splits per output tile (>= 1)
    int32_t k_blocks;     // ceil(K / BK)
    int64_t num_units;    // batch * tiles_m * tiles_n * splits
    int32_t group_m;      // tile-row group of the rasterisation
    int32_t a_mn;         // 1: A's M dimension is contiguous (column-major A)
    int32_t b_k;          // 1: B's K dimension is contiguous (column-major B)
    int32_t a_bcast;      // 1: A has batch stride 0 (same A for every problem)
    int32_t b_bcast;      // 1: B has batch stride 0
    int32_t epi_tma;      // 1: TMA store of C; 0: plain masked stores
    void *C;              // plain-store epilogue target (fp32, or bf16 when out_bf16)
    int64_t ldc, strideC;
    // Fused epilogue (fused == 1): D = act(alpha * acc + bias[j]) + beta * R,
    // applied once to the final fp32 value; D and R are bf16 when out_bf16.
    int32_t fused, act, out_bf16;
    float alpha, beta;
    const float *bias;
    int64_t bias_stride;
    const void *residual;
    int64_t ldr, strideR;
    float *partials;      // split-K partial tiles
    int32_t *counters;    // split-K arrival counters, one per output tile
    uint32_t *err;        // device error word
    uint64_t timeout_ns;
    int32_t debug_stall;  // 1: watchdog self-test; 2 (TG_DEBUG_CHECKS builds): planted failed check
    // extents of the split-K scratch, for the consistency checks of
    // TG_DEBUG_CHECKS builds: floats of partial tiles, int32 tile counters
    int64_t partial_floats;
    int64_t counter_count;
    // Stream-K schedule (stream_k == 1): every worker takes dp_waves whole
    // tiles (tile = worker + i * workers), then the k-block range
    // [w * sk_iters / workers, (w + 1) * sk_iters / workers) of the sk_tiles
    // tiles that follow; a tile covered by several ranges is combined from
    // per-range partials.  maxparts = partial slots per tile (split-K: splits).
    int32_t stream_k;
    int32_t dp_waves;
    int32_t sk_first_tile;
    int32_t maxparts;
    int64_t sk_iters;
    // Workers that take a stream-K range: P * sk_tiles when each shared tile
    // is cut into P >= 2 equal parts (each range inside one tile), else all.
    int32_t sk_workers;
    unsigned long long *trace;  // grid x 8 timestamps, or null
    uint32_t mma_fmt;           // 8-/4-bit operands: A format << 7 | B format << 10
    // Block-scaled operands: E8M0 scales pre-arranged in 512-byte blocks,
    // for problem z, 128-row (A) or BN-column (B) tile t and k-block kb the
    // blocks ((z * tiles + t) * k_blocks + kb) * halves * subs + h * subs + sub
    // (h: which four runs of the k-block; sub: which 128 rows or columns).
    const uint8_t *sfa;
    const uint8_t *sfb;
};

// Shared-memory budget of one tile width.  PAIR: the tile is computed by a
// cluster of two CTAs on two SMs (tcgen05 cta_group::2): each CTA holds its
// own 128 rows of A and half of the BN columns of B.  HALF_A (one CTA per
// tile, outputs of at most 64 rows): a ring slot holds 64 rows of A, so more
// slots fit; the MMA still reads 128 rows, the upper 64 from the memory
// after the slot, and the accumulator rows they produce are never stored.
template <int BN, bool PAIR = false, bool HALF_A = false>
struct Geometry {
    static constexpr int B_COLS = PAIR ? BN / 2 : BN;     // B columns this CTA loads
    static constexpr int A_ROWS = HALF_A ? BM / 2 : BM;   // A rows a slot holds
    static constexpr int A_STAGE = A_ROWS * BK * 2;       // 16 KB (8 KB)
    static constexpr int B_STAGE = BK * B_COLS * 2;       // B_COLS * 128 B
    static constexpr int STAGE = A_STAGE + B_STAGE;
    static constexpr int EPI_BYTES = 4 * EPI_BUFS * EPI_CHUNK * EPI_CHUNK * 4;  // 32 KB
    static constexpr int BAR_BYTES = 512;
    // Block-scaled operands: the scale blocks of one slot - A's 512 bytes,
    // then B's 512 bytes per 128 columns of the tile.
    static constexpr int SF_B_BLOCKS = (BN + 127) / 128;
    static constexpr int SF_STAGE = 512 * (1 + SF_B_BLOCKS);
    static constexpr int ALIGN_SLACK = 1024;
    static constexpr int MAX_STAGES_RAW = (SMEM_LIMIT - EPI_BYTES - BAR_BYTES - ALIGN_SLACK) / STAGE;
    static constexpr int MAX_STAGES = MAX_STAGES_RAW > 8 ? 8 : MAX_STAGES_RAW;
    static constexpr int TMEM_COLS = (2 * BN <= 128) ? 128 : (2 * BN <= 256) ? 256 : 512;
    // At least 120 KB, so that two CTAs never share an SM: the persistent
    // kernel assumes it owns the SM's tensor memory (up to all 512 columns).
    static constexpr int ONE_CTA_PER_SM = 120 * 1024;
    static constexpr int smem_bytes(int stages) {
        return stages * STAGE + EPI_BYTES + BAR_BYTES + ALIGN_SLACK > ONE_CTA_PER_SM
                   ? stages * STAGE + EPI_BYTES + BAR_BYTES + ALIGN_SLACK
                   : ONE_CTA_PER_SM;
    }
    // halves: scale blocks per 128 rows and k-block (1: 8-bit elements, four
    // runs of 32 a k-block; 2: packed 4-bit elements, eight runs)
    static constexpr int smem_bytes_mx(int stages, int halves = 1)
    {
        return smem_bytes(stages) + stages * SF_STAGE * halves;
    }
};

// Block-scaled element families (the `mx` argument of the launches).
enum : int { MX_NONE = 0, MX_FP8 = 1, MX_FP4 = 2 };

// Launch of the persistent GEMM kernel for one tile width (defined in the
// per-width translation units).  pair: two-SM tiles (grid counts CTAs, a
// multiple of 2); f8: 8-bit floating-point operands (or, with mx == MX_FP4,
// packed 4-bit ones, which the kernel moves as bytes); mx: block-scaled
// operands (one CTA per tile).  Returns the launch's cudaError_t.
#define TG_DECLARE_LAUNCH(BN_)                                                                   \
    cudaError_t launch_gemm_bn##BN_(const CUtensorMap &ta, const CUtensorMap &tb,                \
                                    const CUtensorMap &tc, const KernelParams &p, int stages,   \
                                    bool pair, bool f8, int mx, int grid, cudaStream_t s);      \
    int max_pairs_bn##BN_(int stages, bool f8);
TG_DECLARE_LAUNCH(64)
TG_DECLARE_LAUNCH(128)
// Half-height A slots (outputs of at most 64 rows): width 128 with 8 slots
// and width 192 with 6; f8 as above.
cudaError_t launch_gemm_bn128_half_a(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                                     const KernelParams &p, bool f8, int grid, cudaStream_t s);
cudaError_t launch_gemm_bn192_half_a(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                                     const KernelParams &p, bool f8, int grid, cudaStream_t s);
TG_DECLARE_LAUNCH(192)
TG_DECLARE_LAUNCH(256)
#undef TG_DECLARE_LAUNCH
// Block-scaled operands (mx: MX_FP8 or MX_FP4) on 224-wide one-CTA tiles.
cudaError_t launch_gemm_mx224(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                              const KernelParams &p, int stages, int mx, int grid, cudaStream_t s);

}  // namespace tg
