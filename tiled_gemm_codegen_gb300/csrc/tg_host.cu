// Host side of the C ABI declared in include/tg_gemm.h: argument checks,
// planning, per-stream workspaces, TMA descriptors, and the two small
// kernels of the path besides the GEMM itself (the pack pass that realigns
// operands TMA cannot address, and the zero fill of the K == 0 case).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "tg_epilogue.cuh"
#include "tg_gemm.h"
#include "tg_internal.h"
#include "tg_direct.h"
#include "tg_plan.h"
#include "tg_ptx.cuh"

#define TG_API extern "C" __attribute__((visibility("default")))

namespace tg {
namespace {

constexpr uint64_t DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s

// TG_TRACE=1 prints each call's plan to stderr (read once).
bool trace_enabled()
{
    static const bool on = std::getenv("TG_TRACE") != nullptr;
    return on;
}
constexpr int64_t EXTENT_LIMIT = INT32_MAX;

// ------------------------------------------------------------ small kernels
// Pack (the realign pass): copy a batch of rows x cols bf16 matrices with
// arbitrary element strides into a dense buffer whose rows are padded to a
// multiple of 64 elements (pack_pitch: 128 bytes, so rows start on cache
// lines; TMA itself needs only 16-byte rows).  The
// pad columns are written as 0; the GEMM never reads them (its tensor map
// extent is the true column count).  One launch packs A and B (two jobs).
//
// Each thread writes one 16-byte chunk (8 elements).  Its source is read
// with the widest aligned loads the source address allows: one 16-byte,
// two 8-byte or four 4-byte loads, or, for a 2-byte-aligned source, five
// aligned 4-byte words realigned with funnel shifts.  A wider load is used
// only when every byte it touches lies inside the operand's span
// [span_begin, span_end); otherwise, and in a row's ragged tail, elements
// are read one by one.
struct PackJob {
    const uint16_t *src;
    uint16_t *dst;
    int64_t rows, cols, ld_src, s_src, ld_dst, chunks;
    uintptr_t span_begin, span_end;  // bytes of the source this job may read
};

__device__ __forceinline__ uint32_t pack_pair(uint16_t lo, uint16_t hi)
{
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ uint4 load8_bf16(const uint16_t *s, const PackJob &j)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(s);
    if ((a & 15u) == 0) return *reinterpret_cast<const uint4 *>(s);
    if ((a & 7u) == 0) {
        const uint2 lo = *reinterpret_cast<const uint2 *>(s);
        const uint2 hi = *reinterpret_cast<const uint2 *>(s + 4);
        return make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    if ((a & 3u) == 0) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(s);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (a - 2 >= j.span_begin && a + 18 <= j.span_end) {
        // words at a-2, a+2, .., a+14: element e of s sits in the high half
        // of word (e+1)/2 (e odd: low half of word (e+1)/2)
        const uint32_t *w = reinterpret_cast<const uint32_t *>(a - 2);
        const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
        return make_uint4(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16),
                          __funnelshift_r(w2, w3, 16), __funnelshift_r(w3, w4, 16));
    }
    return make_uint4(pack_pair(s[0], s[1]), pack_pair(s[2], s[3]), pack_pair(s[4], s[5]),
                      pack_pair(s[6], s[7]));
}

__global__ void pack_bf16_kernel(PackJob ja, PackJob jb, int blocks_a)
{
    // the GEMM that follows may be scheduled now: it waits for this grid to
    // complete before it reads the packed operands
    ptx::griddep_launch_dependents();
    const bool is_a = static_cast<int>(blockIdx.x) < blocks_a;
    const PackJob j = is_a ? ja : jb;
    const int64_t bid = is_a ? blockIdx.x : blockIdx.x - blocks_a;
    const int64_t nblocks = is_a ? blocks_a : gridDim.x - blocks_a;
    const int64_t chunks_per_row = j.ld_dst / 8;
    for (int64_t c = bid * blockDim.x + threadIdx.x; c < j.chunks; c += nblocks * blockDim.x) {
        const int64_t row_g = c / chunks_per_row;
        const int64_t col0 = (c - row_g * chunks_per_row) * 8;
        const int64_t b = row_g / j.rows;
        const int64_t r = row_g - b * j.rows;
        const uint16_t *s = j.src + b * j.s_src + r * j.ld_src + col0;
        uint4 out;
        if (col0 + 8 <= j.cols) {
            out = load8_bf16(s, j);
        } else {
            uint16_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = (col0 + e < j.cols) ? s[e] : static_cast<uint16_t>(0);
            out = make_uint4(pack_pair(v[0], v[1]), pack_pair(v[2], v[3]), pack_pair(v[4], v[5]),
                             pack_pair(v[6], v[7]));
        }
        *reinterpret_cast<uint4 *>(j.dst + row_g * j.ld_dst + col0) = out;
    }
}

// Block-scaled operands: re-arrange one operand's E8M0 scales (rows x
// ceil(K/32) bytes a problem, any pitch) into the blocks the GEMM kernel
// copies with each k-block: 512 bytes per 128 rows and four runs of 32
// elements of K, the byte of row 32g + l and run j of the four at
// l * 16 + g * 4 + j (tensor-memory lane l of cell column g after the warpx4
// copy; TVM "Tensor Layout", Case study: Blackwell tensor memory, the
// scale-factor atom of 32 rows on lanes, 4 scales per 32-bit column cell,
// replicated over the four lane quadrants).  A k-block of 8-bit elements has
// four runs (halves = 1), one of packed 4-bit elements eight (halves = 2:
// runs 0-3, then 4-7).  Rows and runs past the operand read as 127 (2^0):
// their operand elements are the TMA unit's zero fill.  A tile of
// `tile_rows` rows (128, or B's tile width) has `subs` = ceil(tile_rows /
// 128) blocks per half; tile rows past tile_rows read as 127 too.  Order:
// for problem z, tile t and k-block kb, the blocks
// ((z * tiles + t) * k_blocks + kb) * halves * subs + h * subs + sub.
struct ScaleJob {
    const uint8_t *src;
    uint8_t *dst;
    int64_t rows, runs, ld, stride;  // stride: between problems (0: shared)
    int64_t problems, tiles, k_blocks, tile_rows, subs, halves;
};

// One CTA re-arranges the scales of one 128-row block (sub) of one tile for
// SC_RUNS consecutive runs (16 8-bit or 8 4-bit k-blocks): the 128 rows x
// SC_RUNS runs are read with coalesced byte loads into shared memory (rows
// SC_PITCH bytes apart, so the 32 rows a warp reads next fall in 32
// different banks), then each warp writes whole 512-byte blocks, lane l's 16
// bytes holding rows l, 32 + l, 64 + l and 96 + l.
constexpr int SC_RUNS = 64;
constexpr int SC_PITCH = SC_RUNS + 4;
constexpr int SC_THREADS = 256;

__host__ __device__ inline int64_t scale_kb_per_cta(const ScaleJob &j) { return SC_RUNS / (4 * j.halves); }

inline int64_t scale_blocks(const ScaleJob &j)
{
    const int64_t kpc = scale_kb_per_cta(j);
    return j.problems * j.tiles * j.subs * ((j.k_blocks + kpc - 1) / kpc);
}

__global__ void __launch_bounds__(SC_THREADS) scale_tile_kernel(ScaleJob ja, ScaleJob jb, int64_t blocks_a)
{
    ptx::griddep_launch_dependents();
    __shared__ __align__(16) uint8_t slab[128 * SC_PITCH];
    const bool is_a = static_cast<int64_t>(blockIdx.x) < blocks_a;
    const ScaleJob j = is_a ? ja : jb;
    int64_t bid = is_a ? blockIdx.x : blockIdx.x - blocks_a;
    const int64_t kpc = scale_kb_per_cta(j);
    const int64_t kchunks = (j.k_blocks + kpc - 1) / kpc;
    const int64_t kc = bid % kchunks;
    bid /= kchunks;
    const int64_t sub = bid % j.subs;
    bid /= j.subs;
    const int64_t t = bid % j.tiles;
    const int64_t z = bid / j.tiles;
    const uint8_t *src = j.src + z * j.stride;
    const int64_t run0 = kc * SC_RUNS;
    // all of a thread's loads in flight at once (the sources are cold)
    constexpr int PER_THREAD = 128 * SC_RUNS / SC_THREADS;
    uint8_t v[PER_THREAD];
#pragma unroll
    for (int u = 0; u < PER_THREAD; ++u) {
        const int i = static_cast<int>(threadIdx.x) + u * SC_THREADS;
        const int r = i / SC_RUNS, c = i % SC_RUNS;
        const int64_t in_tile = sub * 128 + r;
        const int64_t row = t * j.tile_rows + in_tile;
        const int64_t run = run0 + c;
        const bool ok = in_tile < j.tile_rows && row < j.rows && run < j.runs;
        v[u] = ok ? src[row * j.ld + run] : static_cast<uint8_t>(127);
    }
#pragma unroll
    for (int u = 0; u < PER_THREAD; ++u) {
        const int i = static_cast<int>(threadIdx.x) + u * SC_THREADS;
        slab[(i / SC_RUNS) * SC_PITCH + i % SC_RUNS] = v[u];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // item = (k-block, half) of this CTA's runs, four runs each
    for (int item = warp; item < SC_RUNS / 4; item += SC_THREADS / 32) {
        const int64_t kbg = kc * kpc + item / j.halves;
        const int64_t h = item % j.halves;
        if (kbg >= j.k_blocks) break;
        uint32_t w[4];
#pragma unroll
        for (int g = 0; g < 4; ++g)
            w[g] = *reinterpret_cast<const uint32_t *>(slab + (32 * g + lane) * SC_PITCH + 4 * item);
        const int64_t blk = ((z * j.tiles + t) * j.k_blocks + kbg) * j.halves * j.subs + h * j.subs + sub;
        *reinterpret_cast<uint4 *>(j.dst + blk * 512 + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// K == 0: every entry of C is the empty sum.
__global__ void zero_c_kernel(float *C, int64_t M, int64_t N, int64_t ldc, int64_t sC,
                              int64_t total)
{
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = e / (M * N);
        const int64_t r = e - b * M * N;
        const int64_t i = r / N;
        const int64_t j = r - i * N;
        C[b * sC + i * ldc + j] = 0.0f;
    }
}

// ------------------------------------------------------------ argument checks
struct Args {
    const void *A;
    const void *B;
    void *C;  // C (fp32), or D of the fused epilogue (fp32 or bf16)
    int64_t M, N, K, lda, ldb, ldc, batch, sA, sB, sC;
    int64_t c_bytes = 4;  // element size of C
    int64_t ab_bytes = 2; // element size of A and B (1: 8-bit floating point)
    uint32_t mma_fmt = 0; // 8-bit operands: instruction-descriptor format fields
    bool a_cm = false;    // A stored K x M (column-major)
    bool b_cm = false;    // B stored N x K (column-major)
    // block-scaled operands: E8M0 scales per 32 elements of K
    bool mx = false;
    // packed 4-bit elements (two a byte): K, lda, ldb and the operand batch
    // strides above are then in BYTES (element counts / 2)
    bool fp4 = false;
    int64_t k_elems() const { return fp4 ? 2 * K : K; }
    const uint8_t *sfa = nullptr, *sfb = nullptr;
    int64_t ld_sfa = 0, s_sfa = 0, ld_sfb = 0, s_sfb = 0;
    // stored (rows, columns) of A and B
    int64_t a_rows() const { return a_cm ? K : M; }
    int64_t a_cols() const { return a_cm ? M : K; }
    int64_t b_rows() const { return b_cm ? N : K; }
    int64_t b_cols() const { return b_cm ? K : N; }
};

// Args with the operand layouts of `opt` (the layout fields are part of the
// operation, not tuning).
Args with_layout(Args a, const tg_options *opt)
{
    if (opt) {
        a.a_cm = opt->a_col_major != 0;
        a.b_cm = opt->b_col_major != 0;
    }
    return a;
}

// Elements spanned by one operand over all problems (0 if empty).  Callers
// have bounded every factor (extents < 2^31, strides <= 2^40) and checked
// the total against SPAN_LIMIT in 128-bit arithmetic first.
int64_t span_elems(int64_t rows, int64_t cols, int64_t ld, int64_t batch, int64_t stride)
{
    if (rows == 0 || cols == 0) return 0;
    return (batch - 1) * stride + (rows - 1) * ld + cols;
}

constexpr __int128 SPAN_LIMIT = static_cast<__int128>(1) << 56;  // elements

bool span_ok(int64_t rows, int64_t cols, int64_t ld, int64_t batch, int64_t stride)
{
    if (rows == 0 || cols == 0) return true;
    const __int128 s = static_cast<__int128>(batch - 1) * stride +
                       static_cast<__int128>(rows - 1) * ld + cols;
    return s < SPAN_LIMIT;
}

bool ranges_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1)
{
    return a0 < b1 && b0 < a1;
}

// Checks everything the header promises, before any CUDA call.
tg_status validate(const Args &a)
{
    if (a.M < 0 || a.N < 0 || a.K < 0 || a.batch < 1) return TG_ERR_INVALID_ARG;
    if (a.M > EXTENT_LIMIT || a.N > EXTENT_LIMIT || a.K > EXTENT_LIMIT || a.batch > EXTENT_LIMIT)
        return TG_ERR_INVALID_ARG;
    if (a.sA < 0 || a.sB < 0 || a.sC < 0) return TG_ERR_INVALID_ARG;
    if (a.lda < a.a_cols() || a.ldb < a.b_cols() || a.ldc < a.N) return TG_ERR_INVALID_ARG;
    // strides beyond 2^40 elements are not addressable in any case
    const int64_t STRIDE_LIMIT = int64_t(1) << 40;
    if (a.lda > STRIDE_LIMIT || a.ldb > STRIDE_LIMIT || a.ldc > STRIDE_LIMIT ||
        a.sA > STRIDE_LIMIT || a.sB > STRIDE_LIMIT || a.sC > STRIDE_LIMIT)
        return TG_ERR_INVALID_ARG;
    if (a.M == 0 || a.N == 0) return TG_OK;
    if (!span_ok(a.M, a.N, a.ldc, a.batch, a.sC) || !span_ok(a.a_rows(), a.a_cols(), a.lda, a.batch, a.sA) ||
        !span_ok(a.b_rows(), a.b_cols(), a.ldb, a.batch, a.sB))
        return TG_ERR_INVALID_ARG;
    if (a.C == nullptr) return TG_ERR_INVALID_ARG;
    if (a.K > 0 && (a.A == nullptr || a.B == nullptr)) return TG_ERR_INVALID_ARG;
    // distinct problems may not share an element of C
    const int64_t one_c = (a.M - 1) * a.ldc + a.N;
    if (a.batch > 1 && a.sC < one_c) return TG_ERR_INVALID_ARG;
    if (a.K > 0) {
        const uintptr_t c0 = reinterpret_cast<uintptr_t>(a.C);
        const uintptr_t c1 =
            c0 + static_cast<uintptr_t>(a.c_bytes) * static_cast<uintptr_t>(span_elems(a.M, a.N, a.ldc, a.batch, a.sC));
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.A);
        const uintptr_t a1 =
            a0 + static_cast<uintptr_t>(a.ab_bytes) *
                     static_cast<uintptr_t>(span_elems(a.a_rows(), a.a_cols(), a.lda, a.batch, a.sA));
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(a.B);
        const uintptr_t b1 =
            b0 + static_cast<uintptr_t>(a.ab_bytes) *
                     static_cast<uintptr_t>(span_elems(a.b_rows(), a.b_cols(), a.ldb, a.batch, a.sB));
        if (ranges_overlap(c0, c1, a0, a1) || ranges_overlap(c0, c1, b0, b1))
            return TG_ERR_INVALID_ARG;
    }
    return TG_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PlanInput plan_input(const Args &a, int sms, const tg_options *opt)
{
    PlanInput in{};
    in.M = a.M;
    in.N = a.N;
    in.K = a.K;
    in.batch = a.batch;
    in.a_bcast = a.batch > 1 && a.sA == 0;
    in.b_bcast = a.batch > 1 && a.sB == 0;
    const bool batched_a = a.batch > 1 && !in.a_bcast;
    const bool batched_b = a.batch > 1 && !in.b_bcast;
    const int64_t eb = a.ab_bytes;
    in.a_tma_ok = aligned16(a.A) && (a.lda * eb) % 16 == 0 && (!batched_a || (a.sA * eb) % 16 == 0);
    in.b_tma_ok = aligned16(a.B) && (a.ldb * eb) % 16 == 0 && (!batched_b || (a.sB * eb) % 16 == 0);
    in.f8 = a.ab_bytes == 1;
    in.mx = a.mx;
    in.fp4 = a.fp4;
    in.c_tma_ok = aligned16(a.C) && (a.ldc * a.c_bytes) % 16 == 0 &&
                  (a.batch == 1 || (a.sC * a.c_bytes) % 16 == 0);
    in.sm_count = sms;
    in.a_cm = a.a_cm;
    in.b_cm = a.b_cm;
    if (opt) {
        in.block_n = opt->block_n;
        in.stages = opt->stages;
        in.split_k = opt->split_k;
        in.force_pack = opt->force_pack;
        in.epilogue = opt->epilogue;
        in.max_ctas = opt->max_ctas;
        in.cta_pair = opt->cta_pair;
        in.stream_k = opt->stream_k;
        in.direct = opt->direct;
    }
    return in;
}

void fill_info(const Plan &p, tg_plan_info *out)
{
    std::memset(out, 0, sizeof(*out));
    out->block_m = p.pair ? 2 * BM : p.half_a ? BM / 2 : BM;
    out->cta_pair = p.pair ? 2 : 1;
    out->stream_k = p.stream_k ? 2 : 1;
    out->sk_tiles = static_cast<int32_t>(p.sk_tiles);
    out->block_n = p.bn;
    out->block_k = p.fp4 ? 4 * BK : p.f8 ? 2 * BK : BK;  // elements of K a k-block
    out->stages = p.stages;
    out->tiles_m = p.tiles_m;
    out->tiles_n = p.tiles_n;
    out->k_blocks = p.k_blocks;
    out->split_k = p.splits;
    out->num_units = p.units;
    out->grid = p.grid;
    out->pack_a = p.pack_a ? 1 : 0;
    out->pack_b = p.pack_b ? 1 : 0;
    out->epilogue = p.epilogue;
    out->smem_bytes = p.smem;
    out->tmem_cols = p.tmem;
    out->workspace_bytes = p.workspace();
    out->direct = p.direct ? 2 : 1;
}

// ------------------------------------------------------------ device state
struct DeviceInfo {
    int sms = 0;
};

struct Workspace {
    int device = -1;
    void *arena = nullptr;  // pack copies + split-K partials
    size_t arena_cap = 0;
    int32_t *counters = nullptr;  // split-K arrival counters (kept zero between calls)
    size_t counters_cap = 0;
    uint32_t *err = nullptr;  // device error word of this stream
    void *host_arena = nullptr;  // device copies of tg_gemm_host operands
    size_t host_cap = 0;
    // tg_gemm_host's copy streams and events (created on first use)
    cudaStream_t h2d = nullptr, d2h = nullptr;
    static constexpr int HOST_EVENTS = 1 + 3 * HOST_MAX_PIECES;
    cudaEvent_t ev[HOST_EVENTS] = {};
};

std::mutex g_mutex;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

tg_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return TG_OK;
    if (e == cudaErrorMemoryAllocation) return TG_ERR_OOM;
    return TG_ERR_CUDA;
}

tg_status device_sms(int dev, int *sms)
{
    auto it = g_devices.find(dev);
    if (it != g_devices.end()) {
        *sms = it->second.sms;
        return TG_OK;
    }
    int v = 0;
    cudaError_t e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
    g_devices[dev].sms = v;
    *sms = v;
    return TG_OK;
}

Workspace &workspace_for(int dev, cudaStream_t stream)
{
    Workspace &w = g_workspaces[{dev, stream}];
    w.device = dev;
    return w;
}

// Grows a device buffer; waits for the stream first so that no kernel still
// uses the old one.
tg_status grow(void **buf, size_t *cap, size_t need, cudaStream_t stream)
{
    if (need <= *cap) return TG_OK;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_status(e);
    if (*buf) cudaFree(*buf);
    *buf = nullptr;
    *cap = 0;
    const size_t want = need + need / 4;
    e = cudaMalloc(buf, want);
    if (e != cudaSuccess) {
        *buf = nullptr;
        return cuda_status(e);
    }
    *cap = want;
    return TG_OK;
}

tg_status ensure_err_word(Workspace &w, cudaStream_t stream)
{
    if (w.err) return TG_OK;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&w.err), 256);
    if (e != cudaSuccess) {
        w.err = nullptr;
        return cuda_status(e);
    }
    e = cudaMemsetAsync(w.err, 0, 256, stream);
    return cuda_status(e);
}

tg_status ensure_counters(Workspace &w, size_t bytes, cudaStream_t stream)
{
    if (bytes <= w.counters_cap) return TG_OK;
    void *p = w.counters;
    tg_status st = grow(&p, &w.counters_cap, bytes, stream);
    w.counters = static_cast<int32_t *>(p);
    if (st != TG_OK) return st;
    return cuda_status(cudaMemsetAsync(w.counters, 0, w.counters_cap, stream));
}

// ------------------------------------------------------------ TMA descriptors
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn query_encode_fn()
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
}

// The driver's encoder, looked up once.  A function-local static with an
// initialiser: C++ runs the lookup exactly once and every caller, from any
// thread, sees the finished pointer (some callers hold no library mutex).
EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = query_encode_fn();
    return fn;
}

// Recently encoded tensor maps (per host thread): repeated calls on the same
// buffers skip the driver's encode.
struct MapKey {
    const void *base;
    int dt;
    uint64_t d0, d1, d2, s1, s2;
    uint32_t b0, b1;
    bool operator==(const MapKey &o) const
    {
        return base == o.base && dt == o.dt && d0 == o.d0 && d1 == o.d1 && d2 == o.d2 &&
               s1 == o.s1 && s2 == o.s2 && b0 == o.b0 && b1 == o.b1;
    }
};
struct MapCache {
    static constexpr int N = 32;
    MapKey key[N];
    CUtensorMap map[N];
    bool used[N] = {};
    int next = 0;
};
thread_local MapCache t_maps;

// A rank-3 tiled map: dim0 contiguous (d0 elements), dim1 rows (stride1
// bytes), dim2 problems (stride2 bytes); box {box0, box1, 1}; 128B swizzle;
// out-of-range elements read as zero.
bool encode_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t d0, uint64_t d1,
               uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const MapKey k{base, static_cast<int>(dt) * 16 + static_cast<int>(swz), d0, d1, d2, stride1, stride2,
                   box0, box1};
    for (int i = 0; i < MapCache::N; ++i)
        if (t_maps.used[i] && t_maps.key[i] == k) {
            *m = t_maps.map[i];
            return true;
        }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    const int slot = t_maps.next;
    t_maps.next = (slot + 1) % MapCache::N;
    t_maps.key[slot] = k;
    t_maps.map[slot] = *m;
    t_maps.used[slot] = true;
    return true;
}

// Stride of the problem dimension when there is only one problem (any valid
// value; never used to step).
uint64_t single_problem_stride(uint64_t rows, uint64_t stride1)
{
    const uint64_t s = rows * stride1;
    return (s + 15) / 16 * 16;
}

cudaError_t launch_gemm(int bn, bool pair, bool f8, int mx, const CUtensorMap &ta, const CUtensorMap &tb,
                        const CUtensorMap &tc, const KernelParams &p, int stages, int grid,
                        cudaStream_t s)
{
    if (mx != MX_NONE && bn == 224)
        return pair || !f8 ? cudaErrorInvalidValue : launch_gemm_mx224(ta, tb, tc, p, stages, mx, grid, s);
    switch (bn) {
        case 64: return launch_gemm_bn64(ta, tb, tc, p, stages, pair, f8, mx, grid, s);
        case 128: return launch_gemm_bn128(ta, tb, tc, p, stages, pair, f8, mx, grid, s);
        case 192: return launch_gemm_bn192(ta, tb, tc, p, stages, pair, f8, mx, grid, s);
        case 256: return launch_gemm_bn256(ta, tb, tc, p, stages, pair, f8, mx, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

// Half-height A slots (one CTA per tile): widths 128 (8 slots) and 192 (6).
cudaError_t launch_gemm_half_a(int bn, bool f8, const CUtensorMap &ta, const CUtensorMap &tb,
                               const CUtensorMap &tc, const KernelParams &p, int stages, int grid, cudaStream_t s)
{
    if (stages != half_a_stages(bn)) return cudaErrorInvalidValue;
    switch (bn) {
        case 128: return launch_gemm_bn128_half_a(ta, tb, tc, p, f8, grid, s);
        case 192: return launch_gemm_bn192_half_a(ta, tb, tc, p, f8, grid, s);
        default: return cudaErrorInvalidValue;
    }
}

// Co-resident two-CTA clusters of a pair configuration, cached per device.
int max_pairs(int dev, int bn, int stages, bool f8)
{
    static std::map<std::tuple<int, int, int, bool>, int> cache;
    const auto key = std::make_tuple(dev, bn, stages, f8);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int n = 0;
    switch (bn) {
        case 128: n = max_pairs_bn128(stages, f8); break;
        case 256: n = max_pairs_bn256(stages, f8); break;
        default: n = 0;
    }
    cache[key] = n;
    return n;
}

// Fused-epilogue fields of the kernel parameters.
void fill_epilogue(KernelParams &p, const Args &a, const tg_epilogue *ep)
{
    p.C = a.C;
    p.ldc = a.ldc;
    p.strideC = a.sC;
    p.M = static_cast<int32_t>(a.M);
    p.N = static_cast<int32_t>(a.N);
    p.fused = 1;
    p.act = ep->activation;
    p.out_bf16 = ep->out_type == TG_BF16 ? 1 : 0;
    p.alpha = ep->alpha;
    p.beta = ep->beta;
    p.bias = ep->bias;
    p.bias_stride = ep->bias_stride;
    p.residual = ep->residual;
    p.ldr = ep->ldr;
    p.strideR = ep->strideR;
}

// K == 0 with an epilogue: D = act(bias) + beta * R (the empty sum is 0).
__global__ void epilogue_only_kernel(const KernelParams p, int64_t total)
{
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t b = e / (static_cast<int64_t>(p.M) * p.N);
        const int64_t r = e - b * p.M * p.N;
        const int64_t i = r / p.N;
        const int64_t j = r - i * p.N;
        float x = __fmul_rn(p.alpha, 0.0f);
        if (p.bias) x = __fadd_rn(x, p.bias[b * p.bias_stride + j]);
        x = activation(x, p.act);
        const int64_t ro = b * p.strideR + i * p.ldr + j;
        const int64_t o = b * p.strideC + i * p.ldc + j;
        if (p.out_bf16) {
            if (p.residual) {
                const float rv = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t *>(p.residual)[ro]) << 16);
                x = __fadd_rn(x, __fmul_rn(p.beta, rv));
            }
            static_cast<__nv_bfloat16 *>(p.C)[o] = __float2bfloat16_rn(x);
        } else {
            if (p.residual) x = __fadd_rn(x, __fmul_rn(p.beta, static_cast<const float *>(p.residual)[ro]));
            static_cast<float *>(p.C)[o] = x;
        }
    }
}

int grid_for(int64_t work, int sms)
{
    int64_t g = (work + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sms) * 8;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

// The pack job of one operand: rows x cols bf16 (batch nb, element stride
// between problems), into dst with rows padded to 8 elements.
PackJob pack_job(const void *src, uint16_t *dst, int64_t rows, int64_t cols, int64_t ld, int64_t nb,
                 int64_t stride)
{
    const int64_t ld2 = pack_pitch(cols);
    const uintptr_t base = reinterpret_cast<uintptr_t>(src);
    return PackJob{static_cast<const uint16_t *>(src), dst, rows, cols, ld, stride, ld2, nb * rows * (ld2 / 8), base,
                   base + 2u * static_cast<uintptr_t>(span_elems(rows, cols, ld, nb, stride))};
}

// The whole device-side path of one call (arguments already validated).
tg_status run_gemm(const Args &a, cudaStream_t stream, const tg_options *opt,
                   const tg_epilogue *ep = nullptr)
{
    if (a.M == 0 || a.N == 0) return TG_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    std::lock_guard<std::mutex> lock(g_mutex);
    int sms = 0;
    tg_status st = device_sms(dev, &sms);
    if (st != TG_OK) return st;

    if (a.K == 0) {
        const int64_t total = a.batch * a.M * a.N;
        if (ep) {
            KernelParams p{};
            fill_epilogue(p, a, ep);
            epilogue_only_kernel<<<grid_for(total, sms), 256, 0, stream>>>(p, total);
        } else {
            zero_c_kernel<<<grid_for(total, sms), 256, 0, stream>>>(static_cast<float *>(a.C), a.M, a.N,
                                                                     a.ldc, a.sC, total);
        }
        return cuda_status(cudaGetLastError());
    }

    PlanInput in = plan_input(a, sms, opt);
    Plan plan;
    if (!make_plan(in, plan)) return TG_ERR_INVALID_ARG;

    Workspace &w = workspace_for(dev, stream);
    st = ensure_err_word(w, stream);
    if (st != TG_OK) return st;

    if (plan.direct) {
        KernelParams p{};
        p.M = static_cast<int32_t>(a.M);
        p.N = static_cast<int32_t>(a.N);
        p.K = static_cast<int32_t>(a.K);
        p.batch = static_cast<int32_t>(a.batch);
        p.tiles_m = plan.tiles_m;
        p.tiles_n = plan.tiles_n;
        p.splits = 1;
        p.k_blocks = plan.k_blocks;
        p.num_units = plan.units;
        p.a_mn = a.a_cm ? 1 : 0;
        p.b_k = a.b_cm ? 1 : 0;
        p.C = a.C;
        p.ldc = a.ldc;
        p.strideC = a.sC;
        if (ep) fill_epilogue(p, a, ep);
        p.err = w.err;
        p.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : DEFAULT_TIMEOUT_NS;
        p.debug_stall = (opt && opt->debug_stall) ? (opt->debug_stall == 2 ? 2 : 1) : 0;
        p.trace = opt ? reinterpret_cast<unsigned long long *>(opt->trace_buffer) : nullptr;
        if (trace_enabled())
            std::fprintf(stderr, "tg_gemm M=%lld N=%lld K=%lld batch=%lld: direct tiles=%dx%d kb=%d chunk=%d grid=%d\n",
                         (long long)a.M, (long long)a.N, (long long)a.K, (long long)a.batch, plan.tiles_m,
                         plan.tiles_n, plan.k_blocks, plan.stages, plan.grid);
        const int64_t dsA = in.a_bcast || a.batch == 1 ? 0 : a.sA, dsB = in.b_bcast || a.batch == 1 ? 0 : a.sB;
        // contiguous extents: K of a row-major A or column-major B, else M or N
        const bool vec = direct_vec_ok(a.A, a.lda, dsA, a.a_cm ? a.M : a.K) &&
                         direct_vec_ok(a.B, a.ldb, dsB, a.b_cm ? a.K : a.N);
        e = launch_direct(p, a.A, a.B, a.lda, a.ldb, dsA, dsB, plan.stages, vec, plan.grid, stream);
        return cuda_status(e);
    }

    const void *A = a.A;
    const void *B = a.B;
    int64_t lda = a.lda, ldb = a.ldb, sA = a.sA, sB = a.sB;

    // Encode the operand maps; an operand TMA cannot describe is packed.
    CUtensorMap ta{}, tb{}, tc{};
    // Row-major A: boxes [128 rows x 64 k] ([64 rows x 64 k] for half-height
    // A slots); column-major A: [64 k x 64 rows].
    // Row-major B: [64 k x 64 columns]; column-major B: [B columns x 64 k].
    const uint32_t b_cols_cta = static_cast<uint32_t>(plan.pair ? plan.bn / 2 : plan.bn);
    // Element type and the K extent of a 128-byte box row: 64 bf16 or 128
    // 8-bit elements (8-bit operands are K-major: row-major A, column-major B).
    const int64_t eb = a.ab_bytes;
    const CUtensorMapDataType dt = eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t kbox = static_cast<uint32_t>(128 / eb);
    auto encode_a = [&]() {
        const uint64_t z = in.a_bcast || a.batch == 1 ? 1 : static_cast<uint64_t>(a.batch);
        const uint64_t s2 = z == 1 ? single_problem_stride(a.a_rows(), lda * eb) : static_cast<uint64_t>(sA) * eb;
        if (a.a_cm) return encode_3d(&ta, dt, A, a.M, a.K, z, lda * eb, s2, 64, BK);
        return encode_3d(&ta, dt, A, a.K, a.M, z, lda * eb, s2, kbox, plan.half_a ? BM / 2 : BM);
    };
    auto encode_b = [&]() {
        const uint64_t z = in.b_bcast || a.batch == 1 ? 1 : static_cast<uint64_t>(a.batch);
        const uint64_t s2 = z == 1 ? single_problem_stride(a.b_rows(), ldb * eb) : static_cast<uint64_t>(sB) * eb;
        if (a.b_cm) return encode_3d(&tb, dt, B, a.K, a.N, z, ldb * eb, s2, kbox, b_cols_cta);
        return encode_3d(&tb, dt, B, a.N, a.K, z, ldb * eb, s2, 64, BK);
    };
    if (!encode_fn()) return TG_ERR_CUDA;
    // 8-bit operands are never packed (the entry point requires 16-byte rows)
    if (plan.f8 && (plan.pack_a || plan.pack_b || !encode_a() || !encode_b())) return TG_ERR_UNSUPPORTED;
    if (!plan.pack_a && !encode_a()) {
        plan.pack_a = true;
        plan.ws_pack_a = round_up((in.a_bcast ? 1 : a.batch) * a.a_rows() * pack_pitch(a.a_cols()) * 2, 256);
    }
    if (!plan.pack_b && !encode_b()) {
        plan.pack_b = true;
        plan.ws_pack_b = round_up((in.b_bcast ? 1 : a.batch) * a.b_rows() * pack_pitch(a.b_cols()) * 2, 256);
    }

    // The persistent grid actually launched: two-SM tiles never use more
    // clusters than can be resident at once; the stream-K ranges follow it.
    int grid = plan.grid;
    if (plan.pair) {
        const int pairs = max_pairs(dev, plan.bn, plan.stages, plan.f8);
        if (pairs <= 0) return TG_ERR_UNSUPPORTED;
        if (grid > 2 * pairs) grid = 2 * pairs;
        if (trace_enabled())
            std::fprintf(stderr, "tg_gemm: co-resident CTA pairs %d, launch grid %d\n", pairs, grid);
        if (grid != plan.grid) replan_stream_k(in, plan, grid);
    }

    const size_t arena_need = static_cast<size_t>(plan.ws_pack_a + plan.ws_pack_b + plan.ws_partials +
                                                  plan.ws_scales_a + plan.ws_scales_b);
    if (arena_need > 0) {
        st = grow(&w.arena, &w.arena_cap, arena_need, stream);
        if (st != TG_OK) return st;
    }
    if (plan.ws_counters > 0) {
        st = ensure_counters(w, static_cast<size_t>(plan.ws_counters), stream);
        if (st != TG_OK) return st;
    }
    uint8_t *arena = static_cast<uint8_t *>(w.arena);
    uint16_t *pack_a_buf = reinterpret_cast<uint16_t *>(arena);
    uint16_t *pack_b_buf = reinterpret_cast<uint16_t *>(arena + plan.ws_pack_a);
    float *partials = reinterpret_cast<float *>(arena + plan.ws_pack_a + plan.ws_pack_b);
    uint8_t *scales_a = arena + plan.ws_pack_a + plan.ws_pack_b + plan.ws_partials;
    uint8_t *scales_b = scales_a + plan.ws_scales_a;
    if (plan.mx) {
        const int64_t runs = ceil_div(a.k_elems(), 32);
        const int64_t za = in.a_bcast ? 1 : a.batch, zb = in.b_bcast ? 1 : a.batch;
        const int64_t subs_b = ceil_div(plan.bn, 128);
        const int64_t halves = plan.fp4 ? 2 : 1;
        const ScaleJob ja{a.sfa, scales_a, a.M, runs, a.ld_sfa, a.batch > 1 ? a.s_sfa : 0, za, plan.tiles_m,
                          plan.k_blocks, 128, 1, halves};
        const ScaleJob jb{a.sfb, scales_b, a.N, runs, a.ld_sfb, a.batch > 1 ? a.s_sfb : 0, zb, plan.tiles_n,
                          plan.k_blocks, plan.bn, subs_b, halves};
        const int64_t blocks_a = scale_blocks(ja), blocks_b = scale_blocks(jb);
        if (blocks_a + blocks_b > INT32_MAX) return TG_ERR_UNSUPPORTED;
        scale_tile_kernel<<<static_cast<unsigned>(blocks_a + blocks_b), SC_THREADS, 0, stream>>>(ja, jb, blocks_a);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
    }

    if (plan.pack_a || plan.pack_b) {
        PackJob ja{}, jb{};
        if (plan.pack_a)
            ja = pack_job(a.A, pack_a_buf, a.a_rows(), a.a_cols(), a.lda, in.a_bcast ? 1 : a.batch, a.sA);
        if (plan.pack_b)
            jb = pack_job(a.B, pack_b_buf, a.b_rows(), a.b_cols(), a.ldb, in.b_bcast ? 1 : a.batch, a.sB);
        const int blocks_a = plan.pack_a ? grid_for(ja.chunks, sms) : 0;
        const int blocks_b = plan.pack_b ? grid_for(jb.chunks, sms) : 0;
        pack_bf16_kernel<<<blocks_a + blocks_b, 256, 0, stream>>>(ja, jb, blocks_a);
        if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
        if (plan.pack_a) {
            A = pack_a_buf;
            lda = ja.ld_dst;
            sA = in.a_bcast ? 0 : a.a_rows() * ja.ld_dst;
            if (!encode_a()) return TG_ERR_CUDA;
        }
        if (plan.pack_b) {
            B = pack_b_buf;
            ldb = jb.ld_dst;
            sB = in.b_bcast ? 0 : a.b_rows() * jb.ld_dst;
            if (!encode_b()) return TG_ERR_CUDA;
        }
    }
    if (plan.epilogue == 1) {
        const uint64_t z = static_cast<uint64_t>(a.batch);
        const uint64_t s2 = z == 1 ? single_problem_stride(a.M, a.ldc * a.c_bytes)
                                   : static_cast<uint64_t>(a.sC) * a.c_bytes;
        const bool bf16 = a.c_bytes == 2;
        if (!encode_3d(&tc, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.C,
                       a.N, a.M, z, a.ldc * a.c_bytes, s2, EPI_CHUNK, EPI_CHUNK,
                       bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B)) {
            if (opt && opt->epilogue == 1) return TG_ERR_UNSUPPORTED;
            plan.epilogue = 2;
        }
    }
    if (plan.epilogue != 1) tc = ta;  // unused by the kernel; any valid map

    KernelParams p{};
    p.M = static_cast<int32_t>(a.M);
    p.N = static_cast<int32_t>(a.N);
    p.K = static_cast<int32_t>(a.K);
    p.batch = static_cast<int32_t>(a.batch);
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.splits = plan.splits;
    p.k_blocks = plan.k_blocks;
    p.num_units = plan.units;
    p.group_m = plan.group_m;
    p.a_bcast = in.a_bcast ? 1 : 0;
    p.b_bcast = in.b_bcast ? 1 : 0;
    p.a_mn = a.a_cm ? 1 : 0;
    p.b_k = a.b_cm ? 1 : 0;
    p.epi_tma = plan.epilogue == 1 ? 1 : 0;
    p.C = a.C;
    p.ldc = a.ldc;
    p.strideC = a.sC;
    if (ep) fill_epilogue(p, a, ep);
    const bool partial_tiles = plan.splits > 1 || plan.stream_k;
    p.partials = partial_tiles ? partials : nullptr;
    p.counters = partial_tiles ? w.counters : nullptr;
    p.stream_k = plan.stream_k ? 1 : 0;
    p.dp_waves = plan.dp_waves;
    p.sk_first_tile = static_cast<int32_t>(plan.sk_first_tile);
    p.sk_iters = plan.sk_iters;
    p.sk_workers = plan.sk_workers;
    p.maxparts = plan.maxparts;
    p.err = w.err;
    p.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : DEFAULT_TIMEOUT_NS;
    p.debug_stall = (opt && opt->debug_stall) ? (opt->debug_stall == 2 ? 2 : 1) : 0;
    p.partial_floats = partial_tiles ? plan.ws_partials / 4 : 0;
    p.counter_count = partial_tiles ? plan.ws_counters / 4 : 0;
    p.trace = opt ? reinterpret_cast<unsigned long long *>(opt->trace_buffer) : nullptr;

    if (trace_enabled())
        std::fprintf(stderr,
                     "tg_gemm M=%lld N=%lld K=%lld batch=%lld: BN=%d stages=%d tiles=%dx%d kb=%d "
                     "split=%d pair=%d stream_k=%d (dp_waves=%d sk_tiles=%lld maxparts=%d) units=%lld grid=%d "
                     "pack=%d/%d epi=%d\n",
                     (long long)a.M, (long long)a.N, (long long)a.K, (long long)a.batch, plan.bn,
                     plan.stages, plan.tiles_m, plan.tiles_n, plan.k_blocks, plan.splits, plan.pair ? 2 : 1,
                     plan.stream_k ? 1 : 0, plan.dp_waves, (long long)plan.sk_tiles, plan.maxparts,
                     (long long)plan.units, plan.grid, plan.pack_a, plan.pack_b, plan.epilogue);

    p.mma_fmt = a.mma_fmt;
    p.sfa = plan.mx ? scales_a : nullptr;
    p.sfb = plan.mx ? scales_b : nullptr;
    const int mx_kind = plan.fp4 ? MX_FP4 : plan.mx ? MX_FP8 : MX_NONE;
    e = plan.half_a ? launch_gemm_half_a(plan.bn, plan.f8, ta, tb, tc, p, plan.stages, grid, stream)
                    : launch_gemm(plan.bn, plan.pair, plan.f8, mx_kind, ta, tb, tc, p, plan.stages, grid, stream);
    return cuda_status(e);
}

}  // namespace

// Helpers shared with other translation units of the library (declared in
// tg_internal.h); thin wrappers over the functions above.
int shared_validate(const void *A, const void *B, const float *C, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t sA, int64_t sB,
                    int64_t sC)
{
    return validate(Args{A, B, const_cast<float *>(C), M, N, K, lda, ldb, ldc, batch, sA, sB, sC});
}

bool shared_plan(const void *A, const void *B, const float *C, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t sA, int64_t sB,
                 int64_t sC, int sms, const tg_options *opt, Plan *out, PlanInput *in_out)
{
    PlanInput in =
        plan_input(Args{A, B, const_cast<float *>(C), M, N, K, lda, ldb, ldc, batch, sA, sB, sC}, sms, opt);
    in.half_a_ok = false;  // the static entry point launches full-height A slots
    if (in_out) *in_out = in;
    return make_plan(in, *out);
}

bool shared_encode_3d(CUtensorMap *m, bool fp32, const void *base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1)
{
    return encode_3d(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     base, d0, d1, d2, stride1, stride2, box0, box1);
}

uint64_t shared_single_problem_stride(uint64_t rows, uint64_t stride1)
{
    return single_problem_stride(rows, stride1);
}

cudaError_t shared_launch_gemm(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                               const CUtensorMap &tc, const KernelParams &p, int stages, int grid,
                               cudaStream_t s)
{
    return launch_gemm(bn, false, false, MX_NONE, ta, tb, tc, p, stages, grid, s);
}

cudaError_t shared_zero_fill(float *C, int64_t M, int64_t N, int64_t ldc, int64_t sC, int64_t batch,
                             int sms, cudaStream_t s)
{
    const int64_t total = batch * M * N;
    zero_c_kernel<<<grid_for(total, sms), 256, 0, s>>>(C, M, N, ldc, sC, total);
    return cudaGetLastError();
}

}  // namespace tg

using namespace tg;

TG_API const char *tg_status_string(tg_status s)
{
    switch (s) {
        case TG_OK: return "ok";
        case TG_ERR_INVALID_ARG: return "invalid argument";
        case TG_ERR_UNSUPPORTED: return "unsupported";
        case TG_ERR_CUDA: return "CUDA error";
        case TG_ERR_OOM: return "out of device memory";
        case TG_ERR_TIMEOUT: return "device wait timed out";
        case TG_ERR_DEVICE_CHECK: return "device-side consistency check failed";
        default: return "unknown status";
    }
}

TG_API tg_status tg_gemm_ex(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t strideA,
                            int64_t strideB, int64_t strideC, tg_stream_t stream,
                            const tg_options *opt)
{
    const Args a = with_layout(Args{A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC}, opt);
    tg_status st = validate(a);
    if (st != TG_OK) return st;
    if (opt) {
        // option ranges are checked here too, before anything is enqueued
        PlanInput in = plan_input(a, 148, opt);
        Plan pl;
        if (M > 0 && N > 0 && K > 0 && !make_plan(in, pl)) return TG_ERR_INVALID_ARG;
    }
    return run_gemm(a, reinterpret_cast<cudaStream_t>(stream), opt);
}

// Run-time plan search: every instantiated (width, two-SM, ring depth)
// with stream-K on or off and, when there are fewer tiles than workers,
// split-K factors; each timed `reps` times with events on the caller's
// stream, the median kept, the fastest returned.
TG_API tg_status tg_tune(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K, int64_t lda,
                         int64_t ldb, int64_t ldc, int64_t batch, int64_t strideA, int64_t strideB,
                         int64_t strideC, tg_stream_t stream_, const tg_options *base, int32_t reps,
                         tg_options *best, float *best_us)
{
    using namespace tg;
    if (!best || reps < 1 || reps > 100) return TG_ERR_INVALID_ARG;
    const Args a = with_layout(Args{A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC}, base);
    tg_status st = validate(a);
    if (st != TG_OK) return st;
    tg_options start{};
    if (base) start = *base;
    *best = start;
    if (best_us) *best_us = 0.0f;
    if (M == 0 || N == 0 || K == 0) return TG_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if ((st = device_sms(dev, &sms)) != TG_OK) return st;
    }
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess || (e = cudaEventCreate(&e1)) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        return cuda_status(e);
    }
    float best_t = -1.0f;
    tg_options best_o = start;
    st = TG_OK;
    // Median time of one candidate over `reps` calls (after a warm-up call
    // that also sizes the workspaces); the fastest is kept.
    auto time_candidate = [&](const tg_options &o) {
        float ts[100];
        st = run_gemm(a, stream, &o);
        for (int r = 0; r < reps && st == TG_OK; ++r) {
            cudaEventRecord(e0, stream);
            st = run_gemm(a, stream, &o);
            cudaEventRecord(e1, stream);
            if ((e = cudaEventSynchronize(e1)) != cudaSuccess) st = cuda_status(e);
            if (st == TG_OK) cudaEventElapsedTime(&ts[r], e0, e1);
        }
        if (st != TG_OK) return;
        std::sort(ts, ts + reps);
        const float t = ts[reps / 2] * 1000.0f;
        if (best_t < 0.0f || t < best_t) {
            best_t = t;
            best_o = o;
        }
    };
    {
        // the direct-load kernel, where it applies
        tg_options o = start;
        o.direct = 2;
        PlanInput in = plan_input(a, sms, &o);
        Plan pl;
        if (make_plan(in, pl)) time_candidate(o);
    }
    const int widths[4] = {64, 128, 192, 256};
    const int depths[5] = {2, 3, 4, 6, 8};
    const int splits[6] = {1, 2, 3, 4, 6, 8};
    for (int wi = 0; wi < 4 && st == TG_OK; ++wi) {
        for (int pr = 1; pr <= 2 && st == TG_OK; ++pr) {
            const bool pair = pr == 2;
            if (pair && !pair_width(widths[wi])) continue;
            for (int di = 0; di < 5 && st == TG_OK; ++di) {
                // outputs of at most 64 rows also have rings of 64-row A slots
                const bool half_a = !pair && a.M <= BM / 2 && depths[di] == half_a_stages(widths[wi]);
                if (!stage_supported(widths[wi], depths[di], pair) && !half_a) continue;
                for (int si = 0; si < 6 && st == TG_OK; ++si) {
                    for (int sk = 1; sk <= 2 && st == TG_OK; ++sk) {
                        if (sk == 2 && splits[si] > 1) continue;
                        tg_options o = start;
                        o.direct = 1;
                        o.block_n = widths[wi];
                        o.cta_pair = pr;
                        o.stages = depths[di];
                        o.split_k = splits[si];
                        o.stream_k = sk;
                        PlanInput in = plan_input(a, sms, &o);
                        Plan pl;
                        if (!make_plan(in, pl)) continue;
                        // keep split-K to the cases it exists for: fewer units than workers
                        const int64_t workers = pair ? sms / 2 : sms;
                        if (splits[si] > 1 && pl.units / splits[si] >= workers) continue;
                        if (sk == 2 && !pl.stream_k) continue;  // same plan as stream_k = 1
                        // the deeper half of the instantiated ring depths
                        if (depths[di] < max_stages(widths[wi], pair) / 2) continue;
                        time_candidate(o);
                        if (st != TG_OK) break;
                    }
                }
            }
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != TG_OK) return st;
    *best = best_o;
    if (best_us) *best_us = best_t;
    return TG_OK;
}

TG_API tg_status tg_gemm(const void *A, const void *B, float *C, int64_t M, int64_t N, int64_t K,
                         int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t strideA,
                         int64_t strideB, int64_t strideC, tg_stream_t stream)
{
    return tg_gemm_ex(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, stream,
                      nullptr);
}

namespace tg {
namespace {

// The fused-epilogue arguments against a validated call.
tg_status check_epilogue(const Args &a, const tg_epilogue *ep)
{
    if (ep->activation < TG_ACT_NONE || ep->activation > TG_ACT_SILU) return TG_ERR_INVALID_ARG;
    if (ep->bias_stride < 0) return TG_ERR_INVALID_ARG;
    if (ep->residual) {
        if (ep->ldr < a.N || ep->strideR < 0) return TG_ERR_INVALID_ARG;
        if (a.batch > 1 && ep->strideR < (a.M - 1) * ep->ldr + a.N && ep->strideR != 0) return TG_ERR_INVALID_ARG;
        const bool same = ep->residual == a.C && ep->ldr == a.ldc && ep->strideR == a.sC;
        if (!same) {
            const uintptr_t d0 = reinterpret_cast<uintptr_t>(a.C);
            const uintptr_t d1 = d0 + a.c_bytes * static_cast<uintptr_t>(span_elems(a.M, a.N, a.ldc, a.batch, a.sC));
            const uintptr_t r0 = reinterpret_cast<uintptr_t>(ep->residual);
            const uintptr_t r1 =
                r0 + a.c_bytes * static_cast<uintptr_t>(span_elems(a.M, a.N, ep->ldr, a.batch, ep->strideR));
            if (ranges_overlap(d0, d1, r0, r1)) return TG_ERR_INVALID_ARG;
        }
    }
    return TG_OK;
}

}  // namespace
}  // namespace tg

TG_API tg_status tg_gemm_fused(const void *A, const void *B, void *D, int64_t M, int64_t N,
                               int64_t K, int64_t lda, int64_t ldb, int64_t ldd, int64_t batch,
                               int64_t strideA, int64_t strideB, int64_t strideD, const tg_epilogue *ep,
                               tg_stream_t stream, const tg_options *opt)
{
    using namespace tg;
    if (!ep) return TG_ERR_INVALID_ARG;
    if (ep->out_type != TG_F32 && ep->out_type != TG_BF16) return TG_ERR_INVALID_ARG;
    Args a = with_layout(Args{A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD}, opt);
    a.c_bytes = ep->out_type == TG_BF16 ? 2 : 4;
    tg_status st = validate(a);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    if ((st = check_epilogue(a, ep)) != TG_OK) return st;
    if (opt) {
        PlanInput in = plan_input(a, 148, opt);
        Plan pl;
        if (K > 0 && !make_plan(in, pl)) return TG_ERR_INVALID_ARG;
    }
    return run_gemm(a, reinterpret_cast<cudaStream_t>(stream), opt, ep);
}

namespace tg {
namespace {

// The shared part of the 8-bit entry points: the layout, formats and
// requirements of tg_gemm_fp8, then the call.  `a` holds the operands, D and
// (block-scaled) the scales; its checks of the scales are the caller's.
tg_status run_fp8(Args a, int32_t a_format, int32_t b_format, const tg_epilogue *ep, cudaStream_t stream,
                  const tg_options *opt)
{
    if (!a.fp4) {
        if (a_format != TG_FP8_E4M3 && a_format != TG_FP8_E5M2) return TG_ERR_INVALID_ARG;
        if (b_format != TG_FP8_E4M3 && b_format != TG_FP8_E5M2) return TG_ERR_INVALID_ARG;
    }
    if (opt && (opt->a_col_major || opt->b_col_major || opt->force_pack)) return TG_ERR_INVALID_ARG;
    if (ep && ep->out_type != TG_F32 && ep->out_type != TG_BF16) return TG_ERR_INVALID_ARG;
    // A row-major M x K, B stored N x K (column-major K x N): both K-major
    a.b_cm = true;
    a.ab_bytes = 1;
    a.c_bytes = ep && ep->out_type == TG_BF16 ? 2 : 4;
    // kind::f8f6f4 / kind::mxf8f6f4 operand formats: E4M3 = 0, E5M2 = 1
    // (bits 7-9 A, 10-12 B); kind::mxf4: E2M1 = 1 in both fields
    a.mma_fmt = a.fp4 ? ((1u << 7) | (1u << 10))
                      : (static_cast<uint32_t>(a_format) << 7) | (static_cast<uint32_t>(b_format) << 10);
    tg_status st = validate(a);
    if (st != TG_OK) return st;
    if (a.M == 0 || a.N == 0) return TG_OK;
    if (ep && (st = check_epilogue(a, ep)) != TG_OK) return st;
    if (a.mx && a.K > 0) {
        // the scale matrices lie apart from D
        const int64_t runs = ceil_div(a.k_elems(), 32);
        if (!span_ok(a.M, runs, a.ld_sfa, a.batch, a.s_sfa) || !span_ok(a.N, runs, a.ld_sfb, a.batch, a.s_sfb))
            return TG_ERR_INVALID_ARG;
        const uintptr_t d0 = reinterpret_cast<uintptr_t>(a.C);
        const uintptr_t d1 = d0 + a.c_bytes * static_cast<uintptr_t>(span_elems(a.M, a.N, a.ldc, a.batch, a.sC));
        const uintptr_t f0 = reinterpret_cast<uintptr_t>(a.sfa);
        const uintptr_t f1 = f0 + static_cast<uintptr_t>(span_elems(a.M, runs, a.ld_sfa, a.batch, a.s_sfa));
        const uintptr_t g0 = reinterpret_cast<uintptr_t>(a.sfb);
        const uintptr_t g1 = g0 + static_cast<uintptr_t>(span_elems(a.N, runs, a.ld_sfb, a.batch, a.s_sfb));
        if (ranges_overlap(d0, d1, f0, f1) || ranges_overlap(d0, d1, g0, g1)) return TG_ERR_INVALID_ARG;
    }
    if (a.K > 0) {
        // 16-byte rows: the TMA unit loads the operands as they are
        const bool batched_a = a.batch > 1 && a.sA != 0, batched_b = a.batch > 1 && a.sB != 0;
        if ((reinterpret_cast<uintptr_t>(a.A) & 15u) || (reinterpret_cast<uintptr_t>(a.B) & 15u) || a.lda % 16 ||
            a.ldb % 16 || (batched_a && a.sA % 16) || (batched_b && a.sB % 16))
            return TG_ERR_UNSUPPORTED;
        // the plan exists (checked with a nominal SM count before any CUDA call)
        PlanInput in = plan_input(a, 148, opt);
        Plan pl;
        if (!make_plan(in, pl)) return TG_ERR_INVALID_ARG;
    }
    return run_gemm(a, stream, opt, ep);
}

}  // namespace
}  // namespace tg

TG_API tg_status tg_gemm_fp8(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldd, int64_t batch, int64_t strideA,
                             int64_t strideB, int64_t strideD, int32_t a_format, int32_t b_format,
                             const tg_epilogue *ep, tg_stream_t stream, const tg_options *opt)
{
    using namespace tg;
    const Args a{A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD};
    return run_fp8(a, a_format, b_format, ep, reinterpret_cast<cudaStream_t>(stream), opt);
}

namespace tg {
namespace {

// The scale arguments shared by both block-scaled entry points (K counts
// elements); returns TG_OK or the status to report.
tg_status check_scale_args(int64_t K, int64_t batch, int64_t strideA, int64_t strideB, const uint8_t *SFA,
                           int64_t ld_sfa, int64_t stride_sfa, const uint8_t *SFB, int64_t ld_sfb,
                           int64_t stride_sfb, const tg_options *opt, bool fp4)
{
    if (opt && ((opt->block_n != 0 && opt->block_n != 128 && opt->block_n != 192 && opt->block_n != 224) ||
                opt->cta_pair == 2 || (opt->stages != 0 && opt->stages != 2 && opt->stages != 4) ||
                (fp4 && opt->block_n == 224 && opt->stages == 4)))
        return TG_ERR_INVALID_ARG;
    if (stride_sfa < 0 || stride_sfb < 0 || K < 0) return TG_ERR_INVALID_ARG;
    if (K > 0) {
        const int64_t runs = (K + 31) / 32;
        if (!SFA || !SFB || ld_sfa < runs || ld_sfb < runs) return TG_ERR_INVALID_ARG;
        const int64_t LIMIT = int64_t(1) << 40;
        if (ld_sfa > LIMIT || ld_sfb > LIMIT || stride_sfa > LIMIT || stride_sfb > LIMIT) return TG_ERR_INVALID_ARG;
        // shared operands have shared scales (the re-arranged scales follow
        // the operand's problem index)
        if (batch > 1 && ((strideA == 0 && stride_sfa != 0) || (strideB == 0 && stride_sfb != 0)))
            return TG_ERR_INVALID_ARG;
    }
    return TG_OK;
}

// Packed 4-bit operands: element counts that address whole bytes.
bool fp4_counts_ok(int64_t K, int64_t lda, int64_t ldb, int64_t strideA, int64_t strideB)
{
    return K % 2 == 0 && lda % 2 == 0 && ldb % 2 == 0 && strideA % 2 == 0 && strideB % 2 == 0;
}

}  // namespace
}  // namespace tg

TG_API tg_status tg_gemm_mxfp8(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldd, int64_t batch, int64_t strideA,
                               int64_t strideB, int64_t strideD, int32_t a_format, int32_t b_format,
                               const uint8_t *SFA, int64_t ld_sfa, int64_t stride_sfa, const uint8_t *SFB,
                               int64_t ld_sfb, int64_t stride_sfb, const tg_epilogue *ep, tg_stream_t stream,
                               const tg_options *opt)
{
    using namespace tg;
    Args a{A, B, D, M, N, K, lda, ldb, ldd, batch, strideA, strideB, strideD};
    a.mx = true;
    a.sfa = SFA;
    a.sfb = SFB;
    a.ld_sfa = ld_sfa;
    a.s_sfa = stride_sfa;
    a.ld_sfb = ld_sfb;
    a.s_sfb = stride_sfb;
    const tg_status st = check_scale_args(K, batch, strideA, strideB, SFA, ld_sfa, stride_sfa, SFB, ld_sfb,
                                          stride_sfb, opt, false);
    if (st != TG_OK) return st;
    return run_fp8(a, a_format, b_format, ep, reinterpret_cast<cudaStream_t>(stream), opt);
}


TG_API tg_status tg_gemm_mxfp4(const void *A, const void *B, void *D, int64_t M, int64_t N, int64_t K,
                               int64_t lda, int64_t ldb, int64_t ldd, int64_t batch, int64_t strideA,
                               int64_t strideB, int64_t strideD, const uint8_t *SFA, int64_t ld_sfa,
                               int64_t stride_sfa, const uint8_t *SFB, int64_t ld_sfb, int64_t stride_sfb,
                               const tg_epilogue *ep, tg_stream_t stream, const tg_options *opt)
{
    using namespace tg;
    if (K < 0 || lda < 0 || ldb < 0 || strideA < 0 || strideB < 0) return TG_ERR_INVALID_ARG;
    if (!fp4_counts_ok(K, lda, ldb, strideA, strideB)) return TG_ERR_INVALID_ARG;
    tg_status st = check_scale_args(K, batch, strideA, strideB, SFA, ld_sfa, stride_sfa, SFB, ld_sfb, stride_sfb,
                                    opt, true);
    if (st != TG_OK) return st;
    // from here on the operands are byte matrices: K / 2 bytes a row
    Args a{A, B, D, M, N, K / 2, lda / 2, ldb / 2, ldd, batch, strideA / 2, strideB / 2, strideD};
    a.mx = true;
    a.fp4 = true;
    a.sfa = SFA;
    a.sfb = SFB;
    a.ld_sfa = ld_sfa;
    a.s_sfa = stride_sfa;
    a.ld_sfb = ld_sfb;
    a.s_sfb = stride_sfb;
    return run_fp8(a, 0, 0, ep, reinterpret_cast<cudaStream_t>(stream), opt);
}

TG_API tg_status tg_plan(const void *A, const void *B, const float *C, int64_t M, int64_t N,
                         int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int64_t batch,
                         int64_t strideA, int64_t strideB, int64_t strideC, int32_t sm_count,
                         const tg_options *opt, tg_plan_info *out)
{
    if (!out || sm_count < 0) return TG_ERR_INVALID_ARG;
    const int32_t family = opt ? opt->operands : 0;
    if (family < 0 || family > 3) return TG_ERR_INVALID_ARG;
    Args a = with_layout(Args{A, B, const_cast<float *>(C), M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC},
                         opt);
    if (family != 0) {
        // the 8-/4-bit entry points' layout: A row-major, B stored N x K
        if (opt->a_col_major || opt->b_col_major || opt->force_pack) return TG_ERR_INVALID_ARG;
        a.b_cm = true;
        a.ab_bytes = 1;
        a.mx = family >= 2;
        if (family == 3) {
            // packed 4-bit elements: planned on the operands' bytes
            if (K < 0 || lda < 0 || ldb < 0 || strideA < 0 || strideB < 0) return TG_ERR_INVALID_ARG;
            if (!fp4_counts_ok(K, lda, ldb, strideA, strideB)) return TG_ERR_INVALID_ARG;
            a.fp4 = true;
            a.K = K / 2;
            a.lda = lda / 2;
            a.ldb = ldb / 2;
            a.sA = strideA / 2;
            a.sB = strideB / 2;
        }
    }
    tg_status st = validate(a);
    if (st != TG_OK) return st;
    if (family != 0 && K > 0) {
        // 16-byte rows (counted in bytes)
        const bool batched_a = batch > 1 && a.sA != 0, batched_b = batch > 1 && a.sB != 0;
        if ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) || a.lda % 16 ||
            a.ldb % 16 || (batched_a && a.sA % 16) || (batched_b && a.sB % 16))
            return TG_ERR_UNSUPPORTED;
    }
    int sms = sm_count;
    if (sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_status(e);
        std::lock_guard<std::mutex> lock(g_mutex);
        st = device_sms(dev, &sms);
        if (st != TG_OK) return st;
    }
    std::memset(out, 0, sizeof(*out));
    if (M == 0 || N == 0 || K == 0) return TG_OK;  // nothing (or only a zero fill) to plan
    Plan p;
    if (!make_plan(plan_input(a, sms, opt), p)) return TG_ERR_INVALID_ARG;
    fill_info(p, out);
    return TG_OK;
}

namespace tg {
namespace {

// Copy rows [r0, r0 + nrows) x columns [c0, c0 + ncols) of a matrix between
// two pitches (elements of `eb` bytes).
cudaError_t copy_block(void *dst, int64_t dpitch, const void *src, int64_t spitch, int64_t r0, int64_t nrows,
                       int64_t c0, int64_t ncols, int64_t eb, cudaMemcpyKind kind, cudaStream_t s)
{
    if (nrows <= 0 || ncols <= 0) return cudaSuccess;
    auto *d = static_cast<uint8_t *>(dst) + (r0 * dpitch + c0) * eb;
    const auto *x = static_cast<const uint8_t *>(src) + (r0 * spitch + c0) * eb;
    if (ncols == dpitch && ncols == spitch)
        return cudaMemcpyAsync(d, x, static_cast<size_t>(nrows * ncols * eb), kind, s);
    return cudaMemcpy2DAsync(d, static_cast<size_t>(dpitch * eb), x, static_cast<size_t>(spitch * eb),
                             static_cast<size_t>(ncols * eb), static_cast<size_t>(nrows), kind, s);
}

// Problems [b0, b1) of a batch: one copy when the problems are stacked
// (stride = rows * pitch on both sides), else one per problem.
cudaError_t copy_problems(void *dst, int64_t dpitch, int64_t dstride, const void *src, int64_t spitch,
                          int64_t sstride, int64_t b0, int64_t b1, int64_t r0, int64_t nrows, int64_t rows,
                          int64_t c0, int64_t ncols, int64_t eb, cudaMemcpyKind kind, cudaStream_t s)
{
    if (b1 - b0 > 1 && nrows == rows && dstride == rows * dpitch && sstride == rows * spitch) {
        auto *d = static_cast<uint8_t *>(dst) + b0 * dstride * eb;
        const auto *x = static_cast<const uint8_t *>(src) + b0 * sstride * eb;
        return copy_block(d, dpitch, x, spitch, 0, (b1 - b0) * rows, c0, ncols, eb, kind, s);
    }
    for (int64_t b = b0; b < b1; ++b) {
        cudaError_t e = copy_block(static_cast<uint8_t *>(dst) + b * dstride * eb, dpitch,
                                   static_cast<const uint8_t *>(src) + b * sstride * eb, spitch, r0, nrows, c0,
                                   ncols, eb, kind, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

tg_status host_streams(Workspace &w)
{
    cudaError_t e = cudaSuccess;
    if (!w.h2d && (e = cudaStreamCreateWithFlags(&w.h2d, cudaStreamNonBlocking)) != cudaSuccess) return cuda_status(e);
    if (!w.d2h && (e = cudaStreamCreateWithFlags(&w.d2h, cudaStreamNonBlocking)) != cudaSuccess) return cuda_status(e);
    for (cudaEvent_t &ev : w.ev)
        if (!ev && (e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_status(e);
    return TG_OK;
}

}  // namespace
}  // namespace tg

// Host buffers in, host buffer out.  The operands are copied to the device
// as they are laid out on the host (contiguous spans, so every copy is a
// plain 1-D copy at full link speed; strided 2-D copies of host memory run
// up to ~40% slower), C is written to a device buffer with 16-byte rows (so
// the epilogue stores with the tensor memory accelerator) and copied back
// row by row into the host layout.  The work is pipelined over pieces that
// are contiguous on the host (see host_pieces): one stream copies operand
// pieces in, the caller's stream multiplies each piece as soon as it has
// landed, a third stream copies each finished piece of C out, so the copies
// in both directions overlap the GEMMs and each other.  An operand copied
// whole whose rows are not 16-byte aligned is realigned once on the device.
TG_API tg_status tg_gemm_host(const void *A_host, const void *B_host, float *C_host, int64_t M,
                              int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                              tg_stream_t stream_, const tg_options *opt)
{
    using namespace tg;
    const Args a =
        with_layout(Args{A_host, B_host, C_host, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC}, opt);
    tg_status st = validate(a);
    if (st != TG_OK) return st;
    if (M == 0 || N == 0) return TG_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    int sms = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        if ((st = device_sms(dev, &sms)) != TG_OK) return st;
    }

    const bool a_bcast = batch > 1 && strideA == 0, b_bcast = batch > 1 && strideB == 0;
    const int64_t a_rows = a.a_rows(), a_cols = a.a_cols(), b_rows = a.b_rows(), b_cols = a.b_cols();
    // device copies of A and B keep the host's element offsets: the span of
    // every operand is copied from its first element
    const int64_t na = K > 0 ? span_elems(a_rows, a_cols, lda, a_bcast ? 1 : batch, strideA) : 0;
    const int64_t nb = K > 0 ? span_elems(b_rows, b_cols, ldb, b_bcast ? 1 : batch, strideB) : 0;
    const int64_t ldc_d = round_up(N, 4), sC_d = M * ldc_d;
    const HostPieces hp = host_pieces(M, N, K, batch, a_bcast, b_bcast, a.a_cm, a.b_cm,
                                      strideA == a_rows * lda, strideB == b_rows * ldb);
    // the operand copied whole is realigned once if its rows are not 16-byte
    // aligned - unless the whole problem goes to the direct-load kernel,
    // which reads any pitch in place (the device copies start on 256 bytes)
    bool direct = false;
    if (K > 0 && hp.pieces == 1) {
        Args dev_args = a;
        dev_args.A = reinterpret_cast<const void *>(uintptr_t{256});
        dev_args.B = reinterpret_cast<const void *>(uintptr_t{512});
        dev_args.C = reinterpret_cast<float *>(uintptr_t{768});
        dev_args.ldc = ldc_d;
        dev_args.sC = sC_d;
        Plan pl;
        direct = make_plan(plan_input(dev_args, sms, opt), pl) && pl.direct;
    }
    const bool a_whole = hp.dim == 0 || hp.dim == 3, b_whole = hp.dim == 0 || hp.dim == 2;
    const bool a_fix =
        !direct && K > 0 && a_whole && (lda % 8 != 0 || (batch > 1 && !a_bcast && strideA % 8 != 0));
    const bool b_fix =
        !direct && K > 0 && b_whole && (ldb % 8 != 0 || (batch > 1 && !b_bcast && strideB % 8 != 0));
    const int64_t lda_f = pack_pitch(a_cols), ldb_f = pack_pitch(b_cols);
    const int64_t sA_f = a_bcast ? 0 : a_rows * lda_f, sB_f = b_bcast ? 0 : b_rows * ldb_f;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += static_cast<size_t>(round_up(static_cast<int64_t>(bytes), 256));
        return o;
    };
    const size_t off_a = take(na * 2), off_b = take(nb * 2), off_c = take(batch * sC_d * 4);
    const size_t off_af = a_fix ? take((a_bcast ? 1 : batch) * a_rows * lda_f * 2) : 0;
    const size_t off_bf = b_fix ? take((b_bcast ? 1 : batch) * b_rows * ldb_f * 2) : 0;
    uint8_t *dbuf = nullptr;
    Workspace *wp = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        Workspace &w = workspace_for(dev, stream);
        st = grow(&w.host_arena, &w.host_cap, off, stream);
        if (st == TG_OK) st = host_streams(w);
        if (st != TG_OK) return st;
        dbuf = static_cast<uint8_t *>(w.host_arena);
        wp = &w;  // map nodes are stable; calls on one stream are serial
    }
    Workspace &w = *wp;
    const uint16_t *dA = reinterpret_cast<uint16_t *>(dbuf + off_a);
    const uint16_t *dB = reinterpret_cast<uint16_t *>(dbuf + off_b);
    float *dC = reinterpret_cast<float *>(dbuf + off_c);
    const cudaMemcpyKind H2D = cudaMemcpyHostToDevice;

    // One piece: everything on the caller's stream (cross-stream events would
    // only add latency).  Several: the copy streams start after the caller's
    // earlier work.
    const bool overlap = hp.pieces > 1;
    cudaStream_t s_in = overlap ? w.h2d : stream, s_out = overlap ? w.d2h : stream;
    if (overlap) {
        if ((e = cudaEventRecord(w.ev[0], stream)) != cudaSuccess) return cuda_status(e);
        if ((e = cudaStreamWaitEvent(w.h2d, w.ev[0], 0)) != cudaSuccess) return cuda_status(e);
        if ((e = cudaStreamWaitEvent(w.d2h, w.ev[0], 0)) != cudaSuccess) return cuda_status(e);
    }
    // elements [e0, e1) of an operand's span, host -> device
    auto copy_in = [&](const uint16_t *dst, const void *src, int64_t e0, int64_t e1) {
        if (e1 <= e0) return cudaSuccess;
        return cudaMemcpyAsync(const_cast<uint16_t *>(dst) + e0, static_cast<const uint16_t *>(src) + e0,
                               static_cast<size_t>((e1 - e0) * 2), H2D, s_in);
    };
    // the span of problems [b0, b1), or of rows [r0, r1) of one problem
    auto span = [&](int64_t rows, int64_t cols, int64_t ld, int64_t stride, int64_t b0, int64_t b1, int64_t r0,
                    int64_t r1) {
        const int64_t lo = b0 * stride + r0 * ld;
        const int64_t hi = (b1 - 1) * stride + (r1 - 1) * ld + cols;
        (void)rows;
        return std::make_pair(lo, hi);
    };
    const uint16_t *A_use = dA, *B_use = dB;
    int64_t lda_use = lda, ldb_use = ldb, sA_use = a_bcast ? 0 : strideA, sB_use = b_bcast ? 0 : strideB;
    if (K > 0 && a_whole) {
        const auto sp = span(a_rows, a_cols, lda, strideA, 0, a_bcast ? 1 : batch, 0, a_rows);
        if ((e = copy_in(dA, A_host, sp.first, sp.second)) != cudaSuccess) return cuda_status(e);
        if (a_fix) {
            uint16_t *dst = reinterpret_cast<uint16_t *>(dbuf + off_af);
            const PackJob j = pack_job(dA, dst, a_rows, a_cols, lda, a_bcast ? 1 : batch, strideA);
            pack_bf16_kernel<<<grid_for(j.chunks, sms), 256, 0, s_in>>>(j, PackJob{}, grid_for(j.chunks, sms));
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
            A_use = dst, lda_use = lda_f, sA_use = sA_f;
        }
    }
    if (K > 0 && b_whole) {
        const auto sp = span(b_rows, b_cols, ldb, strideB, 0, b_bcast ? 1 : batch, 0, b_rows);
        if ((e = copy_in(dB, B_host, sp.first, sp.second)) != cudaSuccess) return cuda_status(e);
        if (b_fix) {
            uint16_t *dst = reinterpret_cast<uint16_t *>(dbuf + off_bf);
            const PackJob j = pack_job(dB, dst, b_rows, b_cols, ldb, b_bcast ? 1 : batch, strideB);
            pack_bf16_kernel<<<grid_for(j.chunks, sms), 256, 0, s_in>>>(j, PackJob{}, grid_for(j.chunks, sms));
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
            B_use = dst, ldb_use = ldb_f, sB_use = sB_f;
        }
    }
    cudaEvent_t last_out = nullptr;
    for (int i = 0; i < hp.pieces; ++i) {
        const int64_t lo = hp.dim ? hp.bound(i) : 0, hi = hp.dim ? hp.bound(i + 1) : 0;
        int64_t b0 = 0, b1 = batch, m0 = 0, m1 = M, n0 = 0, n1 = N;
        if (hp.dim == 1) { b0 = lo; b1 = hi; }
        if (hp.dim == 2) { m0 = lo; m1 = hi; }
        if (hp.dim == 3) { n0 = lo; n1 = hi; }
        if (b1 <= b0 || m1 <= m0 || n1 <= n0) continue;
        if (hp.dim == 1) {
            const auto sa = span(a_rows, a_cols, lda, strideA, b0, b1, 0, a_rows);
            const auto sb = span(b_rows, b_cols, ldb, strideB, b0, b1, 0, b_rows);
            e = copy_in(dA, A_host, sa.first, sa.second);
            if (e == cudaSuccess) e = copy_in(dB, B_host, sb.first, sb.second);
        } else if (hp.dim == 2) {  // rows m0..m1 of a row-major A
            const auto sa = span(a_rows, a_cols, lda, strideA, 0, 1, m0, m1);
            e = copy_in(dA, A_host, sa.first, sa.second);
        } else if (hp.dim == 3) {  // columns n0..n1 of B: rows of a column-major B
            const auto sb = span(b_rows, b_cols, ldb, strideB, 0, 1, n0, n1);
            e = copy_in(dB, B_host, sb.first, sb.second);
        }
        cudaEvent_t ev_in = w.ev[1 + 3 * i], ev_gemm = w.ev[2 + 3 * i], ev_out = w.ev[3 + 3 * i];
        if (e == cudaSuccess && overlap) e = cudaEventRecord(ev_in, w.h2d);
        if (e == cudaSuccess && overlap) e = cudaStreamWaitEvent(stream, ev_in, 0);
        if (e != cudaSuccess) return cuda_status(e);
        // the piece's GEMM on the device copies
        const int64_t a_off = a.a_cm ? m0 : m0 * lda_use;
        const int64_t b_off = a.b_cm ? n0 * ldb_use : n0;
        Args piece{A_use + b0 * sA_use + a_off, B_use + b0 * sB_use + b_off, dC + b0 * sC_d + m0 * ldc_d + n0,
                   m1 - m0, n1 - n0, K, lda_use, ldb_use, ldc_d, b1 - b0, sA_use, sB_use, sC_d};
        st = run_gemm(with_layout(piece, opt), stream, opt);
        if (st != TG_OK) return st;
        if (overlap && (e = cudaEventRecord(ev_gemm, stream)) != cudaSuccess) return cuda_status(e);
        if (overlap && (e = cudaStreamWaitEvent(w.d2h, ev_gemm, 0)) != cudaSuccess) return cuda_status(e);
        // only the M x N block of every problem goes back (gaps keep host data)
        e = copy_problems(C_host, ldc, strideC, dC, ldc_d, sC_d, b0, b1, m0, m1 - m0, M, n0, n1 - n0, 4,
                          cudaMemcpyDeviceToHost, s_out);
        if (e == cudaSuccess && overlap) e = cudaEventRecord(ev_out, w.d2h);
        if (e != cudaSuccess) return cuda_status(e);
        if (overlap) last_out = ev_out;
    }
    // the caller's stream resumes after the last piece of C is home
    if (last_out && (e = cudaStreamWaitEvent(stream, last_out, 0)) != cudaSuccess) return cuda_status(e);
    e = cudaStreamSynchronize(stream);
    return cuda_status(e);
}

TG_API tg_status tg_device_error(tg_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return TG_ERR_CUDA;
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return TG_ERR_CUDA;
    // The static-scratch entry point's own word (one per device, shared by
    // all its calls): read and cleared here as well.
    uint32_t static_word = ERR_NONE;
    if (static_error_take(dev, stream, &static_word) != cudaSuccess) return TG_ERR_CUDA;
    const tg_status static_status = static_word == ERR_NONE          ? TG_OK
                                    : static_word == ERR_DEBUG_CHECK ? TG_ERR_DEVICE_CHECK
                                                                     : TG_ERR_TIMEOUT;
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_workspaces.find({dev, stream});
    if (it == g_workspaces.end() || !it->second.err) return static_status;
    Workspace &w = it->second;
    uint32_t word = 0;
    if ((e = cudaMemcpyAsync(&word, w.err, 4, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
        return TG_ERR_CUDA;
    if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return TG_ERR_CUDA;
    if (word == ERR_NONE) return static_status;
    // Clear the word (and the detail word after it), and the split-K
    // counters an aborted kernel may have left part-way.
    cudaMemsetAsync(w.err, 0, 8, stream);
    if (w.counters) cudaMemsetAsync(w.counters, 0, w.counters_cap, stream);
    cudaStreamSynchronize(stream);
    return word == ERR_DEBUG_CHECK ? TG_ERR_DEVICE_CHECK : TG_ERR_TIMEOUT;
}

TG_API void tg_shutdown(void)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &kv : g_workspaces) {
        Workspace &w = kv.second;
        cudaSetDevice(w.device);
        if (w.arena) cudaFree(w.arena);
        if (w.counters) cudaFree(w.counters);
        if (w.err) cudaFree(w.err);
        if (w.host_arena) cudaFree(w.host_arena);
        if (w.h2d) cudaStreamDestroy(w.h2d);
        if (w.d2h) cudaStreamDestroy(w.d2h);
        for (cudaEvent_t ev : w.ev)
            if (ev) cudaEventDestroy(ev);
    }
    g_workspaces.clear();
    g_devices.clear();
    cudaSetDevice(cur);
}
