// tg_gemm_splitk_static: the split-K GEMM with its scratch in a static
// device array instead of memory allocated at run time.
//
// For callers that cannot allocate device memory: plugins inside a host
// framework whose pool owns the device memory, and services that must not
// call cudaMalloc/cudaFree after start-up (both may synchronise the device
// and take unbounded time).  The kernel is the library's persistent GEMM
// kernel unchanged; only where its split-K partial tiles, tile counters and
// error word live differs.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "tg_gemm.h"
#include "tg_internal.h"
#include "tg_plan.h"

#define TG_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr size_t PARTIAL_BYTES = size_t(16) << 20;   // 16 MiB of fp32 partial tiles
constexpr int64_t MAX_TILES = 4096;                  // one int32 counter per tile
constexpr size_t COUNTER_BYTES = MAX_TILES * 4;      // 16 KiB
constexpr size_t ERR_BYTES = 256;
constexpr size_t SCRATCH_BYTES = PARTIAL_BYTES + COUNTER_BYTES + ERR_BYTES;
constexpr int MAX_DEVICES = 64;

}  // namespace

// The scratch.  In host code this name is only a host-side stand-in: its
// device address comes from cudaGetSymbolAddress below and is what the
// kernel receives.
static __device__ __align__(256) uint8_t tg_static_scratch[SCRATCH_BYTES];

namespace {

std::mutex g_setup_mutex;
void *g_scratch_addr[MAX_DEVICES] = {};

// Once per device, with that device current: the array's device address.
tg_status scratch_address(int dev, uint8_t **out)
{
    if (dev < 0 || dev >= MAX_DEVICES) return TG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, tg_static_scratch);
        if (e != cudaSuccess || p == nullptr) return TG_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(g_scratch_addr[dev]);
    return TG_OK;
}

// The array's error word on device `dev`, or null if no call has set the
// device up yet (then no kernel of this entry point has run there).
uint32_t *error_word(int dev)
{
    if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    uint8_t *base = static_cast<uint8_t *>(g_scratch_addr[dev]);
    return base ? reinterpret_cast<uint32_t *>(base + PARTIAL_BYTES + COUNTER_BYTES) : nullptr;
}

// Watchdog self-test of this entry point: with TG_DEBUG_STALL_NS set to a
// positive number of nanoseconds, the kernel's epilogue first waits on a
// barrier that nothing completes, with that limit, so the wait must expire
// and tg_device_error() must report it.  Read on every call (tests set and
// unset it within one process).
uint64_t debug_stall_ns()
{
    const char *v = std::getenv("TG_DEBUG_STALL_NS");
    if (!v || !*v) return 0;
    char *end = nullptr;
    const unsigned long long ns = std::strtoull(v, &end, 10);
    return (end && *end == '\0') ? static_cast<uint64_t>(ns) : 0;
}

}  // namespace

namespace tg {

// Reads the array's error word on device `dev` after `stream` has been
// synchronised by the caller; a nonzero word is cleared (with the detail
// word after it) and returned in *code (ERR_NONE otherwise).  Reads nothing
// on a device where the entry point has never run.  Allocates nothing: the
// word goes through one 4-byte copy into a host variable.
cudaError_t static_error_take(int dev, cudaStream_t stream, uint32_t *code)
{
    *code = ERR_NONE;
    uint32_t *err = error_word(dev);
    if (!err) return cudaSuccess;
    uint32_t word = 0;
    cudaError_t e = cudaMemcpyAsync(&word, err, 4, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || word == ERR_NONE) return e;
    *code = word;
    e = cudaMemsetAsync(err, 0, 8, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e;
}

}  // namespace tg

TG_API tg_status tg_gemm_splitk_static(const void *A, const void *B, float *C, int64_t M,
                                       int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                       int64_t batch, int64_t strideA, int64_t strideB,
                                       int64_t strideC, int32_t split_k, tg_stream_t stream_)
{
    using namespace tg;
    const int v = shared_validate(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC);
    if (v != TG_OK) return static_cast<tg_status>(v);
    if (split_k < 1) return TG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return TG_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TG_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TG_ERR_CUDA;
    if (K == 0)
        return shared_zero_fill(C, M, N, ldc, strideC, batch, sms, stream) == cudaSuccess ? TG_OK
                                                                                          : TG_ERR_CUDA;
    if (split_k > (K + BK - 1) / BK) return TG_ERR_INVALID_ARG;

    tg_options opt{};
    opt.split_k = split_k;
    opt.cta_pair = 1;  // one CTA per tile: the launch below is the single-CTA kernel
    opt.stream_k = 1;  // the split factor is the caller's
    Plan plan;
    PlanInput in;
    if (!shared_plan(A, B, C, M, N, K, lda, ldb, ldc, batch, strideA, strideB, strideC, sms, &opt, &plan, &in))
        return TG_ERR_INVALID_ARG;
    const int64_t tiles = batch * plan.tiles_m * static_cast<int64_t>(plan.tiles_n);
    if (plan.pack_a || plan.pack_b) return TG_ERR_UNSUPPORTED;  // no scratch for a pack copy
    if (tiles > MAX_TILES || plan.ws_partials > static_cast<int64_t>(PARTIAL_BYTES))
        return TG_ERR_UNSUPPORTED;

    uint8_t *scratch = nullptr;
    tg_status st = scratch_address(dev, &scratch);
    if (st != TG_OK) return st;
    float *partials = reinterpret_cast<float *>(scratch);
    int32_t *counters = reinterpret_cast<int32_t *>(scratch + PARTIAL_BYTES);
    uint32_t *err = reinterpret_cast<uint32_t *>(scratch + PARTIAL_BYTES + COUNTER_BYTES);
    // What must start at zero: this call's tile counters (an earlier call
    // that timed out may have left some part-way).  The error word is not
    // cleared here: like the per-stream word, it keeps the first expiry
    // until tg_device_error() reads and clears it (it starts at zero: global
    // variables without an initializer are zero-initialised when the module
    // loads).
    if (cudaMemsetAsync(counters, 0, static_cast<size_t>(tiles) * 4, stream) != cudaSuccess) return TG_ERR_CUDA;

    CUtensorMap ta{}, tb{}, tc{};
    const uint64_t za = in.a_bcast || batch == 1 ? 1 : static_cast<uint64_t>(batch);
    const uint64_t zb = in.b_bcast || batch == 1 ? 1 : static_cast<uint64_t>(batch);
    const uint64_t sa2 = za == 1 ? shared_single_problem_stride(M, lda * 2) : static_cast<uint64_t>(strideA) * 2;
    const uint64_t sb2 = zb == 1 ? shared_single_problem_stride(K, ldb * 2) : static_cast<uint64_t>(strideB) * 2;
    if (!shared_encode_3d(&ta, false, A, K, M, za, lda * 2, sa2, BK, BM)) return TG_ERR_UNSUPPORTED;
    if (!shared_encode_3d(&tb, false, B, N, K, zb, ldb * 2, sb2, 64, BK)) return TG_ERR_UNSUPPORTED;
    bool epi_tma = plan.epilogue == 1;
    if (epi_tma) {
        const uint64_t zc = static_cast<uint64_t>(batch);
        const uint64_t sc2 = zc == 1 ? shared_single_problem_stride(M, ldc * 4) : static_cast<uint64_t>(strideC) * 4;
        epi_tma = shared_encode_3d(&tc, true, C, N, M, zc, ldc * 4, sc2, EPI_CHUNK, EPI_CHUNK);
    }
    if (!epi_tma) tc = ta;  // unused by the kernel

    KernelParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.batch = static_cast<int32_t>(batch);
    p.tiles_m = plan.tiles_m;
    p.tiles_n = plan.tiles_n;
    p.splits = plan.splits;
    p.k_blocks = plan.k_blocks;
    p.num_units = plan.units;
    p.group_m = plan.group_m;
    p.a_bcast = in.a_bcast ? 1 : 0;
    p.b_bcast = in.b_bcast ? 1 : 0;
    p.epi_tma = epi_tma ? 1 : 0;
    p.C = C;
    p.ldc = ldc;
    p.strideC = strideC;
    p.partials = partials;
    p.maxparts = plan.splits;
    p.counters = counters;
    p.err = err;
    p.partial_floats = static_cast<int64_t>(PARTIAL_BYTES / 4);
    p.counter_count = MAX_TILES;
    const uint64_t stall_ns = debug_stall_ns();
    p.timeout_ns = stall_ns ? stall_ns : 2000000000ull;
    p.debug_stall = stall_ns ? 1 : 0;
    const cudaError_t e = shared_launch_gemm(plan.bn, ta, tb, tc, p, plan.stages, plan.grid, stream);
    return e == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}
