// Direct-load GEMM for small problems: one CTA of sixteen warps per 128 x 64
// output tile, no persistent schedule, no tensor maps.
//
// OCANNL "Module Ir.Schedule", Stage with a cooperative copy: every thread
// of the block takes part in moving the operand tiles into shared memory;
// and Pad-to-tile: the staged fringe (rows past M or N, k past K) is stored
// as zeros.  The copy uses plain loads - 16-byte units when both operands
// are 16-byte aligned with a contiguous extent that is a multiple of 8,
// else single elements - so an operand of any pitch and alignment is read
// where it lies: no realign pass and no second launch.  It writes the
// 128-byte-swizzled images the persistent kernel's TMA loads write: K-major
// for an operand stored K-contiguous (row-major A, column-major B), M/N-major
// for one stored M/N-contiguous, so that neighbouring threads read
// neighbouring elements and write neighbouring bytes, and both kernels issue
// the same MMAs on the same values.  Up to DIRECT_KB k-blocks are staged at
// once.  Every thread first issues all of its loads of a round and only then
// stores them, so one memory round trip stages a whole chunk in 16-byte units
// (at most 12 loads a thread) or two k-blocks element by element (48 loads
// a thread); the chunk's MMAs go out as one batch and the next chunk's copy
// waits for their commit.
// Eight warps then read the 128 x 64 accumulator from tensor memory, one
// 32 x 32 block each, and store it through a shared-memory transpose, so
// that every store instruction writes 32 consecutive columns of one row.
//
// The point is latency: a problem of a few tiles and k-blocks is done in
// one launch whose code path is short, where the persistent kernel would
// add the realign pass of misaligned operands and its producer / consumer
// machinery.
#include "tg_direct.h"
#include "tg_kernel.cuh"
#include "tg_plan.h"

namespace tg {
namespace {

constexpr uint32_t D_A_KB = BM * BK * 2;         // bytes of A's image per k-block: 16 KB
constexpr uint32_t D_B_KB = DIRECT_BN * BK * 2;  // bytes of B's image per k-block: 8 KB

static_assert(DIRECT_THREADS == 512 && DIRECT_BN == 64, "16 warps; the epilogue's 8: 4 lane quadrants x 2 column blocks");

// Bounded wait on an mbarrier phase (false after timeout_ns).
__device__ __forceinline__ bool direct_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0 && ptx::global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// 16-bit load issued only when `pred` holds (0 otherwise).  Volatile, so the
// loads of a batch keep their order and all go out before the first store.
__device__ __forceinline__ uint32_t ld_u16_pred(const uint16_t *src, bool pred)
{
    uint16_t v;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %2, 0;\n\t"
        "mov.b16 %0, 0;\n\t"
        "@p ld.global.nc.u16 %0, [%1];\n\t}"
        : "=h"(v)
        : "l"(src), "r"(static_cast<uint32_t>(pred))
        : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(static_cast<uint16_t>(v)) : "memory");
}

// 16-byte load (8 elements) issued only when `pred` holds (zeros otherwise).
__device__ __forceinline__ uint4 ld_v4_pred(const uint16_t *src, bool pred)
{
    uint4 v;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\tmov.b32 %3, 0;\n\t"
        "@p ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];\n\t}"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(src), "r"(static_cast<uint32_t>(pred))
        : "memory");
    return v;
}

// One operand as the copy sees it: element (row r, k) at
// base[r * s_row + k * s_k] for rows [0, rows) and k [0, K).
struct DirectOperand {
    const uint16_t *base;
    int64_t s_row, s_k;
    int32_t rows;
};

// This thread's share of one operand's k-block image of ROWS rows x 64 k
// (ROWS * 64 / 512 elements).  K-major image (operand stored K-contiguous):
// thread t takes k = t mod 64 of rows t / 64 + 8j, so a warp reads 32
// consecutive k of one row; 16-byte unit u of image row r sits at
// u ^ (r mod 8).  M/N-major image (stored M/N-contiguous): thread t takes
// row t mod ROWS at k = t / ROWS + (512 / ROWS) j, so a warp reads 32
// consecutive rows; the image is atoms of 64 rows x 64 k, one 128-byte k
// row of 64 elements each, unit u of k row kk at u ^ (kk mod 8), atoms 8 KB
// apart.  kbase: the image's first k.
template <int ROWS, bool KC>
__device__ __forceinline__ void load_image(const DirectOperand &o, int32_t kbase, int32_t K, int32_t tid,
                                           uint32_t (&v)[ROWS * BK / DIRECT_THREADS])
{
    constexpr int PER = ROWS * BK / DIRECT_THREADS;
    // Element j is inside the operand exactly when j < nj (a prefix), so each
    // load's predicate is one compare with a constant.
    const uint16_t *src;
    int64_t step;
    int32_t nj;
    if constexpr (KC) {
        const int32_t r0 = tid >> 6, k = kbase + (tid & 63);
        src = o.base + static_cast<int64_t>(r0) * o.s_row + k;
        step = 8 * o.s_row;
        nj = k < K ? min(PER, max(0, (o.rows - r0 + 7) >> 3)) : 0;
    } else {
        constexpr int KSTEP = DIRECT_THREADS / ROWS;
        const int32_t r = tid & (ROWS - 1), k0 = kbase + tid / ROWS;
        src = o.base + r + static_cast<int64_t>(k0) * o.s_k;
        step = KSTEP * o.s_k;
        nj = (r < o.rows && k0 < K) ? min(PER, (K - k0 + KSTEP - 1) / KSTEP) : 0;
    }
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        v[j] = ld_u16_pred(src, j < nj);
        src += step;
    }
}

template <int ROWS, bool KC>
__device__ __forceinline__ void store_image(uint32_t img, int32_t tid, const uint32_t (&v)[ROWS * BK / DIRECT_THREADS])
{
    constexpr int PER = ROWS * BK / DIRECT_THREADS;
    if constexpr (KC) {
        const uint32_t r0 = static_cast<uint32_t>(tid) >> 6, k = static_cast<uint32_t>(tid) & 63u;
        const uint32_t base = img + r0 * 128u + (((k >> 3) ^ (r0 & 7u)) << 4) + (k & 7u) * 2u;
#pragma unroll
        for (int j = 0; j < PER; ++j) st_shared_u16(base + static_cast<uint32_t>(j) * 1024u, v[j]);
    } else {
        constexpr uint32_t KSTEP = DIRECT_THREADS / ROWS;
        const uint32_t r = static_cast<uint32_t>(tid) & (ROWS - 1), k0 = static_cast<uint32_t>(tid) / ROWS;
        const uint32_t base = img + (r >> 6) * 8192u + (r & 7u) * 2u;
        const uint32_t u = (r & 63u) >> 3;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const uint32_t k = k0 + KSTEP * j;
            st_shared_u16(base + k * 128u + ((u ^ (k & 7u)) << 4), v[j]);
        }
    }
}

// The same images in 16-byte units (8 elements along the stored-contiguous
// dimension), for an operand whose base, pitch and batch stride are 16-byte
// aligned and whose contiguous extent (K for a K-major image, M or N for an
// M/N-major one) is a multiple of 8, so that every unit lies wholly inside
// or wholly outside it.  ROWS * 8 units an image, UNITS = ROWS / 64 a thread:
// unit t + 512 j.  K-major: unit (row r, k group c) at r * 128 + ((c ^ (r mod
// 8)) << 4).  M/N-major: unit (k row kk, row group g) at (g / 8) * 8192 +
// kk * 128 + (((g mod 8) ^ (kk mod 8)) << 4).
template <int ROWS, bool KC>
__device__ __forceinline__ void load_image_v4(const DirectOperand &o, int32_t kbase, int32_t K, int32_t tid,
                                              uint4 (&u)[ROWS / 64])
{
#pragma unroll
    for (int j = 0; j < ROWS / 64; ++j) {
        const int32_t id = tid + DIRECT_THREADS * j;
        if constexpr (KC) {
            const int32_t r = id >> 3, k = kbase + 8 * (id & 7);
            u[j] = ld_v4_pred(o.base + static_cast<int64_t>(r) * o.s_row + k, r < o.rows && k < K);
        } else {
            constexpr int RG = ROWS / 8;
            const int32_t k = kbase + id / RG, g = id % RG;
            u[j] = ld_v4_pred(o.base + 8 * g + static_cast<int64_t>(k) * o.s_k, 8 * g < o.rows && k < K);
        }
    }
}

template <int ROWS, bool KC>
__device__ __forceinline__ void store_image_v4(uint32_t img, int32_t tid, const uint4 (&u)[ROWS / 64])
{
#pragma unroll
    for (int j = 0; j < ROWS / 64; ++j) {
        const uint32_t id = static_cast<uint32_t>(tid + DIRECT_THREADS * j);
        uint32_t off;
        if constexpr (KC) {
            const uint32_t r = id >> 3, c = id & 7u;
            off = r * 128u + ((c ^ (r & 7u)) << 4);
        } else {
            constexpr uint32_t RG = ROWS / 8;
            const uint32_t kk = id / RG, g = id % RG;
            off = (g >> 3) * 8192u + kk * 128u + (((g & 7u) ^ (kk & 7u)) << 4);
        }
        ptx::st_shared_v4(img + off, u[j].x, u[j].y, u[j].z, u[j].w);
    }
}

struct DirectArgs {
    const void *A, *B;
    int64_t lda, ldb, sA, sB;  // element pitches and batch strides (0: shared operand)
    int32_t chunk_kb;          // k-blocks staged at once (1 .. DIRECT_KB)
    int32_t vec;               // both operands staged in 16-byte units (see load_image_v4)
};

// A_KC / B_KC: A stored row-major / B stored column-major (K-contiguous);
// FUSED: the fused epilogue.  One instance per combination keeps each
// kernel's code to its own path (a call this small runs largely from a cold
// instruction cache).
template <bool A_KC, bool B_KC, bool FUSED>
__global__ void __launch_bounds__(DIRECT_THREADS, 1) direct_gemm_kernel(const KernelParams p, const DirectArgs d)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const int chunk_kb = d.chunk_kb;
    const uint32_t sA = raw + pad;                                      // chunk_kb x 16 KB
    const uint32_t sB = sA + static_cast<uint32_t>(chunk_kb) * D_A_KB;  // chunk_kb x 8 KB
    const uint32_t stage_bytes = static_cast<uint32_t>(chunk_kb) * (D_A_KB + D_B_KB);
    const uint32_t epi_bytes = 8u * EPI_CHUNK * EPI_CHUNK * 4;
    const uint32_t bar0 = sA + (stage_bytes > epi_bytes ? stage_bytes : epi_bytes);
    const uint32_t mma_bar = bar0, stall_bar = bar0 + 8;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + pad + (bar0 - sA) + 16);

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int32_t tid = static_cast<int32_t>(threadIdx.x);
    unsigned long long *trace = p.trace ? p.trace + 8ull * blockIdx.x : nullptr;
    auto stamp = [&](int k) {
        if (trace) trace[k] = ptx::global_timer_ns();
    };
    if (tid == 0) {
        stamp(0);
        ptx::mbar_init(mma_bar, 1);
        ptx::mbar_init(stall_bar, 1);
        ptx::fence_barrier_init();
    }
    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), DIRECT_TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    ptx::griddep_wait();  // operands and C only after the previous kernels of the stream
    if (tid == 0) stamp(1);

    // output tile of this CTA
    const int64_t per_batch = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    const int32_t b = static_cast<int32_t>(blockIdx.x / per_batch);
    const int32_t rem = static_cast<int32_t>(blockIdx.x % per_batch);
    const int32_t tm = rem / p.tiles_n, tn = rem % p.tiles_n;
    const int32_t m0 = tm * BM, n0 = tn * DIRECT_BN;
    // A (M x K) staged by its rows m0 + r, B (K x N) by its columns n0 + r.
    const uint16_t *Ab = static_cast<const uint16_t *>(d.A) + static_cast<int64_t>(b) * d.sA;
    const uint16_t *Bb = static_cast<const uint16_t *>(d.B) + static_cast<int64_t>(b) * d.sB;
    constexpr bool a_kc = A_KC, b_kc = B_KC;
    const DirectOperand opA{Ab + (a_kc ? static_cast<int64_t>(m0) * d.lda : static_cast<int64_t>(m0)),
                            a_kc ? d.lda : 1, a_kc ? 1 : d.lda, p.M - m0};
    const DirectOperand opB{Bb + (b_kc ? static_cast<int64_t>(n0) * d.ldb : static_cast<int64_t>(n0)),
                            b_kc ? d.ldb : 1, b_kc ? 1 : d.ldb, p.N - n0};

    // The persistent kernel's descriptors for the same images: a K-major
    // operand steps 32 B per 16 k, an M/N-major one 16 k rows (2 KB) with
    // its 64-row atoms 8 KB apart.
    const uint32_t idesc = instr_desc_bf16<BM, DIRECT_BN>(!a_kc, !b_kc);
    const uint64_t a_desc0 = smem_desc_sw128(0, a_kc ? 16 : BK * 128, 1024);
    const uint64_t b_desc0 = smem_desc_sw128(0, b_kc ? 16 : BK * 128, 1024);
    const uint32_t a_step = a_kc ? 32u : 2048u, b_step = b_kc ? 32u : 2048u;
    bool ok = true;
    const int32_t n_chunks = (p.k_blocks + chunk_kb - 1) / chunk_kb;
#pragma unroll 1
    for (int32_t ch = 0; ch < n_chunks; ++ch) {
        const int32_t kb0 = ch * chunk_kb;
        const int32_t nkb = min(chunk_kb, p.k_blocks - kb0);
        if (d.vec) {
            // The whole chunk in one round: at most 3 x DIRECT_KB 16-byte
            // loads a thread, then the stores.
            uint4 ua[DIRECT_KB][BM / 64], ub[DIRECT_KB][DIRECT_BN / 64];
#pragma unroll
            for (int32_t kb = 0; kb < DIRECT_KB; ++kb) {
                if (kb < nkb) {  // uniform
                    load_image_v4<BM, A_KC>(opA, (kb0 + kb) * BK, p.K, tid, ua[kb]);
                    load_image_v4<DIRECT_BN, B_KC>(opB, (kb0 + kb) * BK, p.K, tid, ub[kb]);
                }
            }
#pragma unroll
            for (int32_t kb = 0; kb < DIRECT_KB; ++kb) {
                if (kb < nkb) {
                    store_image_v4<BM, A_KC>(sA + static_cast<uint32_t>(kb) * D_A_KB, tid, ua[kb]);
                    store_image_v4<DIRECT_BN, B_KC>(sB + static_cast<uint32_t>(kb) * D_B_KB, tid, ub[kb]);
                }
            }
        }
        // Otherwise two k-blocks a round: all 48 loads of this thread, then its stores.
#pragma unroll 1
        for (int32_t kb = 0; kb < (d.vec ? 0 : nkb); kb += 2) {
            const bool two = kb + 1 < nkb;  // uniform
            const int32_t kbase = (kb0 + kb) * BK;
            uint32_t va0[BM * BK / DIRECT_THREADS], vb0[DIRECT_BN * BK / DIRECT_THREADS];
            uint32_t va1[BM * BK / DIRECT_THREADS], vb1[DIRECT_BN * BK / DIRECT_THREADS];
            load_image<BM, A_KC>(opA, kbase, p.K, tid, va0);
            load_image<DIRECT_BN, B_KC>(opB, kbase, p.K, tid, vb0);
            if (two) {
                load_image<BM, A_KC>(opA, kbase + BK, p.K, tid, va1);
                load_image<DIRECT_BN, B_KC>(opB, kbase + BK, p.K, tid, vb1);
            }
            store_image<BM, A_KC>(sA + static_cast<uint32_t>(kb) * D_A_KB, tid, va0);
            store_image<DIRECT_BN, B_KC>(sB + static_cast<uint32_t>(kb) * D_B_KB, tid, vb0);
            if (two) {
                store_image<BM, A_KC>(sA + static_cast<uint32_t>(kb + 1) * D_A_KB, tid, va1);
                store_image<DIRECT_BN, B_KC>(sB + static_cast<uint32_t>(kb + 1) * D_B_KB, tid, vb1);
            }
        }
        ptx::fence_proxy_async_smem();  // the generic-proxy writes, before the MMAs read them
        __syncthreads();
        if (ch == 0 && tid == 0) stamp(2);
        if (warp == 0) {
            if (ptx::elect_one()) {
                ptx::tc_fence_after();
                for (int32_t kb = 0; kb < nkb; ++kb) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = a_desc0 | (((sA + kb * D_A_KB + kk * a_step) >> 4) & 0x3FFFu);
                        const uint64_t bd = b_desc0 | (((sB + kb * D_B_KB + kk * b_step) >> 4) & 0x3FFFu);
                        ptx::mma_bf16(tmem_base, ad, bd, idesc, (ch > 0 || kb > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                ptx::mma_commit(mma_bar);
            }
            __syncwarp();
        }
        // The commit also frees the staging area for the next chunk.
        ok = __syncthreads_and(direct_wait(mma_bar, static_cast<uint32_t>(ch) & 1u, p.timeout_ns) ? 1 : 0) != 0;
        if (!ok) {
            if (tid == 0) atomicCAS(p.err, 0u, static_cast<uint32_t>(ERR_TIMEOUT_MMA));
            break;
        }
        ptx::tc_fence_after();
    }
    if (tid == 0) stamp(3);

    if (ok && DEBUG_CHECKS && p.debug_stall == 2) {
        // Self-test of the consistency checks' reporting path (a planted
        // failed check): nothing is stored.
        if (tid == 0 && atomicCAS(p.err, 0u, static_cast<uint32_t>(ERR_DEBUG_CHECK)) == 0u)
            atomicExch(p.err + 1, static_cast<uint32_t>(CHK_PLANTED));
        ok = false;
    } else if (ok && p.debug_stall) {
        // Watchdog self-test: a barrier that nothing ever completes.
        ok = __syncthreads_and(direct_wait(stall_bar, 0, p.timeout_ns) ? 1 : 0) != 0;
        if (!ok && tid == 0) atomicCAS(p.err, 0u, static_cast<uint32_t>(ERR_TIMEOUT_EPILOGUE));
    }
    if (ok && warp < 8) {
        if (tid == 0) stamp(4);
        // warp w: tensor-memory lanes (rows) 32 (w mod 4) .., columns 32 (w / 4) ..
        const int q = warp & 3, cb = warp >> 2;
        uint32_t v[32];
        ptx::tmem_load_32cols(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(cb * 32), v);
        const int32_t row0 = m0 + q * 32, col0 = n0 + cb * 32;
        if (row0 < p.M && col0 < p.N) {
            if constexpr (FUSED) apply_epilogue(p, v, row0 + lane, col0, b);
            // Transpose through this warp's 4 KB box (the staging area is
            // free: every MMA that read it has completed): row `lane` of the
            // block goes in as eight 16-byte units (unit j at j ^ (lane mod 8)),
            // then lane l reads column l of each row.
            const uint32_t box = sA + static_cast<uint32_t>(warp) * (EPI_CHUNK * EPI_CHUNK * 4);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ptx::st_shared_v4(box + lane * 128 + ((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                  v[4 * j + 3]);
            __syncwarp();
            const int32_t col = col0 + lane;
            const int32_t nrows = min(32, p.M - row0);
            const uint32_t src = box + ((lane >> 2) << 4) + ((lane & 3) << 2);
            const int64_t off = static_cast<int64_t>(b) * p.strideC + static_cast<int64_t>(row0) * p.ldc + col;
#pragma unroll 1
            for (int r0 = 0; r0 < 32; r0 += 8) {
                float vals[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) vals[r] = ld_shared_f32((src ^ (((r0 + r) & 7) << 4)) + (r0 + r) * 128);
                if (col < p.N) {
                    if (FUSED && p.out_bf16) {  // bf16 output only through the fused epilogue
                        uint16_t *dst = static_cast<uint16_t *>(p.C) + off;
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            if (r0 + r < nrows)
                                dst[static_cast<int64_t>(r0 + r) * p.ldc] = __bfloat16_as_ushort(__float2bfloat16_rn(vals[r]));
                    } else {
                        float *dst = static_cast<float *>(p.C) + off;
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            if (r0 + r < nrows) dst[static_cast<int64_t>(r0 + r) * p.ldc] = vals[r];
                    }
                }
            }
        }
        if (tid == 0) stamp(5);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, DIRECT_TMEM_COLS);
    }
    if (tid == 0) {
        stamp(6);
        stamp(7);
    }
}

}  // namespace

cudaError_t launch_direct(const KernelParams &p, const void *A, const void *B, int64_t lda, int64_t ldb,
                          int64_t sA, int64_t sB, int chunk_kb, bool vec, int64_t grid, cudaStream_t s)
{
    if (chunk_kb < 1 || chunk_kb > DIRECT_KB || grid < 1 || grid > INT32_MAX) return cudaErrorInvalidValue;
    const int smem = direct_smem_bytes(chunk_kb);
    using Kern = void (*)(const KernelParams, const DirectArgs);
    static const Kern kernels[8] = {
        direct_gemm_kernel<false, false, false>, direct_gemm_kernel<false, false, true>,
        direct_gemm_kernel<false, true, false>,  direct_gemm_kernel<false, true, true>,
        direct_gemm_kernel<true, false, false>,  direct_gemm_kernel<true, false, true>,
        direct_gemm_kernel<true, true, false>,   direct_gemm_kernel<true, true, true>};
    const int which = (p.a_mn == 0 ? 4 : 0) + (p.b_k != 0 ? 2 : 0) + (p.fused ? 1 : 0);
    const Kern kern = kernels[which];
    // the shared-memory opt-in is per kernel and device; set it once
    static std::atomic<unsigned long long> configured[8] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(configured[which].load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, direct_smem_bytes(DIRECT_KB));
        if (e != cudaSuccess) return e;
        configured[which].fetch_or(bit, std::memory_order_acq_rel);
    }
    const DirectArgs d{A, B, lda, ldb, sA, sB, chunk_kb, vec ? 1 : 0};
    // Programmatic dependent launch, as for the persistent kernel: set-up
    // (barriers, tensor memory) may overlap the previous kernel's tail.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(DIRECT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, d);
}

}  // namespace tg
