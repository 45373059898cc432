// Persistent, warp-specialised bf16 -> fp32 GEMM kernel for sm_103a.
//
// One CTA per SM (or one two-CTA cluster per SM pair, PAIR) walks a static
// list of work units (output tile x K split).  Roles (the "Active subsets"
// of one accumulator's producers and consumers, LuisaCompute "Execution
// Nests and coordinates", Logical anchor and execution frontier):
//   warp 0         : TMA producer.  Loads this CTA's A rows [128 x BK]
//                    (K-major) and its B columns [BK x BN or BN/2] (N-major)
//                    of k-block kb into ring slot kb mod STAGES with the
//                    128-byte swizzle; boxes that run past M, N or K are
//                    zero-filled by the TMA unit (OCANNL "Module
//                    Ir.Schedule", Pad-to-tile and Stage: out-of-range slots
//                    hold the additive identity 0).
//   warp 1         : MMA issuer (the leader CTA of a pair).  BK/16
//                    tcgen05.mma per slot into a tensor-memory accumulator;
//                    the first one of a unit overwrites (the zero-initialised
//                    accumulator of OCANNL Privatize).
//                    Both run their loop on all 32 lanes (barrier waits by
//                    every lane, lane 0's result for all: warp-uniform
//                    control flow) and issue from one elect.sync lane.
//   warps 2..5     : epilogue.  tcgen05.ld of the accumulator (warp w reads
//                    TMEM lanes 32*(w%4) ..) into a 128B-swizzled 32 x 32
//                    fp32 box in shared memory, then a TMA store of the box
//                    (clipped at M and N by the hardware) or, when C is not
//                    16-byte aligned, coalesced masked stores of its rows.
// Synchronisation is the issue / completion / release protocol of
// LuisaCompute "Pipelines and stage boundaries" (section "Issue, completion
// and release are different events"):
//   full[s]       : the TMA bytes of slot s landed (expect_tx); in a pair the
//                   leader's full[s] counts the bytes of both CTAs
//   empty[s]      : tcgen05.commit after the slot's MMAs -> TMA may refill s
//                   (pair: multicast to both CTAs)
//   tfull[b]      : tcgen05.commit after a unit's last MMA -> epilogue may
//                   read accumulator buffer b (pair: multicast)
//   tempty[b]     : one arrival per epilogue warp (pair: of both CTAs, on
//                   the leader) after its last tcgen05.ld -> MMA may reuse b
// The ring of STAGES slots generalises OCANNL's pipeline_depth: slot and
// phase are (it mod STAGES, (it / STAGES) & 1), and the values the MMA reads
// do not depend on STAGES, so the result is bitwise independent of it.
//
// Two-SM tiles (PAIR): a cluster of two CTAs computes a 256 x BN tile with
// tcgen05.mma.cta_group::2 (M = 256): each CTA loads its own 128 rows of A
// and half of B's BN columns into its own shared memory (the copies of both
// CTAs complete on the leader's full barrier), and receives its 128 x BN
// accumulator in its own tensor memory.  Per SM this halves the B bytes of
// every k-block (no TMA multicast is used).
//
// Split-K and stream-K (OCANNL "Module Ir.Schedule", Deterministic two-pass
// split reduction): every contributor to a tile writes its fp32 partial
// (half-)tile to scratch, then the last to arrive at the tile's counter sums
// all partials in the fixed k order 0, 1, ..., nparts-1 and stores C.  No
// contributor ever waits for another, so the combine needs no grid-wide
// barrier, and the result is deterministic for a given plan.
//
// Every mbarrier wait is bounded (timeout_ns, %globaltimer).  On expiry the
// waiting role records an error code in the device error word, raises the
// abort flag of its CTA (and of the peer CTA) that makes the other roles
// leave their loops, and every CTA then waits (bounded) for its own TMA
// loads, MMAs and TMA stores in flight, frees its tensor memory and returns.
#pragma once

#include <atomic>

#include "tg_epilogue.cuh"
#include "tg_internal.h"
#include "tg_ptx.cuh"

namespace tg {

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle.
//   bits  0-13 start address >> 4     bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4   bit 46 descriptor version (1)
//   bits 49-51 base offset (0: atoms are 1024-byte aligned)
//   bits 61-63 swizzle mode (2 = 128B)
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma.kind::f16: D fp32 (bits 4-5 = 1),
// A bf16 (bits 7-9 = 1), B bf16 (bits 10-12 = 1), bit 15 = A MN-major,
// bit 16 = B MN-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int M, int N>
__host__ __device__ constexpr uint32_t instr_desc_bf16(bool a_mn, bool b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

struct Unit {
    int32_t b, tm, tn, kb0, kb1;
    int32_t nparts;  // contributors to this output tile (1: store C directly)
    int32_t part;    // this contributor's index, in k order
    int64_t slot;    // tile index of the partial slots and arrival counter
};

// Output tile t -> (problem, tile row, tile column).  Tiles are rasterised in
// groups of group_m tile rows so that concurrently running workers share A
// and B panels in L2.
__device__ __forceinline__ void decode_tile(const KernelParams &p, int64_t t, Unit &w)
{
    const int64_t per_batch = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    w.b = static_cast<int32_t>(t / per_batch);
    const int64_t r = t % per_batch;
    const int64_t group_tiles = static_cast<int64_t>(p.group_m) * p.tiles_n;
    const int32_t g = static_cast<int32_t>(r / group_tiles);
    const int32_t first_m = g * p.group_m;
    const int32_t gsize = min(p.tiles_m - first_m, p.group_m);
    const int32_t in = static_cast<int32_t>(r % group_tiles);
    w.tm = first_m + in % gsize;
    w.tn = in / gsize;
}

// The sequence of work units one worker (a CTA, or a CTA pair) processes.
// Every role of the worker walks its own copy of this iterator and sees the
// same sequence.
//  - split-K / plain: units u = worker + i * workers over tiles x splits;
//    split s of a tile covers k-blocks [s*KB/S, (s+1)*KB/S) (OCANNL two-pass
//    split reduction).
//  - stream-K: first the worker's contiguous range of the stream-K tiles'
//    k-blocks, cut at tile boundaries (the parts of a tile are numbered by
//    the order of their k ranges), then its dp_waves whole tiles.  Only the
//    first sk_workers workers take a range: with P * sk_tiles of them every
//    shared tile is cut into P equal parts and no range crosses a tile.  Shared
//    tiles come first so that their partial writes and combines run in the
//    epilogue while the MMA works on the whole tiles.
struct WorkIter {
    int64_t i;
    int64_t sk_pos, sk_end;
};

__device__ __forceinline__ void work_begin(const KernelParams &p, int64_t worker, int64_t workers,
                                           WorkIter &it)
{
    it.i = 0;
    // workers past sk_workers have no stream-K range
    const int64_t sw = p.sk_workers;
    it.sk_pos = (p.stream_k && worker < sw) ? worker * p.sk_iters / sw : 0;
    it.sk_end = (p.stream_k && worker < sw) ? (worker + 1) * p.sk_iters / sw : 0;
}

// The worker whose stream-K range holds position x (ranges may be empty).
__device__ __forceinline__ int64_t sk_owner(const KernelParams &p, int64_t x, int64_t workers)
{
    const int64_t w = ((x + 1) * workers - 1) / p.sk_iters;
    return w < workers - 1 ? w : workers - 1;
}

__device__ __forceinline__ bool work_next(const KernelParams &p, int64_t worker, int64_t workers,
                                          WorkIter &it, Unit &w)
{
    const int64_t KB = p.k_blocks;
    if (!p.stream_k) {
        const int64_t u = worker + it.i * workers;
        if (u >= p.num_units) return false;
        ++it.i;
        const int32_t split = static_cast<int32_t>(u % p.splits);
        const int64_t t = u / p.splits;
        decode_tile(p, t, w);
        w.kb0 = static_cast<int32_t>((static_cast<int64_t>(split) * KB) / p.splits);
        w.kb1 = static_cast<int32_t>((static_cast<int64_t>(split + 1) * KB) / p.splits);
        w.nparts = p.splits;
        w.part = split;
        w.slot = t;
        return true;
    }
    if (it.sk_pos < it.sk_end) {
        const int64_t ts = it.sk_pos / KB;
        const int64_t tile_end = (ts + 1) * KB;
        const int64_t end = it.sk_end < tile_end ? it.sk_end : tile_end;
        decode_tile(p, p.sk_first_tile + ts, w);
        w.kb0 = static_cast<int32_t>(it.sk_pos - ts * KB);
        w.kb1 = static_cast<int32_t>(end - ts * KB);
        const int64_t first = sk_owner(p, ts * KB, p.sk_workers);
        const int64_t last = sk_owner(p, tile_end - 1, p.sk_workers);
        w.nparts = static_cast<int32_t>(last - first + 1);
        w.part = static_cast<int32_t>(worker - first);
        w.slot = ts;
        it.sk_pos = end;
        return true;
    }
    if (it.i >= p.dp_waves) return false;
    const int64_t t = worker + it.i * workers;
    ++it.i;
    decode_tile(p, t, w);
    w.kb0 = 0;
    w.kb1 = static_cast<int32_t>(KB);
    w.nparts = 1;
    w.part = 0;
    w.slot = t;
    return true;
}

enum WaitResult : int { WAIT_OK = 0, WAIT_TIMEOUT = 1, WAIT_ABORTED = 2 };

struct Watchdog {
    uint64_t timeout_ns;
    volatile int32_t *abort_flag;
    uint32_t *err;
    uint32_t peer_abort;  // cluster address of the peer CTA's abort flag (0: none)
};

// Bounded wait for the phase of parity `parity` of mbarrier `bar`.
__device__ __forceinline__ int wait_bounded(uint32_t bar, uint32_t parity, const Watchdog &wd)
{
    if (ptx::mbar_try_wait(bar, parity)) return WAIT_OK;
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return WAIT_OK;
        if ((it & 15u) == 0) {
            if (*wd.abort_flag) return WAIT_ABORTED;
            if (ptx::global_timer_ns() - t0 > wd.timeout_ns) return WAIT_TIMEOUT;
        }
    }
}

// Bounded wait that ignores the abort flag: used to drain this CTA's own
// asynchronous operations before it exits.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, const Watchdog &wd)
{
    const uint64_t t0 = ptx::global_timer_ns();
    for (uint32_t it = 0;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 15u && ptx::global_timer_ns() - t0 > wd.timeout_ns) {
            atomicCAS(wd.err, 0u, static_cast<uint32_t>(ERR_TIMEOUT_DRAIN));
            return false;
        }
    }
}

// wait_bounded by every lane of a warp, with lane 0's result for all: the
// warp leaves (or stays in) its loop as one.
__device__ __forceinline__ int wait_bounded_warp(uint32_t bar, uint32_t parity, const Watchdog &wd)
{
    const int r = wait_bounded(bar, parity, wd);
    return __shfl_sync(0xffffffffu, r, 0);
}

__device__ __forceinline__ void raise_abort(const Watchdog &wd, uint32_t code)
{
    atomicCAS(wd.err, 0u, code);
    *wd.abort_flag = 1;
    if (wd.peer_abort) ptx::st_cluster_u32(wd.peer_abort, 1u);
    __threadfence_block();
}

#ifdef TG_DEBUG_CHECKS
constexpr bool DEBUG_CHECKS = true;
#else
constexpr bool DEBUG_CHECKS = false;
#endif

// Device-side consistency checks of a library built with TG_DEBUG_CHECKS
// (compiled out otherwise).  A failed check records ERR_DEBUG_CHECK in the
// error word and the check's number in the word after it, and raises the
// abort flag of this CTA (and of the peer CTA); the caller skips the access
// the check guarded and leaves its loop, so the CTA exits through the same
// path as a watchdog expiry.  No trap, no assertion, and the out-of-range
// access itself never happens.
enum : uint32_t {
    CHK_UNIT = 1,           // work unit: k range, tile and problem indices
    CHK_SMEM = 2,           // shared-memory layout inside the dynamic allocation
    CHK_ACC_COLS = 3,       // MMA accumulator columns inside the tensor-memory allocation
    CHK_SCALE_COLS = 4,     // block-scale columns of a ring slot inside the allocation
    CHK_SLOT = 5,           // ring slot index below the ring depth
    CHK_EPI_COLS = 6,       // epilogue tensor-memory loads inside the allocation
    CHK_PARTIAL_WRITE = 7,  // split-K / stream-K partial tile inside the scratch
    CHK_PARTIAL_READ = 8,   // the combine's reads inside the scratch
    CHK_COUNTER = 9,        // tile arrival counter inside the scratch
    CHK_PLANTED = 99,       // debug_stall == 2: a planted failure (tests of the reporting path)
};

__device__ __forceinline__ bool dbg_ok(bool cond, uint32_t which, const Watchdog &wd)
{
    if constexpr (!DEBUG_CHECKS) {
        return true;
    } else {
        if (cond) return true;
        if (atomicCAS(wd.err, 0u, static_cast<uint32_t>(ERR_DEBUG_CHECK)) == 0u) atomicExch(wd.err + 1, which);
        *wd.abort_flag = 1;
        if (wd.peer_abort) ptx::st_cluster_u32(wd.peer_abort, 1u);
        __threadfence_block();
        return false;
    }
}

// All 128 epilogue threads agree on a predicate (named barrier 1).
__device__ __forceinline__ bool epi_all(bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

// OCANNL "Module Ir.Schedule", Epilogue fusion: the elementwise tail of the
// reduction, applied to the final fp32 values of one thread's 32 columns:
//   D = act(alpha * acc + bias[col]) + beta * R[row][col]
// The products and sums are rounded one by one (no fused multiply-add), so
// with no activation or relu the fused result equals, bit for bit, the same
// formula applied in fp32 to the stored product.  Each step is one unrolled
// loop over the 32 values behind a single uniform branch (the activation's
// switch sits outside its loop): this code runs from the instruction cache
// between the accumulator loads, and an unrolled loop with every activation
// inlined into each of its 32 bodies would not fit there.
__device__ __forceinline__ void apply_epilogue(const KernelParams &p, uint32_t (&v)[32], int32_t row,
                                               int32_t col0, int32_t b)
{
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = __fmul_rn(p.alpha, __uint_as_float(v[j]));
    if (p.bias) {
        const float *bp = p.bias + static_cast<int64_t>(b) * p.bias_stride + col0;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (col0 + j < p.N) x[j] = __fadd_rn(x[j], __ldg(bp + j));
    }
    switch (p.act) {
        case 1:
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = activation(x[j], 1);
            break;
        case 2:
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = activation(x[j], 2);
            break;
        case 3:
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = activation(x[j], 3);
            break;
        default:
            break;
    }
    // Rows past M are never stored: their residual is not read.
    if (p.residual && row < p.M) {
        const int64_t off = static_cast<int64_t>(b) * p.strideR + static_cast<int64_t>(row) * p.ldr + col0;
        if (p.out_bf16) {
            const uint16_t *rp = static_cast<const uint16_t *>(p.residual) + off;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (col0 + j < p.N)
                    x[j] = __fadd_rn(x[j], __fmul_rn(p.beta, __uint_as_float(static_cast<uint32_t>(rp[j]) << 16)));
        } else {
            const float *rp = static_cast<const float *>(p.residual) + off;
            if ((reinterpret_cast<uintptr_t>(rp) & 15u) == 0 && col0 + 32 <= p.N) {
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(rp + j);
                    x[j] = __fadd_rn(x[j], __fmul_rn(p.beta, t.x));
                    x[j + 1] = __fadd_rn(x[j + 1], __fmul_rn(p.beta, t.y));
                    x[j + 2] = __fadd_rn(x[j + 2], __fmul_rn(p.beta, t.z));
                    x[j + 3] = __fadd_rn(x[j + 3], __fmul_rn(p.beta, t.w));
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N) x[j] = __fadd_rn(x[j], __fmul_rn(p.beta, rp[j]));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(x[j]);
}

// F8: 8-bit floating-point operands (tcgen05 kind::f8f6f4, formats in
// p.mma_fmt), K-major A and B only; a k-block is then 128 elements (still
// 128 bytes a row) and each of its 4 MMAs takes K = 32.
// MX (with F8, one-CTA tiles 128 rows x 128, 192 or 224 columns): block-scaled
// operands (kind::mxf8f6f4): every 32 consecutive elements of a row of A
// (of a column of B) along K share one E8M0 power-of-two scale.  The scales
// of a k-block come pre-arranged as one 512-byte block per 128 rows of A and
// per 128 columns of B's tile (the byte of row 32g + l and K group j at
// l * 16 + g * 4 + j); the producer bulk-copies them with the slot's
// operands, and the MMA thread moves them to tensor memory (tcgen05.cp)
// ahead of the slot's four MMAs, the j-th of which reads byte j of each
// 32-bit scale cell.  Tensor memory holds the two accumulators (2 x BN
// columns) and every slot's scales (4 columns per block), which is why a
// block-scaled tile is at most 224 wide: 2 x 224 + 4 x 12 = 496 of the 512
// columns (TVM "Tensor Layout", Case study: Blackwell tensor memory).
// FP4 (with MX and F8): packed E2M1 operands, two elements a byte
// (tcgen05 kind::mxf4).  A k-block is still 128 bytes a row, now 256
// elements and eight runs of 32, so each slot carries two scale blocks per
// 128 rows or columns (runs 0-3 and 4-7) and every slot takes twice the
// scale columns; the j-th K = 64 MMA reads block j / 2, bytes 2 (j % 2) and
// 2 (j % 2) + 1 of each cell.  Two accumulators and the scales then fit
// 2 x 224 + 2 x 24 columns with a two-slot ring at width 224.
// HALF_A (outputs of at most 64 rows, one CTA per tile): ring slots of 64
// rows of A (Geometry), loaded as one 64-row box; the MMAs are unchanged.
template <int BN, int STAGES, bool PAIR, bool F8 = false, bool MX = false, bool FP4 = false, bool HALF_A = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const KernelParams p)
{
    using G = Geometry<BN, PAIR, HALF_A>;
    static_assert(!HALF_A || (!PAIR && !MX), "half-height A slots: one CTA per tile");
    // widths that are not a multiple of 64 only with K-major 8-bit B (one box)
    static_assert((BN % 64 == 0 || (F8 && BN % 32 == 0)) && BN >= 64 && BN <= 256, "tile width");
    static_assert(!PAIR || G::B_COLS % 64 == 0, "two-SM tiles need 64-column halves of B");
    static_assert(G::smem_bytes(STAGES) <= SMEM_LIMIT, "shared memory budget");
    static_assert(!MX || (F8 && !PAIR && (BN == 128 || BN == 192 || BN == 224)),
                  "block scaling: one-CTA 128-, 192- or 224-wide tiles");
    static_assert(!FP4 || MX, "4-bit operands are block-scaled");
    constexpr int SF_HALVES = FP4 ? 2 : 1;  // scale blocks per 128 rows and k-block
    static_assert(!MX || G::smem_bytes_mx(STAGES, SF_HALVES) <= SMEM_LIMIT, "shared memory budget (scales)");
    constexpr int TILE_M = PAIR ? 2 * BM : BM;
    constexpr int B_BOXES = G::B_COLS / 64;
    constexpr uint32_t B_BOX_BYTES = BK * 64 * 2;  // one 64-column box of B: 8 KB
    constexpr uint32_t EPI_BOX_BYTES = EPI_CHUNK * EPI_CHUNK * 4;  // 4 KB
    constexpr uint32_t EPI_WARPS_TOTAL = PAIR ? 8 : 4;  // arrivals on tempty per tile
    constexpr int KBLK = F8 ? 2 * BK : BK;              // elements of K per k-block (128 bytes)
    // MX: the scale blocks of a slot (A's 512 B, B's 512 B per 128 columns)
    // travel with its operands; tensor memory holds both accumulators
    // (columns 0 .. 2 BN - 1) and the slots' scales (SF_COLS columns a slot
    // from 2 BN: A's 4, then B's 4 per block).
    constexpr uint32_t SF_STAGE = G::SF_STAGE * SF_HALVES;  // scale bytes a slot
    constexpr uint32_t TX_BYTES = G::STAGE + (MX ? SF_STAGE : 0);
    constexpr uint32_t TMEM_ALLOC = MX ? 512u : static_cast<uint32_t>(G::TMEM_COLS);
    constexpr uint32_t SF_COL0 = 2 * BN;
    constexpr uint32_t SF_COLS = 4 * (1 + G::SF_B_BLOCKS) * SF_HALVES;
    constexpr uint32_t SF_B_COL = 4 * SF_HALVES;  // B's scale columns after A's
    static_assert(!MX || SF_COL0 + SF_COLS * STAGES <= TMEM_ALLOC, "scale columns");

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sA = raw + pad;                  // STAGES x [BM x BK] bf16
    const uint32_t sB = sA + STAGES * G::A_STAGE;   // STAGES x [BK x B_COLS] bf16
    const uint32_t sE = sB + STAGES * G::B_STAGE;   // 4 warps x EPI_BUFS x 4 KB
    uint8_t *bar_area = smem + STAGES * G::STAGE + G::EPI_BYTES;
    const uint32_t bar0 = ptx::smem_addr(bar_area);
    const uint32_t sSF = bar0 + G::BAR_BYTES;  // MX: STAGES x SF_STAGE bytes of scales
    // barrier k lives at bar0 + 8k:
    //   [0, S) full   [S, 2S) empty   2S+{0,1} tfull   2S+{2,3} tempty
    //   2S+4 mma-done   2S+5 stall (never completed)
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t stall_bar = bar0 + 8u * (2 * STAGES + 5);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_area + 8 * (2 * STAGES + 6));
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);
    volatile int32_t *last_flag = reinterpret_cast<volatile int32_t *>(tmem_slot + 2);
    uint32_t *issued_slot = tmem_slot + 3;  // k-block loads this CTA's producer issued
    auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](uint32_t b) { return bar0 + 8u * (2 * STAGES + 2 + b); };

    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = static_cast<int>(threadIdx.x & 31);
    // optional timeline: 8 %globaltimer stamps per CTA
    unsigned long long *trace = p.trace ? p.trace + 8ull * blockIdx.x : nullptr;
    auto stamp = [&](int k) {
        if (trace) trace[k] = ptx::global_timer_ns();
    };
    if (threadIdx.x == 0) stamp(0);
    const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
    const bool leader = rank == 0;
    const int64_t worker = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
    const int64_t n_workers = PAIR ? (gridDim.x >> 1) : gridDim.x;

    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), EPI_WARPS_TOTAL);
        }
        ptx::mbar_init(done_bar, 1);
        ptx::mbar_init(stall_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        *issued_slot = 0;
        ptx::fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB);
        if (p.epi_tma) ptx::prefetch_tensormap(&tmC);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_slot), TMEM_ALLOC);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_slot), TMEM_ALLOC);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync_all();  // both CTAs' barriers exist
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touched only this CTA's shared and tensor memory (and
    // the optional trace); A, B, C and the workspace only after the kernels
    // before this one in the stream are complete and visible.
    ptx::griddep_wait();
    const uint32_t peer_abort =
        PAIR ? ptx::map_to_cta(ptx::smem_addr(const_cast<int32_t *>(abort_flag)), rank ^ 1u) : 0u;
    const Watchdog wd{p.timeout_ns, abort_flag, p.err, peer_abort};
    if (threadIdx.x == 0) stamp(1);
    bool skip_all = false;  // TG_DEBUG_CHECKS: the layout check failed, touch nothing
    if constexpr (DEBUG_CHECKS) {
        if (threadIdx.x == 0) {
            uint32_t dyn = 0;
            asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
            const uint32_t end = MX ? sSF + STAGES * SF_STAGE : bar0 + static_cast<uint32_t>(G::BAR_BYTES);
            dbg_ok(end <= raw + dyn && 8u * (2 * STAGES + 6) + 16u <= static_cast<uint32_t>(G::BAR_BYTES) &&
                       sE + 4u * EPI_BUFS * EPI_BOX_BYTES <= bar0,
                   CHK_SMEM, wd);
        }
        __syncthreads();
        skip_all = *abort_flag != 0;
    }

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        // The whole warp runs the loop (warp-uniform control flow); one
        // elected lane issues the barrier arrivals and the copies.
        {
            uint32_t it = 0;
            bool ok = true;
            // pair: both CTAs' copies complete on the leader's full barrier
            const uint32_t full0 = PAIR ? ptx::map_to_cta(full_bar(0), 0u) : full_bar(0);
            WorkIter wi;
            work_begin(p, worker, n_workers, wi);
            Unit w;
            while (ok && !skip_all && work_next(p, worker, n_workers, wi, w)) {
                if (!dbg_ok(w.kb0 >= 0 && w.kb0 < w.kb1 && w.kb1 <= p.k_blocks && w.tm >= 0 && w.tm < p.tiles_m &&
                                w.tn >= 0 && w.tn < p.tiles_n && w.b >= 0 && w.b < p.batch,
                            CHK_UNIT, wd))
                    break;
                const int32_t zA = p.a_bcast ? 0 : w.b;
                const int32_t zB = p.b_bcast ? 0 : w.b;
                const int32_t m_rows = w.tm * TILE_M + static_cast<int32_t>(rank) * BM;
                const int32_t n_cols = w.tn * BN + static_cast<int32_t>(rank) * G::B_COLS;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    const int r = wait_bounded_warp(empty_bar(s), ph ^ 1u, wd);
                    if (r != WAIT_OK) {
                        if (r == WAIT_TIMEOUT && lane == 0) raise_abort(wd, ERR_TIMEOUT_PRODUCER);
                        ok = false;
                        break;
                    }
                    if (!dbg_ok(s < STAGES, CHK_SLOT, wd)) {
                        ok = false;
                        break;
                    }
                    if (ptx::elect_one()) {
                        // One copy: this CTA's own barrier; a pair: the leader's.
                        uint32_t fb;
                        if constexpr (PAIR) {
                            if (leader) ptx::mbar_arrive_expect_tx(full_bar(s), 2 * G::STAGE);
                            fb = full0 + 8u * s;
                        } else {
                            ptx::mbar_arrive_expect_tx(full_bar(s), TX_BYTES);
                            fb = full_bar(s);
                        }
                        auto load = [&](uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1, int32_t c2) {
                            if constexpr (PAIR)
                                ptx::tma_load_3d_pair(dst, map, fb, c0, c1, c2);
                            else
                                ptx::tma_load_3d(dst, map, fb, c0, c1, c2);
                        };
                        const uint32_t a_dst = sA + s * G::A_STAGE;
                        const uint32_t b_dst = sB + s * G::B_STAGE;
                        if (!p.a_mn) {
                            // A row-major: one box [128 rows x 64 k], K-major atoms
                            load(a_dst, &tmA, kb * KBLK, m_rows, zA);
                        } else {
                            // A column-major: two boxes [64 k x 64 rows], MN-major atoms
                            // (HALF_A: the first only)
                            load(a_dst, &tmA, m_rows, kb * KBLK, zA);
                            if constexpr (!HALF_A) load(a_dst + B_BOX_BYTES, &tmA, m_rows + 64, kb * KBLK, zA);
                        }
                        if (!p.b_k) {
                            // B row-major: boxes [64 k x 64 columns], MN-major atoms
#pragma unroll
                            for (int j = 0; j < B_BOXES; ++j)
                                load(b_dst + j * B_BOX_BYTES, &tmB, n_cols + 64 * j, kb * KBLK, zB);
                        } else {
                            // B column-major: one box [B_COLS columns x 64 k], K-major atoms
                            load(b_dst, &tmB, kb * KBLK, n_cols, zB);
                        }
                        if constexpr (MX) {
                            const int64_t fa = (static_cast<int64_t>(zA) * p.tiles_m + w.tm) * p.k_blocks + kb;
                            const int64_t fbk = (static_cast<int64_t>(zB) * p.tiles_n + w.tn) * p.k_blocks + kb;
                            constexpr uint32_t SFA_BYTES = 512 * SF_HALVES;
                            constexpr uint32_t SFB_BYTES = 512 * G::SF_B_BLOCKS * SF_HALVES;
                            ptx::bulk_load(sSF + s * SF_STAGE, p.sfa + fa * SFA_BYTES, SFA_BYTES, fb);
                            ptx::bulk_load(sSF + s * SF_STAGE + SFA_BYTES, p.sfb + fbk * SFB_BYTES, SFB_BYTES, fb);
                        }
                    }
                    __syncwarp();
                }
            }
            if (lane == 0) {
                *issued_slot = it;
                if constexpr (!PAIR) {
                    // Drain: the last load issued into every slot has landed.
                    const uint32_t first = it > STAGES ? it - STAGES : 0u;
                    for (uint32_t j = first; j < it; ++j)
                        if (!wait_drain(full_bar(j % STAGES), (j / STAGES) & 1u, wd)) break;
                }
            }
            __syncwarp();
        }
    } else if (warp == 1) {
        if (!PAIR || leader) {
            // ------------------------------------------------ MMA issuer
            // The whole warp runs the issue loop, so its control flow is
            // warp-uniform; one elected lane issues the tcgen05 instructions.
            // kind::f8f6f4 keeps the layout of the descriptor; only the A and
            // B format fields (bits 7-12) differ
            const uint32_t idesc_bf16 = instr_desc_bf16<TILE_M, BN>(p.a_mn != 0, p.b_k == 0);
            const uint32_t idesc = F8 ? ((idesc_bf16 & ~(0x3Fu << 7)) | p.mma_fmt) : idesc_bf16;
            // kind::mxf8f6f4: no D format field (bits 4-5 hold B's scale
            // byte), scale type E8M0 (bit 23), A's scale byte at bits 29-30
            const uint32_t idesc_mx = p.mma_fmt | (static_cast<uint32_t>(BN >> 3) << 17) | (1u << 23) |
                                      (static_cast<uint32_t>(TILE_M >> 4) << 24);
            // Layout-dependent descriptor parts, fixed for the whole kernel:
            // a K-major operand steps 32 B per 16 k (leading offset unused);
            // an MN-major one steps 16 rows x 128 B and its 64-element atoms
            // sit one box (BK x 128 B) apart.  Per MMA only the start address
            // changes.
            const uint64_t a_desc0 = smem_desc_sw128(0, p.a_mn ? BK * 128 : 16, 1024);
            const uint64_t b_desc0 = smem_desc_sw128(0, p.b_k ? 16 : BK * 128, 1024);
            const uint32_t a_step = p.a_mn ? 2048u : 32u;
            const uint32_t b_step = p.b_k ? 32u : 2048u;
            uint32_t it = 0, t = 0;
            bool ok = true;
            WorkIter wi;
            work_begin(p, worker, n_workers, wi);
            Unit w;
            for (; ok && !skip_all && work_next(p, worker, n_workers, wi, w); ++t) {
                const uint32_t buf = t & 1u;
                const uint32_t tph = (t >> 1) & 1u;
                if (!dbg_ok(buf * BN + BN <= TMEM_ALLOC, CHK_ACC_COLS, wd)) break;
                int r = wait_bounded_warp(tempty_bar(buf), tph ^ 1u, wd);
                if (r != WAIT_OK) {
                    if (r == WAIT_TIMEOUT && lane == 0) raise_abort(wd, ERR_TIMEOUT_MMA);
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int32_t kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const uint32_t s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    r = wait_bounded_warp(full_bar(s), ph, wd);
                    if (r != WAIT_OK) {
                        if (r == WAIT_TIMEOUT && lane == 0) raise_abort(wd, ERR_TIMEOUT_MMA);
                        ok = false;
                        break;
                    }
                    if (it == 0 && lane == 0) stamp(2);
                    if (!dbg_ok(s < STAGES && (!MX || SF_COL0 + SF_COLS * (s + 1) <= TMEM_ALLOC), CHK_SCALE_COLS, wd)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    if (ptx::elect_one()) {
                        const uint32_t a_addr = sA + s * G::A_STAGE;
                        const uint32_t b_addr = sB + s * G::B_STAGE;
                        const uint32_t sf_tmem = tmem_base + SF_COL0 + SF_COLS * s;
                        if constexpr (MX) {
                            // no-swizzle descriptors of the 512-byte scale
                            // blocks: 8-row core matrices 128 B apart.  A's
                            // blocks (one per half) to columns 4h, then B's
                            // blocks [half][128 columns] to the columns after
                            // them: the slot's blocks in their order in
                            // shared memory, 4 columns each.
                            const uint64_t sf_desc = (static_cast<uint64_t>(128 >> 4) << 16) |
                                                     (static_cast<uint64_t>(128 >> 4) << 32) | (1ull << 46);
                            const uint32_t sf_smem = sSF + s * SF_STAGE;
#pragma unroll
                            for (int j = 0; j < (1 + G::SF_B_BLOCKS) * SF_HALVES; ++j)
                                ptx::tmem_cp_32x128b_x4(sf_tmem + 4 * j, sf_desc | (((sf_smem + 512 * j) >> 4) & 0x3FFFu));
                        }
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk) {
                            const uint64_t ad = a_desc0 | (((a_addr + kk * a_step) >> 4) & 0x3FFFu);
                            const uint64_t bd = b_desc0 | (((b_addr + kk * b_step) >> 4) & 0x3FFFu);
                            const uint32_t acc = (kb > w.kb0 || kk > 0) ? 1u : 0u;
                            if constexpr (FP4) {
                                const uint32_t h = static_cast<uint32_t>(kk) >> 1;
                                const uint32_t id = 2u * (static_cast<uint32_t>(kk) & 1u);
                                ptx::mma_mxf4(d_tmem, ad, bd, idesc_mx | (id << 29) | (id << 4), sf_tmem + 4 * h,
                                              sf_tmem + SF_B_COL + 4 * G::SF_B_BLOCKS * h, acc);
                            } else if constexpr (MX)
                                ptx::mma_mx(d_tmem, ad, bd,
                                            idesc_mx | (static_cast<uint32_t>(kk) << 29) | (static_cast<uint32_t>(kk) << 4),
                                            sf_tmem, sf_tmem + SF_B_COL, acc);
                            else if constexpr (PAIR && F8)
                                ptx::mma_f8_pair(d_tmem, ad, bd, idesc, acc);
                            else if constexpr (PAIR)
                                ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, acc);
                            else if constexpr (F8)
                                ptx::mma_f8(d_tmem, ad, bd, idesc, acc);
                            else
                                ptx::mma_bf16(d_tmem, ad, bd, idesc, acc);
                        }
                        if constexpr (PAIR)
                            ptx::mma_commit_pair_multicast(empty_bar(s), 0x3);
                        else
                            ptx::mma_commit(empty_bar(s));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                // every tcgen05 instruction of the loop comes from the elected
                // lane (elect.sync on the converged warp: the same lane each
                // time), so each commit covers the MMAs before it
                if (ptx::elect_one()) {
                    if constexpr (PAIR)
                        ptx::mma_commit_pair_multicast(tfull_bar(buf), 0x3);
                    else
                        ptx::mma_commit(tfull_bar(buf));
                }
                __syncwarp();
            }
            if (ptx::elect_one()) {
                stamp(3);
                // Every MMA issued above completes before tensor memory is freed.
                if constexpr (PAIR)
                    ptx::mma_commit_pair_multicast(done_bar, 0x1);
                else
                    ptx::mma_commit(done_bar);
                wait_drain(done_bar, 0, wd);
            }
            __syncwarp();
        }
    } else {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // tensor-memory lane quadrant of this warp
        const int row = q * 32 + lane;
        const uint32_t stage_base = sE + static_cast<uint32_t>(q * EPI_BUFS) * EPI_BOX_BYTES;
        const uint32_t tempty_leader0 = PAIR ? ptx::map_to_cta(tempty_bar(0), 0u) : tempty_bar(0);
        uint32_t st_cnt = 0;
        bool ok = true;
        if (DEBUG_CHECKS && p.debug_stall == 2) {
            // Self-test of the consistency checks' reporting path.
            ok = epi_all(dbg_ok(false, CHK_PLANTED, wd));
        } else if (p.debug_stall) {
            // Watchdog self-test: a barrier that nothing ever completes.
            const int r = wait_bounded(stall_bar, 0, wd);
            if (r == WAIT_TIMEOUT) raise_abort(wd, ERR_TIMEOUT_EPILOGUE);
            ok = epi_all(r == WAIT_OK);
        }
        if (skip_all) ok = false;

        // One 32 x 32 fp32 chunk (rows m_base + 32q .., columns col0 ..) of
        // this warp's accumulator rows -> C.
        auto store_chunk = [&](uint32_t (&v)[32], int32_t m_base, int32_t col0, int32_t b) {
            const int32_t row0 = m_base + q * 32;
            if (row0 >= p.M || col0 >= p.N) return;  // warp-uniform
            if (p.fused) apply_epilogue(p, v, row0 + lane, col0, b);
            const uint32_t box = stage_base + (st_cnt % EPI_BUFS) * EPI_BOX_BYTES;
            ++st_cnt;
            if (p.epi_tma && lane == 0) ptx::bulk_wait_group_read<EPI_BUFS - 1>();
            __syncwarp();
            const int32_t col = col0 + lane;
            const int32_t nrows = min(32, p.M - row0);
            // A TMA store clips the row at 16-byte granularity: the box that
            // holds the row's last column writes on to the next 16-byte
            // boundary, into the caller's row padding, unless N ends on one.
            // That box goes out with plain stores instead.
            const int32_t per16 = p.out_bf16 ? 8 : 4;
            const bool tma = p.epi_tma && (col0 + EPI_CHUNK <= p.N || p.N % per16 == 0);
            if (!p.out_bf16) {
                // Row `lane` of the box; its 16-byte unit jj is stored at unit
                // jj ^ (lane mod 8): the 128B swizzle (Swizzle(2,3,3) on fp32).
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    ptx::st_shared_v4(box + lane * 128 + ((jj ^ (lane & 7)) << 4), v[4 * jj],
                                      v[4 * jj + 1], v[4 * jj + 2], v[4 * jj + 3]);
                if (tma) {
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_3d(&tmC, box, col0, row0, b);
                        ptx::bulk_commit_group();
                    }
                } else {
                    __syncwarp();
                    // Coalesced: lane l writes column col0 + l of each row.  Eight
                    // rows a step: their values are read from the box first,
                    // then their stores go out back to back.  The loop is kept
                    // rolled: a small tile's epilogue runs its code once, from a
                    // cold instruction cache.
                    const uint32_t src = box + ((lane >> 2) << 4) + ((lane & 3) << 2);
                    float *dst = static_cast<float *>(p.C) + static_cast<int64_t>(b) * p.strideC +
                                 static_cast<int64_t>(row0) * p.ldc + col;
#pragma unroll 1
                    for (int r0 = 0; r0 < 32; r0 += 8) {
                        float vals[8];
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            vals[r] = ld_shared_f32((src ^ (((r0 + r) & 7) << 4)) + (r0 + r) * 128);
                        if (col < p.N) {
#pragma unroll
                            for (int r = 0; r < 8; ++r)
                                if (r0 + r < nrows) dst[static_cast<int64_t>(r0 + r) * p.ldc] = vals[r];
                        }
                    }
                }
            } else {
                // bf16 output (round to nearest even): a 32 x 32 box of 64-byte
                // rows with the 64B swizzle (Swizzle(3,2,3) on bf16): 16-byte
                // unit u of row r sits at unit u ^ ((r / 2) mod 4).
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(v[2 * k], v[2 * k + 1]);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    ptx::st_shared_v4(box + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4), w[4 * u],
                                      w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                if (tma) {
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_3d(&tmC, box, col0, row0, b);
                        ptx::bulk_commit_group();
                    }
                } else {
                    __syncwarp();
                    const uint32_t src = box + ((lane >> 3) << 4) + ((lane & 7) << 1);
                    uint16_t *dst = static_cast<uint16_t *>(p.C) + static_cast<int64_t>(b) * p.strideC +
                                    static_cast<int64_t>(row0) * p.ldc + col;
#pragma unroll 1
                    for (int r0 = 0; r0 < 32; r0 += 8) {
                        uint16_t vals[8];
#pragma unroll
                        for (int r = 0; r < 8; ++r)
                            vals[r] = ld_shared_u16((src ^ ((((r0 + r) >> 1) & 3) << 4)) + (r0 + r) * 64);
                        if (col < p.N) {
#pragma unroll
                            for (int r = 0; r < 8; ++r)
                                if (r0 + r < nrows) dst[static_cast<int64_t>(r0 + r) * p.ldc] = vals[r];
                        }
                    }
                }
            }
        };

        // Frees accumulator buffer `buf` for the MMA issuer (after this
        // warp's last tcgen05.ld of it).
        auto release_tmem = [&](uint32_t buf) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR)
                    ptx::mbar_arrive_cluster(tempty_leader0 + 8u * buf);
                else
                    ptx::mbar_arrive(tempty_bar(buf));
            }
        };

        uint32_t t = 0;
        WorkIter wi;
        work_begin(p, worker, n_workers, wi);
        Unit w;
        for (; ok && work_next(p, worker, n_workers, wi, w); ++t) {
            const uint32_t buf = t & 1u;
            const uint32_t tph = (t >> 1) & 1u;
            const int r = wait_bounded(tfull_bar(buf), tph, wd);
            if (r == WAIT_TIMEOUT) raise_abort(wd, ERR_TIMEOUT_EPILOGUE);
            if (!epi_all(r == WAIT_OK)) break;
            if (t == 0 && warp == 2 && lane == 0) stamp(4);
            if (!dbg_ok(buf * BN + BN <= TMEM_ALLOC, CHK_EPI_COLS, wd)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
            const int32_t m_base = w.tm * TILE_M + static_cast<int32_t>(rank) * BM;
            const int32_t n_base = w.tn * BN;
            if (w.nparts == 1) {
                // Two register sets: the load of chunk c+1 is in flight while
                // chunk c is staged and stored.
                constexpr int NCH = BN / EPI_CHUNK;
                uint32_t va[32], vb[32];
                ptx::tmem_load_32cols(taddr, va);
#pragma unroll 1
                for (int c = 0; c + 1 < NCH; c += 2) {
                    ptx::tmem_load_32cols_async(taddr + (c + 1) * EPI_CHUNK, vb);
                    store_chunk(va, m_base, n_base + c * EPI_CHUNK, w.b);
                    ptx::tmem_wait_ld(vb);
                    if (c + 2 < NCH) ptx::tmem_load_32cols_async(taddr + (c + 2) * EPI_CHUNK, va);
                    else release_tmem(buf);
                    store_chunk(vb, m_base, n_base + (c + 1) * EPI_CHUNK, w.b);
                    if (c + 2 < NCH) ptx::tmem_wait_ld(va);
                }
                if constexpr (NCH % 2 != 0) {
                    // odd chunk count: the last chunk is in va, loaded above
                    release_tmem(buf);
                    store_chunk(va, m_base, n_base + (NCH - 1) * EPI_CHUNK, w.b);
                }
            } else {
                // Partial (half-)tile -> scratch.  Layout inside one part:
                // [chunk c][column quad j4][row][4 columns], so a warp's 32
                // rows of one column quad are 512 contiguous bytes and every
                // access below is a coalesced 16-byte vector per thread.
                const int64_t half = w.slot * (PAIR ? 2 : 1) + rank;
                constexpr int64_t PART_FLOATS = static_cast<int64_t>(BM) * BN;
                if (!dbg_ok(w.part >= 0 && w.part < w.nparts && w.nparts <= p.maxparts &&
                                (half * p.maxparts + w.part + 1) * PART_FLOATS <= p.partial_floats,
                            CHK_PARTIAL_WRITE, wd) ||
                    !dbg_ok((half * p.maxparts + w.nparts) * PART_FLOATS <= p.partial_floats, CHK_PARTIAL_READ, wd) ||
                    !dbg_ok(half >= 0 && half < p.counter_count, CHK_COUNTER, wd))
                    break;
                const bool row_ok = (m_base + row) < p.M;
                const float4 *ws0 = reinterpret_cast<const float4 *>(
                    p.partials + half * static_cast<int64_t>(p.maxparts) * (BM * BN));
                float4 *mine = reinterpret_cast<float4 *>(p.partials) +
                               (half * static_cast<int64_t>(p.maxparts) + w.part) * (BM * BN / 4);
                constexpr int64_t PART4 = BM * BN / 4;  // float4s per part
#pragma unroll 1
                for (int c = 0; c < BN / EPI_CHUNK; ++c) {
                    uint32_t v[32];
                    ptx::tmem_load_32cols(taddr + c * EPI_CHUNK, v);
                    if (c == BN / EPI_CHUNK - 1) release_tmem(buf);
                    if (row_ok) {
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4)
                            __stcg(mine + (c * 8 + j4) * BM + row,
                                   make_float4(__uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]),
                                               __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3])));
                    }
                }
                __threadfence();
                ptx::named_barrier_sync(1, 128);
                if (warp == 2 && lane == 0) {
                    const int32_t old = atomicAdd(p.counters + half, 1);
                    const int32_t last = (old == w.nparts - 1) ? 1 : 0;
                    if (last) atomicExch(p.counters + half, 0);  // ready for the next call
                    *last_flag = last;
                }
                ptx::named_barrier_sync(1, 128);
                if (*last_flag) {
                    __threadfence();
#pragma unroll 1
                    for (int c = 0; c < BN / EPI_CHUNK; ++c) {
                        float4 acc[8];
                        const float4 *src = ws0 + c * 8 * BM + row;
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4)
                            acc[j4] = row_ok ? __ldcg(src + j4 * BM) : make_float4(0.f, 0.f, 0.f, 0.f);
                        // parts 1 .. nparts-1 in order, two parts' loads in flight
                        int s = 1;
                        for (; row_ok && s + 1 < w.nparts; s += 2) {
                            float4 t0[8], t1[8];
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                t0[j4] = __ldcg(src + s * PART4 + j4 * BM);
                                t1[j4] = __ldcg(src + (s + 1) * PART4 + j4 * BM);
                            }
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                acc[j4].x += t0[j4].x; acc[j4].y += t0[j4].y;
                                acc[j4].z += t0[j4].z; acc[j4].w += t0[j4].w;
                                acc[j4].x += t1[j4].x; acc[j4].y += t1[j4].y;
                                acc[j4].z += t1[j4].z; acc[j4].w += t1[j4].w;
                            }
                        }
                        if (row_ok && s < w.nparts) {
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 t0 = __ldcg(src + s * PART4 + j4 * BM);
                                acc[j4].x += t0.x; acc[j4].y += t0.y; acc[j4].z += t0.z; acc[j4].w += t0.w;
                            }
                        }
                        uint32_t v[32];
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            v[4 * j4] = __float_as_uint(acc[j4].x);
                            v[4 * j4 + 1] = __float_as_uint(acc[j4].y);
                            v[4 * j4 + 2] = __float_as_uint(acc[j4].z);
                            v[4 * j4 + 3] = __float_as_uint(acc[j4].w);
                        }
                        store_chunk(v, m_base, n_base + c * EPI_CHUNK, w.b);
                    }
                }
                ptx::named_barrier_sync(1, 128);
            }
        }
        if (warp == 2 && lane == 0) stamp(5);
        // Every TMA store issued by this warp has read its shared-memory
        // source (the global writes complete with the grid).
        if (lane == 0) ptx::bulk_wait_group_read<0>();
        __syncwarp();
        if (warp == 2 && lane == 0) stamp(6);
    }

    __syncthreads();
    if constexpr (PAIR) {
        // Neither CTA leaves (or frees tensor memory) while the other may
        // still signal its barriers, the leader's MMAs may write its TMEM, or
        // a copy of either CTA may still be landing.  Both producers' issue
        // counts are final after the first cluster barrier; the leader then
        // waits for the latest phase of every slot of its full barriers.  If
        // an abort left the two producers at different counts, it first
        // settles the phases only one of them issued: peer bytes that will
        // never come are counted with complete_tx, and a missing leader
        // arrival is made with expect_tx of the peer's bytes alone.
        ptx::cluster_sync_all();
        if (leader && warp == 0 && lane == 0) {
            const uint32_t i_l = *issued_slot;
            const uint32_t i_p = ptx::ld_cluster_u32(ptx::map_to_cta(ptx::smem_addr(issued_slot), 1u));
            const uint32_t hi = i_l > i_p ? i_l : i_p;
            const uint32_t lo = hi > STAGES ? hi - STAGES : 0u;
            for (uint32_t j = lo; j < hi; ++j) {
                const uint32_t s = j % STAGES;
                if (j < i_l && j >= i_p)
                    ptx::mbar_complete_tx(full_bar(s), G::STAGE);
                else if (j >= i_l && j < i_p)
                    ptx::mbar_arrive_expect_tx(full_bar(s), G::STAGE);
                if (!wait_drain(full_bar(s), (j / STAGES) & 1u, wd)) break;
            }
        }
        ptx::cluster_sync_all();
    }
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        if constexpr (PAIR)
            ptx::tmem_dealloc_pair(tmem_base, TMEM_ALLOC);
        else
            ptx::tmem_dealloc(tmem_base, TMEM_ALLOC);
    }
    if (threadIdx.x == 0) stamp(7);
}

template <int BN, int STAGES, bool PAIR, bool F8 = false, bool MX = false, bool FP4 = false, bool HALF_A = false>
cudaError_t launch_fixed(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                         const KernelParams &p, int grid, cudaStream_t s)
{
    constexpr int smem = MX ? Geometry<BN, PAIR>::smem_bytes_mx(STAGES, FP4 ? 2 : 1)
                            : Geometry<BN, PAIR, HALF_A>::smem_bytes(STAGES);
    static_assert(smem <= SMEM_LIMIT, "shared memory budget");
    auto kern = gemm_kernel<BN, STAGES, PAIR, F8, MX, FP4, HALF_A>;
    // the shared-memory opt-in is per device; set it once per device
    static std::atomic<unsigned long long> configured{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    // Programmatic dependent launch: the kernel may start while the previous
    // kernel of the stream finishes; it sets up (barriers, tensor memory,
    // cluster) and then waits on the grid dependency before its first access
    // to any operand or workspace.
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PAIR ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
}

// Largest number of two-CTA clusters of this configuration that can be
// resident at once (0 if the query fails).
template <int BN, int STAGES, bool F8 = false>
int max_active_pairs()
{
    constexpr int smem = Geometry<BN, true>::smem_bytes(STAGES);
    auto kern = gemm_kernel<BN, STAGES, true, F8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace tg
