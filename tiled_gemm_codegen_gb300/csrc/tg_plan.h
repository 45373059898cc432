// Host-side planning of one GEMM call: tile width, ring depth, K splits,
// persistent grid, pack and epilogue decisions.  Pure integer logic, no CUDA
// calls, so tg_plan() can run (and be tested) on a machine without a GPU.
//
// Tiling is OCANNL "Module Ir.Schedule" Split applied to the three loops:
// ceil(M/BM) x ceil(N/BN) output tiles per problem and ceil(K/BK) k-blocks;
// the fringe tiles are padded to the tile (Pad-to-tile) by TMA zero fill.
// The K split is the two-pass split reduction of the same page: k-blocks
// [floor(s*KB/S), floor((s+1)*KB/S)) go to split s.
#pragma once

#include <algorithm>
#include <climits>
#include <cstdint>

#include "tg_internal.h"

namespace tg {

// Widths that have a two-SM (cta_group::2) variant: each CTA of the pair
// loads BN/2 columns of B, which must be whole 64-column boxes.
constexpr bool pair_width(int bn) { return bn == 128 || bn == 256; }

// Ring depths instantiated for each tile width (kept small for build time).
// 8-bit operands (f8): two-SM tiles of width 256 and one-CTA tiles of widths
// 128, 192 and 256 only.
constexpr bool stage_supported(int bn, int s, bool pair = false, bool f8 = false)
{
    if (f8) {
        if (pair) return bn == 256 && (s == 2 || s == 4 || s == 6);
        return (bn == 128 && (s == 2 || s == 4 || s == 6)) || (bn == 192 && (s == 2 || s == 4)) ||
               (bn == 256 && (s == 2 || s == 4));
    }
    if (pair) {
        switch (bn) {
            case 128: return s == 2 || s == 4 || s == 8;
            case 256: return s == 2 || s == 4 || s == 6;
            default: return false;
        }
    }
    switch (bn) {
        case 64: return s == 2 || s == 4 || s == 6 || s == 8;
        case 128: return s == 2 || s == 3 || s == 4 || s == 6;
        case 192: return s == 2 || s == 3 || s == 4;
        case 256: return s == 2 || s == 3 || s == 4;
        default: return false;
    }
}

// Outputs of at most 64 rows (one CTA per tile, bf16 or unscaled 8-bit):
// ring slots of 64 rows of A, as deep as shared memory allows - 8 slots at
// width 128, 6 at width 192 (0: no such instance).
constexpr int half_a_stages(int bn) { return bn == 128 ? 8 : bn == 192 ? 6 : 0; }

// Block-scaled operands: one-CTA tiles of widths 128, 192 and 224, rings 2
// and 4; with packed 4-bit elements (fp4) the 224-wide tiles ring 2 only
// (every slot's scales take twice the tensor-memory columns).
constexpr bool mx_stage_supported(int bn, int s, bool pair = false, bool fp4 = false)
{
    if (pair || !(bn == 128 || bn == 192 || bn == 224) || !(s == 2 || s == 4)) return false;
    return !(fp4 && bn == 224 && s != 2);
}

template <bool PAIR>
constexpr int max_stages_t(int bn)
{
    return bn == 64 ? Geometry<64, PAIR>::MAX_STAGES
           : bn == 128 ? Geometry<128, PAIR>::MAX_STAGES
           : bn == 192 ? Geometry<192, PAIR>::MAX_STAGES
           : bn == 256 ? Geometry<256, PAIR>::MAX_STAGES
                       : 0;
}

constexpr int max_stages(int bn, bool pair = false)
{
    return pair ? max_stages_t<true>(bn) : max_stages_t<false>(bn);
}

static_assert(stage_supported(64, max_stages(64)), "deepest ring of BN=64 instantiated");
static_assert(stage_supported(128, max_stages(128)), "deepest ring of BN=128 instantiated");
static_assert(stage_supported(192, max_stages(192)), "deepest ring of BN=192 instantiated");
static_assert(stage_supported(256, max_stages(256)), "deepest ring of BN=256 instantiated");
static_assert(stage_supported(128, max_stages(128, true), true), "deepest pair ring of BN=128");
static_assert(stage_supported(256, max_stages(256, true), true), "deepest pair ring of BN=256");
static_assert(Geometry<128, false, true>::smem_bytes(8) <= SMEM_LIMIT, "half-height A ring, width 128");
static_assert(Geometry<192, false, true>::smem_bytes(6) <= SMEM_LIMIT, "half-height A ring, width 192");

template <bool PAIR>
constexpr int smem_bytes_t(int bn, int stages)
{
    return bn == 64 ? Geometry<64, PAIR>::smem_bytes(stages)
           : bn == 128 ? Geometry<128, PAIR>::smem_bytes(stages)
           : bn == 192 ? Geometry<192, PAIR>::smem_bytes(stages)
                       : Geometry<256, PAIR>::smem_bytes(stages);
}

constexpr int smem_bytes_for(int bn, int stages, bool pair = false)
{
    return pair ? smem_bytes_t<true>(bn, stages) : smem_bytes_t<false>(bn, stages);
}

constexpr int tmem_cols_for(int bn)
{
    return bn == 64 ? Geometry<64>::TMEM_COLS
           : bn == 128 ? Geometry<128>::TMEM_COLS
           : bn == 192 ? Geometry<192>::TMEM_COLS
                       : Geometry<256>::TMEM_COLS;
}

// Direct-load kernel (tg_direct.cu) for small problems: one CTA of 512
// threads per 128 x 64 output tile, the operands copied into shared memory
// by the threads themselves (any pitch and alignment), DIRECT_KB k-blocks at
// a time, the accumulator in 64 tensor-memory columns.
constexpr int DIRECT_BN = 64;
constexpr int DIRECT_KB = 4;
constexpr int DIRECT_THREADS = 512;
constexpr int DIRECT_TMEM_COLS = 64;
// Staging area (or the epilogue's eight 4 KB transpose boxes, which reuse
// it), 1 KB of alignment slack, two barriers and the tensor-memory address.
constexpr int direct_smem_bytes(int chunk_kb)
{
    const int stage = chunk_kb * (BM * BK * 2 + DIRECT_BN * BK * 2);
    const int epi = 8 * EPI_CHUNK * EPI_CHUNK * 4;
    return (stage > epi ? stage : epi) + 1024 + 64;
}
// At least 33 KB of shared memory a CTA keeps the CTAs resident on one SM
// (228 KB of shared memory, 1 KB reserved per CTA) at most 6, so their
// tensor-memory allocations never exceed the SM's 512 columns (an
// allocation would otherwise wait for another CTA to free its columns).
static_assert((233472 / (direct_smem_bytes(1) + 1024)) * DIRECT_TMEM_COLS <= 512, "direct kernel: tensor memory");
static_assert(direct_smem_bytes(DIRECT_KB) <= SMEM_LIMIT, "direct kernel: shared memory");

struct PlanInput {
    int64_t M, N, K, batch;
    bool a_tma_ok, b_tma_ok, c_tma_ok;  // 16-byte alignment of base and strides
    bool a_bcast, b_bcast;               // batch stride 0 with batch > 1
    int sm_count;
    // overrides (0 = choose)
    int block_n, stages, split_k, force_pack, epilogue, max_ctas;
    int cta_pair;  // 0 = choose, 1 = one CTA per tile, 2 = two-SM tiles
    int stream_k;  // 0 = choose, 1 = off, 2 = on (when the last wave is partial)
    bool a_cm = false, b_cm = false;  // column-major (transposed) operand storage
    bool f8 = false;                  // 8-bit floating-point A and B (K-major)
    bool mx = false;                  // f8 with per-32-element E8M0 block scales
    bool fp4 = false;                 // mx with packed 4-bit elements (K, lda, ldb in bytes)
    bool half_a_ok = true;            // M <= 64 may use slots of 64 rows of A
    int direct = 0;                   // direct-load kernel: 0 = choose, 1 = off, 2 = on
};

struct Plan {
    bool pair = false;  // two-SM tiles (256 rows, cluster of 2)
    bool f8 = false;    // 8-bit operands: 128 elements of K per k-block
    bool mx = false;    // block-scaled 8-bit operands
    bool fp4 = false;   // block-scaled packed 4-bit operands (a k-block: 256 elements)
    bool half_a = false;  // ring slots of 64 rows of A (M <= 64, one CTA per tile)
    bool direct = false;  // direct-load kernel (stages = k-blocks staged at once)
    int bn = 0, stages = 0;
    int tiles_m = 0, tiles_n = 0, k_blocks = 0, splits = 1;
    int64_t units = 0;
    int grid = 0;
    bool pack_a = false, pack_b = false;
    int epilogue = 1;  // 1 TMA store, 2 plain stores
    int smem = 0, tmem = 0;
    int group_m = 8;
    // stream-K schedule (see KernelParams)
    bool stream_k = false;
    int dp_waves = 0, maxparts = 1, sk_workers = 0;
    int64_t sk_first_tile = 0, sk_tiles = 0, sk_iters = 0;
    int64_t ws_pack_a = 0, ws_pack_b = 0, ws_partials = 0, ws_counters = 0;
    // block-scaled operands: the scales re-arranged into 512-byte blocks
    // (one per 128 rows or columns, k-block and four runs), A's then B's
    int64_t ws_scales_a = 0, ws_scales_b = 0;
    int64_t workspace() const
    {
        return ws_pack_a + ws_pack_b + ws_partials + ws_counters + ws_scales_a + ws_scales_b;
    }
};

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Row pitch (elements) of a packed bf16 operand: a multiple of 64 elements,
// so that every row starts on a 128-byte line.  A 16-byte-aligned pitch is
// enough for the TMA unit, but rows that straddle lines cost the loads an
// extra sector each (4096^3 with A rows of 8208 bytes instead of 8192: 4.4
// us slower).
inline int64_t pack_pitch(int64_t cols) { return round_up(cols, 64); }

// Stream-K schedule of `tiles` tiles of `kb` k-blocks on `workers` workers:
// whole tiles for dp_waves full waves, then the remaining sk_tiles tiles'
// k-blocks split into sk_workers contiguous ranges.  When P = workers /
// sk_tiles is at least 2, sk_workers = P * sk_tiles: every shared tile is cut
// into P equal parts and no range crosses a tile (each of those workers has
// one partial unit); otherwise all workers share the k-blocks evenly.
// Measured on GB300 against the even split over all workers: 4096^3 81.9 ->
// 79.9 us, 4096 x 1536 x 4096 49.2 -> 41.0, 4096 x 2816 x 4096 61.4 -> 59.4,
// 8192^3 501.8 -> 499.7; E4M3 4096^3 65.5 -> 53.3 (55.3 without stream-K).
// maxparts = the largest number of ranges one tile meets (its partial
// slots).  Returns false when the last wave is already full.
struct SkSchedule {
    int dp_waves = 0, maxparts = 1, sk_workers = 0;
    int64_t sk_first_tile = 0, sk_tiles = 0, sk_iters = 0;
};

inline int64_t sk_owner_host(int64_t x, int64_t workers, int64_t iters)
{
    const int64_t w = ((x + 1) * workers - 1) / iters;
    return w < workers - 1 ? w : workers - 1;
}

inline bool sk_schedule(int64_t tiles, int64_t kb, int64_t workers, SkSchedule &out)
{
    if (workers <= 1 || tiles % workers == 0 || kb < 1) return false;
    SkSchedule s;
    s.dp_waves = static_cast<int>(tiles / workers);
    s.sk_first_tile = static_cast<int64_t>(s.dp_waves) * workers;
    s.sk_tiles = tiles - s.sk_first_tile;
    s.sk_iters = s.sk_tiles * kb;
    const int64_t parts = std::min<int64_t>(workers / s.sk_tiles, kb);
    s.sk_workers = static_cast<int>(parts >= 2 ? parts * s.sk_tiles : workers);
    int maxp = 1;
    for (int64_t ts = 0; ts < s.sk_tiles; ++ts) {
        const int64_t first = sk_owner_host(ts * kb, s.sk_workers, s.sk_iters);
        const int64_t last = sk_owner_host((ts + 1) * kb - 1, s.sk_workers, s.sk_iters);
        maxp = std::max<int>(maxp, static_cast<int>(last - first + 1));
    }
    s.maxparts = maxp;
    out = s;
    return true;
}

// Cost model (nanoseconds) used to rank candidate plans.  The MMA time of a
// k-block is 2*BM*BN*BK flops per SM at the SM's share of the dense bf16
// peak, divided by an efficiency.  One-CTA efficiencies are the measured
// in-wave rates on GB300 (4096^3): a k-block costs a near-constant ~250 ns of
// operand ingest plus the MMA time, so narrow tiles waste most of it.  A
// two-SM tile halves the B bytes each SM ingests per k-block.  Work is
// spread over `workers` = SMs (one CTA per tile) or SMs/2 (two-SM tiles).
// The memory time is the unique A/B/C bytes plus split-K partial traffic at
// the lower of HBM bandwidth and what the active SMs can pull.
// 8-bit operands: a k-block holds twice the K at twice the MMA rate, so its
// ideal time is the bf16 one; their measured rates (E4M3, GB300) favour
// two-SM 256-wide tiles once K >= 2048 and the tiles fill a wave (4096^3
// 8% faster, 8192^3 and 8192x8192x2048 4% faster), one-CTA 256-wide tiles
// below that (K = 1024: two-SM tiles 12% slower; 2048^3, under one wave of
// pairs: 9% slower).
inline double tile_efficiency(int bn, bool pair, bool f8 = false, int k_blocks = 0)
{
    if (f8) {
        if (pair) return bn >= 256 ? (k_blocks >= 16 ? 0.89 : 0.78) : 0.50;
        return bn >= 256 ? 0.80 : bn >= 224 ? 0.75 : bn >= 192 ? 0.70 : 0.62;
    }
    // measured in-wave rates on GB300 (fraction of the measured bf16 peak)
    if (pair) return bn >= 256 ? 0.97 : 0.53;
    return bn >= 256 ? 0.80 : bn >= 192 ? 0.645 : bn >= 128 ? 0.54 : 0.29;
}

inline double plan_cost_ns(const PlanInput &in, int bn, bool pair, int splits, int k_blocks,
                           int64_t tiles, int sms, bool stream_k = false)
{
    const double sm_flops = 1.95e15 / 152.0;  // per-SM dense bf16, flop/s
    const double kb_ns = (2.0 * BM * bn * BK) / sm_flops * 1e9 / tile_efficiency(bn, pair, in.f8, k_blocks);
    const int64_t workers = pair ? std::max(1, sms / 2) : sms;
    const int64_t units = tiles * splits;
    double t_mma = 0.0, partial = 0.0;
    if (stream_k) {
        // whole waves, then the busiest share of the remaining k-blocks:
        // a P-th of a tile when they are cut into P >= 2 parts a tile
        // (sk_schedule), else an even share over all workers
        const int64_t dp = tiles / workers;
        const int64_t sk_tiles = tiles - dp * workers;
        const int64_t parts = sk_tiles > 0 ? std::min<int64_t>(workers / sk_tiles, k_blocks) : 0;
        const int64_t share = parts >= 2 ? ceil_div(k_blocks, parts) : ceil_div(sk_tiles * k_blocks, workers);
        t_mma = (static_cast<double>(dp * k_blocks) + static_cast<double>(share)) * kb_ns;
        partial = 2.0 * 4.0 * (pair ? 2 : 1) * BM * bn * 2.0 * static_cast<double>(tiles - dp * workers);
    } else {
        const int64_t waves = ceil_div(units, workers);
        const int64_t kb_unit = ceil_div(k_blocks, splits);
        t_mma = static_cast<double>(waves) * static_cast<double>(kb_unit) * kb_ns;
        partial = splits > 1 ? 2.0 * 4.0 * in.batch * in.M * in.N * splits : 0.0;
    }
    const double ab = (in.f8 ? 1.0 : 2.0) * in.batch * (in.M * in.K + in.K * in.N);
    const double c = 4.0 * in.batch * in.M * in.N;
    const int64_t active_sms = std::min<int64_t>(units, workers) * (pair ? 2 : 1);
    const double bw = std::min(6.5e12, static_cast<double>(active_sms) * 50e9);
    const double t_mem = (ab + c + partial) / bw * 1e9;
    const double fixup = (splits > 1 || stream_k) ? 2000.0 : 0.0;
    return (t_mma > t_mem ? t_mma : t_mem) + fixup;
}

// Whether the planner may pick two-SM tiles on its own (otherwise only when
// asked with cta_pair = 2).
constexpr bool PAIR_BY_DEFAULT = true;

// Split-K / stream-K scratch, kept per 128-row (half-)tile.
inline void set_partial_workspace(const PlanInput &in, Plan &p)
{
    const int64_t per_tile = p.pair ? 2 : 1;
    int64_t slot_tiles = 0;
    if (p.stream_k)
        slot_tiles = p.sk_tiles;
    else if (p.splits > 1)
        slot_tiles = in.batch * p.tiles_m * static_cast<int64_t>(p.tiles_n);
    p.ws_partials = slot_tiles * per_tile * p.maxparts * BM * static_cast<int64_t>(p.bn) * 4;
    p.ws_counters = slot_tiles > 0 ? round_up(slot_tiles * per_tile * 4, 256) : 0;
}

// Re-derives the stream-K schedule for the grid actually launched (the
// co-resident cluster limit can lower it); false if it no longer applies.
inline void replan_stream_k(const PlanInput &in, Plan &p, int grid)
{
    if (!p.stream_k) return;
    const int64_t workers = grid / (p.pair ? 2 : 1);
    const int64_t tiles_total = in.batch * p.tiles_m * static_cast<int64_t>(p.tiles_n);
    SkSchedule sk;
    if (sk_schedule(tiles_total, p.k_blocks, workers, sk)) {
        p.dp_waves = sk.dp_waves;
        p.sk_first_tile = sk.sk_first_tile;
        p.sk_tiles = sk.sk_tiles;
        p.sk_iters = sk.sk_iters;
        p.maxparts = sk.maxparts;
        p.sk_workers = sk.sk_workers;
    } else {
        p.stream_k = false;
        p.maxparts = p.splits;
    }
    set_partial_workspace(in, p);
}

// The planner's own choice of the direct-load kernel: at most one tile per
// SM and few k-blocks, where one short launch beats the persistent kernel's
// set-up and, for operands the TMA unit cannot address, its realign pass.
// How many k-blocks pay depends on how the kernel stages the operands:
// 16-byte units when both are 16-byte aligned with a contiguous extent that
// is a multiple of 8 elements, else single elements (~1.2 us a k-block).
// Measured (GB300, CUDA events, L2 flushed; direct / persistent, us):
// 16-byte units - 128^3 8.2 / 12.3, 256^3 10.1 / 12.3, 512^3 12.3 / 14.3,
// 1024 x 1024 x 256 10.2 / 12.3, 64 x 4096 x 512 12.3 / 12.3, 128 x 128 x
// 1024 (16 k-blocks) 16.4 / 16.4, 256 x 256 x 2048 24.6 / 16.4, 2048^2 x 128
// (512 tiles) 20.5 / 16.4; single elements with operands the TMA unit
// cannot address (odd pitches) - 197 x 131 x 77 10.2 / 16.4, 129 x 65 x 257
// (5 k-blocks) 12.3 / 16.4, 100 x 300 x 500 (8) 20.5 / 16.3; single
// elements with operands it can - 256^3 (4 k-blocks) 14.3 / 12.3.
inline bool direct_vec(const PlanInput &in)
{
    return in.a_tma_ok && in.b_tma_ok && (in.a_cm ? in.M : in.K) % 8 == 0 && (in.b_cm ? in.K : in.N) % 8 == 0;
}

inline bool direct_pays(const PlanInput &in, int k_blocks, int64_t units, int sms)
{
    if (units > sms) return false;
    if (direct_vec(in)) return k_blocks <= 8;
    const bool realign = !in.a_tma_ok || !in.b_tma_ok;
    return k_blocks <= (realign ? 5 : 2);
}

// Returns false (and leaves `out` unspecified) for an invalid override.
inline bool make_plan(const PlanInput &in, Plan &out)
{
    Plan p;
    p.f8 = in.f8;
    p.mx = in.mx;
    p.fp4 = in.fp4;
    if (in.mx && !in.f8) return false;
    if (in.fp4 && !in.mx) return false;
    const int sms = in.sm_count > 0 ? in.sm_count : 1;
    const int64_t kb = ceil_div(in.K, in.f8 ? 2 * BK : BK);  // a k-block is 128 bytes of K
    if (in.f8 && (in.a_cm || !in.b_cm || in.force_pack || !in.a_tma_ok || !in.b_tma_ok)) return false;
    if (kb > INT32_MAX) return false;
    p.k_blocks = static_cast<int>(kb);

    if (in.block_n != 0 && in.block_n != 64 && in.block_n != 128 && in.block_n != 192 &&
        in.block_n != 256 && !(in.mx && in.block_n == 224))
        return false;
    if (in.mx && in.block_n != 0 && !mx_stage_supported(in.block_n, 2, false, in.fp4)) return false;
    if (in.split_k < 0 || in.stages < 0 || in.max_ctas < 0) return false;
    if (in.epilogue < 0 || in.epilogue > 2) return false;
    if (in.cta_pair < 0 || in.cta_pair > 2) return false;
    if (in.stream_k < 0 || in.stream_k > 2) return false;
    if (in.stream_k == 2 && in.split_k > 1) return false;  // one way of splitting K at a time
    if (in.split_k > 0 && in.split_k > p.k_blocks) return false;
    if (in.cta_pair == 2 && in.block_n != 0 && !pair_width(in.block_n)) return false;

    // Direct-load kernel: bf16 operands and no override but the operand
    // layouts (direct = 2 with another override is an invalid request).
    if (in.direct < 0 || in.direct > 2) return false;
    const int64_t d_tiles_m = ceil_div(in.M, BM), d_tiles_n = ceil_div(in.N, DIRECT_BN);
    const int64_t d_units = in.batch * d_tiles_m * d_tiles_n;
    const bool no_override = in.block_n == 0 && in.stages == 0 && in.split_k == 0 && !in.force_pack &&
                             in.epilogue == 0 && in.cta_pair == 0 && in.stream_k == 0 && in.max_ctas == 0;
    const bool direct_ok = !in.f8 && p.k_blocks >= 1 && d_units <= INT32_MAX &&
                           (in.block_n == 0 || in.block_n == DIRECT_BN) && in.stages == 0 && in.split_k <= 1 &&
                           !in.force_pack && in.epilogue != 1 && in.cta_pair != 2 && in.stream_k != 2 &&
                           in.max_ctas == 0;
    if (in.direct == 2 && !direct_ok) return false;
    if (in.direct == 2 || (in.direct == 0 && direct_ok && no_override && direct_pays(in, p.k_blocks, d_units, sms))) {
        p.direct = true;
        p.bn = DIRECT_BN;
        p.stages = std::min(p.k_blocks, DIRECT_KB);
        p.tiles_m = static_cast<int>(d_tiles_m);
        p.tiles_n = static_cast<int>(d_tiles_n);
        p.splits = 1;
        p.maxparts = 1;
        p.units = d_units;
        p.grid = static_cast<int>(d_units);
        p.epilogue = 2;
        p.smem = direct_smem_bytes(p.stages);
        p.tmem = DIRECT_TMEM_COLS;
        out = p;
        return true;
    }

    struct Cand {
        int bn;
        bool pair;
    };
    // block-scaled: at most 224 columns (two accumulators and the scales
    // fill tensor memory); the cost model picks among the instantiated widths
    const Cand cands_mx[3] = {{224, false}, {192, false}, {128, false}};
    const Cand cands_all[6] = {{256, true}, {128, true}, {256, false}, {192, false}, {128, false}, {64, false}};
    const Cand *cands = in.mx ? cands_mx : cands_all;
    const int n_cands = in.mx ? 3 : 6;
    // The narrowest one-CTA width of this operand family that holds all of N
    // in one tile column (0: none does).
    int cover_bn = 0;
    for (int ci = 0; ci < n_cands; ++ci) {
        const Cand &cd = cands[ci];
        if (cd.pair || cd.bn < in.N) continue;
        if (in.mx ? !mx_stage_supported(cd.bn, 2, false, in.fp4) : !stage_supported(cd.bn, 2, false, in.f8)) continue;
        if (cover_bn == 0 || cd.bn < cover_bn) cover_bn = cd.bn;
    }
    double best = 0.0;
    bool have = false;
    for (int ci = 0; ci < n_cands; ++ci) {
        const Cand &cd = cands[ci];
        if (in.block_n != 0 && cd.bn != in.block_n) continue;
        if (in.cta_pair == 1 && cd.pair) continue;
        if (in.cta_pair == 2 && !cd.pair) continue;
        if (in.cta_pair == 0 && cd.pair && !PAIR_BY_DEFAULT) continue;
        if (in.f8 && !in.mx && !stage_supported(cd.bn, 2, cd.pair, true)) continue;  // no 8-bit instance
        if (in.mx && !mx_stage_supported(cd.bn, 2, cd.pair, in.fp4)) continue;
        // 4-bit block-scaled: 224-wide tiles keep a two-slot ring (every
        // slot's scales take twice the tensor-memory columns), which measured
        // slower than 192-wide tiles with four slots on every shape tried
        // (4096^3 55.3 vs 47.1 us, 8192^3 384 vs 258 us): taken on request only
        if (in.fp4 && cd.bn == 224 && in.block_n != 224) continue;
        if (!in.mx && cd.bn == 224) continue;
        // the planner's own choice of 8-bit two-SM tiles needs a full wave
        // of pairs (measured, see tile_efficiency)
        if (in.f8 && cd.pair && in.cta_pair == 0 &&
            in.batch * ceil_div(in.M, 2 * BM) * ceil_div(in.N, cd.bn) < std::max(1, sms / 2))
            continue;
        // Rules from the default plan against the run-time tuner's best on
        // 20 bf16 and 12 8-bit shapes (GB300), for the planner's own choices
        // only.  Two-SM tiles lost where the pair's 256 rows were half
        // padding (M = 128: 32.8 vs 22.5 us) or a tile has few k-blocks
        // (bf16 batches of 512^3 and 256^3: 24.6 vs 20.5 us; 8-bit 16384^2 x
        // 512: 327 vs 281 us, 2048 x 8192 x 2048: 43.0 vs 39.0 us).  An
        // 8-bit k-block takes half the MMA time of a bf16 one, so the
        // pair's fixed cost per tile needs twice as many of them.  A tile
        // wider than the narrowest width that holds N lost to it (bf16
        // N = 128 in 256-wide tiles: 30.8 vs 22.5 us; 8-bit N = 128 in
        // 192-wide ones: 24.5 vs 20.5 us; MXFP8 N = 128 in 224-wide ones:
        // 30.7 vs 26.3 us), for every operand family.  A two-SM tile that
        // spans all of N shares no B tile worth the pairing (bf16 N = 160 in
        // two-SM 256-wide tiles: 32.8 vs 24.6 us; N = 128 in two-SM 128-wide
        // ones: 26.6 vs 22.5 us).
        if (!in.mx && in.cta_pair == 0 && cd.pair && (in.M <= BM || p.k_blocks < (in.f8 ? 20 : 10))) continue;
        if (!in.mx && in.cta_pair == 0 && cd.pair && in.N <= cd.bn) continue;
        if (in.block_n == 0 && in.cta_pair != 2 && cover_bn != 0 && cd.bn > cover_bn) continue;
        const int tile_m = cd.pair ? 2 * BM : BM;
        const int64_t tiles_m = ceil_div(in.M, tile_m);
        const int64_t tiles_n = ceil_div(in.N, cd.bn);
        const int64_t tiles = in.batch * tiles_m * tiles_n;
        const int64_t workers = cd.pair ? std::max(1, sms / 2) : sms;
        int split_lo = 1, split_hi = 1;
        if (in.split_k > 0) {
            split_lo = split_hi = in.split_k;
        } else if (tiles < workers) {
            // Few tiles: consider splitting K so the grid fills the SMs,
            // keeping at least 8 k-blocks per split.
            split_hi = static_cast<int>(std::min<int64_t>(16, std::max<int64_t>(1, p.k_blocks / 8)));
        }
        for (int s = split_lo; s <= split_hi; ++s) {
            for (int sk = 0; sk < 2; ++sk) {
                const bool use_sk = sk == 1;
                if (use_sk && (s > 1 || in.stream_k == 1 || tiles % workers == 0)) continue;
                // stream-K pays for its partial units only when they are
                // long enough.  Shared tiles cut into P >= 2 parts: at least
                // 16 k-blocks a part (bf16 2048 x 8192 x 2048, 32 k-blocks in
                // halves: 55.3 -> 51.2 us; 4096 x 1536 x 2048 in thirds:
                // 32.8 -> 34.8; E4M3 4096^3 in halves: 55.3 -> 53.3).  An
                // even split over all workers: bf16 with at least 48 k-blocks
                // a tile (64: 90 -> 84 us; 32: 55.2 -> 63.5 and 88.1 -> 96.3),
                // never for 8-bit operands (E4M3 4096^3: 55.3 -> 65.5).
                if (use_sk && in.stream_k != 2) {
                    const int64_t sk_tiles = tiles % workers;
                    const int64_t parts = sk_tiles > 0 ? std::min<int64_t>(workers / sk_tiles, p.k_blocks) : 0;
                    const bool pays = parts >= 2 ? p.k_blocks / parts >= 16 : (!in.f8 && p.k_blocks >= 48);
                    if (!pays) continue;
                }
                if (!use_sk && in.stream_k == 2 && tiles % workers != 0) continue;
                const double c = plan_cost_ns(in, cd.bn, cd.pair, s, p.k_blocks, tiles, sms, use_sk);
                if (!have || c < best * 0.999) {
                    have = true;
                    best = c;
                    p.bn = cd.bn;
                    p.pair = cd.pair;
                    p.splits = s;
                    p.stream_k = use_sk;
                    p.tiles_m = static_cast<int>(tiles_m);
                    p.tiles_n = static_cast<int>(tiles_n);
                }
            }
        }
    }
    if (!have) return false;

    // Ring depth: the deepest instantiated one unless overridden.
    if (in.mx) {
        if (in.stages != 0 && !mx_stage_supported(p.bn, in.stages, p.pair, in.fp4)) return false;
        p.stages = in.stages != 0 ? in.stages : (mx_stage_supported(p.bn, 4, p.pair, in.fp4) ? 4 : 2);
    } else if (in.half_a_ok && in.M <= BM / 2 && !p.pair && half_a_stages(p.bn) != 0 &&
               (in.stages == 0 || in.stages == half_a_stages(p.bn))) {
        // at most 64 rows: half-height A slots, half again as many of them
        // (the ring then keeps ~50% more of B in flight)
        p.half_a = true;
        p.stages = half_a_stages(p.bn);
    } else if (in.stages != 0) {
        if (!stage_supported(p.bn, in.stages, p.pair, in.f8)) return false;
        p.stages = in.stages;
    } else {
        p.stages = max_stages(p.bn, p.pair);
        while (in.f8 && p.stages > 2 && !stage_supported(p.bn, p.stages, p.pair, true)) --p.stages;
    }
    p.units = in.batch * p.tiles_m * static_cast<int64_t>(p.tiles_n) * p.splits;
    const int64_t workers = p.pair ? std::max(1, sms / 2) : sms;
    int64_t w = p.units < workers ? p.units : workers;
    if (in.max_ctas > 0) {
        const int64_t cap = p.pair ? std::max(1, in.max_ctas / 2) : in.max_ctas;
        if (w > cap) w = cap;
    }
    p.grid = static_cast<int>(w * (p.pair ? 2 : 1));
    p.group_m = 8;
    if (p.stream_k) {
        SkSchedule sk;
        const int64_t tiles_total = in.batch * p.tiles_m * static_cast<int64_t>(p.tiles_n);
        if (!sk_schedule(tiles_total, p.k_blocks, w, sk)) {
            p.stream_k = false;  // e.g. max_ctas made the last wave full
        } else {
            p.dp_waves = sk.dp_waves;
            p.sk_first_tile = sk.sk_first_tile;
            p.sk_tiles = sk.sk_tiles;
            p.sk_iters = sk.sk_iters;
            p.maxparts = sk.maxparts;
            p.sk_workers = sk.sk_workers;
        }
    }
    if (!p.stream_k) p.maxparts = p.splits;

    p.pack_a = in.force_pack || !in.a_tma_ok;
    p.pack_b = in.force_pack || !in.b_tma_ok;
    if (in.epilogue == 1 && !in.c_tma_ok) return false;
    p.epilogue = in.epilogue != 0 ? in.epilogue : (in.c_tma_ok ? 1 : 2);
    p.smem = p.half_a ? (p.bn == 128 ? Geometry<128, false, true>::smem_bytes(p.stages)
                                     : Geometry<192, false, true>::smem_bytes(p.stages))
                      : smem_bytes_for(p.bn, p.stages, p.pair);
    p.tmem = tmem_cols_for(p.bn);
    if (p.mx) {
        const int halves = p.fp4 ? 2 : 1;
        p.smem = p.bn == 224   ? Geometry<224>::smem_bytes_mx(p.stages, halves)
                 : p.bn == 192 ? Geometry<192>::smem_bytes_mx(p.stages, halves)
                               : Geometry<128>::smem_bytes_mx(p.stages, halves);
        p.tmem = 512;  // accumulators and the slots' scales
    }

    const int64_t batch_a = in.a_bcast ? 1 : in.batch;
    const int64_t batch_b = in.b_bcast ? 1 : in.batch;
    // pack copies keep the stored layout: rows x pack_pitch(columns)
    const int64_t a_rows = in.a_cm ? in.K : in.M, a_cols = in.a_cm ? in.M : in.K;
    const int64_t b_rows = in.b_cm ? in.N : in.K, b_cols = in.b_cm ? in.K : in.N;
    p.ws_pack_a = p.pack_a ? round_up(batch_a * a_rows * pack_pitch(a_cols) * 2, 256) : 0;
    p.ws_pack_b = p.pack_b ? round_up(batch_b * b_rows * pack_pitch(b_cols) * 2, 256) : 0;
    if (p.mx) {
        const int64_t halves = p.fp4 ? 2 : 1;
        p.ws_scales_a = round_up(batch_a * p.tiles_m * static_cast<int64_t>(p.k_blocks) * 512 * halves, 256);
        p.ws_scales_b = round_up(batch_b * p.tiles_n * static_cast<int64_t>(p.k_blocks) * 512 * halves * ceil_div(p.bn, 128), 256);
    }
    set_partial_workspace(in, p);
    out = p;
    return true;
}

// Pieces of the host-buffer entry point's pipeline: while piece p is
// multiplied, piece p+1 of the streamed operand is copied in and the C of
// piece p-1 copied out.  A piece is always contiguous in host memory, so
// its copy is one 1-D copy: stacked batches split by problem; a single
// problem streams its larger operand if that operand's pieces are
// contiguous - A (row-major) by rows of M, B (column-major) by columns of
// N - in at most MAX_PIECES pieces of at least PIECE_MIN (boundaries on
// multiples of 256, a tile edge).  Otherwise, or for K == 0 or small
// extents: one piece.
struct HostPieces {
    int dim = 0;         // 0 one piece, 1 batch, 2 M (rows of A and C), 3 N (columns of B and C)
    int pieces = 1;
    int64_t extent = 0;  // extent of the split dimension
    int64_t bound(int i) const  // start of piece i (bound(pieces) == extent)
    {
        if (dim == 1) return extent * i / pieces;
        const int64_t b = (extent * i / pieces + 255) / 256 * 256;
        return b < extent ? b : extent;
    }
};

// Most pieces of the host-buffer pipeline (it keeps three events a piece).
constexpr int HOST_MAX_PIECES = 8;

inline HostPieces host_pieces(int64_t M, int64_t N, int64_t K, int64_t batch, bool a_bcast, bool b_bcast,
                              bool a_cm, bool b_cm, bool a_stacked, bool b_stacked)
{
    constexpr int MAX_PIECES = HOST_MAX_PIECES;
    constexpr int64_t PIECE_MIN = 512;
    HostPieces h;
    if (K == 0 || M == 0 || N == 0) return h;
    if (batch > 1) {
        if (a_bcast || b_bcast || !a_stacked || !b_stacked) return h;
        h.dim = 1;
        h.extent = batch;
        h.pieces = static_cast<int>(std::min<int64_t>(batch, MAX_PIECES));
        return h;
    }
    const bool by_m = M * K >= K * N;
    if (by_m ? a_cm : !b_cm) return h;  // that operand's pieces would be strided
    const int64_t ext = by_m ? M : N;
    const int64_t p = std::min<int64_t>(ext / PIECE_MIN, MAX_PIECES);
    if (p < 2) return h;
    h.dim = by_m ? 2 : 3;
    h.extent = ext;
    h.pieces = static_cast<int>(p);
    return h;
}

}  // namespace tg

// Host helpers shared between the library's translation units (defined in
// tg_host.cu).
#include "tg_gemm.h"

namespace tg {
int shared_validate(const void *A, const void *B, const float *C, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t sA, int64_t sB,
                    int64_t sC);
bool shared_plan(const void *A, const void *B, const float *C, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldc, int64_t batch, int64_t sA, int64_t sB,
                 int64_t sC, int sms, const tg_options *opt, Plan *out, PlanInput *in_out);
bool shared_encode_3d(CUtensorMap *m, bool fp32, const void *base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0, uint32_t box1);
uint64_t shared_single_problem_stride(uint64_t rows, uint64_t stride1);
cudaError_t shared_launch_gemm(int bn, const CUtensorMap &ta, const CUtensorMap &tb,
                               const CUtensorMap &tc, const KernelParams &p, int stages, int grid,
                               cudaStream_t s);
cudaError_t shared_zero_fill(float *C, int64_t M, int64_t N, int64_t ldc, int64_t sC, int64_t batch,
                             int sms, cudaStream_t s);
// Defined in tg_noalloc.cu: reads (and clears, returning it in *code) the
// static-scratch entry point's error word on device `dev`.
cudaError_t static_error_take(int dev, cudaStream_t stream, uint32_t *code);
}  // namespace tg
