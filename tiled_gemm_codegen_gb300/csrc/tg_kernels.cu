// Instantiations of the persistent GEMM kernel: one translation unit per tile
// width (selected at build time with -DTG_BN=...), so the widths compile in
// parallel.  Each width instantiates a few ring depths, with one CTA per tile
// and (widths 128 and 256) two-SM tiles, for bf16 operands and (a subset)
// 8-bit floating-point ones (block-scaled 8-bit and packed 4-bit ones at
// widths 128, 192 and 224, rings 2 and 4 - 224-wide 4-bit tiles ring 2
// only); stage_supported() and
// mx_stage_supported() in tg_plan.h list them and the host planner only
// picks listed configurations.
#include "tg_kernel.cuh"
#include "tg_plan.h"

#ifndef TG_BN
#error "compile with -DTG_BN=<64|128|192|256>"
#endif

namespace tg {

#define TG_CASE(S, PAIR, F8)                                                        \
    case S:                                                                         \
        if constexpr ((!PAIR || pair_width(TG_BN)) && stage_supported(TG_BN, S, PAIR, F8)) \
            return launch_fixed<TG_BN, S, PAIR, F8>(ta, tb, tc, p, grid, s);        \
        else                                                                        \
            return cudaErrorInvalidValue;

#define TG_CASE_PAIRS(S, F8)                                                        \
    case S:                                                                         \
        if constexpr (pair_width(TG_BN) && stage_supported(TG_BN, S, true, F8))     \
            return max_active_pairs<TG_BN, S, F8>();                                \
        else                                                                        \
            return 0;

#define TG_CAT2(a, b) a##b
#define TG_CAT(a, b) TG_CAT2(a, b)

#define TG_SWITCH(PAIR, F8)                                                         \
    switch (stages) {                                                               \
        TG_CASE(2, PAIR, F8)                                                        \
        TG_CASE(3, PAIR, F8)                                                        \
        TG_CASE(4, PAIR, F8)                                                        \
        TG_CASE(6, PAIR, F8)                                                        \
        TG_CASE(8, PAIR, F8)                                                        \
        default:                                                                    \
            return cudaErrorInvalidValue;                                           \
    }

cudaError_t TG_CAT(launch_gemm_bn, TG_BN)(const CUtensorMap &ta, const CUtensorMap &tb,
                                          const CUtensorMap &tc, const KernelParams &p,
                                          int stages, bool pair, bool f8, int mx, int grid, cudaStream_t s)
{
    if (mx != MX_NONE) {
        // block-scaled operands, one CTA per tile: widths 128 and 192 in
        // their units, width 224 (launch_gemm_mx224) in the width-128 unit
        if (pair || !f8) return cudaErrorInvalidValue;
#if TG_BN == 128 || TG_BN == 192
        if (mx == MX_FP4) {
            switch (stages) {
                case 2: return launch_fixed<TG_BN, 2, false, true, true, true>(ta, tb, tc, p, grid, s);
                case 4: return launch_fixed<TG_BN, 4, false, true, true, true>(ta, tb, tc, p, grid, s);
                default: return cudaErrorInvalidValue;
            }
        }
        if (mx != MX_FP8) return cudaErrorInvalidValue;
        switch (stages) {
            case 2: return launch_fixed<TG_BN, 2, false, true, true>(ta, tb, tc, p, grid, s);
            case 4: return launch_fixed<TG_BN, 4, false, true, true>(ta, tb, tc, p, grid, s);
            default: return cudaErrorInvalidValue;
        }
#else
        return cudaErrorInvalidValue;
#endif
    }
    if (pair && f8) TG_SWITCH(true, true)
    if (pair) TG_SWITCH(true, false)
    if (f8) TG_SWITCH(false, true)
    TG_SWITCH(false, false)
}

#if TG_BN == 128
cudaError_t launch_gemm_mx224(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                              const KernelParams &p, int stages, int mx, int grid, cudaStream_t s)
{
    if (mx == MX_FP4)  // two slots: the scales of a third would not fit tensor memory
        return stages == 2 ? launch_fixed<224, 2, false, true, true, true>(ta, tb, tc, p, grid, s)
                           : cudaErrorInvalidValue;
    if (mx != MX_FP8) return cudaErrorInvalidValue;
    switch (stages) {
        case 2: return launch_fixed<224, 2, false, true, true>(ta, tb, tc, p, grid, s);
        case 4: return launch_fixed<224, 4, false, true, true>(ta, tb, tc, p, grid, s);
        default: return cudaErrorInvalidValue;
    }
}
#endif

#if TG_BN == 128 || TG_BN == 192
cudaError_t TG_CAT(TG_CAT(launch_gemm_bn, TG_BN), _half_a)(const CUtensorMap &ta, const CUtensorMap &tb,
                                                          const CUtensorMap &tc, const KernelParams &p, bool f8,
                                                          int grid, cudaStream_t s)
{
    constexpr int S = half_a_stages(TG_BN);
    if (f8) return launch_fixed<TG_BN, S, false, true, false, false, true>(ta, tb, tc, p, grid, s);
    return launch_fixed<TG_BN, S, false, false, false, false, true>(ta, tb, tc, p, grid, s);
}
#endif

int TG_CAT(max_pairs_bn, TG_BN)(int stages, bool f8)
{
    if (f8) {
        switch (stages) {
            TG_CASE_PAIRS(2, true)
            TG_CASE_PAIRS(4, true)
            TG_CASE_PAIRS(6, true)
            TG_CASE_PAIRS(8, true)
            default:
                return 0;
        }
    }
    switch (stages) {
        TG_CASE_PAIRS(2, false)
        TG_CASE_PAIRS(4, false)
        TG_CASE_PAIRS(6, false)
        TG_CASE_PAIRS(8, false)
        default:
            return 0;
    }
}

}  // namespace tg
