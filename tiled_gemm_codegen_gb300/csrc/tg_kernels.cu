// Instantiations of the persistent GEMM kernel: one translation unit per tile
// width (selected at build time with -DTG_BN=...), so the widths compile in
// parallel.  Each width instantiates a few ring depths, with one CTA per tile
// and (widths 128 and 256) two-SM tiles; stage_supported() in tg_plan.h lists
// them and the host planner only picks listed configurations.
#include "tg_kernel.cuh"
#include "tg_plan.h"

#ifndef TG_BN
#error "compile with -DTG_BN=<64|128|192|256>"
#endif

namespace tg {

#define TG_CASE(S)                                                             \
    case S:                                                                    \
        if constexpr (stage_supported(TG_BN, S, false))                        \
            return launch_fixed<TG_BN, S, false>(ta, tb, tc, p, grid, s);      \
        else                                                                   \
            return cudaErrorInvalidValue;

#define TG_CASE_PAIR(S)                                                        \
    case S:                                                                    \
        if constexpr (pair_width(TG_BN) && stage_supported(TG_BN, S, true))    \
            return launch_fixed<TG_BN, S, true>(ta, tb, tc, p, grid, s);       \
        else                                                                   \
            return cudaErrorInvalidValue;

#define TG_CASE_PAIRS(S)                                                       \
    case S:                                                                    \
        if constexpr (pair_width(TG_BN) && stage_supported(TG_BN, S, true))    \
            return max_active_pairs<TG_BN, S>();                               \
        else                                                                   \
            return 0;

#define TG_CAT2(a, b) a##b
#define TG_CAT(a, b) TG_CAT2(a, b)

cudaError_t TG_CAT(launch_gemm_bn, TG_BN)(const CUtensorMap &ta, const CUtensorMap &tb,
                                          const CUtensorMap &tc, const KernelParams &p,
                                          int stages, bool pair, int grid, cudaStream_t s)
{
    if (pair) {
        switch (stages) {
            TG_CASE_PAIR(2)
            TG_CASE_PAIR(4)
            TG_CASE_PAIR(6)
            TG_CASE_PAIR(8)
            default:
                return cudaErrorInvalidValue;
        }
    }
    switch (stages) {
        TG_CASE(2)
        TG_CASE(3)
        TG_CASE(4)
        TG_CASE(6)
        TG_CASE(8)
        default:
            return cudaErrorInvalidValue;
    }
}

int TG_CAT(max_pairs_bn, TG_BN)(int stages)
{
    switch (stages) {
        TG_CASE_PAIRS(2)
        TG_CASE_PAIRS(4)
        TG_CASE_PAIRS(6)
        TG_CASE_PAIRS(8)
        default:
            return 0;
    }
}

}  // namespace tg
