// Instantiations of the persistent GEMM kernel: one translation unit per tile
// width (selected at build time with -DTG_BN=...), so the widths compile in
// parallel.  Each width instantiates a few ring depths; stage_supported()
// in tg_plan.h lists them and the host planner only picks listed depths.
#include "tg_kernel.cuh"
#include "tg_plan.h"

#ifndef TG_BN
#error "compile with -DTG_BN=<64|128|192|256>"
#endif

namespace tg {

#define TG_CASE(S)                                                          \
    case S:                                                                 \
        if constexpr (stage_supported(TG_BN, S))                            \
            return launch_fixed<TG_BN, S>(ta, tb, tc, p, grid, s);          \
        else                                                                \
            return cudaErrorInvalidValue;

#define TG_CAT2(a, b) a##b
#define TG_CAT(a, b) TG_CAT2(a, b)

cudaError_t TG_CAT(launch_gemm_bn, TG_BN)(const CUtensorMap &ta, const CUtensorMap &tb,
                                          const CUtensorMap &tc, const KernelParams &p,
                                          int stages, int grid, cudaStream_t s)
{
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

}  // namespace tg
