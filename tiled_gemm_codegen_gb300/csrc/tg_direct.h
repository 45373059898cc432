// Launch of the direct-load kernel (tg_direct.cu), the host library's path
// for small problems.  Not part of the public ABI.
#pragma once

#include "tg_internal.h"

namespace tg {

// One CTA per 128 x 64 tile of C, `grid` CTAs; A and B read in place
// (element pitches lda / ldb, batch strides sA / sB, 0 for an operand shared
// by every problem; layouts as in p.a_mn / p.b_k); chunk_kb k-blocks staged
// at once (1 .. DIRECT_KB).  Returns the launch's cudaError_t.
cudaError_t launch_direct(const KernelParams &p, const void *A, const void *B, int64_t lda, int64_t ldb,
                          int64_t sA, int64_t sB, int chunk_kb, int64_t grid, cudaStream_t s);

}  // namespace tg
