// Launch of the direct-load kernel (tg_direct.cu), the host library's path
// for small problems.  Not part of the public ABI.
#pragma once

#include "tg_internal.h"

namespace tg {

// One CTA per 128 x 64 tile of C, `grid` CTAs; A and B read in place
// (element pitches lda / ldb, batch strides sA / sB, 0 for an operand shared
// by every problem; layouts as in p.a_mn / p.b_k); chunk_kb k-blocks staged
// at once (1 .. DIRECT_KB); vec: both operands may be staged in 16-byte
// units (direct_vec_ok).  Returns the launch's cudaError_t.
cudaError_t launch_direct(const KernelParams &p, const void *A, const void *B, int64_t lda, int64_t ldb,
                          int64_t sA, int64_t sB, int chunk_kb, bool vec, int64_t grid, cudaStream_t s);

// An operand the direct-load kernel may stage in 16-byte units: base, pitch
// and batch stride (elements; 0 for a shared operand) 16-byte aligned, and
// the extent along its contiguous dimension a multiple of 8 elements.
inline bool direct_vec_ok(const void *base, int64_t ld, int64_t stride, int64_t contiguous_extent)
{
    return (reinterpret_cast<uintptr_t>(base) & 15u) == 0 && ld % 8 == 0 && stride % 8 == 0 &&
           contiguous_extent % 8 == 0;
}

}  // namespace tg
