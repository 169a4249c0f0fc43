// Host-side declarations of the fused op with transposed codes (tk_transpose_kernels.cu).
#pragma once

#include "tk_internal.h"

namespace tk {

// Fused op with the codes written transposed (E4M3, groups of 32/64/128).
// prefetch: 0 none, 1 the first tile, 2 the first and then each next tile
const void *transpose_kernel_fn(int scale_fmt, bool clamp, int prefetch);
int transpose_threads();
cudaError_t launch_transpose(const void *fn, int grid, const SwigluArgs &a, const OutArgs &o, const RowShape &sh,
                             int64_t ldq, cudaStream_t stream);

}  // namespace tk
