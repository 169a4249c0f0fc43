// Host-side declarations of the SwiGLU backward (tk_backward_kernels.cu).
#pragma once

#include "tk_internal.h"

namespace tk {

// SwiGLU backward (optionally recomputing the forward's codes and scales).
struct BackwardArgs {
    const uint16_t *x;    // [T, 2H] bf16, gate half first
    const uint16_t *dy;   // [T, H] bf16
    const float *w;       // [T] or null (weight 1)
    uint16_t *dx;         // [T, 2H] bf16: dgate, then dup
    float *dw;            // [T] or null
    float limit;          // clamp limit (clamping instantiations)
    int32_t H;
    uint32_t limit2;      // the limit as bf16 in both halves (clamp on bf16 pairs)
};
// clamp: 0 none, 1 in fp32 (any limit), 2 on bf16 pairs (a limit that is a bf16 value)
// prefetch: 0 none, 1 the first row block, 2 the first and then each next one
const void *backward_kernel_fn(int clamp, bool recompute, int out_fmt, int scale_fmt, int prefetch);
cudaError_t launch_backward(const void *fn, int grid, int block, const BackwardArgs &a, const OutArgs &o,
                            const RowShape &sh, cudaStream_t stream);

}  // namespace tk
