// Host-side declarations shared by the C-ABI implementation and the
// translation units that instantiate the kernels.
#pragma once

#include <cuda_runtime.h>

#include "tk_kernels.cuh"

namespace tk {

// Kernel entry for a (format, scale, clamp, reduction) combination of the
// fused op, or nullptr if there is none.
const void *swiglu_kernel_fn(int out_fmt, int scale_fmt, bool clamp, bool cta_reduce);
cudaError_t launch_swiglu(const void *fn, int grid, int block, const SwigluArgs &a,
                          const OutArgs &o, const RowShape &sh, cudaStream_t stream);

// Same for the standalone cast (in_dtype: 0 bf16, 1 fp32).
const void *cast_kernel_fn(int in_dtype, int out_fmt, int scale_fmt, bool cta_reduce);
cudaError_t launch_cast(const void *fn, int grid, int block, const CastArgs &a,
                        const OutArgs &o, const RowShape &sh, cudaStream_t stream);

}  // namespace tk
