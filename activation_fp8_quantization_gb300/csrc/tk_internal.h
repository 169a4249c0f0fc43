// Host-side declarations shared by the C-ABI implementation and the
// translation units that instantiate the kernels.
#pragma once

#include <cuda_runtime.h>

#include "tk_kernels.cuh"

namespace tk {

// Entry of the fused op's row-block kernel (any width; `prefetch` 1: the form
// that brings its first row block into L2 before waiting on the previous
// kernel; 2 is not built for the fused op), of its warp-stream kernel or of
// its block-ring kernel (widths a multiple of 512) for a format / scale /
// clamp combination; nullptr if there is none.
const void *swiglu_kernel_fn(int out_fmt, int scale_fmt, bool clamp, bool cta_reduce, int prefetch);
const void *swiglu_stream_fn(int out_fmt, int scale_fmt, bool clamp);
const void *swiglu_block_fn(int out_fmt, int scale_fmt, bool clamp);   // block_stream_kernel
cudaError_t launch_swiglu(const void *fn, int grid, int block, size_t smem, const SwigluArgs &a,
                          const OutArgs &o, const RowShape &sh, cudaStream_t stream);

// Same for the standalone cast (in_dtype: 0 bf16, 1 fp32); its row kernel
// also has `prefetch` 2: the first row block and each next one into L2.
const void *cast_kernel_fn(int in_dtype, int out_fmt, int scale_fmt, bool cta_reduce, int prefetch);
const void *cast_stream_fn(int in_dtype, int out_fmt, int scale_fmt);
const void *cast_block_fn(int in_dtype, int out_fmt, int scale_fmt);
cudaError_t launch_cast(const void *fn, int grid, int block, size_t smem, const CastArgs &a,
                        const OutArgs &o, const RowShape &sh, cudaStream_t stream);

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel of the stream drains; it waits for that kernel
// itself (griddepcontrol.wait) before touching global memory.
inline cudaError_t launch_pdl(const void *fn, int grid, int block, size_t smem, void **args, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// One thread waits on an mbarrier nothing arrives at for `tries` tries, then
// sets bit 0 of *fault (the bounded waits' failure path, for tests).
cudaError_t launch_unanswered_wait(unsigned *fault, uint32_t tries, cudaStream_t stream);

// Bytes of one input row per column of H, for the block-ring kernel.
constexpr int kSwigluRowBytesPerCol = SwigluSrc<false>::kRowBytesPerCol;
constexpr int kCastBf16RowBytesPerCol = CastBf16Src::kRowBytesPerCol;
constexpr int kCastF32RowBytesPerCol = CastF32Src::kRowBytesPerCol;

// Bytes of one warp-ring slot of the stream kernels.
constexpr int kSwigluSlotBytes = SwigluSrc<false>::kSpans * SwigluSrc<false>::kSpanBytes;
constexpr int kCastBf16SlotBytes = CastBf16Src::kSpans * CastBf16Src::kSpanBytes;
constexpr int kCastF32SlotBytes = CastF32Src::kSpans * CastF32Src::kSpanBytes;

}  // namespace tk
