// Host-side declarations shared by the C-ABI implementation and the
// translation units that instantiate the kernels.
#pragma once

#include <cuda_runtime.h>

#include "tk_kernels.cuh"

namespace tk {

// Entry of the fused op's row-block kernel (any width; `prefetch`: the form
// that brings its first row block into L2 before waiting on the previous
// kernel), of its warp-stream kernel or of its block-ring kernel (widths a
// multiple of 512) for a format / scale / clamp combination; nullptr if there
// is none.
const void *swiglu_kernel_fn(int out_fmt, int scale_fmt, bool clamp, bool cta_reduce, bool prefetch);
const void *swiglu_stream_fn(int out_fmt, int scale_fmt, bool clamp);
const void *swiglu_block_fn(int out_fmt, int scale_fmt, bool clamp);   // block_stream_kernel
cudaError_t launch_swiglu(const void *fn, int grid, int block, size_t smem, const SwigluArgs &a,
                          const OutArgs &o, const RowShape &sh, cudaStream_t stream);

// Same for the standalone cast (in_dtype: 0 bf16, 1 fp32).
const void *cast_kernel_fn(int in_dtype, int out_fmt, int scale_fmt, bool cta_reduce, bool prefetch);
const void *cast_stream_fn(int in_dtype, int out_fmt, int scale_fmt);
const void *cast_block_fn(int in_dtype, int out_fmt, int scale_fmt);
cudaError_t launch_cast(const void *fn, int grid, int block, size_t smem, const CastArgs &a,
                        const OutArgs &o, const RowShape &sh, cudaStream_t stream);

// Per-channel cast (tk_channel_kernels.cu): the column-amax pass, the scale
// kernel and the quantize pass for an input / code / scale format.
struct ChannelFns {
    const void *amax;
    const void *scale;
    const void *quant;
    const void *chunk;   // the quantize pass on the amax pass's grid, scales reduced in its prologue
    const void *amax_pf;   // the amax pass's form that prefetches its first rows (short slabs)
    const void *amax_keep, *amax_keep_pf;   // the same two with L2 priorities for the chunk quantize pass
};
// One run's launch shape: the amax pass runs (chunks x slabs) CTAs, each over
// slab_rows rows of a 512-column chunk; the quantize pass is a persistent
// grid of quant_grid CTAs of quant_block threads (the row kernel's mapping,
// sh.rpc rows per CTA per iteration).
struct ChannelLaunch {
    int chunks;
    int slabs;
    int64_t slab_rows;
    int quant_grid;
    int quant_block;
    bool split;   // three launches (amax, scale, row quantize) instead of two (amax, chunk quantize)
    int64_t keep_rows;   // two-launch form: rows at the end of each slab the amax pass loads evict_last
};
ChannelFns channel_fns(int in_dtype, int out_fmt, int scale_fmt, int64_t hidden);
int channel_amax_threads();
int channel_scale_threads();
// partial: device fp32 [slabs, H], the caller's workspace.
cudaError_t launch_channel(const ChannelFns &f, const ChannelLaunch &L, const CastArgs &a, const OutArgs &o,
                           const RowShape &sh, float *partial, cudaStream_t stream);

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

// The weighted top-k combine.
enum { kReduceInBf16 = 0, kReduceInE4M3 = 1 };

struct ReduceArgs {
    const void *y;            // [R, H] bf16, or E4M3 codes
    const float *y_scale;     // [R, H / 128] fp32 (E4M3 rows) or null
    int64_t R;                // rows of y
    int32_t H;
    int32_t K;                // slots per token
    const int32_t *pos;       // [T, K]: row of y, or -1 for an empty slot
    const float *w;           // [T, K]
    int64_t T;
    float gs;                 // global scale
    void *out;                // [T, H] bf16
    int32_t tpr, rpc;         // register kernel: threads per token row (H / 16), tokens per CTA step
    unsigned *fault;          // bit 0: a wait gave up; bit 1: a position outside [-1, R) was met (and skipped)
    // bulk kernel: a task is one column chunk of one token
    int32_t nchunks;          // chunks per token
    int32_t wc;               // columns per chunk
    int32_t stages;           // ring slots per CTA
    int32_t slot_bytes;       // bytes per slot (rows, then scales, then the slot's metadata)
    int32_t rb;               // bytes of one row's chunk
    int32_t sb;               // bytes of one row's chunk scales (E4M3), else 0
};

// Bulk kernel: 1 producer warp + kReduceConsumerWarps consumer warps per CTA.
constexpr int kReduceConsumerWarps = 16;
constexpr int kReduceBulkThreads = 32 * (1 + kReduceConsumerWarps);
constexpr int kReduceBulkMaxK = 32;   // one producer lane per slot
constexpr int kReduceMetaBytes = 8 * 32 * 8;   // the producer's metadata ring (8 tasks x 32 lanes x 8 B)
constexpr int kReduceMaxStages = 16;

// Fused op with the codes written transposed (E4M3, groups of 32/64/128).
const void *transpose_kernel_fn(int scale_fmt, bool clamp, bool prefetch);
int transpose_threads();
cudaError_t launch_transpose(const void *fn, int grid, const SwigluArgs &a, const OutArgs &o, const RowShape &sh,
                             int64_t ldq, cudaStream_t stream);

// SwiGLU backward (optionally recomputing the forward's codes and scales).
struct BackwardArgs {
    const uint16_t *x;    // [T, 2H] bf16, gate half first
    const uint16_t *dy;   // [T, H] bf16
    const float *w;       // [T] or null (weight 1)
    uint16_t *dx;         // [T, 2H] bf16: dgate, then dup
    float *dw;            // [T] or null
    float limit;          // clamp limit (clamping instantiations)
    int32_t H;
};
const void *backward_kernel_fn(bool clamp, bool recompute, int out_fmt, int scale_fmt, bool prefetch);
cudaError_t launch_backward(const void *fn, int grid, int block, const BackwardArgs &a, const OutArgs &o,
                            const RowShape &sh, cudaStream_t stream);

// One thread waits on an mbarrier nothing arrives at for `tries` tries, then
// sets bit 0 of *fault (the bounded waits' failure path, for tests).
cudaError_t launch_unanswered_wait(unsigned *fault, uint32_t tries, cudaStream_t stream);

const void *moe_reduce_kernel_fn(int in_fmt, bool prefetch);
const void *moe_reduce_bulk_kernel_fn(int in_fmt, bool prefetch);
cudaError_t launch_moe_reduce(const void *fn, int grid, int block, int smem, const ReduceArgs &a,
                              cudaStream_t stream);

// Bytes of one input row per column of H, for the block-ring kernel.
constexpr int kSwigluRowBytesPerCol = SwigluSrc<false>::kRowBytesPerCol;
constexpr int kCastBf16RowBytesPerCol = CastBf16Src::kRowBytesPerCol;
constexpr int kCastF32RowBytesPerCol = CastF32Src::kRowBytesPerCol;

// Bytes of one warp-ring slot of the stream kernels.
constexpr int kSwigluSlotBytes = SwigluSrc<false>::kSpans * SwigluSrc<false>::kSpanBytes;
constexpr int kCastBf16SlotBytes = CastBf16Src::kSpans * CastBf16Src::kSpanBytes;
constexpr int kCastF32SlotBytes = CastF32Src::kSpans * CastF32Src::kSpanBytes;

}  // namespace tk
