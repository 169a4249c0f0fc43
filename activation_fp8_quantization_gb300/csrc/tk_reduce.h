// Host-side declarations of the weighted top-k combine (tk_reduce_kernels.cu).
#pragma once

#include "tk_internal.h"

namespace tk {

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

const void *moe_reduce_kernel_fn(int in_fmt, bool prefetch);
const void *moe_reduce_bulk_kernel_fn(int in_fmt, bool prefetch);
cudaError_t launch_moe_reduce(const void *fn, int grid, int block, int smem, const ReduceArgs &a,
                              cudaStream_t stream);

}  // namespace tk
