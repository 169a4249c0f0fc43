// Host-side declarations of the per-channel cast (tk_channel_kernels.cu).
#pragma once

#include "tk_internal.h"

namespace tk {

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

}  // namespace tk
