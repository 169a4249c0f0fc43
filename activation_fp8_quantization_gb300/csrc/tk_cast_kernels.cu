// Instantiations of the standalone per-token / per-block cast kernel.
#include "tk_internal.h"

namespace tk {

namespace {
template <class Src, int OUT, int SCALE, bool CTA>
const void *fn(int pf)
{
    if (pf == 2)
        return reinterpret_cast<const void *>(&row_quant_kernel<Src, OUT, SCALE, CTA, 2>);
    return pf == 1 ? reinterpret_cast<const void *>(&row_quant_kernel<Src, OUT, SCALE, CTA, 1>)
                   : reinterpret_cast<const void *>(&row_quant_kernel<Src, OUT, SCALE, CTA, 0>);
}

template <class Src, int OUT>
const void *pick(int scale_fmt, bool cta, int pf)
{
    if (scale_fmt == kScaleF32)
        return cta ? fn<Src, OUT, kScaleF32, true>(pf) : fn<Src, OUT, kScaleF32, false>(pf);
    return cta ? fn<Src, OUT, kScaleUE8M0, true>(pf) : fn<Src, OUT, kScaleUE8M0, false>(pf);
}

template <class Src>
const void *pick_out(int out_fmt, int scale_fmt, bool cta, int pf)
{
    if (out_fmt == kOutE4M3)
        return pick<Src, kOutE4M3>(scale_fmt, cta, pf);
    if (out_fmt == kOutE2M1)
        return pick<Src, kOutE2M1>(scale_fmt, cta, pf);
    return nullptr;
}
template <class Src>
const void *stream_pick(int out_fmt, int scale_fmt)
{
    if (out_fmt == kOutE4M3)
        return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&warp_stream_kernel<Src, kOutE4M3, kScaleF32>)
                                      : reinterpret_cast<const void *>(&warp_stream_kernel<Src, kOutE4M3, kScaleUE8M0>);
    if (out_fmt == kOutE2M1)
        return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&warp_stream_kernel<Src, kOutE2M1, kScaleF32>)
                                      : reinterpret_cast<const void *>(&warp_stream_kernel<Src, kOutE2M1, kScaleUE8M0>);
    return nullptr;
}
template <class Src>
const void *block_pick(int out_fmt, int scale_fmt)
{
    if (out_fmt == kOutE4M3)
        return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&block_stream_kernel<Src, kOutE4M3, kScaleF32>)
                                      : reinterpret_cast<const void *>(&block_stream_kernel<Src, kOutE4M3, kScaleUE8M0>);
    if (out_fmt == kOutE2M1)
        return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&block_stream_kernel<Src, kOutE2M1, kScaleF32>)
                                      : reinterpret_cast<const void *>(&block_stream_kernel<Src, kOutE2M1, kScaleUE8M0>);
    return nullptr;
}
}  // namespace

const void *cast_block_fn(int in_dtype, int out_fmt, int scale_fmt)
{
    if (in_dtype == 0)
        return block_pick<CastBf16Src>(out_fmt, scale_fmt);
    if (in_dtype == 1)
        return block_pick<CastF32Src>(out_fmt, scale_fmt);
    return nullptr;
}

const void *cast_stream_fn(int in_dtype, int out_fmt, int scale_fmt)
{
    if (in_dtype == 0)
        return stream_pick<CastBf16Src>(out_fmt, scale_fmt);
    if (in_dtype == 1)
        return stream_pick<CastF32Src>(out_fmt, scale_fmt);
    return nullptr;
}

const void *cast_kernel_fn(int in_dtype, int out_fmt, int scale_fmt, bool cta_reduce, int prefetch)
{
    if (in_dtype == 0)
        return pick_out<CastBf16Src>(out_fmt, scale_fmt, cta_reduce, prefetch);
    if (in_dtype == 1)
        return pick_out<CastF32Src>(out_fmt, scale_fmt, cta_reduce, prefetch);
    return nullptr;
}

cudaError_t launch_cast(const void *kfn, int grid, int block, size_t smem, const CastArgs &a,
                        const OutArgs &o, const RowShape &sh, cudaStream_t stream)
{
    CastArgs a_ = a;
    OutArgs o_ = o;
    RowShape sh_ = sh;
    void *args[] = {&a_, &o_, &sh_};
    return launch_pdl(kfn, grid, block, smem, args, stream);
}

}  // namespace tk
