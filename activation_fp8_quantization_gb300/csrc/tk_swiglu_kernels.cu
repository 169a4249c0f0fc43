// Instantiations of the fused SwiGLU + top-k weight + cast kernel.
#include "tk_internal.h"

namespace tk {

namespace {
// prefetch 0 or 1 only: the fused op's row kernel already has its next row
// block's loads in flight in registers, and the form that also prefetches
// each next block into L2 was measured slower for it (4-10%, 2048 to 32768
// rows of width 2048).
template <int OUT, int SCALE, bool CLAMP, bool CTA>
const void *fn(int pf)
{
    if (pf == 2)
        return nullptr;
    return pf == 1 ? reinterpret_cast<const void *>(&row_quant_kernel<SwigluSrc<CLAMP>, OUT, SCALE, CTA, 1>)
                   : reinterpret_cast<const void *>(&row_quant_kernel<SwigluSrc<CLAMP>, OUT, SCALE, CTA, 0>);
}

template <int OUT, int SCALE>
const void *pick(bool clamp, bool cta, int pf)
{
    if (clamp)
        return cta ? fn<OUT, SCALE, true, true>(pf) : fn<OUT, SCALE, true, false>(pf);
    return cta ? fn<OUT, SCALE, false, true>(pf) : fn<OUT, SCALE, false, false>(pf);
}
template <int OUT, int SCALE>
const void *stream_fn(bool clamp)
{
    return clamp ? reinterpret_cast<const void *>(&warp_stream_kernel<SwigluSrc<true>, OUT, SCALE>)
                 : reinterpret_cast<const void *>(&warp_stream_kernel<SwigluSrc<false>, OUT, SCALE>);
}
template <int OUT, int SCALE>
const void *block_fn(bool clamp)
{
    return clamp ? reinterpret_cast<const void *>(&block_stream_kernel<SwigluSrc<true>, OUT, SCALE>)
                 : reinterpret_cast<const void *>(&block_stream_kernel<SwigluSrc<false>, OUT, SCALE>);
}
}  // namespace

const void *swiglu_block_fn(int out_fmt, int scale_fmt, bool clamp)
{
    if (out_fmt == kOutE4M3)
        return scale_fmt == kScaleF32 ? block_fn<kOutE4M3, kScaleF32>(clamp) : block_fn<kOutE4M3, kScaleUE8M0>(clamp);
    if (out_fmt == kOutE2M1)
        return scale_fmt == kScaleF32 ? block_fn<kOutE2M1, kScaleF32>(clamp) : block_fn<kOutE2M1, kScaleUE8M0>(clamp);
    return nullptr;
}

const void *swiglu_stream_fn(int out_fmt, int scale_fmt, bool clamp)
{
    if (out_fmt == kOutE4M3)
        return scale_fmt == kScaleF32 ? stream_fn<kOutE4M3, kScaleF32>(clamp) : stream_fn<kOutE4M3, kScaleUE8M0>(clamp);
    if (out_fmt == kOutE2M1)
        return scale_fmt == kScaleF32 ? stream_fn<kOutE2M1, kScaleF32>(clamp) : stream_fn<kOutE2M1, kScaleUE8M0>(clamp);
    return nullptr;
}

const void *swiglu_kernel_fn(int out_fmt, int scale_fmt, bool clamp, bool cta_reduce, int prefetch)
{
    if (out_fmt == kOutE4M3)
        return scale_fmt == kScaleF32 ? pick<kOutE4M3, kScaleF32>(clamp, cta_reduce, prefetch)
                                      : pick<kOutE4M3, kScaleUE8M0>(clamp, cta_reduce, prefetch);
    if (out_fmt == kOutE2M1)
        return scale_fmt == kScaleF32 ? pick<kOutE2M1, kScaleF32>(clamp, cta_reduce, prefetch)
                                      : pick<kOutE2M1, kScaleUE8M0>(clamp, cta_reduce, prefetch);
    return nullptr;
}

cudaError_t launch_swiglu(const void *kfn, int grid, int block, size_t smem, const SwigluArgs &a,
                          const OutArgs &o, const RowShape &sh, cudaStream_t stream)
{
    SwigluArgs a_ = a;
    OutArgs o_ = o;
    RowShape sh_ = sh;
    void *args[] = {&a_, &o_, &sh_};
    return launch_pdl(kfn, grid, block, smem, args, stream);
}

}  // namespace tk
