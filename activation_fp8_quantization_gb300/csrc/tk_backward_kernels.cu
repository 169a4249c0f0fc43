// SwiGLU backward with the forward's FP8 codes recomputed, sm_103a.
//
// Not described on the pages (they give the forward only): the plain
// derivation of y = silu(g') * u' * w, g' = min(g, L), u' = clamp(u, -L, L):
//   dgate = dy * w * u' * silu'(g')   (0 where g > L)
//   dup   = dy * w * silu(g')         (0 where |u| > L)
//   dw    = sum over the row of dy * silu(g') * u'
// with silu'(g) = s (1 + g (1 - s)), s = sigmoid(g). Optionally the forward's
// codes and scales are recomputed from the same read of x, bit-identical to
// tk_swiglu_quant_run's, for a following GEMM that needs the activation.
//
// A thread owns 16 columns of one row (as the forward's row kernel): it
// reads 32 bytes each of the gate, the up half and dy, and writes 32 bytes
// each of dgate and dup. With t = e^{-|g'|} (computed as h * h, h =
// 2^{-|g'| log2(e) / 2}, as in the forward) and r = 1 / (1 + t):
//   s = r and 1 - s = t r for g' >= 0;  s = t r and 1 - s = r for g' < 0
//   silu = max(g' t, g') r                 (the forward's expression)
//   silu' = (silu * q + p) * r             p = s / r, q = (1 - s) / r
// dw's row sum is reduced in a fixed order (xor shuffles within a warp,
// then the warps of a row in index order through shared memory), so it is
// deterministic.
#include "tk_backward.h"

namespace tk {

namespace {

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// CLAMP: 0 none; 1 in fp32 (any limit); 2 on the bf16 pairs (a limit that
// is a bf16 value, so the clamp is exact there): two lanes per instruction,
// and the lanes past the limit kept as 16-bit masks that zero their bf16
// gradients at the end (+0, as the fp32 form writes).
// Registers are capped at 64 (two 512-thread or four 256-thread CTAs per SM):
// left to itself the compiler gives the clamping, recomputing forms over 100,
// which halves the CTAs per SM and was measured 25% slower than the few
// bytes of spills the cap costs.
template <int CLAMP, bool RECOMPUTE, int OUT, int SCALE, int PREFETCH>
__global__ void __launch_bounds__(512, 2) swiglu_backward_kernel(BackwardArgs a, OutArgs o, RowShape sh)
{
    __shared__ float red[2][16];   // per-warp partial dw, double-buffered by row block
    int buf = 0;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int slot = tid / sh.tpr;
    const int lr = tid - slot * sh.tpr;
    const bool slot_ok = slot < sh.rpc;
    const int col0 = lr * kEPT;
    const int tpg_mask = (1 << sh.tpg_log2) - 1;
    const int64_t nrb = (sh.T + sh.rpc - 1) / sh.rpc;
    const int width = sh.tpr < 32 ? sh.tpr : 32;   // lanes of one row within a warp
    const int nwr = sh.tpr > 32 ? sh.tpr / 32 : 1;  // warps per row
    const float L = a.limit;
    constexpr float kNegHalfLog2e = -0.72134752044448170368f;  // -log2(e) / 2
    const bool wide = aligned32(a.dx);   // uniform: a row's halves stay 32-byte aligned (H % 16 == 0)
    // PREFETCH >= 1 (the plan's choice where a CTA has few row blocks): the first
    // row block's x and dy into L2 before waiting on the previous kernel
    if (PREFETCH >= 1 && slot_ok && (int64_t)blockIdx.x < nrb && (int64_t)blockIdx.x * sh.rpc + slot < sh.T) {
        const int64_t row = (int64_t)blockIdx.x * sh.rpc + slot;
        prefetch_l2(a.x + row * (2 * (int64_t)a.H) + col0);
        prefetch_l2(a.x + row * (2 * (int64_t)a.H) + a.H + col0);
        prefetch_l2(a.dy + row * (int64_t)a.H + col0);
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t rb = blockIdx.x; rb < nrb; rb += gridDim.x) {
        const int64_t row = rb * sh.rpc + slot;
        const bool ok = slot_ok && row < sh.T;
        uint32_t gr[8], ur[8], dr[8];
        float w = 1.0f;
        if (ok) {
            const uint16_t *xr = a.x + row * (2 * (int64_t)a.H) + col0;
            ld_stream_256(xr, gr);
            ld_stream_256(xr + a.H, ur);
            ld_stream_256(a.dy + row * (int64_t)a.H + col0, dr);
            if (a.w)
                w = __ldg(a.w + row);
            // PREFETCH == 2: the CTA's next row block into L2 while this one
            // is worked on
            const int64_t nrow = row + (int64_t)gridDim.x * sh.rpc;
            if (PREFETCH == 2 && nrow < sh.T) {
                prefetch_l2(xr + (int64_t)gridDim.x * sh.rpc * (2 * (int64_t)a.H));
                prefetch_l2(xr + (int64_t)gridDim.x * sh.rpc * (2 * (int64_t)a.H) + a.H);
                prefetch_l2(a.dy + nrow * (int64_t)a.H + col0);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                gr[i] = ur[i] = dr[i] = 0u;
        }
        const uint64_t w2 = splat(w);
        const uint64_t w2n = splat(-w);
        uint32_t og[8], ou[8];
        uint64_t ny[kEPT / 2];
        uint64_t acc = 0;
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t gi = gr[i], ui = ur[i], mg = 0u, mu = 0u;
            if (CLAMP == 2) {
                const uint32_t gc = bf16x2_min(gi, a.limit2);
                const uint32_t uc = bf16x2_max(bf16x2_min(ui, a.limit2), a.limit2 ^ 0x80008000u);
                mg = bf16x2_ne_mask(gc, gi);   // g > L
                mu = bf16x2_ne_mask(uc, ui);   // |u| > L
                gi = gc;
                ui = uc;
            }
            float g0 = bf16_lo(gi), g1 = bf16_hi(gi);
            float u0 = bf16_lo(ui), u1 = bf16_hi(ui);
            bool pg0 = true, pg1 = true, pu0 = true, pu1 = true;
            if (CLAMP == 1) {
                pg0 = !(g0 > L);
                pg1 = !(g1 > L);
                pu0 = !(fabsf(u0) > L);
                pu1 = !(fabsf(u1) > L);
                g0 = fminf(g0, L);
                g1 = fminf(g1, L);
                u0 = fminf(fmaxf(u0, -L), L);
                u1 = fminf(fmaxf(u1, -L), L);
            }
            // the forward's silu, operation for operation
            const uint64_t h = pk(ex2_ftz(__fmul_rn(fabsf(g0), kNegHalfLog2e)),
                                  ex2_ftz(__fmul_rn(fabsf(g1), kNegHalfLog2e)));
            const uint64_t t = mul2(h, h);
            const uint64_t gt = mul2(pk(g0, g1), t);
            const uint64_t num = pk(fmaxf(plo(gt), g0), fmaxf(phi(gt), g1));
            const uint64_t den = add2(t, splat(1.0f));
            const uint64_t r = pk(rcp_ftz(plo(den)), rcp_ftz(phi(den)));
            const uint64_t silu = mul2(num, r);
            const uint64_t uu = pk(u0, u1);
            const uint64_t su = mul2(silu, uu);
            if (RECOMPUTE) {
                ny[i] = mul2(su, w2n);   // -y, as the forward computes it
                amax = fmaxf(amax, fmaxf(fabsf(plo(ny[i])), fabsf(phi(ny[i]))));
            }
            // silu' = (silu * q + p) * r
            const float t0 = plo(t), t1 = phi(t);
            const uint64_t p = pk(g0 >= 0.0f ? 1.0f : t0, g1 >= 0.0f ? 1.0f : t1);
            const uint64_t q = pk(g0 >= 0.0f ? t0 : 1.0f, g1 >= 0.0f ? t1 : 1.0f);
            const uint64_t dsilu = mul2(fma2(silu, q, p), r);
            const uint64_t d = pk(bf16_lo(dr[i]), bf16_hi(dr[i]));
            const uint64_t dw_ = mul2(d, w2);
            uint64_t dg = mul2(mul2(dw_, uu), dsilu);
            uint64_t du = mul2(dw_, silu);
            if (CLAMP == 1) {
                dg = pk(pg0 ? plo(dg) : 0.0f, pg1 ? phi(dg) : 0.0f);
                du = pk(pu0 ? plo(du) : 0.0f, pu1 ? phi(du) : 0.0f);
            }
            og[i] = bf16x2_rn(plo(dg), phi(dg)) & ~mg;
            ou[i] = bf16x2_rn(plo(du), phi(du)) & ~mu;
            acc = fma2(d, su, acc);
        }
        if (ok) {
            uint16_t *dxr = a.dx + row * (2 * (int64_t)a.H) + col0;
            if (wide) {   // dx 32-byte aligned: every thread's 32 bytes are
                          // one sector
                st_stream_256(dxr, og);
                st_stream_256(dxr + a.H, ou);
            } else {
                st_stream_128(dxr, og[0], og[1], og[2], og[3]);
                st_stream_128(dxr + 8, og[4], og[5], og[6], og[7]);
                st_stream_128(dxr + a.H, ou[0], ou[1], ou[2], ou[3]);
                st_stream_128(dxr + a.H + 8, ou[4], ou[5], ou[6], ou[7]);
            }
        }
        if (a.dw) {
            float part = plo(acc) + phi(acc);
            for (int off = width >> 1; off >= 1; off >>= 1)
                part += __shfl_xor_sync(kFull, part, off);
            if (nwr == 1) {
                if (ok && lr == 0)
                    a.dw[row] = part;
            } else {
                // red[buf] is rewritten two row blocks later, after the next
                // block's barrier, which the reading thread reaches only after
                // its read: one barrier per row block suffices.
                if ((tid & 31) == 0)
                    red[buf][warp] = part;
                __syncthreads();
                if (ok && lr == 0) {
                    float s = red[buf][slot * nwr];
                    for (int j = 1; j < nwr; ++j)
                        s += red[buf][slot * nwr + j];
                    a.dw[row] = s;
                }
                buf ^= 1;
            }
        }
        if (RECOMPUTE) {
            amax = group_max(amax, tpg_mask);
            if (ok)
                quantize_store<OUT, SCALE>(ny, amax, row, col0, lr >> sh.tpg_log2, (lr & tpg_mask) == 0, sh, o);
        }
    }
}

template <int CLAMP, int PF>
const void *pick_recompute(int out_fmt, int scale_fmt)
{
    if (out_fmt == kOutE4M3)
        return scale_fmt == kScaleF32
                   ? reinterpret_cast<const void *>(&swiglu_backward_kernel<CLAMP, true, kOutE4M3, kScaleF32, PF>)
                   : reinterpret_cast<const void *>(&swiglu_backward_kernel<CLAMP, true, kOutE4M3, kScaleUE8M0, PF>);
    return scale_fmt == kScaleF32
               ? reinterpret_cast<const void *>(&swiglu_backward_kernel<CLAMP, true, kOutE2M1, kScaleF32, PF>)
               : reinterpret_cast<const void *>(&swiglu_backward_kernel<CLAMP, true, kOutE2M1, kScaleUE8M0, PF>);
}

template <int CLAMP, int PF>
const void *pick_plain(bool recompute, int out_fmt, int scale_fmt)
{
    if (!recompute)
        return reinterpret_cast<const void *>(&swiglu_backward_kernel<CLAMP, false, kOutE4M3, kScaleF32, PF>);
    return pick_recompute<CLAMP, PF>(out_fmt, scale_fmt);
}

template <int PF>
const void *pick_backward(int clamp, bool recompute, int out_fmt, int scale_fmt)
{
    if (clamp == 2)
        return pick_plain<2, PF>(recompute, out_fmt, scale_fmt);
    if (clamp == 1)
        return pick_plain<1, PF>(recompute, out_fmt, scale_fmt);
    return pick_plain<0, PF>(recompute, out_fmt, scale_fmt);
}

}  // namespace

const void *backward_kernel_fn(int clamp, bool recompute, int out_fmt, int scale_fmt, int prefetch)
{
    if (prefetch == 2)
        return pick_backward<2>(clamp, recompute, out_fmt, scale_fmt);
    return prefetch == 1 ? pick_backward<1>(clamp, recompute, out_fmt, scale_fmt)
                         : pick_backward<0>(clamp, recompute, out_fmt, scale_fmt);
}

cudaError_t launch_backward(const void *fn, int grid, int block, const BackwardArgs &a, const OutArgs &o,
                            const RowShape &sh, cudaStream_t stream)
{
    BackwardArgs a_ = a;
    OutArgs o_ = o;
    RowShape sh_ = sh;
    void *args[] = {&a_, &o_, &sh_};
    return launch_pdl(fn, grid, block, 0, args, stream);
}

}  // namespace tk
