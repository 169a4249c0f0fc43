// Device side of the fused SwiGLU + top-k weight + FP8/FP4 cast, sm_103a.
//
// One persistent, grid-strided kernel template serves both entry points. A
// thread owns 16 consecutive columns of one row: for the fused op that is one
// 32-byte vector of the gate half and one of the up half ("TileKernels from
// Beginner to Master", zhichai.net/en/topic/177618752, chapter 1: 32-byte
// vectors on SM100-class parts; chapter 2: both halves of a row reached by a
// `hidden` offset). The activation stays in registers from load to code store
// (chapter 2, "operator fusion, three stages"); group absmax is a butterfly of
// warp shuffles over the threads of one group, or a CTA reduction through
// shared memory for one-scale-per-row at widths a warp cannot cover.
//
// The schedule is persistent (chapter 2, "Persistent Kernel": a fixed grid
// that stays resident while rows stream through): the host sizes the grid to
// the CTAs that fit on all SMs at once, each CTA walks row blocks with a grid
// stride, and the next row block's loads are issued before the current one is
// computed so that every thread keeps 64 bytes of HBM reads in flight.
//
// Numerics (IEEE, no fast-math, no FMA contraction: the library is built with
// -fmad=false and every fused multiply-add below is written out):
//   silu(g) = g * sigmoid(g) with e^{-|g|} from ex2.approx and the reciprocal
//   from rcp.approx; y = (silu(g') * u') * w in fp32. The scale and the
//   quotient y / s are the IEEE fp32 results: s = amax / Qmax by correctly
//   rounded division; y / s either by an exact power-of-two multiply (UE8M0)
//   or by a reciprocal with one Markstein correction step, which returns the
//   correctly rounded quotient. Codes come from the hardware's
//   round-to-nearest-even, saturating e4m3x2 / e2m1x2 conversions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace tk {

constexpr int kEPT = 16;                 // columns per thread
constexpr int kMaxThreads = 1024;
constexpr unsigned kFull = 0xffffffffu;

enum { kOutE4M3 = 0, kOutE2M1 = 1 };
enum { kScaleF32 = 0, kScaleUE8M0 = 1 };

// Row geometry shared by every variant.
struct RowShape {
    int64_t T;          // rows
    int32_t H;          // columns of the activation
    int32_t tpr;        // threads per row = H / 16
    int32_t tpg_log2;   // log2(threads per group); unused by the CTA-reduction variant
    int32_t rpc;        // rows per CTA per iteration
    int32_t groups;     // scales per row
};

struct OutArgs {
    uint8_t *q;
    void *scales;
};

// ----------------------------------------------------------------- memory

__device__ __forceinline__ void ld_stream_256(const void *p, uint32_t (&r)[8])
{
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]),
          "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "l"(p));
}

__device__ __forceinline__ void st_stream_128(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void st_stream_64(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.L1::no_allocate.v2.b32 [%0], {%1,%2};"
                 :: "l"(p), "r"(a), "r"(b) : "memory");
}

// bf16 is the upper half of an fp32: widening is a shift or a mask.
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// ---------------------------------------------------------------- arithmetic

__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// silu(g) = g / (1 + e^{-g}). With t = e^{-|g|} in (0, 1] nothing overflows:
// for g >= 0 it is g / (1 + t); for g < 0 it is g * t / (1 + t).
__device__ __forceinline__ float silu(float g)
{
    const float t = ex2_approx(__fmul_rn(fabsf(g), -1.4426950408889634f));
    const float num = g < 0.0f ? __fmul_rn(g, t) : g;
    return __fmul_rn(num, rcp_approx(__fadd_rn(1.0f, t)));
}

// Correctly rounded a / b from rb = RN(1/b): q0 = RN(a * rb) is within one
// ulp of a / b, the FMA returns the exact remainder a - b * q0, and one
// correction step RN(q0 + r * rb) is RN(a / b) (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", 1990; see also
// Muller et al., "Handbook of Floating-Point Arithmetic", the chapter on
// division with an FMA). Valid while the remainder does not underflow; the
// caller keeps b >= 2^-80 so that is true whenever |a / b| >= 2^-11, and
// smaller quotients encode to a signed zero whatever their last bits.
// For a = -0 the correction adds +0 and -0, which rounds to +0; b > 0 here,
// so the quotient's sign is a's and is copied back.
__device__ __forceinline__ float div_markstein(float a, float b, float rb)
{
    const float q0 = __fmul_rn(a, rb);
    const float r = __fmaf_rn(-q0, b, a);
    return copysignf(__fmaf_rn(r, rb, q0), a);
}

template <int OUT> struct Fmt;
template <> struct Fmt<kOutE4M3> {
    // 448 = 1.75 * 2^8: exponent 8, fraction bits of 1.75
    static constexpr float kQmax = 448.0f;
    static constexpr int kQE = 8;
    static constexpr uint32_t kQM = 0x600000u;
};
template <> struct Fmt<kOutE2M1> {
    // 6 = 1.5 * 2^2
    static constexpr float kQmax = 6.0f;
    static constexpr int kQE = 2;
    static constexpr uint32_t kQM = 0x400000u;
};

// Smallest k with Qmax * 2^k >= amax, read off amax's bits: with
// amax = m * 2^e (1 <= m < 2) and Qmax = q * 2^QE, k = e - QE when m <= q and
// e - QE + 1 otherwise. Clamped to the finite UE8M0 range [-127, 127];
// amax == 0 gives 0.
template <int OUT>
__device__ __forceinline__ int ue8m0_exponent(float amax)
{
    const uint32_t b = __float_as_uint(amax);
    if (b == 0u)
        return 0;
    int e;
    uint32_t m;
    if (b >= 0x00800000u) {
        e = (int)(b >> 23) - 127;
        m = b & 0x7fffffu;
    } else {  // subnormal: leading one at bit p, value 2^(p-149) * 1.f
        const int p = 31 - __clz((int)b);
        e = p - 149;
        m = (b << (23 - p)) & 0x7fffffu;
    }
    int k = e - Fmt<OUT>::kQE + (m > Fmt<OUT>::kQM ? 1 : 0);
    return k < -127 ? -127 : (k > 127 ? 127 : k);
}

// Two fp32 -> two codes, RNE with saturation to the largest finite value.
// The first operand of the conversion lands in the upper half of the result,
// so `lo` (the lower column) is passed second.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return (uint32_t)h;
}

__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ------------------------------------------------------- quantize and store

// Scale the thread's 16 values by 1/s (s from the group's amax), encode and
// store them; the group's first thread also stores the scale.
template <int OUT, int SCALE>
__device__ __forceinline__ void quantize_store(const float (&y)[kEPT], float amax, int64_t row,
                                               int col0, int group_idx, bool write_scale,
                                               const RowShape &sh, const OutArgs &o)
{
    float v[kEPT];
    if (SCALE == kScaleUE8M0) {
        const int k = ue8m0_exponent<OUT>(amax);
        const float inv = __uint_as_float((uint32_t)(127 - k) << 23);  // 2^-k, k <= 126 here
#pragma unroll
        for (int i = 0; i < kEPT; ++i)
            v[i] = __fmul_rn(y[i], inv);  // exact: a power-of-two scaling, rounded once at most
        if (write_scale)
            static_cast<uint8_t *>(o.scales)[row * sh.groups + group_idx] = (uint8_t)(k + 127);
    } else {
        float s = __fdiv_rn(amax, Fmt<OUT>::kQmax);
        if (s == 0.0f)
            s = 1.0f;
        if (s >= 0x1p-80f) {
            const float rs = __frcp_rn(s);
#pragma unroll
            for (int i = 0; i < kEPT; ++i)
                v[i] = div_markstein(y[i], s, rs);
        } else {
#pragma unroll
            for (int i = 0; i < kEPT; ++i)
                v[i] = __fdiv_rn(y[i], s);
        }
        if (write_scale)
            static_cast<float *>(o.scales)[row * sh.groups + group_idx] = s;
    }
    if (OUT == kOutE4M3) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = cvt_e4m3x2(v[4 * j], v[4 * j + 1]) | (cvt_e4m3x2(v[4 * j + 2], v[4 * j + 3]) << 16);
        st_stream_128(o.q + row * (int64_t)sh.H + col0, w[0], w[1], w[2], w[3]);
    } else {
        uint32_t w[2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
            w[j] = cvt_e2m1x2(v[8 * j], v[8 * j + 1]) | (cvt_e2m1x2(v[8 * j + 2], v[8 * j + 3]) << 8) |
                   (cvt_e2m1x2(v[8 * j + 4], v[8 * j + 5]) << 16) |
                   (cvt_e2m1x2(v[8 * j + 6], v[8 * j + 7]) << 24);
        st_stream_64(o.q + row * (int64_t)(sh.H / 2) + col0 / 2, w[0], w[1]);
    }
}

// ------------------------------------------------------------ the kernel

// Src supplies: Args (kernel argument), Regs (raw loaded data for one row
// slice), load(args, row, col0, regs), produce(args, regs, row, y) -> fills
// y[16] and returns nothing, and finish(args) at kernel exit.
template <class Src, int OUT, int SCALE, bool CTA_REDUCE>
__global__ void __launch_bounds__(kMaxThreads)
row_quant_kernel(typename Src::Args a, OutArgs o, RowShape sh)
{
    __shared__ float red[2][32];
    Src src;
    const int tid = threadIdx.x;
    const int slot = tid / sh.tpr;               // row slot in this CTA
    const int lr = tid - slot * sh.tpr;          // thread index within the row
    const bool slot_ok = slot < sh.rpc;
    const int col0 = lr * kEPT;
    const int64_t nrb = (sh.T + sh.rpc - 1) / sh.rpc;
    const int tpg_mask = (1 << sh.tpg_log2) - 1;
    const int group_idx = CTA_REDUCE ? 0 : (lr >> sh.tpg_log2);
    const bool first_of_group = CTA_REDUCE ? (tid == 0) : ((lr & tpg_mask) == 0);

    typename Src::Regs cur, nxt;
    int64_t rb = blockIdx.x;
    int64_t row = rb * sh.rpc + slot;
    bool ok = slot_ok && rb < nrb && row < sh.T;
    if (ok)
        Src::load(a, row, col0, cur);
    else
        Src::zero(cur);

    int it = 0;
    for (; rb < nrb; rb += gridDim.x, ++it) {
        const int64_t nrow = (rb + gridDim.x) * sh.rpc + slot;
        const bool nok = slot_ok && (rb + gridDim.x) < nrb && nrow < sh.T;
        if (nok)
            Src::load(a, nrow, col0, nxt);
        else
            Src::zero(nxt);

        float y[kEPT];
        src.produce(a, cur, row, ok, y);
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kEPT; ++i)
            amax = fmaxf(amax, fabsf(y[i]));

        if (CTA_REDUCE) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
            float *buf = red[it & 1];
            if ((tid & 31) == 0)
                buf[tid >> 5] = amax;
            __syncthreads();
            const int nwarps = (blockDim.x + 31) >> 5;
            amax = 0.0f;
            for (int w = 0; w < nwarps; ++w)
                amax = fmaxf(amax, buf[w]);
        } else {
            for (int off = 1; off <= tpg_mask; off <<= 1)
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
        }
        if (ok)
            quantize_store<OUT, SCALE>(y, amax, row, col0, group_idx, first_of_group, sh, o);

        cur = nxt;
        row = nrow;
        ok = nok;
    }
    src.finish(a);
}

// ------------------------------------------------------------ sources

struct SwigluArgs {
    const uint16_t *x;            // [T, 2H] bf16 bits
    const float *w;               // [T] or null
    unsigned long long *counts;   // [2] or null
    float limit;
    int32_t H;
};

struct Regs32x2 {
    uint32_t g[8];
    uint32_t u[8];
    float w;
};

template <bool CLAMP>
struct SwigluSrc {
    using Args = SwigluArgs;
    using Regs = Regs32x2;
    unsigned cnt_g = 0, cnt_u = 0;

    __device__ __forceinline__ static void load(const Args &a, int64_t row, int col0, Regs &r)
    {
        const uint16_t *p = a.x + row * (2 * (int64_t)a.H) + col0;
        ld_stream_256(p, r.g);
        ld_stream_256(p + a.H, r.u);
        r.w = a.w ? __ldg(a.w + row) : 1.0f;
    }
    __device__ __forceinline__ static void zero(Regs &r)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            r.g[i] = 0u;
            r.u[i] = 0u;
        }
        r.w = 0.0f;
    }
    __device__ __forceinline__ void produce(const Args &a, const Regs &r, int64_t, bool ok,
                                            float (&y)[kEPT])
    {
        const float L = a.limit;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float g[2] = {bf16_lo(r.g[i]), bf16_hi(r.g[i])};
            float u[2] = {bf16_lo(r.u[i]), bf16_hi(r.u[i])};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (CLAMP) {
                    cnt_g += (ok && g[h] > L) ? 1u : 0u;
                    cnt_u += (ok && fabsf(u[h]) > L) ? 1u : 0u;
                    g[h] = fminf(g[h], L);
                    u[h] = fminf(fmaxf(u[h], -L), L);
                }
                y[2 * i + h] = __fmul_rn(__fmul_rn(silu(g[h]), u[h]), r.w);
            }
        }
    }
    __device__ __forceinline__ void finish(const Args &a)
    {
        if (CLAMP && a.counts) {
            const unsigned sg = __reduce_add_sync(kFull, cnt_g);
            const unsigned su = __reduce_add_sync(kFull, cnt_u);
            if ((threadIdx.x & 31) == 0) {
                if (sg)
                    atomicAdd(a.counts + 0, (unsigned long long)sg);
                if (su)
                    atomicAdd(a.counts + 1, (unsigned long long)su);
            }
        }
    }
};

struct CastArgs {
    const void *x;   // [T, H] bf16 or fp32
    int32_t H;
};

struct CastBf16Src {
    using Args = CastArgs;
    struct Regs { uint32_t v[8]; };
    __device__ __forceinline__ static void load(const Args &a, int64_t row, int col0, Regs &r)
    {
        ld_stream_256(static_cast<const uint16_t *>(a.x) + row * (int64_t)a.H + col0, r.v);
    }
    __device__ __forceinline__ static void zero(Regs &r)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            r.v[i] = 0u;
    }
    __device__ __forceinline__ void produce(const Args &, const Regs &r, int64_t, bool, float (&y)[kEPT])
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[2 * i] = bf16_lo(r.v[i]);
            y[2 * i + 1] = bf16_hi(r.v[i]);
        }
    }
    __device__ __forceinline__ void finish(const Args &) {}
};

struct CastF32Src {
    using Args = CastArgs;
    struct Regs { uint32_t v[16]; };
    __device__ __forceinline__ static void load(const Args &a, int64_t row, int col0, Regs &r)
    {
        const float *p = static_cast<const float *>(a.x) + row * (int64_t)a.H + col0;
        uint32_t (&lo)[8] = *reinterpret_cast<uint32_t (*)[8]>(&r.v[0]);
        uint32_t (&hi)[8] = *reinterpret_cast<uint32_t (*)[8]>(&r.v[8]);
        ld_stream_256(p, lo);
        ld_stream_256(p + 8, hi);
    }
    __device__ __forceinline__ static void zero(Regs &r)
    {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            r.v[i] = 0u;
    }
    __device__ __forceinline__ void produce(const Args &, const Regs &r, int64_t, bool, float (&y)[kEPT])
    {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            y[i] = __uint_as_float(r.v[i]);
    }
    __device__ __forceinline__ void finish(const Args &) {}
};

}  // namespace tk
