// Device side of the fused SwiGLU + top-k weight + FP8/FP4 cast, sm_103a.
//
// Two persistent, grid-strided kernel templates serve both entry points. A
// thread owns 16 consecutive columns of one row: for the fused op that is 32
// bytes of the gate half and 32 of the up half ("TileKernels from Beginner to
// Master", zhichai.net/en/topic/177618752, chapter 1: 32-byte vectors on
// SM100-class parts; chapter 2: both halves of a row reached by a `hidden`
// offset). The activation stays in registers from load to code store
// (chapter 2, "operator fusion, three stages"); group absmax is a butterfly of
// warp shuffles over the threads of one group, or a CTA reduction through
// shared memory for one-scale-per-row at widths a warp cannot cover.
//
// The schedule is persistent (chapter 2, "Persistent Kernel": a fixed grid
// that stays resident while rows stream through): the host sizes the grid to
// the CTAs that fit on all SMs at once.
//
//  - warp_stream_kernel (rows whose width is a multiple of 512): every warp
//    streams 512-column slices of rows through its own ring of shared-memory
//    slots filled by TMA bulk copies (one lane issues them, an mbarrier per
//    slot counts the bytes in), so the bytes in flight are set by the ring
//    depth, not by registers, and no CTA-wide barrier is needed.
//  - row_quant_kernel (any width that is a multiple of 16): CTAs walk row
//    blocks with a grid stride; each thread keeps the next row block's loads
//    (64 bytes) in flight while it computes the current one.
//
// Numerics (IEEE, no fast-math, no FMA contraction: the library is built with
// -fmad=false and every fused multiply-add below is written out). Two columns
// travel together through Blackwell's packed fp32x2 multiply / add / FMA, so
// each instruction does two IEEE operations:
//   silu(g) = max(g * t, g) / (1 + t), t = e^{-|g|} = h * h with
//   h = 2^{-|g| log2(e) / 2} from ex2.approx.ftz (h is a normal number for
//   |g| <= 174, and the multiply rounds a subnormal t correctly, so no
//   subnormal is lost), and the reciprocal of 1 + t in [1, 2] from
//   rcp.approx.ftz; y = (silu(g') * u') * w in fp32. The kernel carries -y
//   (the weight enters as -w, an exact negation), which lets the quotient
//   keep the sign of zero without a fix-up. The scale and the quotient y / s
//   are the IEEE fp32 results: s = amax / Qmax by correctly rounded division;
//   y / s either by an exact power-of-two multiply (UE8M0) or by a reciprocal
//   with one Markstein correction step, which returns the correctly rounded
//   quotient. Codes come from the hardware's round-to-nearest-even,
//   saturating e4m3x2 / e2m1x2 conversions.
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
    int32_t rpc;        // rows per CTA per iteration (block_stream_kernel: rows per ring slot)
    int32_t groups;     // scales per row
    int32_t stages;     // stream kernels: ring slots per warp (warp_stream) or per CTA (block_stream), >= 2
    int32_t wpr;        // stream kernels: 512-column slices per row
    unsigned *fault;    // device word: bit 0 set by a kernel whose bounded wait gave up
    int32_t scale_layout;  // 0 row-major [T, G]; 1 column-major [G, ld]; 2 packed UE8M0 words [G/4, ld]
    int64_t scale_ld;      // column-major layouts: padded rows per column (elements or words)
};

// Element index of the scale of group j of row t (layouts 0 and 1), or byte
// index of its exponent (layout 2, UE8M0).
__device__ __forceinline__ int64_t scale_index(const RowShape &sh, int64_t t, int j)
{
    if (sh.scale_layout == 0)
        return t * sh.groups + j;
    if (sh.scale_layout == 1)
        return (int64_t)j * sh.scale_ld + t;
    return (((int64_t)(j >> 2) * sh.scale_ld + t) << 2) + (j & 3);
}

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

// 32 bytes in one store (32-byte aligned): a lane writes a whole sector, so
// L2 sees one full-sector write instead of two half-sector ones
__device__ __forceinline__ void st_stream_256(void *p, const uint32_t (&w)[8])
{
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

__device__ __forceinline__ void st_stream_64(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.L1::no_allocate.v2.b32 [%0], {%1,%2};"
                 :: "l"(p), "r"(a), "r"(b) : "memory");
}

// Hint: bring the line holding p into L2. Issued before griddepcontrol.wait
// it overlaps a launch's first DRAM latency with the previous kernel's tail;
// it reads nothing into registers or L1, and the real loads come after the
// wait, from L2, the point of coherence, so they see the previous kernel's
// writes whatever the prefetch found.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p));
}

// bf16 is the upper half of an fp32: widening is a shift or a mask.
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// ------------------------------------------- programmatic dependent launch

// Wait until the grid this launch depends on (the previous kernel in the
// stream, if it was launched as a programmatic dependency) has completed and
// its memory is visible; a no-op otherwise. Called before the first global
// access, so results never depend on what ran before.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next kernel in the stream to be scheduled now: its CTAs take SMs
// as this grid's CTAs retire and then wait in pdl_wait() for this grid.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ------------------------------------------------------ TMA and mbarriers

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

// make barrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) writes to the same memory
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// one arrival that also announces `bytes` of incoming transactions
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// bulk copy global -> this CTA's shared memory, completion counted on `bar`;
// both addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// bulk prefetch of [src, src + bytes) into L2 (16-byte aligned, bytes a
// multiple of 16)
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// one plain arrival (release semantics at CTA scope)
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return done != 0;
}

// Each try_wait on a phase that does not complete suspends the thread for a
// hardware-chosen interval (3.5 us on GB300, measured with
// tk_diag_unanswered_wait), so this many tries take about 1.8 s: far beyond
// any legitimate copy, after which the kernel gives up on the barrier instead
// of waiting forever.
constexpr uint32_t kSpinLimit = 1u << 19;

__device__ __forceinline__ bool mbar_wait_tries(uint64_t *bar, uint32_t parity, uint32_t tries)
{
    for (uint32_t i = 0; i < tries; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    return false;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    return mbar_wait_tries(bar, parity, kSpinLimit);
}

// ---------------------------------------------------------------- arithmetic

// A pair of fp32 values in one 64-bit register pair, for the f32x2 forms.
__device__ __forceinline__ uint64_t pk(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float plo(uint64_t v)
{
    float lo;
    asm("{\n\t.reg .f32 hi;\n\tmov.b64 {%0, hi}, %1;\n\t}" : "=f"(lo) : "l"(v));
    return lo;
}
__device__ __forceinline__ float phi(uint64_t v)
{
    float hi;
    asm("{\n\t.reg .f32 lo;\n\tmov.b64 {lo, %0}, %1;\n\t}" : "=f"(hi) : "l"(v));
    return hi;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t splat(float v) { return pk(v, v); }

__device__ __forceinline__ float ex2_ftz(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_ftz(float x)
{
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// -(silu(g) * u * w) for the two columns of a pair; w2n = (-w, -w).
// silu(g) = g / (1 + e^{-g}) = max(g * t, g) / (1 + t) with t = e^{-|g|}:
// for g >= 0, g * t <= g; for g < 0, g * t >= g and g * t is the numerator.
__device__ __forceinline__ uint64_t neg_swiglu2(float g0, float g1, float u0, float u1, uint64_t w2n)
{
    constexpr float kNegHalfLog2e = -0.72134752044448170368f;  // -log2(e) / 2
    const uint64_t h = pk(ex2_ftz(__fmul_rn(fabsf(g0), kNegHalfLog2e)),
                          ex2_ftz(__fmul_rn(fabsf(g1), kNegHalfLog2e)));
    const uint64_t t = mul2(h, h);
    const uint64_t gt = mul2(pk(g0, g1), t);
    const uint64_t num = pk(fmaxf(plo(gt), g0), fmaxf(phi(gt), g1));
    const uint64_t den = add2(t, splat(1.0f));
    const uint64_t silu = mul2(num, pk(rcp_ftz(plo(den)), rcp_ftz(phi(den))));
    return mul2(mul2(silu, pk(u0, u1)), w2n);
}

// Correctly rounded quotients y / b of a pair, from ny = -y, b and
// nrb = -RN(1/b): q0 = RN(y * rb) is within one ulp of y / b, the FMA gives
// the exact q0 * b - y, and one correction step RN(q0 + (y - q0 b) rb) is
// RN(y / b) (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", 1990; Muller et al., "Handbook of
// Floating-Point Arithmetic", division with an FMA). Valid while the
// remainder does not underflow: the caller keeps b >= 2^-73, which covers
// every |y / b| >= 2^-11, and smaller quotients encode to a signed zero
// whatever their last bits. With -y as the addend both zeros keep their sign
// (y = -0: q0 = -0, r = +0, q = -0 + -0 = -0; y = +0: +0).
__device__ __forceinline__ uint64_t div_markstein2(uint64_t ny, uint64_t b2, uint64_t nrb2)
{
    const uint64_t q0 = mul2(ny, nrb2);
    const uint64_t r = fma2(q0, b2, ny);
    return fma2(r, nrb2, q0);
}

template <int OUT> struct Fmt;
template <> struct Fmt<kOutE4M3> {
    // 448 = 1.75 * 2^8: exponent 8, fraction bits of 1.75
    static constexpr float kQmax = 448.0f;
    static constexpr float kRcpQmax = 0x1.24924ap-9f;   // RN(1 / 448)
    static constexpr int kQE = 8;
    static constexpr uint32_t kQM = 0x600000u;
};
template <> struct Fmt<kOutE2M1> {
    // 6 = 1.5 * 2^2
    static constexpr float kQmax = 6.0f;
    static constexpr float kRcpQmax = 0x1.555556p-3f;   // RN(1 / 6)
    static constexpr int kQE = 2;
    static constexpr uint32_t kQM = 0x400000u;
};

// Correctly rounded a / b for one value (the pair form's scalar twin).
__device__ __forceinline__ float div_markstein1(float a, float b, float rb)
{
    const float q0 = __fmul_rn(a, rb);
    const float r = __fmaf_rn(-q0, b, a);
    return __fmaf_rn(r, rb, q0);
}

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

// fp32 -> codes, round-to-nearest-even with saturation to the largest
// finite value. The first source of a packed conversion lands in the upper
// half of its result, so the lower column is passed second.
// four fp32 -> four E4M3 codes in one word, the first column in the low byte
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d)
{
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\tcvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\tmov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// eight fp32 -> eight E2M1 codes in one word, column 2k in the low nibble of
// byte k
__device__ __forceinline__ uint32_t cvt_e2m1x8(uint64_t v0, uint64_t v1, uint64_t v2, uint64_t v3)
{
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .f32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
        "mov.b64 {l0, h0}, %1;\n\tmov.b64 {l1, h1}, %2;\n\t"
        "mov.b64 {l2, h2}, %3;\n\tmov.b64 {l3, h3}, %4;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, h0, l0;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, h1, l1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, h2, l2;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, h3, l3;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r) : "l"(v0), "l"(v1), "l"(v2), "l"(v3));
    return r;
}

// Absmax of a scale group spread over the power-of-two lane group that
// tpg_mask + 1 lanes form: one shuffle for groups of one or two lanes, else
// five with offsets past the group masked to 0 (a shuffle with oneself). The
// branch is uniform across the kernel.
__device__ __forceinline__ float group_max(float v, int tpg_mask)
{
    if (tpg_mask <= 1)
        return fmaxf(v, __shfl_xor_sync(kFull, v, tpg_mask));
#pragma unroll
    for (int off = 1; off < 32; off <<= 1)
        v = fmaxf(v, __shfl_xor_sync(kFull, v, off & tpg_mask));
    return v;
}

// ------------------------------------------------------- quantize and store

// Scale the thread's 16 values (held negated, as 8 pairs) by 1/s, with s
// from the group's amax, encode and store them; the group's first thread
// also stores the scale.
// The quotients y / s of one thread's 16 activations (given as -y pairs) and
// the group's scale: s (fp32 mode) or the UE8M0 exponent k. The codes are the
// format's round-to-nearest-even, saturating conversion of v.
template <int OUT, int SCALE>
__device__ __forceinline__ void quantize_values(const uint64_t (&ny)[kEPT / 2], float amax,
                                                uint64_t (&v)[kEPT / 2], float &s, int &k)
{
    if (SCALE == kScaleUE8M0) {
        k = ue8m0_exponent<OUT>(amax);
        // -2^-k (k <= 126 here): the product is the exact power-of-two scaling
        const uint64_t ninv = splat(-__uint_as_float((uint32_t)(127 - k) << 23));
#pragma unroll
        for (int i = 0; i < kEPT / 2; ++i)
            v[i] = mul2(ny[i], ninv);
    } else {
        // amax >= 2^-64 keeps s >= 2^-73 and every remainder above the
        // subnormal range, so both divisions can take the Markstein step;
        // smaller groups (a uniform branch, never taken by ordinary data) use
        // the IEEE division directly.
        if (amax >= 0x1p-64f) {
            s = div_markstein1(amax, Fmt<OUT>::kQmax, Fmt<OUT>::kRcpQmax);
            const uint64_t s2 = splat(s);
            const uint64_t nrs2 = splat(-__frcp_rn(s));
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i)
                v[i] = div_markstein2(ny[i], s2, nrs2);
        } else {
            s = __fdiv_rn(amax, Fmt<OUT>::kQmax);
            if (s == 0.0f)
                s = 1.0f;
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i)
                v[i] = pk(__fdiv_rn(-plo(ny[i]), s), __fdiv_rn(-phi(ny[i]), s));
        }
    }
}

// Store the group's scale (fp32 s, or the UE8M0 byte k + 127) at its index.
template <int SCALE>
__device__ __forceinline__ void store_scale(const RowShape &sh, const OutArgs &o, int64_t row, int group_idx,
                                            float s, int k)
{
    if (SCALE == kScaleUE8M0)
        static_cast<uint8_t *>(o.scales)[scale_index(sh, row, group_idx)] = (uint8_t)(k + 127);
    else
        static_cast<float *>(o.scales)[scale_index(sh, row, group_idx)] = s;
}

// 16 quotients -> 16 E4M3 codes, column order, in four words
__device__ __forceinline__ void e4m3_words(const uint64_t (&v)[kEPT / 2], uint32_t (&w)[4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w[j] = cvt_e4m3x4(plo(v[2 * j]), phi(v[2 * j]), plo(v[2 * j + 1]), phi(v[2 * j + 1]));
}

template <int OUT, int SCALE>
__device__ __forceinline__ void quantize_store(const uint64_t (&ny)[kEPT / 2], float amax, int64_t row,
                                               int col0, int group_idx, bool write_scale,
                                               const RowShape &sh, const OutArgs &o)
{
    uint64_t v[kEPT / 2];
    float s = 0.0f;
    int k = 0;
    quantize_values<OUT, SCALE>(ny, amax, v, s, k);
    if (write_scale)
        store_scale<SCALE>(sh, o, row, group_idx, s, k);
    if (OUT == kOutE4M3) {
        uint32_t w[4];
        e4m3_words(v, w);
        st_stream_128(o.q + row * (int64_t)sh.H + col0, w[0], w[1], w[2], w[3]);
    } else {
        const uint32_t w0 = cvt_e2m1x8(v[0], v[1], v[2], v[3]);
        const uint32_t w1 = cvt_e2m1x8(v[4], v[5], v[6], v[7]);
        st_stream_64(o.q + row * (int64_t)(sh.H / 2) + col0 / 2, w0, w1);
    }
}

// ------------------------------------------------------------ the kernel

// Src supplies: Args (kernel argument); Regs and load(args, row, col0, regs),
// which issues the thread's loads for one row slice; zero(regs);
// produce(args, regs, ok, ny, amax) -> the 16 activations negated as 8 pairs
// and their absmax; finish(args) at kernel exit.
//
// General form: any H that is a multiple of 16, any group size, and one scale
// per row with a CTA-wide reduction. Each thread keeps the next row block's
// loads (64 bytes) in flight while it computes the current one.
// PREFETCH: 0 none; 1 the first row block into L2 before the dependency
// wait; 2 that and, with each block's loads, the block after it into L2.
template <class Src, int OUT, int SCALE, bool CTA_REDUCE, int PREFETCH = 0>
__global__ void __launch_bounds__(kMaxThreads)
row_quant_kernel(typename Src::Args a, OutArgs o, RowShape sh)
{
    __shared__ float red[2][32];
    Src src;
    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    const int slot = tid / sh.tpr;
    const int lr = tid - slot * sh.tpr;
    const bool slot_ok = slot < sh.rpc;
    const int col0 = lr * kEPT;
    const int64_t nrb = (sh.T + sh.rpc - 1) / sh.rpc;
    const int tpg_mask = (1 << sh.tpg_log2) - 1;
    const int group_idx = CTA_REDUCE ? 0 : (lr >> sh.tpg_log2);
    const bool first_of_group = CTA_REDUCE ? (tid == 0) : ((lr & tpg_mask) == 0);
    // PREFETCH (the plan's choice where a CTA has few row blocks, so that the
    // first one's latency is a visible part of the launch): bring the first
    // row block into L2 before waiting on the previous kernel.
    if (PREFETCH >= 1 && slot_ok && (int64_t)blockIdx.x < nrb && (int64_t)blockIdx.x * sh.rpc + slot < sh.T)
        Src::prefetch(a, (int64_t)blockIdx.x * sh.rpc + slot, col0);
    pdl_wait();
    pdl_launch_dependents();
    // Two register sets in turn: while one row block is computed, the next
    // one's loads land in the other set (no register copies between them).
    typename Src::Regs ra, rb_regs;
    const int64_t step = gridDim.x;
    auto row_of = [&](int64_t b) { return b * sh.rpc + slot; };
    auto valid = [&](int64_t b) { return slot_ok && b < nrb && row_of(b) < sh.T; };
    auto fetch = [&](int64_t b, typename Src::Regs &r) {
        if (valid(b))
            Src::load(a, row_of(b), col0, r);
        else
            Src::zero(r);
        if (PREFETCH == 2 && valid(b + step))
            Src::prefetch(a, row_of(b + step), col0);
    };
    int it = 0;
    auto compute = [&](int64_t b, const typename Src::Regs &r) {
        const int64_t row = row_of(b);
        const bool ok = valid(b);
        uint64_t ny[kEPT / 2];
        float amax = 0.0f;
        src.produce(a, r, ok, ny, amax);
        if (CTA_REDUCE) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
            float *buf = red[it & 1];
            if ((tid & 31) == 0)
                buf[tid >> 5] = amax;
            __syncthreads();
            const int nwarps = (nthr + 31) >> 5;
            amax = 0.0f;
            for (int w = 0; w < nwarps; ++w)
                amax = fmaxf(amax, buf[w]);
        } else {
            amax = group_max(amax, tpg_mask);
        }
        if (ok)
            quantize_store<OUT, SCALE>(ny, amax, row, col0, group_idx, first_of_group, sh, o);
        ++it;
    };
    int64_t b = blockIdx.x;
    fetch(b, ra);
    while (b < nrb) {
        fetch(b + step, rb_regs);
        compute(b, ra);
        b += step;
        if (b >= nrb)
            break;
        fetch(b + step, ra);
        compute(b, rb_regs);
        b += step;
    }
    src.finish(a);
}

// ----------------------------------------------------- warp_stream_kernel

constexpr int kStreamThreads = 256;   // 8 warps per CTA

// Src additionally supplies: kSpans spans of kSpanBytes per warp slice (the
// warp's 512 columns of the gate half and of the up half, or of the cast
// input), span(args, row, col_base, s) -> their global addresses,
// fetch_span(slot, lane, regs) -> the lane's bytes from a filled slot, and
// scalar(args, row) -> the optional per-row fp32 (nullptr if none).
//
// Shared memory: warp w owns `stages` slots of kSpans * kSpanBytes bytes at
// w * stages * slot_bytes, and `stages` mbarriers after all rings.
// Task k of a warp (its k-th slice) uses slot k % stages with parity
// (k / stages) & 1; the slot is refilled with task k + stages as soon as the
// warp has read it, before the arithmetic, so `stages` copies stay in flight.
template <class Src, int OUT, int SCALE>
__global__ void __launch_bounds__(kStreamThreads)
warp_stream_kernel(typename Src::Args a, OutArgs o, RowShape sh)
{
    constexpr uint32_t kSlot = Src::kSpans * Src::kSpanBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    Src src;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = sh.stages;
    const int nwarps = blockDim.x >> 5;
    uint8_t *ring = smem + (size_t)warp * S * kSlot;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)nwarps * S * kSlot) + warp * S;
    const int tpg_mask = (1 << sh.tpg_log2) - 1;

    // Task t of the grid is slice t % wpr of row t / wpr; a warp takes tasks
    // first, first + stride, ... Cursors hold (row, slice) and advance by the
    // stride's quotient and remainder, so no division runs per task.
    const int stride = (int)gridDim.x * nwarps;          // < 2^31: grid <= SMs * CTAs per SM
    const int d_row = stride / sh.wpr;
    const int d_sl = stride - d_row * sh.wpr;
    struct Cursor {
        int64_t row;
        int sl;
    };
    auto advance = [&](Cursor &c) {
        c.row += d_row;
        c.sl += d_sl;
        if (c.sl >= sh.wpr) {
            c.sl -= sh.wpr;
            ++c.row;
        }
    };
    const int first = (int)blockIdx.x * nwarps + warp;
    Cursor cur{first / sh.wpr, first % sh.wpr};

    auto issue = [&](const Cursor &c, int slot) {   // lane 0 only
        uint8_t *dst = ring + (size_t)slot * kSlot;
        mbar_arrive_expect_tx(bars + slot, kSlot);
#pragma unroll
        for (int sp = 0; sp < Src::kSpans; ++sp)
            bulk_g2s(dst + sp * Src::kSpanBytes, Src::span(a, c.row, c.sl * 512, sp), Src::kSpanBytes,
                     bars + slot);
    };

    pdl_wait();
    pdl_launch_dependents();
    Cursor fill = cur;   // the next task to copy in
    if (lane == 0) {
        for (int i = 0; i < S; ++i)
            mbar_init(bars + i, 1);
        fence_mbar_init();
    }
    for (int i = 0; i < S; ++i) {
        if (lane == 0 && fill.row < sh.T)
            issue(fill, i);
        advance(fill);
    }
    __syncwarp();

    const float *wp = cur.row < sh.T ? Src::scalar(a, cur.row) : nullptr;
    float w_next = wp ? __ldg(wp) : 1.0f;
    int slot = 0;
    uint32_t parity = 0;
    while (cur.row < sh.T) {
        const int64_t row = cur.row;
        const int cbase = cur.sl * 512;
        const float w_cur = w_next;
        advance(cur);
        if (cur.row < sh.T) {
            const float *np = Src::scalar(a, cur.row);
            w_next = np ? __ldg(np) : 1.0f;
        }
        if (!mbar_wait_bounded(bars + slot, parity)) {
            // give up: flag it, let the copies already issued land, leave
            if (lane == 0)
                atomicOr(sh.fault, 1u);
            int sl = slot;
            uint32_t par = parity;
            Cursor c = cur;
            for (int i = 1; i < S; ++i) {
                if (++sl == S) {
                    sl = 0;
                    par ^= 1u;
                }
                if (c.row < sh.T)
                    mbar_wait_bounded(bars + sl, par);
                advance(c);
            }
            return;
        }
        typename Src::Regs regs;
        Src::fetch_span(ring + (size_t)slot * kSlot, lane, regs);
        Src::set_scalar(regs, w_cur);
        __syncwarp();
        if (fill.row < sh.T) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(fill, slot);
            }
        }
        advance(fill);

        uint64_t ny[kEPT / 2];
        float amax = 0.0f;
        src.produce(a, regs, true, ny, amax);
        amax = group_max(amax, tpg_mask);
        const int lr = (cbase >> 4) + lane;
        quantize_store<OUT, SCALE>(ny, amax, row, cbase + lane * kEPT, lr >> sh.tpg_log2,
                                   (lr & tpg_mask) == 0, sh, o);
        if (++slot == S) {
            slot = 0;
            parity ^= 1u;
        }
    }
    src.finish(a);
}

// ---------------------------------------------------- block_stream_kernel

constexpr int kBlockConsumerWarps = 8;
constexpr int kBlockThreads = 32 * (kBlockConsumerWarps + 1);   // + 1 producer warp

// Src additionally supplies kRowBytesPerCol (bytes of one input row per
// column of H) and fetch_block(row, H, s, lane, regs): the lane's bytes of
// the row's 512-column slice s from a whole row held in shared memory.
//
// The CTA's kBlockConsumerWarps consumer warps share one ring of `stages`
// slots; a slot holds sh.rpc consecutive whole rows of the input, which lie
// contiguously in memory, so one TMA bulk copy by the producer warp (the
// last warp, one lane) fills it. CTA b takes row blocks b, b + grid, ...;
// a block's rpc * wpr tasks (a task: one 512-column slice of one row) go to
// the consumer warps in turn, and the count runs on across blocks (task t of
// the CTA -> warp t % kBlockConsumerWarps). full[s] completes when the copy
// has landed; empty[s] takes one arrival per task, so it completes once every
// task of the block has been read out of the slot. The plan keeps
// rpc * wpr >= kBlockConsumerWarps: every warp then has a task in every full
// block, so no warp can get a whole ring ahead of a barrier's phase.
// Against warp_stream_kernel this moves the copies off the consumer warps
// and makes them one per block instead of two per slice.
template <class Src, int OUT, int SCALE>
__global__ void __launch_bounds__(kBlockThreads, 3)
block_stream_kernel(typename Src::Args a, OutArgs o, RowShape sh)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = sh.stages;
    const int RB = sh.rpc;
    const uint32_t row_bytes = (uint32_t)Src::kRowBytesPerCol * (uint32_t)sh.H;
    const uint32_t slot_bytes = (uint32_t)RB * row_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * slot_bytes);
    uint64_t *empty = full + S;
    const int64_t nblk = (sh.T + RB - 1) / RB;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, (uint32_t)(RB * sh.wpr));
        }
        fence_mbar_init();
    }
    // the producer's first slots into L2 while the previous kernel drains
    // (a hint: the copies themselves run after the wait)
    if (warp == kBlockConsumerWarps && lane == 0) {
        int64_t blk = blockIdx.x;
        for (int i = 0; i < S && blk < nblk; ++i, blk += gridDim.x) {
            const int64_t left = sh.T - blk * RB;
            const uint32_t bytes = (uint32_t)(left < RB ? left : RB) * row_bytes;
            bulk_prefetch_l2(Src::span(a, blk * RB, 0, 0), bytes);
        }
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    if (warp == kBlockConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane != 0)
            return;
        int slot = 0;
        uint32_t par = 0;   // parity of the slot's current use
        int64_t issued = 0;
        for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
            // the slot's previous block must have been read out entirely
            if (issued >= S && !mbar_wait_bounded(empty + slot, par ^ 1u)) {
                atomicOr(sh.fault, 1u);
                break;
            }
            const int64_t row0 = blk * RB;
            const int64_t left = sh.T - row0;
            const uint32_t bytes = (uint32_t)(left < RB ? left : RB) * row_bytes;
            mbar_arrive_expect_tx(full + slot, bytes);
            bulk_g2s(smem + (size_t)slot * slot_bytes, Src::span(a, row0, 0, 0), bytes, full + slot);
            ++issued;
            if (++slot == S) {
                slot = 0;
                par ^= 1u;
            }
        }
        // every copy this CTA issued lands before its shared memory goes away
        for (int s = 0; s < S && s < issued; ++s) {
            const int64_t last_use = (issued - 1 - s) / S;
            if (!mbar_wait_bounded(full + s, (uint32_t)(last_use & 1)))
                atomicOr(sh.fault, 1u);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    Src src;
    const int wpr = sh.wpr;
    const int tpg_mask = (1 << sh.tpg_log2) - 1;
    const int d_rl = kBlockConsumerWarps / wpr;   // the step of kBlockConsumerWarps tasks
    const int d_s = kBlockConsumerWarps - d_rl * wpr;
    int rl = warp / wpr;   // row within the block
    int s = warp - rl * wpr;   // slice within the row
    int slot = 0;
    uint32_t par = 0;
    int64_t row0 = (int64_t)blockIdx.x * RB;
    const int64_t row_step = (int64_t)gridDim.x * RB;
    while (row0 + rl < sh.T) {
        const int64_t row = row0 + rl;
        const float *wp = Src::scalar(a, row);
        const float w = wp ? __ldg(wp) : 1.0f;
        if (!mbar_wait_bounded(full + slot, par)) {
            if (lane == 0)
                atomicOr(sh.fault, 1u);
            return;
        }
        typename Src::Regs regs;
        Src::fetch_block(smem + (size_t)slot * slot_bytes + (size_t)rl * row_bytes, sh.H, s, lane, regs);
        Src::set_scalar(regs, w);
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty + slot);

        uint64_t ny[kEPT / 2];
        float amax = 0.0f;
        src.produce(a, regs, true, ny, amax);
        amax = group_max(amax, tpg_mask);
        const int lr = s * 32 + lane;   // the lane's 16-column unit within the row
        quantize_store<OUT, SCALE>(ny, amax, row, lr * kEPT, lr >> sh.tpg_log2, (lr & tpg_mask) == 0, sh, o);

        s += d_s;
        if (s >= wpr) {
            s -= wpr;
            ++rl;
        }
        rl += d_rl;
        if (rl >= RB) {   // at most one block further: rpc * wpr >= kBlockConsumerWarps
            rl -= RB;
            row0 += row_step;
            if (++slot == S) {
                slot = 0;
                par ^= 1u;
            }
        }
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
    uint32_t limit2;              // the limit as bf16 in both halves (when packed_clamp)
    int32_t packed_clamp;         // the limit is exact in bf16: clamp and count on packed bf16 pairs
};

// bf16x2 lane-wise min, max and comparisons (all-ones or zero per 16-bit lane)
__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_gt_mask(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t bf16x2_ne_mask(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("set.ne.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// lane-wise max(|a|, |b|), its sign bit the xor of a's and b's
__device__ __forceinline__ uint32_t bf16x2_max_abs(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

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
    __device__ __forceinline__ static void prefetch(const Args &a, int64_t row, int col0)
    {
        const uint16_t *p = a.x + row * (2 * (int64_t)a.H) + col0;
        prefetch_l2(p);
        prefetch_l2(p + a.H);
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

    static constexpr int kSpans = 2;          // the gate half, the up half
    static constexpr int kSpanBytes = 1024;   // 512 bf16 columns

    __device__ __forceinline__ static const void *span(const Args &a, int64_t row, int cbase, int sp)
    {
        return a.x + row * (2 * (int64_t)a.H) + sp * a.H + cbase;
    }
    __device__ __forceinline__ static const float *scalar(const Args &a, int64_t row)
    {
        return a.w ? a.w + row : nullptr;
    }
    __device__ __forceinline__ static void fetch_span(const uint8_t *slot, int lane, Regs &r)
    {
        fetch_pair(slot + lane * 32, slot + 1024 + lane * 32, r);
    }
    // block_stream_kernel: a whole row (H gate columns, then H up columns)
    // sits in shared memory; the lane's 16 columns of its 512-column slice s
    static constexpr int kRowBytesPerCol = 4;
    __device__ __forceinline__ static void fetch_block(const uint8_t *row, int H, int s, int lane, Regs &r)
    {
        fetch_pair(row + s * 1024 + lane * 32, row + 2 * H + s * 1024 + lane * 32, r);
    }
    __device__ __forceinline__ static void fetch_pair(const uint8_t *gp, const uint8_t *up, Regs &r)
    {
        const uint4 *g = reinterpret_cast<const uint4 *>(gp);
        const uint4 *u = reinterpret_cast<const uint4 *>(up);
        const uint4 g0 = g[0], g1 = g[1], u0 = u[0], u1 = u[1];
        r.g[0] = g0.x; r.g[1] = g0.y; r.g[2] = g0.z; r.g[3] = g0.w;
        r.g[4] = g1.x; r.g[5] = g1.y; r.g[6] = g1.z; r.g[7] = g1.w;
        r.u[0] = u0.x; r.u[1] = u0.y; r.u[2] = u0.z; r.u[3] = u0.w;
        r.u[4] = u1.x; r.u[5] = u1.y; r.u[6] = u1.z; r.u[7] = u1.w;
    }
    __device__ __forceinline__ static void set_scalar(Regs &r, float w) { r.w = w; }
    __device__ __forceinline__ void produce(const Args &a, const Regs &r, bool ok,
                                            uint64_t (&ny)[kEPT / 2], float &amax)
    {
        const float L = a.limit;
        const uint64_t w2n = splat(-r.w);
        if (CLAMP && a.packed_clamp) {
            // The limit is a bf16 value, so clamping the bf16 inputs is exact
            // and two lanes go per instruction. Most threads hold no value
            // beyond the limit: the packed max of the gate values, and of the
            // up values' magnitudes, shows that for each half (14 instructions
            // for the thread's 32 inputs), and only a half that has one is
            // clamped and counted. A lane's clamp is recorded as one bit (bit
            // i of its half for pair i); popc counts them.
            const uint32_t L2 = a.limit2, nL2 = a.limit2 ^ 0x80008000u;
            uint32_t g[8], u[8];
            uint32_t gm = r.g[0], um = r.u[0];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                g[i] = r.g[i];
                u[i] = r.u[i];
                if (i) {
                    gm = bf16x2_max(gm, g[i]);
                    um = bf16x2_max_abs(um, u[i]);
                }
            }
            if (bf16x2_gt_mask(gm, L2)) {
                uint32_t mg = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    mg |= bf16x2_gt_mask(g[i], L2) & (0x00010001u << i);
                    g[i] = bf16x2_min(g[i], L2);
                }
                if (ok)
                    cnt_g += __popc(mg);
            }
            if (bf16x2_gt_mask(um & 0x7FFF7FFFu, L2)) {
                uint32_t mu = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t uc = bf16x2_max(bf16x2_min(u[i], L2), nL2);
                    mu |= bf16x2_ne_mask(uc, u[i]) & (0x00010001u << i);
                    u[i] = uc;
                }
                if (ok)
                    cnt_u += __popc(mu);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                ny[i] = neg_swiglu2(bf16_lo(g[i]), bf16_hi(g[i]), bf16_lo(u[i]), bf16_hi(u[i]), w2n);
                amax = fmaxf(amax, fmaxf(fabsf(plo(ny[i])), fabsf(phi(ny[i]))));
            }
            return;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float g0 = bf16_lo(r.g[i]), g1 = bf16_hi(r.g[i]);
            float u0 = bf16_lo(r.u[i]), u1 = bf16_hi(r.u[i]);
            if (CLAMP) {
                cnt_g += (ok && g0 > L) ? 1u : 0u;
                cnt_g += (ok && g1 > L) ? 1u : 0u;
                cnt_u += (ok && fabsf(u0) > L) ? 1u : 0u;
                cnt_u += (ok && fabsf(u1) > L) ? 1u : 0u;
                g0 = fminf(g0, L);
                g1 = fminf(g1, L);
                u0 = fminf(fmaxf(u0, -L), L);
                u1 = fminf(fmaxf(u1, -L), L);
            }
            ny[i] = neg_swiglu2(g0, g1, u0, u1, w2n);
            amax = fmaxf(amax, fmaxf(fabsf(plo(ny[i])), fabsf(phi(ny[i]))));
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
    __device__ __forceinline__ static void prefetch(const Args &a, int64_t row, int col0)
    {
        prefetch_l2(static_cast<const uint16_t *>(a.x) + row * (int64_t)a.H + col0);
    }

    __device__ __forceinline__ static void zero(Regs &r)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            r.v[i] = 0u;
    }

    static constexpr int kSpans = 1;
    static constexpr int kSpanBytes = 1024;   // 512 bf16 columns

    __device__ __forceinline__ static const void *span(const Args &a, int64_t row, int cbase, int)
    {
        return static_cast<const uint16_t *>(a.x) + row * (int64_t)a.H + cbase;
    }
    __device__ __forceinline__ static const float *scalar(const Args &, int64_t) { return nullptr; }
    static constexpr int kRowBytesPerCol = 2;
    __device__ __forceinline__ static void fetch_block(const uint8_t *row, int, int s, int lane, Regs &r)
    {
        fetch_span(row + s * kSpanBytes, lane, r);
    }
    __device__ __forceinline__ static void fetch_span(const uint8_t *slot, int lane, Regs &r)
    {
        const uint4 *p = reinterpret_cast<const uint4 *>(slot + lane * 32);
        const uint4 c0 = p[0], c1 = p[1];
        r.v[0] = c0.x; r.v[1] = c0.y; r.v[2] = c0.z; r.v[3] = c0.w;
        r.v[4] = c1.x; r.v[5] = c1.y; r.v[6] = c1.z; r.v[7] = c1.w;
    }
    __device__ __forceinline__ static void set_scalar(Regs &, float) {}
    __device__ __forceinline__ void produce(const Args &, const Regs &r, bool, uint64_t (&ny)[kEPT / 2],
                                            float &amax)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y0 = bf16_lo(r.v[i]), y1 = bf16_hi(r.v[i]);
            ny[i] = pk(-y0, -y1);
            amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
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
    __device__ __forceinline__ static void prefetch(const Args &a, int64_t row, int col0)
    {
        prefetch_l2(static_cast<const float *>(a.x) + row * (int64_t)a.H + col0);
    }

    __device__ __forceinline__ static void zero(Regs &r)
    {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            r.v[i] = 0u;
    }

    static constexpr int kSpans = 1;
    static constexpr int kSpanBytes = 2048;   // 512 fp32 columns

    __device__ __forceinline__ static const void *span(const Args &a, int64_t row, int cbase, int)
    {
        return static_cast<const float *>(a.x) + row * (int64_t)a.H + cbase;
    }
    __device__ __forceinline__ static const float *scalar(const Args &, int64_t) { return nullptr; }
    static constexpr int kRowBytesPerCol = 4;
    __device__ __forceinline__ static void fetch_block(const uint8_t *row, int, int s, int lane, Regs &r)
    {
        fetch_span(row + s * kSpanBytes, lane, r);
    }
    __device__ __forceinline__ static void fetch_span(const uint8_t *slot, int lane, Regs &r)
    {
        const uint4 *p = reinterpret_cast<const uint4 *>(slot + lane * 64);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 c = p[k];
            r.v[4 * k] = c.x;
            r.v[4 * k + 1] = c.y;
            r.v[4 * k + 2] = c.z;
            r.v[4 * k + 3] = c.w;
        }
    }
    __device__ __forceinline__ static void set_scalar(Regs &, float) {}
    __device__ __forceinline__ void produce(const Args &, const Regs &r, bool, uint64_t (&ny)[kEPT / 2],
                                            float &amax)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y0 = __uint_as_float(r.v[2 * i]), y1 = __uint_as_float(r.v[2 * i + 1]);
            ny[i] = pk(-y0, -y1);
            amax = fmaxf(amax, fmaxf(fabsf(y0), fabsf(y1)));
        }
    }
    __device__ __forceinline__ void finish(const Args &) {}
};

}  // namespace tk
