// Per-channel cast, sm_103a: one scale per column j of x [T, H], from the
// absolute maximum of column j over all T rows; every value of the column is
// scaled by it and encoded ("TileLang + TileKernels：DeepSeek 的 GPU 内核开发新范式",
// zhichai.net/topic/177618740, section "3. Quantization", format table: the
// per-channel granularity of FP8 E4M3).
//
// A column's scale depends on every row, so no row can be encoded before the
// whole input has been read once: the cast reads x twice. Two or three
// launches, chained by programmatic dependent launch (each waits for the
// previous one in griddepcontrol.wait before its first global access):
//
//  1. col_amax_kernel: CTA (c, s) takes the 512-column chunk c of the row
//     slab s; its eight warps take the slab's rows in turn (warp w: rows
//     w, w + 8, ...), a lane 16 columns of each (32-byte loads), two sets of
//     rows in flight, keeping the running |x| maximum in registers (bf16
//     pairs by packed max, exact). The warps' maxima meet in shared memory
//     and the CTA writes one fp32 partial maximum per column: partial[s, col].
//  2. Either col_chunk_quant_kernel on the same grid: CTA (c, s) reduces the
//     partials of its own 512 columns into their scales (the slab-0 CTA also
//     stores them) and encodes its slab of that chunk, last row first, where
//     the amax pass has left the slab's last rows in L2 (evict_last);
//     or col_scale_kernel (one CTA per 32 columns reduces the partials into
//     the scales) followed by col_quant_kernel: the row kernel's mapping (16
//     columns per thread, H / 16 threads per row, a persistent grid over row
//     blocks from the last one back, the next block's loads in flight), each
//     thread holding its 16 column scales. The first saves a launch and suits outputs that L2
//     absorbs; the second writes whole rows in sequence, which large outputs
//     need. Either way a value costs one correctly rounded quotient
//     (Markstein's correction, or an exact power-of-two multiply) and its
//     share of a packed conversion.
#include "tk_channel.h"

namespace tk {

namespace {

constexpr int kAmaxWarps = 8;
constexpr int kAmaxThreads = 32 * kAmaxWarps;
// rows per load set (two sets in flight per warp): 32 bytes of a bf16 row,
// 64 of an fp32 row per lane
template <bool BF16> constexpr int kAmaxUnroll = BF16 ? 4 : 2;

// Running |x| maximum of a lane's 16 columns.
template <bool BF16> struct AbsMax;

template <> struct AbsMax<true> {
    uint32_t m[8];   // bf16 pairs; |x| of a bf16 is its bits without the sign
    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            m[i] = 0u;
    }
    __device__ __forceinline__ void add(const CastBf16Src::Regs &r)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            m[i] = bf16x2_max(m[i], r.v[i] & 0x7fff7fffu);
    }
    __device__ __forceinline__ void out(float (&f)[kEPT]) const
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            f[2 * i] = bf16_lo(m[i]);
            f[2 * i + 1] = bf16_hi(m[i]);
        }
    }
};

template <> struct AbsMax<false> {
    float m[kEPT];
    __device__ __forceinline__ void init()
    {
#pragma unroll
        for (int i = 0; i < kEPT; ++i)
            m[i] = 0.0f;
    }
    __device__ __forceinline__ void add(const CastF32Src::Regs &r)
    {
#pragma unroll
        for (int i = 0; i < kEPT; ++i)
            m[i] = fmaxf(m[i], fabsf(__uint_as_float(r.v[i])));
    }
    __device__ __forceinline__ void out(float (&f)[kEPT]) const
    {
#pragma unroll
        for (int i = 0; i < kEPT; ++i)
            f[i] = m[i];
    }
};

// 32-byte read-only loads with an L2 eviction priority (EV 1: evict_first,
// 2: evict_last). Before the chunk quantize pass, the amax pass marks the
// rows that pass reads first (the end of each slab) evict_last and the rest
// evict_first, so that what L2 keeps between the passes is what is reread
// soonest; the chunk pass reads evict_first, which also takes the kept lines
// back to the lowest priority once they have been used. (Before the row
// quantize pass, whose input does not fit L2 anyway, plain loads measured
// faster than any split of the priorities.)
template <int EV>
__device__ __forceinline__ void ld_ev_256(const void *p, uint32_t (&r)[8])
{
    if (EV == 2)
        asm("ld.global.nc.L1::no_allocate.L2::evict_last.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
            : "l"(p));
    else
        asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
            : "l"(p));
}

template <int EV, class Src>
__device__ __forceinline__ void load_ev(const CastArgs &a, int64_t row, int col0, typename Src::Regs &r)
{
    if constexpr (Src::kRowBytesPerCol == 2) {
        ld_ev_256<EV>(static_cast<const uint16_t *>(a.x) + row * (int64_t)a.H + col0, r.v);
    } else {
        const float *p = static_cast<const float *>(a.x) + row * (int64_t)a.H + col0;
        uint32_t (&lo)[8] = *reinterpret_cast<uint32_t (*)[8]>(&r.v[0]);
        uint32_t (&hi)[8] = *reinterpret_cast<uint32_t (*)[8]>(&r.v[8]);
        ld_ev_256<EV>(p, lo);
        ld_ev_256<EV>(p + 8, hi);
    }
}

template <class Src, bool BF16, bool PREFETCH, bool KEEP>
__global__ void __launch_bounds__(kAmaxThreads, 2) col_amax_kernel(CastArgs a, int64_t T, int64_t slab_rows,
                                                               float *partial, int64_t keep_slab)
{
    __shared__ __align__(16) float red[kAmaxWarps][512];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk0 = (int)blockIdx.x * 512;
    const int col0 = chunk0 + lane * kEPT;
    const bool col_ok = col0 < a.H;
    const int64_t r0 = (int64_t)blockIdx.y * slab_rows;
    const int64_t r1 = (T - r0) < slab_rows ? T : r0 + slab_rows;
    // PREFETCH (short slabs, where the first rows' latency is a visible part
    // of the launch): the warp's first set of rows into L2 before the wait
    if (PREFETCH && col_ok)
        for (int u = 0; u < kAmaxUnroll<BF16>; ++u) {
            const int64_t row = r0 + warp + (int64_t)u * kAmaxWarps;
            if (row < r1)
                Src::prefetch(a, row, col0);
        }
    pdl_wait();
    pdl_launch_dependents();
    AbsMax<BF16> acc;
    acc.init();
    // Two sets of U rows in turn: the next set's loads are issued before the
    // current set is reduced, so 2U rows stay in flight per warp.
    constexpr int U = kAmaxUnroll<BF16>;
    constexpr int64_t kStep = U * kAmaxWarps;
    typename Src::Regs va[U], vb[U];
    auto fetch = [&](int64_t r, typename Src::Regs (&v)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = r + (int64_t)u * kAmaxWarps;
            if (col_ok && row < r1) {
                if (!KEEP)
                    Src::load(a, row, col0, v[u]);
                else if (row - r0 >= slab_rows - keep_slab)
                    load_ev<2, Src>(a, row, col0, v[u]);
                else
                    load_ev<1, Src>(a, row, col0, v[u]);
            } else {
                Src::zero(v[u]);
            }
        }
    };
    auto reduce = [&](const typename Src::Regs (&v)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u)
            acc.add(v[u]);
    };
    int64_t r = r0 + warp;
    fetch(r, va);
    while (r < r1) {
        fetch(r + kStep, vb);
        reduce(va);
        r += kStep;
        if (r >= r1)
            break;
        fetch(r + kStep, va);
        reduce(vb);
        r += kStep;
    }
    float f[kEPT];
    acc.out(f);
    float4 *dst = reinterpret_cast<float4 *>(&red[warp][lane * kEPT]);
#pragma unroll
    for (int k = 0; k < kEPT / 4; ++k)
        dst[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
    __syncthreads();
    for (int c = threadIdx.x; c < 512; c += kAmaxThreads) {
        float m = red[0][c];
#pragma unroll
        for (int w = 1; w < kAmaxWarps; ++w)
            m = fmaxf(m, red[w][c]);
        if (chunk0 + c < a.H)
            partial[(int64_t)blockIdx.y * a.H + chunk0 + c] = m;
    }
}

constexpr int kScaleThreads = 1024;   // 32 columns x 32 partial strides

template <int OUT, int SCALE>
__global__ void __launch_bounds__(kScaleThreads) col_scale_kernel(const float *partial, int slabs, int H,
                                                                   void *scales)
{
    __shared__ float red[32][33];
    const int tx = threadIdx.x & 31;
    const int ty = threadIdx.x >> 5;
    const int c = (int)blockIdx.x * 32 + tx;
    pdl_wait();
    pdl_launch_dependents();
    // independent loads, four at a time, so their latencies overlap
    float m = 0.0f;
    if (c < H) {
        float m1 = 0.0f, m2 = 0.0f, m3 = 0.0f;
        int s = ty;
        for (; s + 96 < slabs; s += 128) {
            const float *p = partial + (int64_t)s * H + c;
            m = fmaxf(m, p[0]);
            m1 = fmaxf(m1, p[32 * (int64_t)H]);
            m2 = fmaxf(m2, p[64 * (int64_t)H]);
            m3 = fmaxf(m3, p[96 * (int64_t)H]);
        }
        for (; s < slabs; s += 32)
            m = fmaxf(m, partial[(int64_t)s * H + c]);
        m = fmaxf(fmaxf(m, m1), fmaxf(m2, m3));
    }
    red[ty][tx] = m;
    __syncthreads();
    if (ty != 0 || c >= H)
        return;
#pragma unroll 8
    for (int k = 1; k < 32; ++k)
        m = fmaxf(m, red[k][tx]);
    if (SCALE == kScaleUE8M0) {
        static_cast<uint8_t *>(scales)[c] = (uint8_t)(ue8m0_exponent<OUT>(m) + 127);
    } else {
        // the per-block cast's rule: correctly rounded m / Qmax, 1 for zero
        float s;
        if (m >= 0x1p-64f) {
            s = div_markstein1(m, Fmt<OUT>::kQmax, Fmt<OUT>::kRcpQmax);
        } else {
            s = __fdiv_rn(m, Fmt<OUT>::kQmax);
            if (s == 0.0f)
                s = 1.0f;
        }
        static_cast<float *>(scales)[c] = s;
    }
}

// The 16 column scales of one thread as pair operands of the quotient:
// s2 = (s_a, s_b) and nr2 = (-RN(1/s_a), -RN(1/s_b)) in fp32 mode, or
// nr2 = (-2^-k_a, -2^-k_b) in UE8M0 mode. Markstein's step needs s >= 2^-73
// (else its remainder can underflow); a column with a smaller scale (its
// maximum is below about 2^-64, never ordinary data) keeps s * 2^100 and
// -RN(1/(s * 2^100)) instead, and its values are multiplied by 2^100 before
// the division. Both scalings are exact (y stays below 448 * 2^27), so the
// quotient is the same real number and its correct rounding the same fp32.
// Bit i of `tiny` marks such a column.
template <int SCALE> struct ColScales {
    uint64_t s2[kEPT / 2];
    uint64_t nr2[kEPT / 2];
    uint32_t tiny;

    __device__ __forceinline__ void load(const void *scales, int col0)
    {
        tiny = 0u;
        if (SCALE == kScaleUE8M0) {
            const uint4 b = *reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(scales) + col0);
            const uint32_t w[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i) {
                const uint32_t byte_a = (w[i >> 1] >> (16 * (i & 1))) & 0xffu;
                const uint32_t byte_b = (w[i >> 1] >> (16 * (i & 1) + 8)) & 0xffu;
                // byte = k + 127, so 2^-k has the biased exponent 254 - byte
                // (byte <= 253 for any finite amax)
                nr2[i] = pk(-__uint_as_float((254u - byte_a) << 23), -__uint_as_float((254u - byte_b) << 23));
                s2[i] = 0;
            }
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(scales) + col0);
            float sc[kEPT];
#pragma unroll
            for (int k = 0; k < kEPT / 4; ++k) {
                const float4 v = p[k];
                sc[4 * k] = v.x;
                sc[4 * k + 1] = v.y;
                sc[4 * k + 2] = v.z;
                sc[4 * k + 3] = v.w;
            }
#pragma unroll
            for (int j = 0; j < kEPT; ++j) {
                if (sc[j] < 0x1p-73f) {
                    sc[j] = __fmul_rn(sc[j], 0x1p100f);
                    tiny |= 1u << j;
                }
            }
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i) {
                s2[i] = pk(sc[2 * i], sc[2 * i + 1]);
                nr2[i] = pk(-__frcp_rn(sc[2 * i]), -__frcp_rn(sc[2 * i + 1]));
            }
        }
    }

    // quotients y / s of the 16 values, given as -y pairs
    __device__ __forceinline__ void divide(const uint64_t (&ny)[kEPT / 2], uint64_t (&v)[kEPT / 2]) const
    {
        if (SCALE == kScaleUE8M0) {
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i)
                v[i] = mul2(ny[i], nr2[i]);
        } else if (tiny == 0u) {
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i)
                v[i] = div_markstein2(ny[i], s2[i], nr2[i]);
        } else {
#pragma unroll
            for (int i = 0; i < kEPT / 2; ++i) {
                const uint64_t k2 = pk((tiny >> (2 * i)) & 1u ? 0x1p100f : 1.0f,
                                       (tiny >> (2 * i + 1)) & 1u ? 0x1p100f : 1.0f);
                v[i] = div_markstein2(mul2(ny[i], k2), s2[i], nr2[i]);
            }
        }
    }
};

template <class Src, int OUT, int SCALE, int MAXT>
__global__ void __launch_bounds__(MAXT) col_quant_kernel(CastArgs a, OutArgs o, RowShape sh)
{
    Src src;
    const int tid = threadIdx.x;
    const int slot = tid / sh.tpr;
    const int lr = tid - slot * sh.tpr;
    const bool slot_ok = slot < sh.rpc;
    const int col0 = lr * kEPT;
    const int64_t nrb = (sh.T + sh.rpc - 1) / sh.rpc;
    pdl_wait();
    pdl_launch_dependents();
    ColScales<SCALE> cs;
    cs.load(o.scales, slot_ok ? col0 : 0);
    typename Src::Regs ra, rb_regs;
    const int64_t step = gridDim.x;
    // the last row block first: the amax pass read the bottom rows last, so
    // those are the ones most likely still in L2
    auto row_of = [&](int64_t b) { return (nrb - 1 - b) * sh.rpc + slot; };
    auto valid = [&](int64_t b) { return slot_ok && b < nrb && row_of(b) < sh.T; };
    auto fetch = [&](int64_t b, typename Src::Regs &r) {
        if (valid(b))
            Src::load(a, row_of(b), col0, r);
        else
            Src::zero(r);
    };
    auto compute = [&](int64_t b, const typename Src::Regs &r) {
        if (!valid(b))
            return;
        const int64_t row = row_of(b);
        uint64_t ny[kEPT / 2];
        float amax_unused = 0.0f;
        src.produce(a, r, true, ny, amax_unused);
        uint64_t v[kEPT / 2];
        cs.divide(ny, v);
        if (OUT == kOutE4M3) {
            uint32_t w[4];
            e4m3_words(v, w);
            st_stream_128(o.q + row * (int64_t)sh.H + col0, w[0], w[1], w[2], w[3]);
        } else {
            const uint32_t w0 = cvt_e2m1x8(v[0], v[1], v[2], v[3]);
            const uint32_t w1 = cvt_e2m1x8(v[4], v[5], v[6], v[7]);
            st_stream_64(o.q + row * (int64_t)(sh.H / 2) + col0 / 2, w0, w1);
        }
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
}

// Rows per load set of the chunk quantize pass (two sets in flight per
// warp): what the registers allow beside the 16 column scales.
template <bool BF16, int SCALE>
constexpr int kChunkUnroll = BF16 ? (SCALE == kScaleUE8M0 ? 3 : 2) : (SCALE == kScaleUE8M0 ? 2 : 1);

// The quantize pass over the amax pass's grid: CTA (c, s) takes the same
// 512-column chunk c and row slab s. It first reduces the slabs' partial
// maxima of its own 512 columns (warp w reads slabs w, w + 8, ...; the warps
// meet in shared memory) into the chunk's scales, which the slab-0 CTA of the
// chunk also writes out; so no separate scale kernel runs. It then walks its
// slab from the last row back: the amax pass read each slab front to back,
// so the rows it read last, the ones most likely still in L2, come first.
template <class Src, bool BF16, int OUT, int SCALE>
__global__ void __launch_bounds__(kAmaxThreads, 2) col_chunk_quant_kernel(CastArgs a, int64_t T, int64_t slab_rows,
                                                                        const float *partial, int slabs, OutArgs o)
{
    __shared__ __align__(16) float red[kAmaxWarps][512];
    __shared__ __align__(16) uint8_t sclbuf[512 * 4];   // the chunk's scales, in the output's format
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int chunk0 = (int)blockIdx.x * 512;
    const int col0 = chunk0 + lane * kEPT;
    const bool col_ok = col0 < a.H;
    const int64_t r0 = (int64_t)blockIdx.y * slab_rows;
    const int64_t r1 = (T - r0) < slab_rows ? T : r0 + slab_rows;
    pdl_wait();
    pdl_launch_dependents();

    // 1. the chunk's column maxima over every slab's partial
    {
        float m[kEPT];
#pragma unroll
        for (int j = 0; j < kEPT; ++j)
            m[j] = 0.0f;
        if (col_ok)
            for (int sl = warp; sl < slabs; sl += kAmaxWarps) {
                const float4 *p = reinterpret_cast<const float4 *>(partial + (int64_t)sl * a.H + col0);
#pragma unroll
                for (int k = 0; k < kEPT / 4; ++k) {
                    const float4 v = p[k];
                    m[4 * k] = fmaxf(m[4 * k], v.x);
                    m[4 * k + 1] = fmaxf(m[4 * k + 1], v.y);
                    m[4 * k + 2] = fmaxf(m[4 * k + 2], v.z);
                    m[4 * k + 3] = fmaxf(m[4 * k + 3], v.w);
                }
            }
        float4 *dst = reinterpret_cast<float4 *>(&red[warp][lane * kEPT]);
#pragma unroll
        for (int k = 0; k < kEPT / 4; ++k)
            dst[k] = make_float4(m[4 * k], m[4 * k + 1], m[4 * k + 2], m[4 * k + 3]);
    }
    __syncthreads();
    // 2. amax -> scale, by the per-block cast's rules
    for (int c = threadIdx.x; c < 512; c += kAmaxThreads) {
        float m = red[0][c];
#pragma unroll
        for (int w = 1; w < kAmaxWarps; ++w)
            m = fmaxf(m, red[w][c]);
        const bool out_col = blockIdx.y == 0 && chunk0 + c < a.H;
        if (SCALE == kScaleUE8M0) {
            const uint8_t byte = (uint8_t)(ue8m0_exponent<OUT>(m) + 127);
            sclbuf[c] = byte;
            if (out_col)
                static_cast<uint8_t *>(o.scales)[chunk0 + c] = byte;
        } else {
            float sc;
            if (m >= 0x1p-64f) {
                sc = div_markstein1(m, Fmt<OUT>::kQmax, Fmt<OUT>::kRcpQmax);
            } else {
                sc = __fdiv_rn(m, Fmt<OUT>::kQmax);
                if (sc == 0.0f)
                    sc = 1.0f;
            }
            reinterpret_cast<float *>(sclbuf)[c] = sc;
            if (out_col)
                static_cast<float *>(o.scales)[chunk0 + c] = sc;
        }
    }
    __syncthreads();
    ColScales<SCALE> cs;
    cs.load(sclbuf, lane * kEPT);

    // 3. the slab's rows, last first; warp w takes rows r1-1-w, r1-1-w-8, ...
    Src src;
    constexpr int U = kChunkUnroll<BF16, SCALE>;
    constexpr int64_t kStep = (int64_t)U * kAmaxWarps;
    typename Src::Regs va[U], vb[U];
    auto row_of = [&](int64_t j, int u) { return r1 - 1 - warp - (j + u) * kAmaxWarps; };
    auto fetch = [&](int64_t j, typename Src::Regs (&v)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = row_of(j, u);
            if (col_ok && row >= r0)
                load_ev<1, Src>(a, row, col0, v[u]);
            else
                Src::zero(v[u]);
        }
    };
    auto encode = [&](int64_t j, const typename Src::Regs (&v)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t row = row_of(j, u);
            if (!col_ok || row < r0)
                continue;
            uint64_t ny[kEPT / 2];
            float amax_unused = 0.0f;
            src.produce(a, v[u], true, ny, amax_unused);
            uint64_t q[kEPT / 2];
            cs.divide(ny, q);
            if (OUT == kOutE4M3) {
                uint32_t w[4];
                e4m3_words(q, w);
                st_stream_128(o.q + row * (int64_t)a.H + col0, w[0], w[1], w[2], w[3]);
            } else {
                const uint32_t w0 = cvt_e2m1x8(q[0], q[1], q[2], q[3]);
                const uint32_t w1 = cvt_e2m1x8(q[4], q[5], q[6], q[7]);
                st_stream_64(o.q + row * (int64_t)(a.H / 2) + col0 / 2, w0, w1);
            }
        }
    };
    // rows per warp: ceil((r1 - r0 - warp) / 8)
    const int64_t nrow = (r1 - r0 - warp + kAmaxWarps - 1) / kAmaxWarps;
    int64_t j = 0;
    fetch(j, va);
    while (j < nrow) {
        fetch(j + U, vb);
        encode(j, va);
        j += U;
        if (j >= nrow)
            break;
        fetch(j + U, va);
        encode(j, vb);
        j += U;
    }
}

template <class Src, bool BF16, int OUT>
const void *chunk_pick(int scale_fmt)
{
    return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&col_chunk_quant_kernel<Src, BF16, OUT, kScaleF32>)
                                  : reinterpret_cast<const void *>(&col_chunk_quant_kernel<Src, BF16, OUT, kScaleUE8M0>);
}

template <class Src, int OUT, int MAXT>
const void *quant_pick(int scale_fmt)
{
    return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&col_quant_kernel<Src, OUT, kScaleF32, MAXT>)
                                  : reinterpret_cast<const void *>(&col_quant_kernel<Src, OUT, kScaleUE8M0, MAXT>);
}

template <class Src>
const void *quant_pick_out(int out_fmt, int scale_fmt, bool wide)
{
    if (out_fmt == kOutE4M3)
        return wide ? quant_pick<Src, kOutE4M3, kMaxThreads>(scale_fmt) : quant_pick<Src, kOutE4M3, 512>(scale_fmt);
    return wide ? quant_pick<Src, kOutE2M1, kMaxThreads>(scale_fmt) : quant_pick<Src, kOutE2M1, 512>(scale_fmt);
}

template <int OUT>
const void *scale_pick(int scale_fmt)
{
    return scale_fmt == kScaleF32 ? reinterpret_cast<const void *>(&col_scale_kernel<OUT, kScaleF32>)
                                  : reinterpret_cast<const void *>(&col_scale_kernel<OUT, kScaleUE8M0>);
}

cudaError_t launch_grid(const void *fn, dim3 grid, int block, void **args, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

ChannelFns channel_fns(int in_dtype, int out_fmt, int scale_fmt, int64_t hidden)
{
    ChannelFns f{};
    if (in_dtype != 0 && in_dtype != 1)
        return f;
    if (out_fmt != kOutE4M3 && out_fmt != kOutE2M1)
        return f;
    if (scale_fmt != kScaleF32 && scale_fmt != kScaleUE8M0)
        return f;
    f.amax = in_dtype == 0 ? reinterpret_cast<const void *>(&col_amax_kernel<CastBf16Src, true, false, false>)
                           : reinterpret_cast<const void *>(&col_amax_kernel<CastF32Src, false, false, false>);
    f.amax_pf = in_dtype == 0 ? reinterpret_cast<const void *>(&col_amax_kernel<CastBf16Src, true, true, false>)
                              : reinterpret_cast<const void *>(&col_amax_kernel<CastF32Src, false, true, false>);
    f.amax_keep = in_dtype == 0 ? reinterpret_cast<const void *>(&col_amax_kernel<CastBf16Src, true, false, true>)
                                : reinterpret_cast<const void *>(&col_amax_kernel<CastF32Src, false, false, true>);
    f.amax_keep_pf = in_dtype == 0 ? reinterpret_cast<const void *>(&col_amax_kernel<CastBf16Src, true, true, true>)
                                   : reinterpret_cast<const void *>(&col_amax_kernel<CastF32Src, false, true, true>);
    f.scale = out_fmt == kOutE4M3 ? scale_pick<kOutE4M3>(scale_fmt) : scale_pick<kOutE2M1>(scale_fmt);
    const bool wide = hidden > 8192;   // more than 512 threads per row
    f.quant = in_dtype == 0 ? quant_pick_out<CastBf16Src>(out_fmt, scale_fmt, wide)
                            : quant_pick_out<CastF32Src>(out_fmt, scale_fmt, wide);
    if (in_dtype == 0)
        f.chunk = out_fmt == kOutE4M3 ? chunk_pick<CastBf16Src, true, kOutE4M3>(scale_fmt)
                                      : chunk_pick<CastBf16Src, true, kOutE2M1>(scale_fmt);
    else
        f.chunk = out_fmt == kOutE4M3 ? chunk_pick<CastF32Src, false, kOutE4M3>(scale_fmt)
                                      : chunk_pick<CastF32Src, false, kOutE2M1>(scale_fmt);
    return f;
}

int channel_amax_threads() { return kAmaxThreads; }
int channel_scale_threads() { return kScaleThreads; }

cudaError_t launch_channel(const ChannelFns &f, const ChannelLaunch &L, const CastArgs &a, const OutArgs &o,
                           const RowShape &sh, float *partial, cudaStream_t stream)
{
    CastArgs a_ = a;
    int64_t T = sh.T, slab_rows = L.slab_rows;
    float *part = partial;
    int64_t keep_slab = L.keep_rows;
    void *args1[] = {&a_, &T, &slab_rows, &part, &keep_slab};
    // short slabs (each warp at most eight row sets): the prefetching form;
    // before the chunk quantize pass, the form that sets L2 priorities
    const bool pf = slab_rows <= 8 * 4 * kAmaxWarps;
    const void *amax = L.split ? (pf ? f.amax_pf : f.amax) : (pf ? f.amax_keep_pf : f.amax_keep);
    cudaError_t e = launch_grid(amax, dim3(L.chunks, L.slabs), kAmaxThreads, args1, stream);
    if (e != cudaSuccess)
        return e;
    const int nparts = L.slabs;   // partial maxima per column
    if (!L.split) {
        const float *cpart = partial;
        int slabs = nparts;
        OutArgs o_ = o;
        void *args2[] = {&a_, &T, &slab_rows, &cpart, &slabs, &o_};
        return launch_grid(f.chunk, dim3(L.chunks, L.slabs), kAmaxThreads, args2, stream);
    }
    const float *cpart = partial;
    int slabs = nparts, H = a.H;
    void *sc = o.scales;
    void *args2[] = {&cpart, &slabs, &H, &sc};
    e = launch_grid(f.scale, dim3((H + 31) / 32), kScaleThreads, args2, stream);
    if (e != cudaSuccess)
        return e;
    OutArgs o_ = o;
    RowShape sh_ = sh;
    void *args3[] = {&a_, &o_, &sh_};
    return launch_grid(f.quant, dim3(L.quant_grid), L.quant_block, args3, stream);
}

}  // namespace tk
