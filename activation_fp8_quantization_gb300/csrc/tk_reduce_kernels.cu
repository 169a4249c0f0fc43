// The weighted top-k combine after the expert GEMMs, sm_103a.
//
// out[t, :] = gs * sum_{k, pos[t,k] valid} w[t,k] * deq(y[pos[t,k], :]):
// the expert rows are gathered through token_topk_to_pos, scaled by the
// routing weight and (for E4M3 rows) their 1x128 quantization factor,
// accumulated in fp32 registers and written once as bf16 ("TileKernels从入门到
// 精通", zhichai.net/topic/177618752, ch.3 "结算中心的减法工程": weights, quant
// factors and the global scale held in registers, one read and one write;
// "动态寻址": gathering through token_topk_to_pos).
//
// A thread owns 16 columns of one token; a CTA handles max(1, 256 / (H/16))
// tokens per step of a persistent grid stride. Each token's K positions and
// weights are read first, then the expert slices four at a time so that four
// 32-byte (bf16) or 16-byte (E4M3) loads are in flight per thread.
// Accumulation is acc = fma(w, y, acc) in k order on packed fp32 pairs; the
// result is gs * acc rounded to nearest even bf16. A position outside
// [0, num_rows) is treated as an empty slot and sets bit 1 of the fault word
// (the kernel never reads through it).
#include <cuda_fp16.h>

#include "tk_internal.h"

namespace tk {

namespace {

constexpr int kBatch = 4;

template <int IN>
struct RowSlice;

template <>
struct RowSlice<kReduceInBf16> {
    uint32_t v[8];   // 16 bf16
    __device__ __forceinline__ void load(const ReduceArgs &a, int32_t r, int col0)
    {
        ld_stream_256(static_cast<const uint16_t *>(a.y) + (int64_t)r * a.H + col0, v);
    }
    // acc += w * deq(row)
    __device__ __forceinline__ void accumulate(const ReduceArgs &, int32_t, int, float w, uint64_t (&acc)[8]) const
    {
        const uint64_t w2 = splat(w);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = fma2(w2, pk(bf16_lo(v[i]), bf16_hi(v[i])), acc[i]);
    }
};

template <>
struct RowSlice<kReduceInE4M3> {
    uint32_t v[4];   // 16 E4M3 codes
    __device__ __forceinline__ void load(const ReduceArgs &a, int32_t r, int col0)
    {
        const uint4 c = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint8_t *>(a.y) + (int64_t)r * a.H + col0));
        v[0] = c.x;
        v[1] = c.y;
        v[2] = c.z;
        v[3] = c.w;
    }
    __device__ __forceinline__ void accumulate(const ReduceArgs &a, int32_t r, int col0, float w,
                                               uint64_t (&acc)[8]) const
    {
        // the 16 columns lie in one 128-column group: one scale per slice
        const float ws = __fmul_rn(w, __ldg(a.y_scale + (int64_t)r * (a.H / 128) + col0 / 128));
        const uint64_t w2 = splat(ws);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // two codes -> f16x2 (exact: every E4M3 value is an f16 value) -> two fp32
            uint32_t lo2, hi2;
            asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
                "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
                : "=r"(lo2), "=r"(hi2) : "r"(v[i]));
            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&lo2));
            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&hi2));
            acc[2 * i] = fma2(w2, pk(f0.x, f0.y), acc[2 * i]);
            acc[2 * i + 1] = fma2(w2, pk(f1.x, f1.y), acc[2 * i + 1]);
        }
    }
};

// two fp32 -> bf16x2, round to nearest even; lo in the low half
__device__ __forceinline__ uint32_t to_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// At most 512 threads per CTA (H <= 8192), which leaves room for four
// slices in flight per thread without spilling.
template <int IN>
__global__ void __launch_bounds__(512) moe_reduce_kernel(ReduceArgs a)
{
    const int tid = threadIdx.x;
    const int slot = tid / a.tpr;
    const int lr = tid - slot * a.tpr;
    const bool slot_ok = slot < a.rpc;
    const int col0 = lr * kEPT;
    const int64_t ntb = (a.T + a.rpc - 1) / a.rpc;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t tb = blockIdx.x; tb < ntb; tb += gridDim.x) {
        const int64_t t = tb * a.rpc + slot;
        if (!slot_ok || t >= a.T)
            continue;
        uint64_t acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[i] = 0;
        const int32_t *pos = a.pos + t * a.K;
        const float *wt = a.w + t * a.K;
        for (int k0 = 0; k0 < a.K; k0 += kBatch) {
            int32_t r[kBatch];   // row of y, or -1
            float wk[kBatch];
            RowSlice<IN> s[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int k = k0 + j;
                const int32_t p = k < a.K ? __ldg(pos + k) : -1;
                wk[j] = k < a.K ? __ldg(wt + k) : 0.0f;
                r[j] = p;
                if (p < -1 || p >= a.R) {   // not a row and not "empty": flag it, skip it
                    if (lr == 0)
                        atomicOr(a.fault, 2u);
                    r[j] = -1;
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (r[j] >= 0)
                    s[j].load(a, r[j], col0);
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (r[j] >= 0)
                    s[j].accumulate(a, r[j], col0, wk[j], acc);
        }
        const uint64_t g2 = splat(a.gs);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint64_t v = mul2(acc[i], g2);
            o[i] = to_bf16x2(plo(v), phi(v));
        }
        uint16_t *dst = static_cast<uint16_t *>(a.out) + t * (int64_t)a.H + col0;
        st_stream_128(dst, o[0], o[1], o[2], o[3]);
        st_stream_128(dst + 8, o[4], o[5], o[6], o[7]);
    }
}

}  // namespace

const void *moe_reduce_kernel_fn(int in_fmt)
{
    if (in_fmt == kReduceInBf16)
        return reinterpret_cast<const void *>(&moe_reduce_kernel<kReduceInBf16>);
    if (in_fmt == kReduceInE4M3)
        return reinterpret_cast<const void *>(&moe_reduce_kernel<kReduceInE4M3>);
    return nullptr;
}

cudaError_t launch_moe_reduce(const void *kfn, int grid, int block, const ReduceArgs &a, cudaStream_t stream)
{
    ReduceArgs a_ = a;
    void *args[] = {&a_};
    return launch_pdl(kfn, grid, block, 0, args, stream);
}

}  // namespace tk
