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
// Both kernels accumulate acc = fma(w, y, acc) in k order on packed fp32
// pairs (E4M3 rows: w is first multiplied by the row's group scale), from
// acc = 0, skipping empty slots, and write gs * acc rounded to nearest even
// bf16, so they give bit-identical outputs. A position outside [0, num_rows)
// other than -1 is treated as an empty slot and sets bit 1 of the fault word
// (neither kernel reads through it).
//
//  - moe_reduce_bulk_kernel (K <= 32, rows of at least 2 KB; E4M3 rows with H
//    a multiple of 512): a task is one column chunk of one token. Warp 0 of
//    each persistent CTA is the producer: lane k fetches the token's k-th
//    position and weight (eight tasks ahead), then copies row k's chunk (and its
//    scales) into a ring slot of shared memory with one TMA bulk copy, an
//    mbarrier per slot counting the bytes in. Sixteen consumer warps wait on the
//    slot, accumulate the chunk from shared memory together, store it as bf16
//    and release the slot on a second mbarrier. The bytes in flight (the
//    ring, ~200 KB per SM) cost no registers.
//  - moe_reduce_kernel (any shape): a thread owns 16 columns of one token;
//    a CTA handles max(1, 256 / (H/16)) tokens per step of a persistent grid
//    stride; each token's K positions and weights are read first, then the
//    expert slices four at a time so that four 32-byte (bf16) or 16-byte
//    (E4M3) loads are in flight per thread.
#include <cuda_fp16.h>

#include "tk_reduce.h"

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
template <int IN, bool PREFETCH>
__global__ void __launch_bounds__(512) moe_reduce_kernel(ReduceArgs a)
{
    const int tid = threadIdx.x;
    const int slot = tid / a.tpr;
    const int lr = tid - slot * a.tpr;
    const bool slot_ok = slot < a.rpc;
    const int col0 = lr * kEPT;
    const int64_t ntb = (a.T + a.rpc - 1) / a.rpc;
    // PREFETCH (the plan's choice where a CTA has few token blocks): the
    // first token block's expert slices into L2 before waiting on the
    // previous kernel. The positions are read past L1 (.cg), so no stale
    // line stays behind for the reads after the wait; an address is only a
    // hint here and is used only when it lies inside y.
    if (PREFETCH && slot_ok && (int64_t)blockIdx.x * a.rpc + slot < a.T) {
        const int64_t t = (int64_t)blockIdx.x * a.rpc + slot;
        for (int k = 0; k < a.K; ++k) {
            const int32_t p = __ldcg(a.pos + t * a.K + k);
            if (p >= 0 && p < a.R)
                prefetch_l2(static_cast<const uint8_t *>(a.y) +
                            ((int64_t)p * a.H + col0) * (IN == kReduceInBf16 ? 2 : 1));
        }
    }
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
        if (aligned32(a.out)) {   // uniform: rows of H % 16 == 0 bf16 keep 32-byte alignment
            st_stream_256(dst, o);
        } else {
            st_stream_128(dst, o[0], o[1], o[2], o[3]);
            st_stream_128(dst + 8, o[4], o[5], o[6], o[7]);
        }
    }
}

// Tasks of metadata (positions, weights) the producer keeps in flight.
constexpr int kMetaAhead = 8;

__device__ __forceinline__ void cp_async_4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// at most kMetaAhead - 1 groups of this thread still pending
__device__ __forceinline__ void cp_async_wait_ahead()
{
    asm volatile("cp.async.wait_group %0;" :: "n"(kMetaAhead - 1) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Bulk kernel. Shared memory: `stages` slots of slot_bytes, each
//   [K rows x rb bytes][K x sb scale bytes][mask (4 B), pad to 16][w[K] fp32]
// then full[stages] and empty[stages] mbarriers, then the producer's
// metadata ring: kMetaAhead x 32 positions and kMetaAhead x 32 weights.
// full[s] takes two arrivals (the producer's lane 0 before and after its
// copies and metadata) plus the copied bytes; empty[s] takes one arrival per
// consumer warp. All consumer warps take every task in turn, so no warp
// waits more than one phase ahead of a barrier.
template <int IN, bool PREFETCH>
__global__ void __launch_bounds__(kReduceBulkThreads, 1) moe_reduce_bulk_kernel(ReduceArgs a)
{
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kElt = IN == kReduceInBf16 ? 2 : 1;
    constexpr int kG = IN == kReduceInBf16 ? 8 : 16;   // columns per consumer step: 16 bytes of y
    const int S = a.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)S * a.slot_bytes);
    uint64_t *empty = full + S;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t ntasks = a.T * a.nchunks;
    const int meta_off = a.K * (a.rb + a.sb);
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full + i, 2);
            mbar_init(empty + i, kReduceConsumerWarps);
        }
        fence_mbar_init();
    }
    // PREFETCH (the plan's choice where a CTA has few tasks): the producer
    // warp sends the chunks of its first `stages` tasks into L2 before
    // waiting on the previous kernel (positions read past L1, as above; a
    // hint only, and only for a position inside y).
    if (PREFETCH && warp == 0 && lane < a.K) {
        for (int i = 0; i < S; ++i) {
            const int64_t task = blockIdx.x + (int64_t)i * gridDim.x;
            if (task >= ntasks)
                break;
            const int64_t t = task / a.nchunks;
            const int c = (int)(task - t * a.nchunks);
            const int32_t p = __ldcg(a.pos + t * a.K + lane);
            if (p >= 0 && p < a.R)
                bulk_prefetch_l2(static_cast<const uint8_t *>(a.y) + ((int64_t)p * a.H + (int64_t)c * a.wc) * kElt,
                                 (uint32_t)a.rb);
        }
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        // Lane k's position and weight for the task kMetaAhead tasks ahead
        // stream into a small shared ring with 4-byte asynchronous copies
        // (one commit group per task), so no load latency sits between a
        // slot's release and its refill.
        const bool in_k = lane < a.K;
        int32_t *mpos = reinterpret_cast<int32_t *>(empty + S);   // [kMetaAhead][32]
        float *mw_ring = reinterpret_cast<float *>(mpos + kMetaAhead * 32);
        auto prefetch = [&](int64_t task, int entry) {
            if (task < ntasks && in_k) {
                const int64_t t = task / a.nchunks;
                cp_async_4(mpos + entry * 32 + lane, a.pos + t * a.K + lane);
                cp_async_4(mw_ring + entry * 32 + lane, a.w + t * a.K + lane);
            }
            cp_async_commit();
        };
#pragma unroll
        for (int i = 0; i < kMetaAhead; ++i)
            prefetch(blockIdx.x + (int64_t)i * gridDim.x, i);
        int slot = 0;
        uint32_t use_par = 0;   // parity of the current use of `slot`
        int64_t issued = 0;
        int entry = 0;
        for (int64_t task = blockIdx.x; task < ntasks; task += gridDim.x) {
            cp_async_wait_ahead();   // this task's group has landed (groups complete in order)
            const int32_t p = in_k ? mpos[entry * 32 + lane] : -1;
            const float wv = in_k ? mw_ring[entry * 32 + lane] : 0.0f;
            const int64_t t = task / a.nchunks;
            const int c = (int)(task - t * a.nchunks);
            const bool valid = in_k && p >= 0 && p < a.R;
            if (in_k && c == 0 && (p < -1 || p >= a.R))
                atomicOr(a.fault, 2u);
            const uint32_t mask = __ballot_sync(kFull, valid);
            if (issued >= S) {   // wait until every consumer warp released the slot's previous use
                bool got = true;
                if (lane == 0)
                    got = mbar_wait_bounded(empty + slot, use_par ^ 1u);
                if (!__shfl_sync(kFull, got ? 1 : 0, 0)) {
                    if (lane == 0)
                        atomicOr(a.fault, 1u);
                    break;
                }
            }
            uint8_t *base = smem + (size_t)slot * a.slot_bytes;
            if (lane == 0)
                mbar_arrive_expect_tx(full + slot, (uint32_t)__popc(mask) * (uint32_t)(a.rb + a.sb));
            __syncwarp();
            if (valid) {
                const int64_t c0 = (int64_t)c * a.wc;
                bulk_g2s(base + lane * a.rb, static_cast<const uint8_t *>(a.y) + ((int64_t)p * a.H + c0) * kElt,
                         (uint32_t)a.rb, full + slot);
                if constexpr (IN == kReduceInE4M3)
                    bulk_g2s(base + a.K * a.rb + lane * a.sb, a.y_scale + (int64_t)p * (a.H / 128) + c0 / 128,
                             (uint32_t)a.sb, full + slot);
            }
            if (in_k)
                reinterpret_cast<float *>(base + meta_off + 16)[lane] = wv;
            if (lane == 0)
                *reinterpret_cast<uint32_t *>(base + meta_off) = mask;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(full + slot);
            ++issued;
            if (++slot == S) {
                slot = 0;
                use_par ^= 1u;
            }
            // refill the metadata entry just used (its values are consumed above)
            prefetch(task + (int64_t)kMetaAhead * gridDim.x, entry);
            if (++entry == kMetaAhead)
                entry = 0;
        }
        // every copy this CTA issued lands before its shared memory goes away
        cp_async_wait_all();
        if (lane == 0) {
            for (int s = 0; s < S && s < issued; ++s) {
                const int64_t last_use = (issued - 1 - s) / S;
                if (!mbar_wait_bounded(full + s, (uint32_t)(last_use & 1)))
                    atomicOr(a.fault, 1u);
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int ctid = threadIdx.x - 32;
    const int ngroups = a.wc / kG;
    const uint64_t g2 = splat(a.gs);
    int slot = 0;
    uint32_t par = 0;
    for (int64_t task = blockIdx.x; task < ntasks; task += gridDim.x) {
        const int64_t t = task / a.nchunks;
        const int c = (int)(task - t * a.nchunks);
        if (!mbar_wait_bounded(full + slot, par)) {
            if (lane == 0)
                atomicOr(a.fault, 1u);
            return;
        }
        
        const uint8_t *base = smem + (size_t)slot * a.slot_bytes;
        const uint32_t mask = *reinterpret_cast<const uint32_t *>(base + meta_off);
        const float *mw = reinterpret_cast<const float *>(base + meta_off + 16);
        uint16_t *orow = static_cast<uint16_t *>(a.out) + t * (int64_t)a.H + (int64_t)c * a.wc;
        for (int g = ctid; g < ngroups; g += kReduceConsumerWarps * 32) {
            uint64_t acc[kG / 2];
#pragma unroll
            for (int q = 0; q < kG / 2; ++q)
                acc[q] = 0;
            for (int k0 = 0; k0 < a.K; k0 += 4) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)   // in-bounds reads of the slot; unused when the slot is empty
                    if (k0 + j < a.K)
                        v[j] = *reinterpret_cast<const uint4 *>(base + (k0 + j) * a.rb + g * 16);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k = k0 + j;
                    if (k >= a.K || !((mask >> k) & 1u))
                        continue;
                    const uint32_t vv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                    if constexpr (IN == kReduceInBf16) {
                        const uint64_t w2 = splat(mw[k]);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            acc[q] = fma2(w2, pk(bf16_lo(vv[q]), bf16_hi(vv[q])), acc[q]);
                    } else {
                        const float sc = reinterpret_cast<const float *>(base + a.K * a.rb + k * a.sb)[g >> 3];
                        const uint64_t w2 = splat(__fmul_rn(mw[k], sc));
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t lo2, hi2;
                            asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
                                "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
                                : "=r"(lo2), "=r"(hi2) : "r"(vv[q]));
                            const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&lo2));
                            const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&hi2));
                            acc[2 * q] = fma2(w2, pk(f0.x, f0.y), acc[2 * q]);
                            acc[2 * q + 1] = fma2(w2, pk(f1.x, f1.y), acc[2 * q + 1]);
                        }
                    }
                }
            }
            uint32_t o[kG / 2];
#pragma unroll
            for (int q = 0; q < kG / 2; ++q) {
                const uint64_t vg = mul2(acc[q], g2);
                o[q] = to_bf16x2(plo(vg), phi(vg));
            }
            uint16_t *dst = orow + g * kG;
            if constexpr (kG == 16) {
                if (aligned32(a.out)) {
                    st_stream_256(dst, o);
                } else {
                    st_stream_128(dst, o[0], o[1], o[2], o[3]);
                    st_stream_128(dst + 8, o[4], o[5], o[6], o[7]);
                }
            } else {
                st_stream_128(dst, o[0], o[1], o[2], o[3]);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(empty + slot);
        if (++slot == S) {
            slot = 0;
            par ^= 1u;
        }
    }
}

}  // namespace

const void *moe_reduce_kernel_fn(int in_fmt, bool prefetch)
{
    if (in_fmt == kReduceInBf16)
        return prefetch ? reinterpret_cast<const void *>(&moe_reduce_kernel<kReduceInBf16, true>)
                        : reinterpret_cast<const void *>(&moe_reduce_kernel<kReduceInBf16, false>);
    if (in_fmt == kReduceInE4M3)
        return prefetch ? reinterpret_cast<const void *>(&moe_reduce_kernel<kReduceInE4M3, true>)
                        : reinterpret_cast<const void *>(&moe_reduce_kernel<kReduceInE4M3, false>);
    return nullptr;
}

const void *moe_reduce_bulk_kernel_fn(int in_fmt, bool prefetch)
{
    if (in_fmt == kReduceInBf16)
        return prefetch ? reinterpret_cast<const void *>(&moe_reduce_bulk_kernel<kReduceInBf16, true>)
                        : reinterpret_cast<const void *>(&moe_reduce_bulk_kernel<kReduceInBf16, false>);
    if (in_fmt == kReduceInE4M3)
        return prefetch ? reinterpret_cast<const void *>(&moe_reduce_bulk_kernel<kReduceInE4M3, true>)
                        : reinterpret_cast<const void *>(&moe_reduce_bulk_kernel<kReduceInE4M3, false>);
    return nullptr;
}

cudaError_t launch_moe_reduce(const void *kfn, int grid, int block, int smem, const ReduceArgs &a,
                              cudaStream_t stream)
{
    ReduceArgs a_ = a;
    void *args[] = {&a_};
    return launch_pdl(kfn, grid, block, smem, args, stream);
}

}  // namespace tk
