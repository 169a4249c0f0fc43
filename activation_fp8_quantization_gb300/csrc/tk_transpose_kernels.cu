// Fused SwiGLU + top-k weight + per-token cast with the codes written
// transposed, sm_103a.
//
// "TileKernels从入门到精通" (zhichai.net/topic/177618752), closing section
// "结语：工程化极致的胜利", looking back on chapter 2: SwiGLU, the per-token
// quant and the transpose fit into one kernel launch, with no intermediate
// tensor written back and read again. Here the grouping, the
// scales and the codes are exactly those of tk_swiglu_quant_run (groups of g
// consecutive columns of one row); only the code matrix is stored as
// qT[H, ldq], element (column i, row t) at i * ldq + t, so that a following
// GEMM that contracts over the rows reads it row-major.
//
// A CTA of 128 threads owns a tile of 32 rows x 128 columns at a time
// (persistent grid stride over tiles; small CTAs, up to eight per SM, so that
// one CTA's loads overlap another's quantization and write-out). Phase 1:
// eight threads per row, 16 columns each, run the fused op and the quantizer
// of the row-major kernels (same arithmetic, same order) for two passes of 16
// rows and store the 16 codes row-major into a shared tile. Phase 2: each
// thread gathers the tile's 32 rows of one column and writes them as one
// 32-byte store (ldq is a multiple of 32, so the sector is aligned), or as two
// 16-byte stores where qT itself is only 16-byte aligned; either way every
// warp writes full 32-byte sectors of 32 rows of qT, but L2 receives one
// full-sector write per thread instead of two half-sector ones. Rows
// T <= t < ldq of the last tile are written as zero codes; nothing at or past
// ldq is written.
#include "tk_transpose.h"

namespace tk {

namespace {

constexpr int kTileRows = 32;
constexpr int kTileCols = 128;
constexpr int kTileStride = 144;   // bytes per shared row: 16-byte aligned, conflict-free in both phases
constexpr int kTransposeThreads = 128;
constexpr int kPassRows = kTransposeThreads / 8;

// PREFETCH: 0 none; 1 the first tile's rows into L2 before the dependency
// wait; 2 that and, at each tile, the CTA's next tile's rows.
template <int SCALE, bool CLAMP, int PREFETCH>
__global__ void __launch_bounds__(kTransposeThreads) transpose_quant_kernel(SwigluArgs a, OutArgs o, RowShape sh,
                                                                              int64_t ldq)
{
    __shared__ __align__(16) uint8_t tile[kTileRows * kTileStride];
    SwigluSrc<CLAMP> src;
    const int tid = threadIdx.x;
    const int rr = tid >> 3;           // row of the pass (0..15)
    const int cc = (tid & 7) * kEPT;   // first column within the tile
    const int tpg_mask = (1 << sh.tpg_log2) - 1;
    const int ncb = sh.H / kTileCols;
    const int64_t ntiles = (sh.T + kTileRows - 1) / kTileRows * ncb;
    const int oc = tid & (kTileCols - 1);   // phase 2: column within the tile
    const int oh = tid >> 7;                // phase 2: rows oh*32 .. oh*32+31 (oh = 0 with 128 threads)
    // uniform: every qT row starts 32-byte aligned, so each thread's 32 rows
    // of one column go out as one sector-sized store
    const bool wide = (ldq & 31) == 0 && aligned32(o.q);
    // PREFETCH >= 1 (the plan's choice where a CTA has few tiles): the first
    // tile's rows into L2 before waiting on the previous kernel
    if (PREFETCH >= 1 && (int64_t)blockIdx.x < ntiles) {
        const int64_t tb = blockIdx.x / ncb;
        const int c0 = (int)(blockIdx.x - tb * ncb) * kTileCols;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int64_t row = tb * kTileRows + p * kPassRows + rr;
            if (row < sh.T)
                SwigluSrc<CLAMP>::prefetch(a, row, c0 + cc);
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x) {
        const int64_t tb = tl / ncb;
        const int c0 = (int)(tl - tb * ncb) * kTileCols;
        const int64_t t0 = tb * kTileRows;
        typename SwigluSrc<CLAMP>::Regs regs[2];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int64_t row = t0 + p * kPassRows + rr;
            if (row < sh.T)
                SwigluSrc<CLAMP>::load(a, row, c0 + cc, regs[p]);
            else
                SwigluSrc<CLAMP>::zero(regs[p]);
        }
        if (PREFETCH == 2) {   // the CTA's next tile into L2 while this one is worked on
            const int64_t tn = tl + gridDim.x;
            if (tn < ntiles) {
                const int64_t tbn = tn / ncb;
                const int c0n = (int)(tn - tbn * ncb) * kTileCols;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int64_t row = tbn * kTileRows + p * kPassRows + rr;
                    if (row < sh.T)
                        SwigluSrc<CLAMP>::prefetch(a, row, c0n + cc);
                }
            }
        }
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            const int64_t row = t0 + p * kPassRows + rr;
            const bool ok = row < sh.T;
            uint64_t ny[kEPT / 2];
            float amax = 0.0f;
            src.produce(a, regs[p], ok, ny, amax);
            amax = group_max(amax, tpg_mask);
            uint64_t v[kEPT / 2];
            float s = 0.0f;
            int k = 0;
            quantize_values<kOutE4M3, SCALE>(ny, amax, v, s, k);
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (ok) {
                e4m3_words(v, w);
                if ((tid & tpg_mask) == 0)
                    store_scale<SCALE>(sh, o, row, (c0 + cc) >> (sh.tpg_log2 + 4), s, k);
            }
            *reinterpret_cast<uint4 *>(tile + (p * kPassRows + rr) * kTileStride + cc) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        __syncthreads();
        uint32_t out[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint8_t *src_col = tile + (oh * 32 + 4 * j) * kTileStride + oc;
            out[j] = (uint32_t)src_col[0] | ((uint32_t)src_col[kTileStride] << 8) |
                     ((uint32_t)src_col[2 * kTileStride] << 16) | ((uint32_t)src_col[3 * kTileStride] << 24);
        }
        const int64_t r0 = t0 + oh * 32;
        uint8_t *dst = o.q + (int64_t)(c0 + oc) * ldq + r0;
        if (wide && r0 + 32 <= ldq) {
            st_stream_256(dst, out);
        } else {
            if (r0 < ldq)
                st_stream_128(dst, out[0], out[1], out[2], out[3]);
            if (r0 + 16 < ldq)
                st_stream_128(dst + 16, out[4], out[5], out[6], out[7]);
        }
        __syncthreads();
    }
    src.finish(a);
}

}  // namespace

namespace {
template <int PF>
const void *transpose_pick(int scale_fmt, bool clamp)
{
    if (scale_fmt == kScaleF32)
        return clamp ? reinterpret_cast<const void *>(&transpose_quant_kernel<kScaleF32, true, PF>)
                     : reinterpret_cast<const void *>(&transpose_quant_kernel<kScaleF32, false, PF>);
    return clamp ? reinterpret_cast<const void *>(&transpose_quant_kernel<kScaleUE8M0, true, PF>)
                 : reinterpret_cast<const void *>(&transpose_quant_kernel<kScaleUE8M0, false, PF>);
}
}  // namespace

const void *transpose_kernel_fn(int scale_fmt, bool clamp, int prefetch)
{
    if (prefetch == 2)
        return transpose_pick<2>(scale_fmt, clamp);
    return prefetch == 1 ? transpose_pick<1>(scale_fmt, clamp) : transpose_pick<0>(scale_fmt, clamp);
}

int transpose_threads() { return kTransposeThreads; }

cudaError_t launch_transpose(const void *fn, int grid, const SwigluArgs &a, const OutArgs &o, const RowShape &sh,
                             int64_t ldq, cudaStream_t stream)
{
    SwigluArgs a_ = a;
    OutArgs o_ = o;
    RowShape sh_ = sh;
    int64_t ldq_ = ldq;
    void *args[] = {&a_, &o_, &sh_, &ldq_};
    return launch_pdl(fn, grid, kTransposeThreads, 0, args, stream);
}

}  // namespace tk
