// C ABI: descriptor validation, plans (launch shape chosen once per device)
// and stream-ordered launches. Declared in include/tk_swiglu_quant.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "tk_backward.h"
#include "tk_channel.h"
#include "tk_internal.h"
#include "tk_reduce.h"
#include "tk_transpose.h"
#include "tk_swiglu_quant.h"

#define TK_API extern "C" __attribute__((visibility("default")))

namespace {

thread_local std::string g_msg;

tk_status fail(tk_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_msg = buf;
    return st;
}

tk_status ok() { return TK_OK; }

tk_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(TK_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int ilog2(int v)
{
    int r = 0;
    while ((1 << r) < v)
        ++r;
    return r;
}

// Shared checks of hidden / group / formats.
tk_status check_geometry(int64_t hidden, int32_t group, int32_t scale_fmt, int32_t out_fmt)
{
    if (hidden <= 0)
        return fail(TK_ERR_INVALID_ARG, "hidden must be positive (got %lld)", (long long)hidden);
    if (hidden % 16 != 0 || hidden > 16384)
        return fail(TK_ERR_UNSUPPORTED, "hidden must be a multiple of 16 in [16, 16384] (got %lld)",
                    (long long)hidden);
    if (group < 0)
        return fail(TK_ERR_INVALID_ARG, "group_size must be >= 0 (got %d)", group);
    if (group != 0) {
        if (!(group == 16 || group == 32 || group == 64 || group == 128 || group == 256 || group == 512))
            return fail(TK_ERR_UNSUPPORTED, "group_size must be 0, 16, 32, 64, 128, 256 or 512 (got %d)", group);
        if (hidden % group != 0)
            return fail(TK_ERR_UNSUPPORTED, "group_size %d does not divide hidden %lld", group,
                        (long long)hidden);
    }
    if (scale_fmt != TK_SCALE_FP32 && scale_fmt != TK_SCALE_UE8M0)
        return fail(TK_ERR_INVALID_ARG, "unknown scale_fmt %d", scale_fmt);
    if (out_fmt != TK_OUT_E4M3 && out_fmt != TK_OUT_E2M1)
        return fail(TK_ERR_INVALID_ARG, "unknown out_fmt %d", out_fmt);
    return TK_OK;
}

bool is_flag(int32_t v) { return v == 0 || v == 1; }

// Launch geometry common to both ops.
struct Geometry {
    int tpr, tpg_log2, rpc, block, groups;
    bool cta_reduce;
};

Geometry geometry(int64_t hidden, int32_t group)
{
    Geometry g{};
    g.tpr = (int)(hidden / tk::kEPT);
    const int gsz = group ? group : (int)hidden;
    g.groups = (int)(hidden / gsz);
    const int tpg = gsz / tk::kEPT;
    g.cta_reduce = !(is_pow2(tpg) && tpg <= 32);
    if (g.cta_reduce) {
        g.rpc = 1;
        g.tpg_log2 = 0;
    } else {
        g.rpc = g.tpr >= 256 ? 1 : 256 / g.tpr;
        g.tpg_log2 = ilog2(tpg);
    }
    g.block = ((g.tpr * g.rpc + 31) / 32) * 32;
    return g;
}

// Guard that makes `device` current and restores the previous device.
struct DeviceScope {
    int prev = -1;
    bool switched = false;
    cudaError_t err = cudaSuccess;
    explicit DeviceScope(int device)
    {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != device) {
            err = cudaSetDevice(device);
            switched = err == cudaSuccess;
        }
    }
    ~DeviceScope()
    {
        if (switched)
            cudaSetDevice(prev);
    }
};

// The kernels a plan can launch.
enum Kind { kRows = TK_KERNEL_ROWS, kWarpStream = TK_KERNEL_WARP_STREAM, kBlockStream = TK_KERNEL_BLOCK_RING };

// Everything a launch needs, fixed when the plan is made.
struct Launch {
    const void *fn;
    const void *fn_pf;   // row kernel only: the form that prefetches its first row block (see row_fn)
    const void *fn_pf2;  // cast row kernel only: the form that also prefetches each next row block
    int kind;          // row_quant_kernel, warp_stream_kernel or block_stream_kernel
    int block;         // threads per CTA
    int rpc;           // row kernel: rows per CTA per iteration; block kernel: rows per ring slot
    int tpr, tpg_log2, groups;
    int wpr, stages;   // stream kernels: 512-column slices per row, ring slots (per warp or per CTA)
    size_t smem;       // dynamic shared memory per CTA
    int max_grid;      // resident CTAs on all SMs
    int num_sms;
    unsigned *fault;   // device address of the fault word
};

// A persistent grid for `units` equal work units taken in grid-stride order:
// the resident CTAs, trimmed so that every CTA takes the same number of
// units, give or take one (rounds = ceil(units / max_grid), grid =
// ceil(units / rounds)); the last round then finds nearly every CTA busy
// instead of a fraction of them. Used by the register combine (bf16
// combine 24.80 -> 24.42 us); the other kernels measured slower with it
// (8192-row fused 14.96 -> 15.72 us, 100003-row 222.4 -> 229.3 us,
// transposed clamp workload 60.8 -> 63.1 us: fewer bytes in flight in every
// round cost more than the last round's idle CTAs), so they keep every
// resident CTA.
int balanced_grid(int64_t units, int max_grid)
{
    if (units <= max_grid)
        return (int)(units > 0 ? units : 1);
    const int64_t rounds = (units + max_grid - 1) / max_grid;
    return (int)((units + rounds - 1) / rounds);
}

int grid_for(const Launch &L, int64_t T)
{
    const int64_t units =
        L.kind == kWarpStream ? (T * L.wpr + (L.block / 32) - 1) / (L.block / 32) : (T + L.rpc - 1) / L.rpc;
    return (int)(units < L.max_grid ? units : L.max_grid);
}

// The row kernel's entry for a run of T rows: the prefetching form where
// each CTA has at most 32 row blocks, so that the first block's latency is a
// visible part of the launch. Measured on GB300: 8192 x 2048 fused 15.2 ->
// 14.9 us, 256 x 512 2.0 -> 1.6 us, the 8192 x 4096 cast 17.8 -> 17.4 us;
// the 16384 x 7168 cast (54 blocks per CTA) was 4% slower with the prefetch
// compiled in, even where the branch was not taken, hence a separate
// instantiation rather than a run-time test in one.
const void *row_fn(const Launch &L, int64_t T, int grid)
{
    if (L.kind != TK_KERNEL_ROWS || !L.fn_pf)
        return L.fn;
    const int64_t nrb = (T + L.rpc - 1) / L.rpc;
    // The cast's row kernel (fn_pf2 set): each next block into L2 too at 4
    // to 32 row blocks per CTA. Measured on GB300 (µs, first block only /
    // each next block too), width 4096: per-token fp32 input 4096 rows
    // 14.00/13.13, 8192 25.91/25.22, 16384 50.23/48.15, 2048 7.45/7.68;
    // 1 x 128 bf16 input 4096 rows 9.47/9.16, 2048 5.41/5.74.
    if (L.fn_pf2 && nrb >= 4 * (int64_t)grid && nrb <= 32 * (int64_t)grid)
        return L.fn_pf2;
    return nrb <= 32 * (int64_t)grid ? L.fn_pf : L.fn;
}

// Padded rows per column of a column-major scale layout (elements, or
// 32-bit words for the packed one): 16 bytes of scale elements.
int64_t scale_ld(int32_t layout, int32_t scale_fmt, int64_t T)
{
    if (layout == TK_SCALE_COL_MAJOR) {
        const int64_t per16 = scale_fmt == TK_SCALE_FP32 ? 4 : 16;
        return (T + per16 - 1) / per16 * per16;
    }
    if (layout == TK_SCALE_COL_MAJOR_PACKED)
        return (T + 3) / 4 * 4;
    return 0;
}

size_t scale_bytes_for(int32_t layout, int32_t scale_fmt, int64_t T, int64_t groups)
{
    const size_t e = scale_fmt == TK_SCALE_FP32 ? 4 : 1;
    if (layout == TK_SCALE_COL_MAJOR)
        return (size_t)groups * (size_t)scale_ld(layout, scale_fmt, T) * e;
    if (layout == TK_SCALE_COL_MAJOR_PACKED)
        return (size_t)(groups / 4) * (size_t)scale_ld(layout, scale_fmt, T) * 4;
    return (size_t)T * (size_t)groups * e;
}

tk::RowShape shape_for(const Launch &L, int64_t T, int64_t hidden, int32_t layout, int32_t scale_fmt)
{
    return tk::RowShape{T, (int32_t)hidden, L.tpr, L.tpg_log2, L.rpc, L.groups, L.stages, L.wpr, L.fault,
                        layout, scale_ld(layout, scale_fmt, T)};
}

// The scale layout must be known, and the packed one needs UE8M0 scales and
// a whole number of four-group words per row.
tk_status check_scale_layout(int32_t layout, int32_t scale_fmt, int64_t hidden, int32_t group)
{
    if (layout != TK_SCALE_ROW_MAJOR && layout != TK_SCALE_COL_MAJOR && layout != TK_SCALE_COL_MAJOR_PACKED)
        return fail(TK_ERR_INVALID_ARG, "unknown scale_layout %d", layout);
    if (layout == TK_SCALE_COL_MAJOR_PACKED) {
        const int64_t groups = group ? hidden / group : 1;
        if (scale_fmt != TK_SCALE_UE8M0)
            return fail(TK_ERR_UNSUPPORTED, "the packed scale layout holds UE8M0 exponents only");
        if (groups % 4 != 0)
            return fail(TK_ERR_UNSUPPORTED, "the packed scale layout needs a multiple of 4 groups per row");
    }
    return TK_OK;
}

// A clamp limit whose fp32 bits end in 16 zeros is a bf16 value: the kernels
// then clamp the bf16 inputs directly, two lanes per instruction.
void set_packed_limit(tk::SwigluArgs &a)
{
    uint32_t bits;
    memcpy(&bits, &a.limit, sizeof bits);
    a.packed_clamp = (bits & 0xffffu) == 0;
    a.limit2 = (bits >> 16) * 0x00010001u;
}

int env_int(const char *name, int dflt)
{
    const char *v = getenv(name);
    return v ? atoi(v) : dflt;
}

// Ring depth of the stream kernel: the most bytes in flight per SM with at
// least 24 resident warps per SM (ties: the shallower ring).
// TK_PIPELINE_STAGES=<n> (2..8) overrides the choice.
tk_status choose_stream_ring(Launch *L, int slot_bytes, int optin)
{
    const int warps = L->block / 32;
    const int forced = env_int("TK_PIPELINE_STAGES", 0);
    long best = -1;
    for (int S = 2; S <= 8; ++S) {
        const size_t smem = (size_t)warps * S * (slot_bytes + 8);
        if (smem > (size_t)optin)
            break;
        int occ = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, L->fn, L->block, smem);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (occ < 1)
            continue;
        const long inflight = (long)occ * warps * S * slot_bytes;
        const bool pick = forced ? S == forced : ((long)occ * warps >= 24 || best < 0) && inflight > best;
        if (pick) {
            best = inflight;
            L->stages = S;
            L->smem = smem;
            L->max_grid = occ;
        }
    }
    if (best < 0)
        return fail(TK_ERR_UNSUPPORTED, "no warp ring fits in shared memory");
    return TK_OK;
}

// Ring of the block-ring kernel. Rows per slot: the fewest that give a block
// at least one slice per consumer warp, times the multiple nearest below
// TK_BLOCK_SLOT_KB (default 32) KB; then the ring depth with the most bytes
// in flight per SM while at least 24 consumer warps per SM stay resident
// (ties: the shallower ring). TK_BLOCK_STAGES=<n> (2..16) forces the depth.
// Measured on GB300 at width 2048: 32 KB slots (four rows, two slots, three
// CTAs per SM) are 3% faster than 16 KB slots four deep; six 16 KB slots
// (two CTAs per SM) are 9% slower.
tk_status choose_block_ring(Launch *L, int64_t row_bytes, int optin)
{
    const int rb_min = (tk::kBlockConsumerWarps + L->wpr - 1) / L->wpr;
    const int64_t target = (int64_t)env_int("TK_BLOCK_SLOT_KB", 32) * 1024;
    int64_t mult = target / (rb_min * row_bytes);
    if (mult < 1)
        mult = 1;
    L->rpc = (int)(rb_min * mult);
    const int64_t slot = (int64_t)L->rpc * row_bytes;
    const int forced = env_int("TK_BLOCK_STAGES", 0);
    long best = -1;
    for (int S = 2; S <= 16; ++S) {
        const int64_t smem = (int64_t)S * (slot + 16);   // the slots, then full[S] and empty[S]
        if (smem > optin)
            break;
        int occ = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, L->fn, L->block, (size_t)smem);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (occ < 1)
            continue;
        const long inflight = (long)occ * S * slot;
        const bool pick =
            forced ? S == forced : ((long)occ * tk::kBlockConsumerWarps >= 24 || best < 0) && inflight > best;
        if (pick) {
            best = inflight;
            L->stages = S;
            L->smem = (size_t)smem;
            L->max_grid = occ;
        }
    }
    if (best < 0)
        return fail(TK_ERR_UNSUPPORTED, "no block ring fits in shared memory");
    return TK_OK;
}

}  // namespace

// Set by a stream kernel that gave up waiting on one of its own copies.
__device__ unsigned int g_tk_fault_word;

namespace {

// The kernels of a plan: the row kernel always, the two stream kernels where
// they apply. TK_KERNEL=rows, =stream or =block (read when the plan is made)
// forces one; otherwise the block-ring kernel runs batches of the fused op
// that give every resident CTA at least block_min row blocks, and the row
// kernel everything else (block_min = 0: never).
struct Launches {
    Launch rows;
    Launch stream;
    Launch block;
    bool has_stream;
    bool has_block;
    int64_t block_min;
    // standalone cast: the block ring runs inputs of block_lo..block_hi bytes
    // (row_bytes per row), the row kernel all others; block_hi = 0: unused
    int64_t block_lo, block_hi, row_bytes;
    int forced;   // 0: by size, 1: rows, 2: warp stream, 3: block ring
};

// Where the block-ring kernel overtakes the row kernel, whose register
// prefetch starts up faster: the row blocks per resident CTA from which the
// block kernel runs. Measured on GB300 (µs, row kernel / block kernel):
//   width 2048 (two rows per row-kernel CTA; 4 rows per block, 456 CTAs):
//     fp32 scales, no clamp: 16384 rows 27.5/29.4, 32768 52.6/53.6, 65536 102.3/102.2
//     UE8M0, clamp 7:        16384 rows 30.7/31.6, 32768 58.8/58.3, 65536 114.1/111.3
//     FP4 1x32, clamp 7:     16384 rows 29.6/30.6, 65536 109.5/107.0
//   width 3072 (one row per row-kernel CTA; 2 rows per block):
//     fp32 scales, no clamp: 25000 rows 62.5/60.4, 100003 240.5/223.9
// so about 32 blocks per CTA without the clamp and 16 with it where the row
// kernel packs two or more rows per CTA, and 8 where it holds one row per CTA
// (wide rows, which it runs less efficiently). The standalone cast, with a
// third of the fused op's arithmetic per byte, is not issue-bound on the row
// kernel; the block ring only shortens its start-up, and on long runs its
// steady rate is lower. Measured on GB300 (bf16 input, us, row kernel /
// block kernel):
//   width 4096, fp32 scales: 4096 rows 9.49/10.59, 8192 17.37/16.91,
//     16384 32.72/31.08, 32768 63.74/59.76, 65536 124.1/127.3 (117.7/134.1)
//   width 7168, UE8M0: 2048 rows 8.62/8.64, 4096 15.86/14.00, 16384
//     55.01/51.91, 24576 81.12/84.59, 32768 107.1/115.6, 49152 158.8/175.7
//   width 2048, fp32 scales: 8192 rows 9.50/10.61, 16384 17.35/16.88
//   width 4096, 1x32 E2M1: 4096 rows 8.27/8.86, 8192 15.11/13.95, 32768
//     54.67/50.82
// and fp32 input, width 4096: 8192 rows 26.00/26.89, 16384 51.96/50.49,
// 32768 103.9/97.5. So the cast takes the block ring for inputs of 48 to
// 288 MiB (bf16) or 160 to 640 MiB (fp32), the row kernel otherwise.
constexpr int64_t kCastBlockLoBf16 = (int64_t)48 << 20, kCastBlockHiBf16 = (int64_t)288 << 20;
constexpr int64_t kCastBlockLoF32 = (int64_t)160 << 20, kCastBlockHiF32 = (int64_t)640 << 20;

int64_t block_min_per_cta(const Launch &rows, bool clamp)
{
    if (rows.rpc < 2)
        return 8;
    return clamp ? 16 : 32;
}

const Launch &pick(const Launches &Ls, int64_t T)
{
    if (Ls.forced == 1)
        return Ls.rows;
    if (Ls.forced == 2)
        return Ls.has_stream ? Ls.stream : Ls.rows;
    if (Ls.forced == 3)
        return Ls.has_block ? Ls.block : Ls.rows;
    if (Ls.has_block && Ls.block_hi > 0) {
        const int64_t in = T * Ls.row_bytes;
        return in >= Ls.block_lo && in <= Ls.block_hi ? Ls.block : Ls.rows;
    }
    if (!Ls.has_block || Ls.block_min <= 0)
        return Ls.rows;
    const int64_t nblk = (T + Ls.block.rpc - 1) / Ls.block.rpc;
    return nblk >= Ls.block_min * Ls.block.max_grid ? Ls.block : Ls.rows;
}

// Validate the device and size one kernel's launch of `kind` (the caller
// checked that it applies): fn is that kernel's entry; slot_bytes the warp
// stream kernel's slot, row_bytes one input row (block kernel).
tk_status make_launch(int device, int64_t hidden, int32_t group, const void *fn, int kind, int slot_bytes,
                      int64_t row_bytes, Launch *L)
{
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= count)
        return fail(TK_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, count);
    DeviceScope scope(device);
    if (scope.err != cudaSuccess)
        return cuda_fail(scope.err, "cudaSetDevice");
    *L = Launch{};
    e = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, device);
    int optin = 0;
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    void *fault = nullptr;
    if (e == cudaSuccess)
        e = cudaGetSymbolAddress(&fault, g_tk_fault_word);
    if (e != cudaSuccess)
        return cuda_fail(e, "querying the device");
    L->fault = static_cast<unsigned *>(fault);

    const Geometry geo = geometry(hidden, group);
    L->tpr = geo.tpr;
    L->tpg_log2 = geo.tpg_log2;
    L->groups = geo.groups;
    L->kind = kind;
    L->fn = fn;
    if (kind == kBlockStream) {
        L->block = tk::kBlockThreads;
        L->wpr = (int)(hidden / 512);
        e = cudaFuncSetAttribute(L->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(L->fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return cuda_fail(e, "configuring the block kernel's shared memory");
        tk_status st = choose_block_ring(L, row_bytes, optin);
        if (st != TK_OK)
            return st;
    } else if (kind == kWarpStream) {
        L->block = tk::kStreamThreads;
        L->rpc = 1;
        L->wpr = (int)(hidden / 512);
        e = cudaFuncSetAttribute(L->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(L->fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess)
            return cuda_fail(e, "configuring the stream kernel's shared memory");
        tk_status st = choose_stream_ring(L, slot_bytes, optin);
        if (st != TK_OK)
            return st;
    } else {
        L->block = geo.block;
        L->rpc = geo.rpc;
        L->stages = 0;
        L->wpr = 0;
        L->smem = 0;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, L->fn, L->block, 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        if (occ < 1)
            return fail(TK_ERR_UNSUPPORTED, "kernel cannot be resident with %d threads per CTA", L->block);
        L->max_grid = occ;
    }
    L->max_grid *= L->num_sms;
    return TK_OK;
}

tk_status make_launches(int device, int64_t hidden, int32_t group, const void *row_fn, const void *stream_fn,
                        const void *block_fn, int slot_bytes, int row_bytes_per_col, Launches *Ls)
{
    *Ls = Launches{};
    const char *force = getenv("TK_KERNEL");
    Ls->forced = !force                       ? 0
                 : strcmp(force, "rows") == 0   ? 1
                 : strcmp(force, "stream") == 0 ? 2
                 : strcmp(force, "block") == 0  ? 3
                                                : 0;
    tk_status st = make_launch(device, hidden, group, row_fn, kRows, 0, 0, &Ls->rows);
    if (st != TK_OK)
        return st;
    const Geometry geo = geometry(hidden, group);
    Ls->has_stream = stream_fn && hidden % 512 == 0 && !geo.cta_reduce;
    if (Ls->has_stream)
        st = make_launch(device, hidden, group, stream_fn, kWarpStream, slot_bytes, 0, &Ls->stream);
    if (st != TK_OK)
        return st;
    Ls->has_block = Ls->has_stream && block_fn;
    if (Ls->has_block)
        st = make_launch(device, hidden, group, block_fn, kBlockStream, 0, (int64_t)row_bytes_per_col * hidden,
                         &Ls->block);
    return st;
}

tk_status check_current_device(int device)
{
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (cur != device)
        return fail(TK_ERR_DEVICE, "current device is %d but the plan was made for device %d", cur, device);
    return TK_OK;
}


}  // namespace

struct tk_swiglu_quant_plan_s {
    tk_swiglu_quant_desc desc;
    int device;
    Launches Ls;
    // transposed-codes kernel (null where the shape does not allow it), and
    // its form that prefetches its first tile (runs with few tiles per CTA)
    const void *tfn;
    const void *tfn_pf;
    const void *tfn_pf2;   // prefetches each next tile too (few tiles per CTA)
    int tgrid;
    int tgrid2;   // resident CTAs of tfn_pf2
    int tpf;      // TK_TRANSPOSE_PF=0|1|2 when the plan was made (forces a form), else -1
};

struct tk_quant_cast_plan_s {
    tk_quant_cast_desc desc;
    int device;
    Launches Ls;       // per-token / per-block plans
    // per-channel plans: the three kernels, the quantize pass's launch shape
    // and the CTAs the amax pass aims at
    tk::ChannelFns cfn;
    Launch cq;
    int amax_ctas;
    int channel_forced;   // TK_CHANNEL_KERNEL when the plan was made: 0 by size, 1 chunk, 2 split
};

// ------------------------------------------------------------------ fused op

TK_API tk_status tk_swiglu_quant_validate(const tk_swiglu_quant_desc *d)
{
    if (!d)
        return fail(TK_ERR_INVALID_ARG, "desc is NULL");
    tk_status st = check_geometry(d->hidden, d->group_size, d->scale_fmt, d->out_fmt);
    if (st != TK_OK)
        return st;
    if (!is_flag(d->has_topk_weights) || !is_flag(d->use_clamp) || !is_flag(d->count_clamped))
        return fail(TK_ERR_INVALID_ARG, "has_topk_weights, use_clamp and count_clamped must be 0 or 1");
    if (d->use_clamp && !(std::isfinite(d->clamp_limit) && d->clamp_limit >= 0.0f))
        return fail(TK_ERR_INVALID_ARG, "clamp_limit must be finite and >= 0 (got %g)", (double)d->clamp_limit);
    if (d->count_clamped && !d->use_clamp)
        return fail(TK_ERR_INVALID_ARG, "count_clamped needs use_clamp");
    return check_scale_layout(d->scale_layout, d->scale_fmt, d->hidden, d->group_size);
}

TK_API tk_status tk_swiglu_quant_plan(const tk_swiglu_quant_desc *d, int device, tk_swiglu_quant_plan_t *plan)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan output pointer is NULL");
    *plan = nullptr;
    tk_status st = tk_swiglu_quant_validate(d);
    if (st != TK_OK)
        return st;
    const Geometry geo = geometry(d->hidden, d->group_size);
    const bool clamp = d->use_clamp != 0;
    const void *row_fn = tk::swiglu_kernel_fn(d->out_fmt, d->scale_fmt, clamp, geo.cta_reduce, 0);
    const void *stream_fn = tk::swiglu_stream_fn(d->out_fmt, d->scale_fmt, clamp);
    const void *block_fn = tk::swiglu_block_fn(d->out_fmt, d->scale_fmt, clamp);
    if (!row_fn)
        return fail(TK_ERR_UNSUPPORTED, "no kernel for this combination");
    Launches Ls{};
    st = make_launches(device, d->hidden, d->group_size, row_fn, stream_fn, block_fn, tk::kSwigluSlotBytes,
                       tk::kSwigluRowBytesPerCol, &Ls);
    if (st != TK_OK)
        return st;
    Ls.block_min = block_min_per_cta(Ls.rows, clamp);
    Ls.rows.fn_pf = tk::swiglu_kernel_fn(d->out_fmt, d->scale_fmt, clamp, geo.cta_reduce, 1);
    // The transposed-codes kernel: E4M3, groups of 32, 64 or 128 columns
    // inside its 128-column tiles.
    const void *tfn = nullptr, *tfn_pf = nullptr, *tfn_pf2 = nullptr;
    int tgrid = 0, tgrid2 = 0;
    if (d->out_fmt == TK_OUT_E4M3 && d->hidden % 128 == 0 &&
        (d->group_size == 32 || d->group_size == 64 || d->group_size == 128)) {
        tfn = tk::transpose_kernel_fn(d->scale_fmt, clamp, 0);
        tfn_pf = tk::transpose_kernel_fn(d->scale_fmt, clamp, 1);
        tfn_pf2 = tk::transpose_kernel_fn(d->scale_fmt, clamp, 2);
        int occ = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, tfn, tk::transpose_threads(), 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "occupancy of the transposed kernel");
        tgrid = occ * Ls.rows.num_sms;
        int occ2 = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, tfn_pf2, tk::transpose_threads(), 0);
        if (e != cudaSuccess)
            return cuda_fail(e, "occupancy of the transposed kernel");
        tgrid2 = occ2 * Ls.rows.num_sms;
        if (tgrid < 1 || tgrid2 < 1)
            tfn = nullptr;
    }
    const int tpf = env_int("TK_TRANSPOSE_PF", -1);
    auto *p = new (std::nothrow) tk_swiglu_quant_plan_s{*d, device, Ls, tfn, tfn_pf, tfn_pf2, tgrid, tgrid2,
                                                        tpf >= 0 && tpf <= 2 ? tpf : -1};
    if (!p)
        return fail(TK_ERR_INVALID_ARG, "out of host memory");
    *plan = p;
    return ok();
}

TK_API tk_status tk_swiglu_quant_plan_destroy(tk_swiglu_quant_plan_t plan)
{
    delete plan;
    return ok();
}

TK_API tk_status tk_swiglu_quant_output_sizes(const tk_swiglu_quant_desc *d, int64_t T, size_t *q_bytes,
                                              size_t *scale_bytes)
{
    tk_status st = tk_swiglu_quant_validate(d);
    if (st != TK_OK)
        return st;
    if (T < 0 || !q_bytes || !scale_bytes)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 and the outputs non-NULL");
    const int64_t groups = d->group_size ? d->hidden / d->group_size : 1;
    *q_bytes = (size_t)T * (size_t)(d->out_fmt == TK_OUT_E4M3 ? d->hidden : d->hidden / 2);
    *scale_bytes = scale_bytes_for(d->scale_layout, d->scale_fmt, T, groups);
    return ok();
}

namespace {

// The argument checks shared by the row-major and the transposed call.
tk_status check_swiglu_args(const tk_swiglu_quant_plan_s *plan, const void *x, const float *topk_weights,
                            const void *q, const void *scales, const int64_t *clamped_count)
{
    const tk_swiglu_quant_desc &d = plan->desc;
    if (!x || !q || !scales)
        return fail(TK_ERR_INVALID_ARG, "x, q and scales must be non-NULL");
    if (d.has_topk_weights && !topk_weights)
        return fail(TK_ERR_INVALID_ARG, "the plan expects topk_weights");
    if (d.count_clamped && !clamped_count)
        return fail(TK_ERR_INVALID_ARG, "the plan expects clamped_count");
    if (!aligned(x, 32))
        return fail(TK_ERR_MISALIGNED, "x must be 32-byte aligned");
    if (!aligned(q, 16))
        return fail(TK_ERR_MISALIGNED, "q must be 16-byte aligned");
    if (d.scale_fmt == TK_SCALE_FP32 && !aligned(scales, 4))
        return fail(TK_ERR_MISALIGNED, "fp32 scales must be 4-byte aligned");
    if (d.scale_layout != TK_SCALE_ROW_MAJOR && !aligned(scales, 16))
        return fail(TK_ERR_MISALIGNED, "column-major scales must be 16-byte aligned");
    if (d.has_topk_weights && !aligned(topk_weights, 4))
        return fail(TK_ERR_MISALIGNED, "topk_weights must be 4-byte aligned");
    if (d.count_clamped && !aligned(clamped_count, 8))
        return fail(TK_ERR_MISALIGNED, "clamped_count must be 8-byte aligned");
    return check_current_device(plan->device);
}

tk::SwigluArgs swiglu_args(const tk_swiglu_quant_desc &d, const void *x, const float *topk_weights,
                           int64_t *clamped_count)
{
    tk::SwigluArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.w = d.has_topk_weights ? topk_weights : nullptr;
    a.counts = d.count_clamped ? reinterpret_cast<unsigned long long *>(clamped_count) : nullptr;
    a.limit = d.use_clamp ? d.clamp_limit : 0.0f;
    a.H = (int32_t)d.hidden;
    set_packed_limit(a);
    return a;
}

}  // namespace

TK_API tk_status tk_swiglu_quant_run(tk_swiglu_quant_plan_t plan, int64_t T, const void *x,
                                     const float *topk_weights, void *q, void *scales,
                                     int64_t *clamped_count, void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    const tk_swiglu_quant_desc &d = plan->desc;
    tk_status st = check_swiglu_args(plan, x, topk_weights, q, scales, clamped_count);
    if (st != TK_OK)
        return st;
    const tk::SwigluArgs a = swiglu_args(d, x, topk_weights, clamped_count);
    tk::OutArgs o{static_cast<uint8_t *>(q), scales};
    const Launch &L = pick(plan->Ls, T);
    cudaError_t e = tk::launch_swiglu(row_fn(L, T, grid_for(L, T)), grid_for(L, T), L.block, L.smem, a, o,
                                      shape_for(L, T, d.hidden, d.scale_layout, d.scale_fmt),
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the fused kernel");
    return ok();
}

namespace {

// The device address of page-locked host memory `p` (null stays null), or an
// error if `p` is not such memory.
tk_status mapped_address(const void *p, const char *what, void **dev)
{
    *dev = nullptr;
    if (!p)
        return TK_OK;
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaPointerGetAttributes");
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer)
        return fail(TK_ERR_INVALID_ARG, "%s must be page-locked host memory the device can address", what);
    *dev = attr.devicePointer;
    return TK_OK;
}

}  // namespace

TK_API tk_status tk_swiglu_quant_run_mapped(tk_swiglu_quant_plan_t plan, int64_t T, const void *x_host,
                                            const float *topk_weights_host, void *q_host, void *scales_host,
                                            int64_t *clamped_count_host, void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    const tk_swiglu_quant_desc &d = plan->desc;
    tk_status st = check_swiglu_args(plan, x_host, topk_weights_host, q_host, scales_host, clamped_count_host);
    if (st != TK_OK)
        return st;
    void *x = nullptr, *w = nullptr, *q = nullptr, *s = nullptr, *c = nullptr;
    if ((st = mapped_address(x_host, "x", &x)) != TK_OK ||
        (st = mapped_address(d.has_topk_weights ? topk_weights_host : nullptr, "topk_weights", &w)) != TK_OK ||
        (st = mapped_address(q_host, "q", &q)) != TK_OK || (st = mapped_address(scales_host, "scales", &s)) != TK_OK ||
        (st = mapped_address(d.count_clamped ? clamped_count_host : nullptr, "clamped_count", &c)) != TK_OK)
        return st;
    const tk::SwigluArgs a = swiglu_args(d, x, static_cast<const float *>(w), static_cast<int64_t *>(c));
    tk::OutArgs o{static_cast<uint8_t *>(q), s};
    const Launch &L = plan->Ls.rows;
    cudaError_t e = tk::launch_swiglu(L.fn, grid_for(L, T), L.block, L.smem, a, o,
                                      shape_for(L, T, d.hidden, d.scale_layout, d.scale_fmt),
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the fused kernel");
    return ok();
}

TK_API tk_status tk_swiglu_quant_transposed_size(tk_swiglu_quant_plan_t plan, int64_t T, size_t *qt_bytes,
                                                 int64_t *ld)
{
    if (!plan || T < 0 || !qt_bytes || !ld)
        return fail(TK_ERR_INVALID_ARG, "plan and outputs must be non-NULL and num_tokens >= 0");
    if (!plan->tfn)
        return fail(TK_ERR_UNSUPPORTED, "transposed codes need E4M3, group_size 32, 64 or 128 and "
                                        "hidden % 128 == 0");
    *ld = (T + 31) / 32 * 32;
    *qt_bytes = (size_t)plan->desc.hidden * (size_t)*ld;
    return ok();
}

TK_API tk_status tk_swiglu_quant_run_transposed(tk_swiglu_quant_plan_t plan, int64_t T, const void *x,
                                                const float *topk_weights, void *qt, void *scales,
                                                int64_t *clamped_count, void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (!plan->tfn)
        return fail(TK_ERR_UNSUPPORTED, "transposed codes need E4M3, group_size 32, 64 or 128 and "
                                        "hidden % 128 == 0");
    if (T == 0)
        return ok();
    const tk_swiglu_quant_desc &d = plan->desc;
    tk_status st = check_swiglu_args(plan, x, topk_weights, qt, scales, clamped_count);
    if (st != TK_OK)
        return st;
    const tk::SwigluArgs a = swiglu_args(d, x, topk_weights, clamped_count);
    tk::OutArgs o{static_cast<uint8_t *>(qt), scales};
    const Launch &L = plan->Ls.rows;
    tk::RowShape sh = shape_for(L, T, d.hidden, d.scale_layout, d.scale_fmt);
    int lg = 0;
    while ((16 << lg) < d.group_size)
        ++lg;
    sh.tpg_log2 = lg;
    sh.groups = (int32_t)(d.hidden / d.group_size);
    const int64_t ldq = (T + 31) / 32 * 32;
    const int64_t tiles = (T + 31) / 32 * (d.hidden / 128);
    // Prefetching forms: without the clamp the first tile and each next one
    // always; with it the same at up to 8 tiles per CTA, the first tile only
    // at up to 32, none beyond. Measured on GB300 (µs; none / first tile only
    // / each next tile too): 8192 rows of width 2048 17.80/17.37/15.89,
    // 100003 rows of width 3072 (70 tiles per CTA) 264.6/264.5/262.3, 32768
    // rows of width 2048 with the clamp and outliers (15 tiles per CTA)
    // -/60.62/62.29; over 2048 to 32768 rows at widths 2048 and 3072 the
    // next-tile form was never slower without the clamp, and with it faster
    // up to 16384 rows (8 tiles per CTA).
    const int mode = plan->tpf >= 0                              ? plan->tpf
                     : !d.use_clamp                              ? 2
                     : tiles <= 8 * (int64_t)plan->tgrid2        ? 2
                     : tiles <= 32 * (int64_t)plan->tgrid        ? 1
                                                                 : 0;
    const int gmax = mode == 2 ? plan->tgrid2 : plan->tgrid;
    const int grid = (int)(tiles < gmax ? tiles : gmax);
    const void *fn = mode == 2 ? plan->tfn_pf2 : mode == 1 ? plan->tfn_pf : plan->tfn;
    cudaError_t e = tk::launch_transpose(fn, grid, a, o, sh, ldq, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the transposed kernel");
    return ok();
}

TK_API tk_status tk_swiglu_quant_launch_info(tk_swiglu_quant_plan_t plan, int64_t T, int *grid, int *block,
                                             int *rows_per_cta, int *num_sms, int *kernel)
{
    if (!plan || T < 0)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL or num_tokens < 0");
    const Launch &L = pick(plan->Ls, T);
    if (grid)
        *grid = T == 0 ? 0 : grid_for(L, T);
    if (block)
        *block = L.block;
    if (rows_per_cta)
        *rows_per_cta = L.kind == kWarpStream ? 0 : L.rpc;
    if (num_sms)
        *num_sms = L.num_sms;
    if (kernel)
        *kernel = L.kind;
    return ok();
}

// -------------------------------------------------------- host-buffer pipe

namespace {
constexpr int kSlots = 3;

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

struct tk_swiglu_quant_host_pipe_s {
    tk_swiglu_quant_plan_t plan;
    int64_t chunk_rows;
    cudaStream_t s_in, s_k, s_out;
    cudaEvent_t ev_entry, ev_exit;
    cudaEvent_t ev_in[kSlots], ev_k[kSlots], ev_out[kSlots];
    size_t x_bytes, w_bytes, q_bytes, s_bytes;  // per slot, unaligned
    size_t slot_bytes, total_bytes;
    size_t q_row, s_row;                        // output bytes per row
};

namespace {
void destroy_pipe_objects(tk_swiglu_quant_host_pipe_s *p)
{
    cudaStream_t ss[3] = {p->s_in, p->s_k, p->s_out};
    for (cudaStream_t st : ss)
        if (st) {
            cudaStreamSynchronize(st);
            cudaStreamDestroy(st);
        }
    cudaEvent_t es[2] = {p->ev_entry, p->ev_exit};
    for (cudaEvent_t e : es)
        if (e)
            cudaEventDestroy(e);
    for (int i = 0; i < kSlots; ++i) {
        if (p->ev_in[i])
            cudaEventDestroy(p->ev_in[i]);
        if (p->ev_k[i])
            cudaEventDestroy(p->ev_k[i]);
        if (p->ev_out[i])
            cudaEventDestroy(p->ev_out[i]);
    }
}
}  // namespace

TK_API tk_status tk_swiglu_quant_host_pipe_create(tk_swiglu_quant_plan_t plan, int64_t chunk_rows,
                                                  tk_swiglu_quant_host_pipe_t *out)
{
    if (!out)
        return fail(TK_ERR_INVALID_ARG, "pipe output pointer is NULL");
    *out = nullptr;
    if (!plan || chunk_rows < 1)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL or chunk_rows < 1");
    const tk_swiglu_quant_desc &d = plan->desc;
    auto *p = new (std::nothrow) tk_swiglu_quant_host_pipe_s{};
    if (!p)
        return fail(TK_ERR_INVALID_ARG, "out of host memory");
    p->plan = plan;
    p->chunk_rows = chunk_rows;
    const size_t groups = d.group_size ? (size_t)(d.hidden / d.group_size) : 1;
    p->q_row = (size_t)(d.out_fmt == TK_OUT_E4M3 ? d.hidden : d.hidden / 2);
    p->s_row = groups * (d.scale_fmt == TK_SCALE_FP32 ? 4u : 1u);
    p->x_bytes = (size_t)chunk_rows * (size_t)d.hidden * 4u;
    p->w_bytes = d.has_topk_weights ? (size_t)chunk_rows * 4u : 0;
    p->q_bytes = (size_t)chunk_rows * p->q_row;
    p->s_bytes = (size_t)chunk_rows * p->s_row;
    p->slot_bytes = align256(p->x_bytes) + align256(p->w_bytes) + align256(p->q_bytes) + align256(p->s_bytes);
    p->total_bytes = kSlots * p->slot_bytes + 256;  // + the clamp counter

    DeviceScope scope(plan->device);
    cudaError_t e = scope.err;
    cudaStream_t *ss[3] = {&p->s_in, &p->s_k, &p->s_out};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
        e = cudaStreamCreateWithFlags(ss[i], cudaStreamNonBlocking);
    cudaEvent_t *es[2 + 3 * kSlots] = {&p->ev_entry, &p->ev_exit};
    for (int i = 0; i < kSlots; ++i) {
        es[2 + i] = &p->ev_in[i];
        es[2 + kSlots + i] = &p->ev_k[i];
        es[2 + 2 * kSlots + i] = &p->ev_out[i];
    }
    for (int i = 0; i < 2 + 3 * kSlots && e == cudaSuccess; ++i)
        e = cudaEventCreateWithFlags(es[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
        destroy_pipe_objects(p);
        delete p;
        return cuda_fail(e, "creating the host pipe's streams and events");
    }
    *out = p;
    return ok();
}

TK_API tk_status tk_swiglu_quant_host_pipe_destroy(tk_swiglu_quant_host_pipe_t pipe)
{
    if (!pipe)
        return ok();
    {
        DeviceScope scope(pipe->plan->device);
        destroy_pipe_objects(pipe);
    }
    delete pipe;
    return ok();
}

TK_API tk_status tk_swiglu_quant_host_workspace_size(tk_swiglu_quant_host_pipe_t pipe, size_t *bytes)
{
    if (!pipe || !bytes)
        return fail(TK_ERR_INVALID_ARG, "pipe or bytes is NULL");
    *bytes = pipe->total_bytes;
    return ok();
}

TK_API tk_status tk_swiglu_quant_run_host(tk_swiglu_quant_host_pipe_t pipe, int64_t T, const void *x_host,
                                          const float *w_host, void *q_host, void *scales_host,
                                          int64_t *count_host, void *workspace, size_t workspace_bytes,
                                          void *stream)
{
    if (!pipe)
        return fail(TK_ERR_INVALID_ARG, "pipe is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    tk_swiglu_quant_plan_t plan = pipe->plan;
    const tk_swiglu_quant_desc &d = plan->desc;
    if (d.scale_layout != TK_SCALE_ROW_MAJOR)
        return fail(TK_ERR_UNSUPPORTED, "the host-buffer call returns row-major scales only");
    if (!x_host || !q_host || !scales_host)
        return fail(TK_ERR_INVALID_ARG, "x_host, q_host and scales_host must be non-NULL");
    if (d.has_topk_weights && !w_host)
        return fail(TK_ERR_INVALID_ARG, "the plan expects topk_weights_host");
    if (d.count_clamped && !count_host)
        return fail(TK_ERR_INVALID_ARG, "the plan expects clamped_count_host");
    if (!workspace || workspace_bytes < pipe->total_bytes)
        return fail(TK_ERR_INVALID_ARG, "workspace must hold %zu bytes (got %zu)", pipe->total_bytes,
                    workspace_bytes);
    if (!aligned(workspace, 256))
        return fail(TK_ERR_MISALIGNED, "workspace must be 256-byte aligned");
    tk_status st = check_current_device(plan->device);
    if (st != TK_OK)
        return st;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int64_t *dcount = reinterpret_cast<int64_t *>(ws + kSlots * pipe->slot_bytes);
    cudaStream_t user = static_cast<cudaStream_t>(stream);
    const size_t x_row = (size_t)d.hidden * 4u;
    cudaError_t e = cudaEventRecord(pipe->ev_entry, user);
    cudaStream_t ss[3] = {pipe->s_in, pipe->s_k, pipe->s_out};
    for (int i = 0; i < 3 && e == cudaSuccess; ++i)
        e = cudaStreamWaitEvent(ss[i], pipe->ev_entry, 0);
    if (e == cudaSuccess && d.count_clamped)
        e = cudaMemcpyAsync(dcount, count_host, 2 * sizeof(int64_t), cudaMemcpyHostToDevice, pipe->s_in);

    const int64_t nchunks = (T + pipe->chunk_rows - 1) / pipe->chunk_rows;
    for (int64_t c = 0; c < nchunks && e == cudaSuccess; ++c) {
        const int slot = (int)(c % kSlots);
        const int64_t r0 = c * pipe->chunk_rows;
        const int64_t rows = (T - r0) < pipe->chunk_rows ? (T - r0) : pipe->chunk_rows;
        uint8_t *sx = ws + slot * pipe->slot_bytes;
        uint8_t *sw = sx + align256(pipe->x_bytes);
        uint8_t *sq = sw + align256(pipe->w_bytes);
        uint8_t *ssc = sq + align256(pipe->q_bytes);
        // copy in, once the slot's previous chunk has been copied out
        if (c >= kSlots)
            e = cudaStreamWaitEvent(pipe->s_in, pipe->ev_out[slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sx, static_cast<const uint8_t *>(x_host) + (size_t)r0 * x_row,
                                (size_t)rows * x_row, cudaMemcpyHostToDevice, pipe->s_in);
        if (e == cudaSuccess && d.has_topk_weights)
            e = cudaMemcpyAsync(sw, w_host + r0, (size_t)rows * 4u, cudaMemcpyHostToDevice, pipe->s_in);
        if (e == cudaSuccess)
            e = cudaEventRecord(pipe->ev_in[slot], pipe->s_in);
        // compute
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(pipe->s_k, pipe->ev_in[slot], 0);
        if (e == cudaSuccess) {
            tk::SwigluArgs a{};
            a.x = reinterpret_cast<const uint16_t *>(sx);
            a.w = d.has_topk_weights ? reinterpret_cast<const float *>(sw) : nullptr;
            a.counts = d.count_clamped ? reinterpret_cast<unsigned long long *>(dcount) : nullptr;
            a.limit = d.use_clamp ? d.clamp_limit : 0.0f;
            a.H = (int32_t)d.hidden;
            set_packed_limit(a);
            tk::OutArgs o{sq, ssc};
            const Launch &L = pick(plan->Ls, rows);
            e = tk::launch_swiglu(row_fn(L, rows, grid_for(L, rows)), grid_for(L, rows), L.block, L.smem, a, o,
                                  shape_for(L, rows, d.hidden, TK_SCALE_ROW_MAJOR, d.scale_fmt), pipe->s_k);
        }
        if (e == cudaSuccess)
            e = cudaEventRecord(pipe->ev_k[slot], pipe->s_k);
        // copy out
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(pipe->s_out, pipe->ev_k[slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint8_t *>(q_host) + (size_t)r0 * pipe->q_row, sq,
                                (size_t)rows * pipe->q_row, cudaMemcpyDeviceToHost, pipe->s_out);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint8_t *>(scales_host) + (size_t)r0 * pipe->s_row, ssc,
                                (size_t)rows * pipe->s_row, cudaMemcpyDeviceToHost, pipe->s_out);
        if (e == cudaSuccess)
            e = cudaEventRecord(pipe->ev_out[slot], pipe->s_out);
    }
    // the last copy-out waited for the last kernel, and kernels run in order
    if (e == cudaSuccess && d.count_clamped)
        e = cudaMemcpyAsync(count_host, dcount, 2 * sizeof(int64_t), cudaMemcpyDeviceToHost, pipe->s_out);
    if (e == cudaSuccess)
        e = cudaEventRecord(pipe->ev_exit, pipe->s_out);
    if (e == cudaSuccess)
        e = cudaStreamWaitEvent(user, pipe->ev_exit, 0);
    if (e != cudaSuccess)
        return cuda_fail(e, "enqueueing the host-buffer pipeline");
    return ok();
}

// ------------------------------------------- host-buffer call without allocation

// The workspace of tk_swiglu_quant_run_host_static: one array per device,
// reserved when the library's module loads, shared by every such call.
static __device__ __align__(256) unsigned char g_tk_static_scratch[TK_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_static_mu;
// Device address of the array, looked up once per device ordinal. The
// address belongs to the context current at the lookup, the device's primary
// context for a runtime-API caller; the cache assumes that context for the
// life of the process.
void *g_static_addr[kMaxDevices] = {};
}  // namespace

TK_API tk_status tk_swiglu_quant_run_host_static(tk_swiglu_quant_host_pipe_t pipe, int64_t T, const void *x_host,
                                                 const float *w_host, void *q_host, void *scales_host,
                                                 int64_t *count_host, void *stream)
{
    if (!pipe)
        return fail(TK_ERR_INVALID_ARG, "pipe is NULL");
    // the same statuses as tk_swiglu_quant_run_host for the row count
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    if (pipe->total_bytes > TK_STATIC_SCRATCH_BYTES)
        return fail(TK_ERR_UNSUPPORTED,
                    "the pipe needs %zu bytes of workspace but the built-in array holds %zu: "
                    "make the pipe with fewer chunk_rows",
                    pipe->total_bytes, (size_t)TK_STATIC_SCRATCH_BYTES);
    const int device = pipe->plan->device;
    if (device < 0 || device >= kMaxDevices)
        return fail(TK_ERR_UNSUPPORTED, "device %d is beyond the %d devices this call supports", device,
                    kMaxDevices);
    tk_status st = check_current_device(device);
    if (st != TK_OK)
        return st;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_addr[device]) {
            // the symbol's host name is only a stand-in; the device address
            // comes from the runtime, with this device current
            cudaError_t e = cudaGetSymbolAddress(&g_static_addr[device], g_tk_static_scratch);
            if (e != cudaSuccess) {
                g_static_addr[device] = nullptr;
                return cuda_fail(e, "cudaGetSymbolAddress of the built-in workspace");
            }
        }
        scratch = g_static_addr[device];
    }
    return tk_swiglu_quant_run_host(pipe, T, x_host, w_host, q_host, scales_host, count_host, scratch,
                                    TK_STATIC_SCRATCH_BYTES, stream);
}

// ------------------------------------------------------------ standalone cast

TK_API tk_status tk_quant_cast_validate(const tk_quant_cast_desc *d)
{
    if (!d)
        return fail(TK_ERR_INVALID_ARG, "desc is NULL");
    tk_status st = check_geometry(d->hidden, d->group_size, d->scale_fmt, d->out_fmt);
    if (st != TK_OK)
        return st;
    if (d->in_dtype != TK_IN_BF16 && d->in_dtype != TK_IN_FP32)
        return fail(TK_ERR_INVALID_ARG, "unknown in_dtype %d", d->in_dtype);
    if (d->granularity != TK_GRAN_GROUPS && d->granularity != TK_GRAN_PER_CHANNEL)
        return fail(TK_ERR_INVALID_ARG, "unknown granularity %d", d->granularity);
    if (d->granularity == TK_GRAN_PER_CHANNEL) {
        if (d->group_size != 0)
            return fail(TK_ERR_INVALID_ARG, "a per-channel cast takes group_size 0 (got %d)", d->group_size);
        if (d->scale_layout != TK_SCALE_ROW_MAJOR && d->scale_layout != TK_SCALE_COL_MAJOR &&
            d->scale_layout != TK_SCALE_COL_MAJOR_PACKED)
            return fail(TK_ERR_INVALID_ARG, "unknown scale_layout %d", d->scale_layout);
        if (d->scale_layout != TK_SCALE_ROW_MAJOR)
            return fail(TK_ERR_UNSUPPORTED, "per-channel scales are one row [H]: row-major layout only");
        return TK_OK;
    }
    return check_scale_layout(d->scale_layout, d->scale_fmt, d->hidden, d->group_size);
}

namespace {

// Codes up to this size take the two-launch form (the chunk quantize pass on
// the amax pass's grid, scales reduced in its prologue); larger outputs the
// three-launch form (scale kernel, then the row quantize pass, whose CTAs
// write whole rows in sequence). Measured on GB300 (fraction of the copy
// bandwidth, chunk / three-launch): 8192 x 4096 E4M3 (33.5 MB of codes)
// 0.842 / 0.785; 32768 x 4096 E2M1 (67 MB) 0.985 / 0.960; 16384 x 7168 E4M3
// (117 MB) 0.788 / 0.881; fp32 input 8192 x 4096 0.929 / 0.930.
constexpr size_t kChannelChunkMaxCodes = (size_t)96 << 20;

// Bytes of x the amax pass marks evict_last for the chunk quantize pass
// (L2 is 126 MB). Measured on GB300 with 0 / 48 / 80 / 112 MB: 8192 x 4096
// bf16 30.5 / 28.7 / 27.5 / 27.5 us, fp32 49.0 / 47.5 / 45.9 / 46.0 us,
// 32768 x 4096 to E2M1 90.0 / 91.0 / 87.9 / 87.2 us; plain loads 28.3,
// 47.4 and 90.6 us.
constexpr size_t kChannelKeepBytes = (size_t)96 << 20;

// Plan the per-channel kernels: the quantize pass sized like the row kernel
// (16 columns per thread, rows per CTA so that a CTA has about 256 threads),
// the amax pass aiming at four CTAs per SM (each keeps 32 KB of loads in
// flight), capped by its occupancy.
tk_status plan_channel(const tk_quant_cast_desc *d, int device, tk_quant_cast_plan_s *p)
{
    p->cfn = tk::channel_fns(d->in_dtype, d->out_fmt, d->scale_fmt, d->hidden);
    if (!p->cfn.amax || !p->cfn.scale || !p->cfn.quant || !p->cfn.chunk)
        return fail(TK_ERR_UNSUPPORTED, "no per-channel kernel for this combination");
    tk_status st = make_launch(device, d->hidden, 16, p->cfn.quant, kRows, 0, 0, &p->cq);
    if (st != TK_OK)
        return st;
    DeviceScope scope(device);
    if (scope.err != cudaSuccess)
        return cuda_fail(scope.err, "cudaSetDevice");
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p->cfn.amax, tk::channel_amax_threads(), 0);
    if (e == cudaSuccess) {
        int occ2 = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, p->cfn.scale, tk::channel_scale_threads(), 0);
        if (e == cudaSuccess && occ2 < 1)
            return fail(TK_ERR_UNSUPPORTED, "the per-channel scale kernel cannot be resident");
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, p->cfn.chunk, tk::channel_amax_threads(), 0);
        if (e == cudaSuccess && occ2 < 1)
            return fail(TK_ERR_UNSUPPORTED, "the per-channel quantize kernel cannot be resident");
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "occupancy of the per-channel kernels");
    if (occ < 1)
        return fail(TK_ERR_UNSUPPORTED, "the per-channel amax kernel cannot be resident");
    p->amax_ctas = (occ < 4 ? occ : 4) * p->cq.num_sms;
    const char *force = getenv("TK_CHANNEL_KERNEL");
    p->channel_forced = !force ? 0 : strcmp(force, "chunk") == 0 ? 1 : strcmp(force, "split") == 0 ? 2 : 0;
    return TK_OK;
}

// Row slabs of the amax pass for T rows: about amax_ctas CTAs in all, at
// least 32 rows per slab (four rows per warp), no empty slab.
tk::ChannelLaunch channel_launch(const tk_quant_cast_plan_s *p, int64_t T)
{
    tk::ChannelLaunch L{};
    L.chunks = (int)((p->desc.hidden + 511) / 512);
    int64_t slabs = (p->amax_ctas + L.chunks - 1) / L.chunks;
    const int64_t by_rows = (T + 31) / 32;
    if (slabs > by_rows)
        slabs = by_rows;
    if (slabs < 1)
        slabs = 1;
    L.slab_rows = (T + slabs - 1) / slabs;
    L.slabs = (int)((T + L.slab_rows - 1) / L.slab_rows);
    L.quant_grid = grid_for(p->cq, T);
    L.quant_block = p->cq.block;
    const size_t q_bytes = (size_t)T * (size_t)(p->desc.out_fmt == TK_OUT_E4M3 ? p->desc.hidden : p->desc.hidden / 2);
    L.split = p->channel_forced ? p->channel_forced == 2 : q_bytes > kChannelChunkMaxCodes;
    // two-launch form: the last rows of each slab, kChannelKeepBytes of x in
    // all, stay in L2 for the chunk quantize pass
    const int64_t row_bytes = p->desc.hidden * (p->desc.in_dtype == TK_IN_BF16 ? 2 : 4);
    const int64_t keep = (int64_t)kChannelKeepBytes / row_bytes / L.slabs;
    L.keep_rows = L.split ? 0 : (keep < L.slab_rows ? keep : L.slab_rows);
    return L;
}

size_t channel_workspace(const tk_quant_cast_plan_s *p, int64_t T)
{
    if (T <= 0)
        return 0;
    const tk::ChannelLaunch L = channel_launch(p, T);
    return (size_t)L.slabs * (size_t)p->desc.hidden * sizeof(float);
}

}  // namespace

TK_API tk_status tk_quant_cast_plan(const tk_quant_cast_desc *d, int device, tk_quant_cast_plan_t *plan)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan output pointer is NULL");
    *plan = nullptr;
    tk_status st = tk_quant_cast_validate(d);
    if (st != TK_OK)
        return st;
    if (d->granularity == TK_GRAN_PER_CHANNEL) {
        auto *p = new (std::nothrow) tk_quant_cast_plan_s{};
        if (!p)
            return fail(TK_ERR_INVALID_ARG, "out of host memory");
        p->desc = *d;
        p->device = device;
        st = plan_channel(d, device, p);
        if (st != TK_OK) {
            delete p;
            return st;
        }
        *plan = p;
        return ok();
    }
    const Geometry geo = geometry(d->hidden, d->group_size);
    const void *row_fn = tk::cast_kernel_fn(d->in_dtype, d->out_fmt, d->scale_fmt, geo.cta_reduce, 0);
    const void *stream_fn = tk::cast_stream_fn(d->in_dtype, d->out_fmt, d->scale_fmt);
    const void *block_fn = tk::cast_block_fn(d->in_dtype, d->out_fmt, d->scale_fmt);
    if (!row_fn)
        return fail(TK_ERR_UNSUPPORTED, "no kernel for this combination");
    Launches Ls{};
    const bool bf16 = d->in_dtype == TK_IN_BF16;
    st = make_launches(device, d->hidden, d->group_size, row_fn, stream_fn, block_fn,
                       bf16 ? tk::kCastBf16SlotBytes : tk::kCastF32SlotBytes,
                       bf16 ? tk::kCastBf16RowBytesPerCol : tk::kCastF32RowBytesPerCol, &Ls);
    if (st != TK_OK)
        return st;
    Ls.rows.fn_pf = tk::cast_kernel_fn(d->in_dtype, d->out_fmt, d->scale_fmt, geo.cta_reduce, 1);
    Ls.rows.fn_pf2 = tk::cast_kernel_fn(d->in_dtype, d->out_fmt, d->scale_fmt, geo.cta_reduce, 2);
    Ls.row_bytes = d->hidden * (bf16 ? 2 : 4);
    Ls.block_lo = bf16 ? kCastBlockLoBf16 : kCastBlockLoF32;
    Ls.block_hi = bf16 ? kCastBlockHiBf16 : kCastBlockHiF32;
    auto *p = new (std::nothrow) tk_quant_cast_plan_s{*d, device, Ls, tk::ChannelFns{}, Launch{}, 0, 0};
    if (!p)
        return fail(TK_ERR_INVALID_ARG, "out of host memory");
    *plan = p;
    return ok();
}

TK_API tk_status tk_quant_cast_output_sizes(const tk_quant_cast_desc *d, int64_t T, size_t *q_bytes,
                                            size_t *scale_bytes_out)
{
    tk_status st = tk_quant_cast_validate(d);
    if (st != TK_OK)
        return st;
    if (T < 0 || !q_bytes || !scale_bytes_out)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 and the outputs non-NULL");
    const int64_t groups = d->group_size ? d->hidden / d->group_size : 1;
    *q_bytes = (size_t)T * (size_t)(d->out_fmt == TK_OUT_E4M3 ? d->hidden : d->hidden / 2);
    if (d->granularity == TK_GRAN_PER_CHANNEL)
        *scale_bytes_out = (size_t)d->hidden * (d->scale_fmt == TK_SCALE_FP32 ? 4u : 1u);
    else
        *scale_bytes_out = scale_bytes_for(d->scale_layout, d->scale_fmt, T, groups);
    return ok();
}

TK_API tk_status tk_quant_cast_plan_destroy(tk_quant_cast_plan_t plan)
{
    delete plan;
    return ok();
}

namespace {

// Host checks shared by both cast calls (T > 0).
tk_status check_cast_args(const tk_quant_cast_plan_s *plan, const void *x, const void *q, const void *scales)
{
    const tk_quant_cast_desc &d = plan->desc;
    if (!x || !q || !scales)
        return fail(TK_ERR_INVALID_ARG, "x, q and scales must be non-NULL");
    if (!aligned(x, 32))
        return fail(TK_ERR_MISALIGNED, "x must be 32-byte aligned");
    if (!aligned(q, 16))
        return fail(TK_ERR_MISALIGNED, "q must be 16-byte aligned");
    if (d.granularity == TK_GRAN_PER_CHANNEL) {
        if (!aligned(scales, 16))
            return fail(TK_ERR_MISALIGNED, "per-channel scales must be 16-byte aligned");
    } else {
        if (d.scale_fmt == TK_SCALE_FP32 && !aligned(scales, 4))
            return fail(TK_ERR_MISALIGNED, "fp32 scales must be 4-byte aligned");
        if (d.scale_layout != TK_SCALE_ROW_MAJOR && !aligned(scales, 16))
            return fail(TK_ERR_MISALIGNED, "column-major scales must be 16-byte aligned");
    }
    return check_current_device(plan->device);
}

tk_status launch_groups_cast(const tk_quant_cast_plan_s *plan, int64_t T, const void *x, void *q, void *scales,
                             void *stream)
{
    const tk_quant_cast_desc &d = plan->desc;
    tk::CastArgs a{x, (int32_t)d.hidden};
    tk::OutArgs o{static_cast<uint8_t *>(q), scales};
    const Launch &L = pick(plan->Ls, T);
    cudaError_t e = tk::launch_cast(row_fn(L, T, grid_for(L, T)), grid_for(L, T), L.block, L.smem, a, o,
                                    shape_for(L, T, d.hidden, d.scale_layout, d.scale_fmt),
                                    static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the cast kernel");
    return ok();
}

}  // namespace

TK_API tk_status tk_quant_cast_run(tk_quant_cast_plan_t plan, int64_t T, const void *x, void *q, void *scales,
                                   void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (plan->desc.granularity == TK_GRAN_PER_CHANNEL)
        return fail(TK_ERR_INVALID_ARG, "a per-channel cast needs device workspace: call tk_quant_cast_run_ws");
    if (T == 0)
        return ok();
    tk_status st = check_cast_args(plan, x, q, scales);
    if (st != TK_OK)
        return st;
    return launch_groups_cast(plan, T, x, q, scales, stream);
}

TK_API tk_status tk_quant_cast_workspace_size(tk_quant_cast_plan_t plan, int64_t T, size_t *bytes)
{
    if (!plan || !bytes || T < 0)
        return fail(TK_ERR_INVALID_ARG, "plan and bytes must be non-NULL and num_tokens >= 0");
    *bytes = plan->desc.granularity == TK_GRAN_PER_CHANNEL ? channel_workspace(plan, T) : 0;
    return ok();
}

TK_API tk_status tk_quant_cast_launch_info(tk_quant_cast_plan_t plan, int64_t T, int *launches, int *form)
{
    if (!plan || T < 0)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL or num_tokens < 0");
    int n = 1, f = TK_CAST_ROWS;
    if (plan->desc.granularity == TK_GRAN_PER_CHANNEL) {
        const bool split = channel_launch(plan, T > 0 ? T : 1).split;
        n = split ? 3 : 2;
        f = split ? TK_CAST_CHANNEL_SPLIT : TK_CAST_CHANNEL_CHUNK;
    } else {
        const Launch &L = pick(plan->Ls, T > 0 ? T : 1);
        f = L.kind == kBlockStream ? TK_CAST_BLOCK_RING : L.kind == kWarpStream ? TK_CAST_WARP_STREAM : TK_CAST_ROWS;
    }
    if (launches)
        *launches = T == 0 ? 0 : n;
    if (form)
        *form = f;
    return ok();
}

TK_API tk_status tk_quant_cast_run_ws(tk_quant_cast_plan_t plan, int64_t T, const void *x, void *q, void *scales,
                                      void *workspace, size_t workspace_bytes, void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    tk_status st = check_cast_args(plan, x, q, scales);
    if (st != TK_OK)
        return st;
    const tk_quant_cast_desc &d = plan->desc;
    if (d.granularity != TK_GRAN_PER_CHANNEL)
        return launch_groups_cast(plan, T, x, q, scales, stream);
    const size_t need = channel_workspace(plan, T);
    if (!workspace || workspace_bytes < need)
        return fail(TK_ERR_INVALID_ARG, "workspace must hold %zu bytes for %lld rows (got %zu)", need,
                    (long long)T, workspace ? workspace_bytes : (size_t)0);
    if (!aligned(workspace, 16))
        return fail(TK_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    const tk::ChannelLaunch L = channel_launch(plan, T);
    tk::CastArgs a{x, (int32_t)d.hidden};
    tk::OutArgs o{static_cast<uint8_t *>(q), scales};
    const tk::RowShape sh = shape_for(plan->cq, T, d.hidden, TK_SCALE_ROW_MAJOR, d.scale_fmt);
    cudaError_t e = tk::launch_channel(plan->cfn, L, a, o, sh, static_cast<float *>(workspace),
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the per-channel cast kernels");
    return ok();
}

// ------------------------------------------------------- weighted top-k combine

struct tk_moe_reduce_plan_s {
    tk_moe_reduce_desc desc;
    int device;
    const void *fn, *fn_pf;   // fn_pf: the form that prefetches its first task into L2
    int block, rpc, tpr, max_grid;
    unsigned *fault;
    // bulk kernel (has_bulk: the shape allows it)
    bool has_bulk;
    int forced;   // 0: by alignment, 1: register kernel, 2: bulk kernel where allowed
    const void *bulk_fn, *bulk_fn_pf;
    int nchunks, wc, stages, slot_bytes, rb, sb, smem, bulk_grid;
};

namespace {

// Chunking of the bulk combine: the fewest equal chunks per token whose slot
// (K row chunks, their scales, the metadata) fits kReduceSlotTarget bytes,
// with every copy 16-byte aligned; then as many slots as shared memory holds,
// up to kReduceMaxStages. Returns false where the bulk kernel does not apply (K > 32, rows
// under 2 KB, E4M3 rows with H not a multiple of 512, fewer than 2 slots).
// TK_REDUCE_SLOT_KB=<n> (read when the plan is made) overrides the target.
// E4M3 rows gather fastest as whole rows (fewer, larger copies per task).
constexpr int kReduceSlotTargetBf16 = 48 << 10;
constexpr int kReduceSlotTargetE4M3 = 64 << 10;

bool plan_reduce_bulk(tk_moe_reduce_plan_s *p, int optin)
{
    const tk_moe_reduce_desc &d = p->desc;
    const bool fp8 = d.in_fmt == TK_REDUCE_IN_E4M3;
    const int64_t elt = fp8 ? 1 : 2;
    if (d.topk > tk::kReduceBulkMaxK || d.hidden * elt < 2048 || (fp8 && d.hidden % 512 != 0))
        return false;
    const int64_t unit = fp8 ? 512 : 8;   // chunk widths keep copies aligned (and E4M3 scale rows)
    const int kb = env_int("TK_REDUCE_SLOT_KB", 0);
    const int64_t target = kb > 0 ? (int64_t)kb << 10 : (fp8 ? kReduceSlotTargetE4M3 : kReduceSlotTargetBf16);
    for (int64_t n = 1; n <= d.hidden / unit; ++n) {
        if (d.hidden % n != 0 || (d.hidden / n) % unit != 0)
            continue;
        const int64_t wc = d.hidden / n;
        const int64_t rb = wc * elt;
        const int64_t sb = fp8 ? wc / 128 * 4 : 0;
        const int64_t meta = 16 + 4 * (int64_t)d.topk;
        const int64_t slot = (d.topk * (rb + sb) + meta + 127) / 128 * 128;
        if (slot > target && n < d.hidden / unit)
            continue;
        const int64_t fit = (optin - 1024 - tk::kReduceMetaBytes) / (slot + 16);   // 1 KB for the runtime's reserve
        const int stages = (int)(fit < tk::kReduceMaxStages ? fit : tk::kReduceMaxStages);
        if (stages < 2)
            return false;
        p->nchunks = (int)n;
        p->wc = (int)wc;
        p->rb = (int)rb;
        p->sb = (int)sb;
        p->slot_bytes = (int)slot;
        p->stages = stages;
        p->smem = stages * (int)slot + 16 * stages + tk::kReduceMetaBytes;
        return true;
    }
    return false;
}

struct ReduceLaunch {
    bool bulk;
    const void *fn;
    int grid, block, smem;
};

// The bulk kernel runs for E4M3 rows where the plan allows it and y and
// y_scale are 16-byte aligned: there it gathers faster than the register
// kernel, whose bytes in flight are capped by registers at 16 bytes of row
// per thread and slot. bf16 rows (32 bytes per thread and slot) go to the
// register kernel, which was the faster of the two for them. Forcing the
// bulk kernel applies it wherever the plan and the alignment allow.
ReduceLaunch reduce_launch(const tk_moe_reduce_plan_s *p, int64_t T, const void *y, const float *y_scale)
{
    const bool fp8 = p->desc.in_fmt == TK_REDUCE_IN_E4M3;
    const bool wanted = p->forced == 2 || (p->forced == 0 && fp8);
    const bool bulk = p->has_bulk && wanted && aligned(y, 16) && (!fp8 || aligned(y_scale, 16));
    ReduceLaunch L{};
    L.bulk = bulk;
    // the prefetching forms where a CTA has at most 32 tasks (its first
    // ones are then a large enough share to be worth sending ahead)
    if (bulk) {
        const int64_t tasks = T * p->nchunks;
        L.grid = (int)(tasks < p->bulk_grid ? (tasks > 0 ? tasks : 1) : p->bulk_grid);
        L.fn = tasks <= 32 * (int64_t)L.grid ? p->bulk_fn_pf : p->bulk_fn;
        L.block = tk::kReduceBulkThreads;
        L.smem = p->smem;
    } else {
        const int64_t ntb = (T + p->rpc - 1) / p->rpc;
        L.grid = balanced_grid(ntb, p->max_grid);
        L.fn = ntb <= 32 * (int64_t)L.grid ? p->fn_pf : p->fn;
        L.block = p->block;
        L.smem = 0;
    }
    return L;
}

}  // namespace

TK_API tk_status tk_moe_reduce_validate(const tk_moe_reduce_desc *d)
{
    if (!d)
        return fail(TK_ERR_INVALID_ARG, "desc is NULL");
    if (d->hidden <= 0 || d->topk <= 0)
        return fail(TK_ERR_INVALID_ARG, "hidden and topk must be positive");
    if (d->hidden % 16 != 0 || d->hidden > 8192)
        return fail(TK_ERR_UNSUPPORTED, "hidden must be a multiple of 16 in [16, 8192] (got %lld)",
                    (long long)d->hidden);
    if (d->topk > 64)
        return fail(TK_ERR_UNSUPPORTED, "topk must be at most 64 (got %d)", d->topk);
    if (d->in_fmt != TK_REDUCE_IN_BF16 && d->in_fmt != TK_REDUCE_IN_E4M3)
        return fail(TK_ERR_INVALID_ARG, "unknown in_fmt %d", d->in_fmt);
    if (d->in_fmt == TK_REDUCE_IN_E4M3 && d->hidden % 128 != 0)
        return fail(TK_ERR_UNSUPPORTED, "E4M3 rows need hidden to be a multiple of 128");
    return ok();
}

TK_API tk_status tk_moe_reduce_plan(const tk_moe_reduce_desc *d, int device, tk_moe_reduce_plan_t *plan)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan output pointer is NULL");
    *plan = nullptr;
    tk_status st = tk_moe_reduce_validate(d);
    if (st != TK_OK)
        return st;
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= count)
        return fail(TK_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, count);
    DeviceScope scope(device);
    if (scope.err != cudaSuccess)
        return cuda_fail(scope.err, "cudaSetDevice");
    tk_moe_reduce_plan_s p{};
    p.desc = *d;
    p.device = device;
    p.fn = tk::moe_reduce_kernel_fn(d->in_fmt, false);
    p.fn_pf = tk::moe_reduce_kernel_fn(d->in_fmt, true);
    p.tpr = (int)(d->hidden / tk::kEPT);
    p.rpc = p.tpr >= 256 ? 1 : 256 / p.tpr;
    p.block = ((p.tpr * p.rpc + 31) / 32) * 32;   // <= 512 for hidden <= 8192
    int num_sms = 0, occ = 0;
    void *fault = nullptr;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p.fn, p.block, 0);
    if (e == cudaSuccess)
        e = cudaGetSymbolAddress(&fault, g_tk_fault_word);
    if (e != cudaSuccess)
        return cuda_fail(e, "querying the device");
    if (occ < 1)
        return fail(TK_ERR_UNSUPPORTED, "kernel cannot be resident with %d threads per CTA", p.block);
    p.max_grid = occ * num_sms;
    p.fault = static_cast<unsigned *>(fault);
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess)
        return cuda_fail(e, "querying the device");
    p.has_bulk = plan_reduce_bulk(&p, optin);
    if (p.has_bulk) {
        p.bulk_fn = tk::moe_reduce_bulk_kernel_fn(d->in_fmt, false);
        p.bulk_fn_pf = tk::moe_reduce_bulk_kernel_fn(d->in_fmt, true);
        e = cudaFuncSetAttribute(p.bulk_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(p.bulk_fn_pf, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
        int bocc = 0;
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bocc, p.bulk_fn, tk::kReduceBulkThreads, p.smem);
        if (e != cudaSuccess)
            return cuda_fail(e, "configuring the bulk combine kernel");
        p.has_bulk = bocc >= 1;
        p.bulk_grid = bocc * num_sms;
    }
    // TK_REDUCE_KERNEL=regs or =bulk (read when the plan is made) forces one
    // kernel where the shape (and, for bulk, the alignment) allows it.
    const char *force = getenv("TK_REDUCE_KERNEL");
    p.forced = !force ? 0 : (strcmp(force, "regs") == 0 ? 1 : (strcmp(force, "bulk") == 0 ? 2 : 0));
    auto *h = new (std::nothrow) tk_moe_reduce_plan_s(p);
    if (!h)
        return fail(TK_ERR_INVALID_ARG, "out of host memory");
    *plan = h;
    return ok();
}

TK_API tk_status tk_moe_reduce_plan_destroy(tk_moe_reduce_plan_t plan)
{
    delete plan;
    return ok();
}

TK_API tk_status tk_moe_reduce_run(tk_moe_reduce_plan_t plan, int64_t T, const void *y, const float *y_scale,
                                   int64_t num_rows, const int32_t *pos, const float *w, float gs, void *out,
                                   void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0 || num_rows < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens and num_rows must be >= 0");
    if (T == 0)
        return ok();
    const tk_moe_reduce_desc &d = plan->desc;
    const bool fp8 = d.in_fmt == TK_REDUCE_IN_E4M3;
    if (!pos || !w || !out || (num_rows > 0 && !y) || (fp8 && num_rows > 0 && !y_scale))
        return fail(TK_ERR_INVALID_ARG, "y, y_scale (E4M3), token_topk_to_pos, topk_weights and out "
                                        "must be non-NULL");
    if (!std::isfinite(gs))
        return fail(TK_ERR_INVALID_ARG, "global_scale must be finite");
    if (y && !aligned(y, fp8 ? 16 : 32))
        return fail(TK_ERR_MISALIGNED, "y must be %d-byte aligned", fp8 ? 16 : 32);
    if (!aligned(out, 16))
        return fail(TK_ERR_MISALIGNED, "out must be 16-byte aligned");
    if (!aligned(pos, 4) || !aligned(w, 4) || (fp8 && y_scale && !aligned(y_scale, 4)))
        return fail(TK_ERR_MISALIGNED, "token_topk_to_pos, topk_weights and y_scale must be 4-byte aligned");
    tk_status st = check_current_device(plan->device);
    if (st != TK_OK)
        return st;
    tk::ReduceArgs a{};
    a.y = y;
    a.y_scale = fp8 ? y_scale : nullptr;
    a.R = num_rows;
    a.H = (int32_t)d.hidden;
    a.K = d.topk;
    a.pos = pos;
    a.w = w;
    a.T = T;
    a.gs = gs;
    a.out = out;
    a.tpr = plan->tpr;
    a.rpc = plan->rpc;
    a.fault = plan->fault;
    const ReduceLaunch L = reduce_launch(plan, T, y, y_scale);
    a.nchunks = plan->nchunks;
    a.wc = plan->wc;
    a.stages = plan->stages;
    a.slot_bytes = plan->slot_bytes;
    a.rb = plan->rb;
    a.sb = plan->sb;
    cudaError_t e = tk::launch_moe_reduce(L.fn, L.grid, L.block, L.smem, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the combine kernel");
    return ok();
}

TK_API tk_status tk_moe_reduce_launch_info(tk_moe_reduce_plan_t plan, int64_t num_tokens, const void *y,
                                           const float *y_scale, int *kernel, int *grid, int *block,
                                           int *smem_bytes)
{
    if (!plan || !kernel || !grid || !block || !smem_bytes)
        return fail(TK_ERR_INVALID_ARG, "plan and outputs must be non-NULL");
    if (num_tokens < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0");
    const ReduceLaunch L = reduce_launch(plan, num_tokens, y, y_scale);
    *kernel = L.bulk ? 1 : 0;
    *grid = L.grid;
    *block = L.block;
    *smem_bytes = L.smem;
    return ok();
}

// ------------------------------------------------------------------ backward

struct tk_swiglu_backward_plan_s {
    tk_swiglu_backward_desc desc;
    int device;
    const void *fn;
    const void *fn_pf;   // the form that prefetches its first row block (runs with few row blocks per CTA)
    const void *fn_pf2;  // the form that also prefetches each next row block
    int pf_forced;       // TK_BACKWARD_PF=0|1|2 when the plan was made, else -1
    int block, tpr, rpc, tpg_log2, groups, max_grid;
    unsigned *fault;
};

TK_API tk_status tk_swiglu_backward_validate(const tk_swiglu_backward_desc *d)
{
    if (!d)
        return fail(TK_ERR_INVALID_ARG, "desc is NULL");
    const int64_t H = d->hidden;
    if (H <= 0)
        return fail(TK_ERR_INVALID_ARG, "hidden must be positive (got %lld)", (long long)H);
    const bool small = H == 16 || H == 32 || H == 64 || H == 128 || H == 256;
    if (!small && !(H % 512 == 0 && H <= 8192))
        return fail(TK_ERR_UNSUPPORTED, "hidden must be 16, 32, 64, 128, 256 or a multiple of 512 up to 8192 "
                                        "(got %lld)", (long long)H);
    if (!is_flag(d->has_topk_weights) || !is_flag(d->use_clamp) || !is_flag(d->recompute_quant))
        return fail(TK_ERR_INVALID_ARG, "has_topk_weights, use_clamp and recompute_quant must be 0 or 1");
    if (d->use_clamp && !(d->clamp_limit > 0.0f && std::isfinite(d->clamp_limit)))
        return fail(TK_ERR_INVALID_ARG, "clamp_limit must be finite and > 0");
    if (d->recompute_quant) {
        if (d->group_size == 0)
            return fail(TK_ERR_UNSUPPORTED, "the recompute needs group_size 16 ... 512 (no per-token scale)");
        tk_swiglu_quant_desc f{};
        f.hidden = H;
        f.group_size = d->group_size;
        f.scale_fmt = d->scale_fmt;
        f.out_fmt = d->out_fmt;
        f.has_topk_weights = d->has_topk_weights;
        f.use_clamp = d->use_clamp;
        f.clamp_limit = d->clamp_limit;
        f.count_clamped = 0;
        f.scale_layout = d->scale_layout;
        return tk_swiglu_quant_validate(&f);
    }
    return ok();
}

TK_API tk_status tk_swiglu_backward_plan(const tk_swiglu_backward_desc *d, int device, tk_swiglu_backward_plan_t *plan)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan output pointer is NULL");
    *plan = nullptr;
    tk_status st = tk_swiglu_backward_validate(d);
    if (st != TK_OK)
        return st;
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= count)
        return fail(TK_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, count);
    DeviceScope scope(device);
    if (scope.err != cudaSuccess)
        return cuda_fail(scope.err, "cudaSetDevice");
    tk_swiglu_backward_plan_s p{};
    p.desc = *d;
    p.device = device;
    uint32_t limit_bits = 0;
    memcpy(&limit_bits, &d->clamp_limit, sizeof limit_bits);
    const int clamp_mode = !d->use_clamp ? 0 : (limit_bits & 0xffffu) == 0 ? 2 : 1;
    p.fn = tk::backward_kernel_fn(clamp_mode, d->recompute_quant != 0, d->out_fmt, d->scale_fmt, 0);
    p.fn_pf = tk::backward_kernel_fn(clamp_mode, d->recompute_quant != 0, d->out_fmt, d->scale_fmt, 1);
    p.fn_pf2 = tk::backward_kernel_fn(clamp_mode, d->recompute_quant != 0, d->out_fmt, d->scale_fmt, 2);
    {
        const int f = env_int("TK_BACKWARD_PF", -1);
        p.pf_forced = f >= 0 && f <= 2 ? f : -1;
    }
    p.tpr = (int)(d->hidden / tk::kEPT);
    p.rpc = p.tpr >= 256 ? 1 : 256 / p.tpr;
    p.block = ((p.tpr * p.rpc + 31) / 32) * 32;   // <= 512 for hidden <= 8192
    if (d->recompute_quant) {
        p.tpg_log2 = ilog2(d->group_size / tk::kEPT);
        p.groups = (int)(d->hidden / d->group_size);
    }
    int num_sms = 0, occ = 0;
    void *fault = nullptr;
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p.fn, p.block, 0);
    if (e == cudaSuccess)
        e = cudaGetSymbolAddress(&fault, g_tk_fault_word);
    if (e != cudaSuccess)
        return cuda_fail(e, "querying the device");
    if (occ < 1)
        return fail(TK_ERR_UNSUPPORTED, "kernel cannot be resident with %d threads per CTA", p.block);
    p.max_grid = occ * num_sms;
    p.fault = static_cast<unsigned *>(fault);
    auto *h = new (std::nothrow) tk_swiglu_backward_plan_s(p);
    if (!h)
        return fail(TK_ERR_INVALID_ARG, "out of host memory");
    *plan = h;
    return ok();
}

TK_API tk_status tk_swiglu_backward_plan_destroy(tk_swiglu_backward_plan_t plan)
{
    delete plan;
    return ok();
}

TK_API tk_status tk_swiglu_backward_run(tk_swiglu_backward_plan_t plan, int64_t T, const void *x,
                                        const float *topk_weights, const void *dy, void *dx, float *dw, void *q,
                                        void *scales, void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    const tk_swiglu_backward_desc &d = plan->desc;
    if (!x || !dy || !dx)
        return fail(TK_ERR_INVALID_ARG, "x, dy and dx must be non-NULL");
    if (d.has_topk_weights && !topk_weights)
        return fail(TK_ERR_INVALID_ARG, "the plan expects topk_weights");
    if (d.recompute_quant && (!q || !scales))
        return fail(TK_ERR_INVALID_ARG, "the plan recomputes the codes: q and scales must be non-NULL");
    if (!aligned(x, 32) || !aligned(dy, 32))
        return fail(TK_ERR_MISALIGNED, "x and dy must be 32-byte aligned");
    if (!aligned(dx, 16))
        return fail(TK_ERR_MISALIGNED, "dx must be 16-byte aligned");
    if ((dw && !aligned(dw, 4)) || (d.has_topk_weights && !aligned(topk_weights, 4)))
        return fail(TK_ERR_MISALIGNED, "dw and topk_weights must be 4-byte aligned");
    if (d.recompute_quant) {
        if (!aligned(q, 16))
            return fail(TK_ERR_MISALIGNED, "q must be 16-byte aligned");
        if ((d.scale_fmt == TK_SCALE_FP32 && !aligned(scales, 4)) ||
            (d.scale_layout != TK_SCALE_ROW_MAJOR && !aligned(scales, 16)))
            return fail(TK_ERR_MISALIGNED, "scales must be 4-byte (fp32) or 16-byte (column-major) aligned");
    }
    tk_status st = check_current_device(plan->device);
    if (st != TK_OK)
        return st;
    tk::BackwardArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.dy = static_cast<const uint16_t *>(dy);
    a.w = d.has_topk_weights ? topk_weights : nullptr;
    a.dx = static_cast<uint16_t *>(dx);
    a.dw = dw;
    a.limit = d.use_clamp ? d.clamp_limit : 0.0f;
    a.H = (int32_t)d.hidden;
    uint32_t limit_bits = 0;
    memcpy(&limit_bits, &a.limit, sizeof limit_bits);
    a.limit2 = (limit_bits >> 16) * 0x00010001u;
    tk::OutArgs o{static_cast<uint8_t *>(q), scales};
    const int32_t layout = d.recompute_quant ? d.scale_layout : TK_SCALE_ROW_MAJOR;
    const tk::RowShape sh{T, (int32_t)d.hidden, plan->tpr, plan->tpg_log2, plan->rpc, plan->groups, 0, 0,
                          plan->fault, layout, scale_ld(layout, d.scale_fmt, T)};
    const int64_t nrb = (T + plan->rpc - 1) / plan->rpc;
    const int grid = (int)(nrb < plan->max_grid ? nrb : plan->max_grid);
    // Prefetching forms by row blocks per CTA: the first block and each next
    // one at up to 8, the first only at up to 32. Measured on GB300 at width
    // 2048 (µs, first block only / each next block too): 8192 rows (6.7
    // blocks per CTA) 30.15/28.68 without the clamp, 32.22/30.80 with it;
    // 32768 rows (27 per CTA) 110.97/129.30 and 110.88/128.91 (UE8M0, clamp):
    // with many blocks per CTA the extra prefetches cost more than they hide.
    const int mode = plan->pf_forced >= 0        ? plan->pf_forced
                     : nrb <= 8 * (int64_t)grid  ? 2
                     : nrb <= 32 * (int64_t)grid ? 1
                                                 : 0;
    const void *fn = mode == 2 ? plan->fn_pf2 : mode == 1 ? plan->fn_pf : plan->fn;
    cudaError_t e = tk::launch_backward(fn, grid, plan->block, a, o, sh, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the backward kernel");
    return ok();
}

// ---------------------------------------------------------------- diagnostics

TK_API tk_status tk_fault_word(int device, uint32_t *value, int clear)
{
    if (!value)
        return fail(TK_ERR_INVALID_ARG, "value is NULL");
    DeviceScope scope(device);
    if (scope.err != cudaSuccess)
        return cuda_fail(scope.err, "cudaSetDevice");
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tk_fault_word, sizeof v);
    if (e == cudaSuccess && clear) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_tk_fault_word, &zero, sizeof zero);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "reading the fault word");
    *value = v;
    return ok();
}


TK_API tk_status tk_diag_unanswered_wait(int device, uint32_t tries, void *stream)
{
    if (tries == 0 || tries > (1u << 22))
        return fail(TK_ERR_INVALID_ARG, "tries must be in [1, 2^22] (got %u)", tries);
    tk_status st = check_current_device(device);
    if (st != TK_OK)
        return st;
    void *fault = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&fault, g_tk_fault_word);
    if (e == cudaSuccess)
        e = tk::launch_unanswered_wait(static_cast<unsigned *>(fault), tries, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the unanswered-wait kernel");
    return ok();
}

TK_API const char *tk_status_string(tk_status s)
{
    switch (s) {
    case TK_OK: return "TK_OK";
    case TK_ERR_INVALID_ARG: return "TK_ERR_INVALID_ARG";
    case TK_ERR_UNSUPPORTED: return "TK_ERR_UNSUPPORTED";
    case TK_ERR_MISALIGNED: return "TK_ERR_MISALIGNED";
    case TK_ERR_CUDA: return "TK_ERR_CUDA";
    case TK_ERR_DEVICE: return "TK_ERR_DEVICE";
    }
    return "TK_ERR_UNKNOWN";
}

TK_API const char *tk_last_error_message(void) { return g_msg.c_str(); }
