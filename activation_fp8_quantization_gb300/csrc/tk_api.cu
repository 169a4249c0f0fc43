// C ABI: descriptor validation, plans (launch shape chosen once per device)
// and stream-ordered launches. Declared in include/tk_swiglu_quant.h.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "tk_internal.h"
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

// Device facts a plan records once.
tk_status query_device(int device, const void *fn, int block, int *num_sms, int *max_grid)
{
    int count = 0;
    cudaError_t e = cudaGetDeviceCount(&count);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDeviceCount");
    if (device < 0 || device >= count)
        return fail(TK_ERR_INVALID_ARG, "device %d out of range (%d devices)", device, count);
    e = cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
    int prev = -1;
    e = cudaGetDevice(&prev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess)
        return cuda_fail(e, "cudaSetDevice");
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, block, 0);
    if (prev != device)
        cudaSetDevice(prev);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (occ < 1)
        return fail(TK_ERR_UNSUPPORTED, "kernel cannot be resident with %d threads per CTA", block);
    *max_grid = *num_sms * occ;
    return TK_OK;
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

int grid_for(int64_t T, int rpc, int max_grid)
{
    const int64_t nrb = (T + rpc - 1) / rpc;
    return (int)(nrb < max_grid ? nrb : max_grid);
}

}  // namespace

struct tk_swiglu_quant_plan_s {
    tk_swiglu_quant_desc desc;
    int device;
    int num_sms;
    int max_grid;
    Geometry geo;
    const void *fn;
};

struct tk_quant_cast_plan_s {
    tk_quant_cast_desc desc;
    int device;
    int num_sms;
    int max_grid;
    Geometry geo;
    const void *fn;
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
    if (d->reserved != 0)
        return fail(TK_ERR_INVALID_ARG, "reserved must be 0");
    return ok();
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
    const void *fn = tk::swiglu_kernel_fn(d->out_fmt, d->scale_fmt, d->use_clamp != 0, geo.cta_reduce);
    if (!fn)
        return fail(TK_ERR_UNSUPPORTED, "no kernel for this combination");
    int num_sms = 0, max_grid = 0;
    st = query_device(device, fn, geo.block, &num_sms, &max_grid);
    if (st != TK_OK)
        return st;
    auto *p = new (std::nothrow) tk_swiglu_quant_plan_s{*d, device, num_sms, max_grid, geo, fn};
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
    *scale_bytes = (size_t)T * (size_t)groups * (d->scale_fmt == TK_SCALE_FP32 ? 4u : 1u);
    return ok();
}

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
    if (d.has_topk_weights && !aligned(topk_weights, 4))
        return fail(TK_ERR_MISALIGNED, "topk_weights must be 4-byte aligned");
    if (d.count_clamped && !aligned(clamped_count, 8))
        return fail(TK_ERR_MISALIGNED, "clamped_count must be 8-byte aligned");
    tk_status st = check_current_device(plan->device);
    if (st != TK_OK)
        return st;

    tk::SwigluArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.w = d.has_topk_weights ? topk_weights : nullptr;
    a.counts = d.count_clamped ? reinterpret_cast<unsigned long long *>(clamped_count) : nullptr;
    a.limit = d.use_clamp ? d.clamp_limit : 0.0f;
    a.H = (int32_t)d.hidden;
    tk::OutArgs o{static_cast<uint8_t *>(q), scales};
    const Geometry &g = plan->geo;
    tk::RowShape sh{T, (int32_t)d.hidden, g.tpr, g.tpg_log2, g.rpc, g.groups};
    const int grid = grid_for(T, g.rpc, plan->max_grid);
    cudaError_t e = tk::launch_swiglu(plan->fn, grid, g.block, a, o, sh, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the fused kernel");
    return ok();
}

TK_API tk_status tk_swiglu_quant_launch_info(tk_swiglu_quant_plan_t plan, int64_t T, int *grid, int *block,
                                             int *rows_per_cta, int *num_sms)
{
    if (!plan || T < 0)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL or num_tokens < 0");
    if (grid)
        *grid = T == 0 ? 0 : grid_for(T, plan->geo.rpc, plan->max_grid);
    if (block)
        *block = plan->geo.block;
    if (rows_per_cta)
        *rows_per_cta = plan->geo.rpc;
    if (num_sms)
        *num_sms = plan->num_sms;
    return ok();
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
    return ok();
}

TK_API tk_status tk_quant_cast_plan(const tk_quant_cast_desc *d, int device, tk_quant_cast_plan_t *plan)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan output pointer is NULL");
    *plan = nullptr;
    tk_status st = tk_quant_cast_validate(d);
    if (st != TK_OK)
        return st;
    const Geometry geo = geometry(d->hidden, d->group_size);
    const void *fn = tk::cast_kernel_fn(d->in_dtype, d->out_fmt, d->scale_fmt, geo.cta_reduce);
    if (!fn)
        return fail(TK_ERR_UNSUPPORTED, "no kernel for this combination");
    int num_sms = 0, max_grid = 0;
    st = query_device(device, fn, geo.block, &num_sms, &max_grid);
    if (st != TK_OK)
        return st;
    auto *p = new (std::nothrow) tk_quant_cast_plan_s{*d, device, num_sms, max_grid, geo, fn};
    if (!p)
        return fail(TK_ERR_INVALID_ARG, "out of host memory");
    *plan = p;
    return ok();
}

TK_API tk_status tk_quant_cast_plan_destroy(tk_quant_cast_plan_t plan)
{
    delete plan;
    return ok();
}

TK_API tk_status tk_quant_cast_run(tk_quant_cast_plan_t plan, int64_t T, const void *x, void *q, void *scales,
                                   void *stream)
{
    if (!plan)
        return fail(TK_ERR_INVALID_ARG, "plan is NULL");
    if (T < 0)
        return fail(TK_ERR_INVALID_ARG, "num_tokens must be >= 0 (got %lld)", (long long)T);
    if (T == 0)
        return ok();
    const tk_quant_cast_desc &d = plan->desc;
    if (!x || !q || !scales)
        return fail(TK_ERR_INVALID_ARG, "x, q and scales must be non-NULL");
    if (!aligned(x, 32))
        return fail(TK_ERR_MISALIGNED, "x must be 32-byte aligned");
    if (!aligned(q, 16))
        return fail(TK_ERR_MISALIGNED, "q must be 16-byte aligned");
    if (d.scale_fmt == TK_SCALE_FP32 && !aligned(scales, 4))
        return fail(TK_ERR_MISALIGNED, "fp32 scales must be 4-byte aligned");
    tk_status st = check_current_device(plan->device);
    if (st != TK_OK)
        return st;
    tk::CastArgs a{x, (int32_t)d.hidden};
    tk::OutArgs o{static_cast<uint8_t *>(q), scales};
    const Geometry &g = plan->geo;
    tk::RowShape sh{T, (int32_t)d.hidden, g.tpr, g.tpg_log2, g.rpc, g.groups};
    const int grid = grid_for(T, g.rpc, plan->max_grid);
    cudaError_t e = tk::launch_cast(plan->fn, grid, g.block, a, o, sh, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "launch of the cast kernel");
    return ok();
}

// ---------------------------------------------------------------- diagnostics

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
