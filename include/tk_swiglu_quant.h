/*
 * tk_swiglu_quant.h -- C ABI of the fused SwiGLU + MoE top-k weight +
 * FP8/FP4 activation cast and the operations around it:
 *   tk_swiglu_quant_*     the fused op (device buffers; host buffers staged
 *                         through device memory, or read and written in place
 *                         by the kernel; codes row-major or transposed)
 *   tk_quant_cast_*       the standalone per-token / per-block / per-channel cast
 *   tk_moe_reduce_*       the weighted top-k combine after the expert GEMMs
 *   tk_swiglu_backward_*  the SwiGLU backward, optionally recomputing the codes
 *   tk_fault_word, tk_diag_unanswered_wait, tk_status_string,
 *   tk_last_error_message                                     diagnostics
 *
 * The operation ("TileKernels从入门到精通" / "TileKernels from Beginner to
 * Master", zhichai.net/topic/177618752 and zhichai.net/en/topic/177618752,
 * chapter 2): every row r of x [T, 2H] (bf16, row-major) is one expanded
 * (token, expert) pair; its gate half g = x[r, 0:H] and up half u = x[r, H:2H]
 * ("conjoined twin" layout) give
 *
 *     y[r, i] = silu(g') * u' * w[r],   silu(z) = z / (1 + exp(-z)),
 *     g' = min(g, L),  u' = clamp(u, -L, L)          (only with use_clamp),
 *
 * computed in fp32 registers. y is cut into groups of `group_size` columns
 * (or one group per row); each group gets a scale from its absolute maximum
 * amax -- fp32 s = amax / Qmax, or UE8M0 s = 2^k with k the smallest integer
 * such that Qmax * 2^k >= amax -- and each value is stored as the
 * round-to-nearest-even, saturating code of y / s in FP8 E4M3 (Qmax = 448) or
 * FP4 E2M1 (Qmax = 6). Formats and granularities: "TileLang + TileKernels：
 * DeepSeek 的 GPU 内核开发新范式" (zhichai.net/topic/177618740), section
 * "3. Quantization", format table. Clamp guard and its counter: same chapter 2,
 * "守门员 Clamp". The standalone cast is the same scaling and encoding applied
 * to an input that is already the activation (ch.1, per_token_cast).
 *
 * Conventions for every entry point:
 *  - Device pointers are CUDA global-memory addresses on the plan's device,
 *    owned by the caller; the library never frees or retains them.
 *  - Calls are stream-ordered and asynchronous: they enqueue work on `stream`
 *    (a cudaStream_t passed as void*, NULL = the legacy default stream) and
 *    return without synchronising. Errors detected on the host are returned
 *    before anything is enqueued.
 *  - A plan is immutable once made and may be used from several host threads
 *    and streams at once. It holds host state only (the descriptor, the device
 *    ordinal, the launch shape); destroying it does not touch device memory.
 *  - On any status other than TK_OK, tk_last_error_message() returns a
 *    description for the calling thread.
 */
#ifndef TK_SWIGLU_QUANT_H
#define TK_SWIGLU_QUANT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tk_status {
    TK_OK = 0,
    TK_ERR_INVALID_ARG = 1,  /* null where a pointer is required, negative size, bad enum */
    TK_ERR_UNSUPPORTED = 2,  /* well-formed but outside what is implemented (e.g. hidden > 16384) */
    TK_ERR_MISALIGNED = 3,   /* a pointer breaks the alignment rules of the call */
    TK_ERR_CUDA = 4,         /* a CUDA runtime call failed (message has the CUDA error) */
    TK_ERR_DEVICE = 5        /* the calling thread's current device is not the plan's device */
} tk_status;

typedef enum tk_scale_fmt {
    TK_SCALE_FP32 = 0,   /* one fp32 per group: amax / Qmax (1.0 if that is zero) */
    TK_SCALE_UE8M0 = 1   /* one byte per group: k + 127, scale 2^k (byte 127 for amax == 0) */
} tk_scale_fmt;

typedef enum tk_out_fmt {
    TK_OUT_E4M3 = 0,     /* one byte per value, OCP FP8 E4M3 (max 448, no inf) */
    TK_OUT_E2M1 = 1      /* two values per byte, OCP FP4 E2M1 (max 6); value 2k in the low nibble */
} tk_out_fmt;

typedef enum tk_in_dtype {
    TK_IN_BF16 = 0,
    TK_IN_FP32 = 1
} tk_in_dtype;

/* Where the scale of group j of row t goes ("TMA-aligned column-major scale
 * factors" and "packed" UE8M0 of the quantization section of "TileLang +
 * TileKernels", zhichai.net/topic/177618740; the exact layouts are this
 * library's reading). G = groups per row. */
typedef enum tk_scale_layout {
    TK_SCALE_ROW_MAJOR = 0,        /* [T, G]: element t*G + j */
    TK_SCALE_COL_MAJOR = 1,        /* [G, Tp]: element j*Tp + t, Tp = T rounded up to a multiple of
                                      16 bytes of scale elements (4 fp32 or 16 UE8M0), so every
                                      column starts on a 16-byte boundary; rows t >= T of the
                                      padding are not written */
    TK_SCALE_COL_MAJOR_PACKED = 2  /* UE8M0 only, G % 4 == 0: 32-bit words [G/4, Tp4], word
                                      m*Tp4 + t holds the exponents of groups 4m..4m+3 of row t,
                                      group 4m in the low byte; Tp4 = T rounded up to 4; padding
                                      words are not written */
} tk_scale_layout;

/* ------------------------------------------------------------------------
 * Fused SwiGLU + top-k weight + cast
 * ---------------------------------------------------------------------- */

typedef struct tk_swiglu_quant_desc {
    int64_t hidden;            /* H: width of the output; x rows hold 2H bf16. 16 <= H <= 16384, H % 16 == 0 */
    int32_t group_size;        /* columns per scale: 16, 32, 64, 128, 256 or 512 (dividing H); 0 = one per row */
    int32_t scale_fmt;         /* tk_scale_fmt */
    int32_t out_fmt;           /* tk_out_fmt */
    int32_t has_topk_weights;  /* 1: run() takes fp32 weights [T]; 0: weight 1 */
    int32_t use_clamp;         /* 1: gate <= clamp_limit, up in [-clamp_limit, clamp_limit] */
    float clamp_limit;         /* finite, >= 0; read only when use_clamp */
    int32_t count_clamped;     /* 1: run() ADDS the clamp counts into a device int64[2]; needs use_clamp */
    int32_t scale_layout;      /* tk_scale_layout */
} tk_swiglu_quant_desc;

typedef struct tk_swiglu_quant_plan_s *tk_swiglu_quant_plan_t;

/* Check a descriptor on the host only (no CUDA call). TK_OK,
 * TK_ERR_INVALID_ARG or TK_ERR_UNSUPPORTED. */
tk_status tk_swiglu_quant_validate(const tk_swiglu_quant_desc *desc);

/* Validate desc, query device `device` (SM count, occupancy) and pick the
 * kernel and launch shape. On TK_OK *plan owns a host allocation released by
 * tk_swiglu_quant_plan_destroy. Does not change the current device. */
tk_status tk_swiglu_quant_plan(const tk_swiglu_quant_desc *desc, int device,
                               tk_swiglu_quant_plan_t *plan);

/* Release a plan (NULL is accepted). The plan must not be used afterwards. */
tk_status tk_swiglu_quant_plan_destroy(tk_swiglu_quant_plan_t plan);

/* Bytes of the code and scale outputs for num_tokens rows (host only):
 * q: T*H (E4M3) or T*H/2 (E2M1); scales, with e = 4 (fp32) or 1 (UE8M0) and
 * G = H / group_size (1 when group_size == 0): T*G*e row-major, G*Tp*e
 * column-major, (G/4)*Tp4*4 packed (see tk_scale_layout). */
tk_status tk_swiglu_quant_output_sizes(const tk_swiglu_quant_desc *desc, int64_t num_tokens,
                                       size_t *q_bytes, size_t *scale_bytes);

/* Enqueue the fused kernel.
 *   x             [T, 2H] bf16, row-major, gate half first; 32-byte aligned
 *   topk_weights  [T] fp32, 4-byte aligned; required iff has_topk_weights, else ignored
 *   q             codes, [T, H] or [T, H/2] bytes, row-major; 16-byte aligned
 *   scales        fp32 or uint8 in the plan's scale layout; 4-byte aligned
 *                 (fp32, row-major), 16-byte aligned (column-major layouts)
 *   clamped_count device int64[2], 8-byte aligned: [0] += gate values above
 *                 the limit, [1] += up values outside [-L, L]; required iff
 *                 count_clamped, else ignored. The caller zeroes it.
 * num_tokens == 0 enqueues nothing and returns TK_OK. The calling thread's
 * current device must be the plan's device (TK_ERR_DEVICE otherwise). Inputs
 * and outputs must not overlap. */
tk_status tk_swiglu_quant_run(tk_swiglu_quant_plan_t plan, int64_t num_tokens,
                              const void *x, const float *topk_weights, void *q,
                              void *scales, int64_t *clamped_count, void *stream);

/* ------------------------------------------------------------------------
 * Fused op with the codes written transposed
 *
 * "TileKernels从入门到精通" (zhichai.net/topic/177618752), closing section
 * "结语：工程化极致的胜利": SwiGLU, the per-token quant and the transpose are
 * fused into one kernel launch. The grouping (g consecutive columns of one
 * row), the scales (in the plan's scale layout) and the codes are exactly
 * those of tk_swiglu_quant_run; only the codes are stored transposed:
 *
 *     qt[i * ld + t] = code of row t, column i      (0 <= i < H, 0 <= t < T)
 *
 * with ld = T rounded up to a multiple of 32, so every row of qt starts
 * 32-byte aligned (each thread of the kernel then writes one whole 32-byte
 * sector of 32 rows with a single store); qt[i * ld + t] for T <= t < ld is
 * written as 0. This is the operand layout of a following GEMM that
 * contracts over the rows.
 * Requires a plan with E4M3 codes, group_size 32, 64 or 128 and H % 128 == 0
 * (TK_ERR_UNSUPPORTED otherwise). Arguments, alignment and errors are those
 * of tk_swiglu_quant_run, with qt (H * ld bytes, 16-byte aligned; 32-byte
 * aligned for the single-store form) in place of q; the clamp counters are
 * added to as there.
 * ---------------------------------------------------------------------- */

/* ld and the bytes of qt for num_tokens rows (host only). */
tk_status tk_swiglu_quant_transposed_size(tk_swiglu_quant_plan_t plan, int64_t num_tokens, size_t *qt_bytes,
                                          int64_t *ld);

tk_status tk_swiglu_quant_run_transposed(tk_swiglu_quant_plan_t plan, int64_t num_tokens, const void *x,
                                         const float *topk_weights, void *qt, void *scales,
                                         int64_t *clamped_count, void *stream);

/* Launch shape a run of num_tokens rows would use (host only): CTAs in the
 * persistent grid, threads per CTA, rows one CTA takes per iteration (the
 * rows of one ring slot for the block-ring kernel; 0 for the warp-stream
 * kernel, whose warps each stream 512-column slices), the SM count, and which
 * kernel (TK_KERNEL_ROWS, TK_KERNEL_WARP_STREAM or TK_KERNEL_BLOCK_RING). Any
 * output pointer may be NULL. Where the width is a multiple of 512 a plan
 * holds the stream kernels too and picks per run by num_tokens: the block-ring
 * kernel once every resident CTA has enough row blocks to stream (32, or 16
 * with the clamp, where the row kernel packs two or more rows per CTA; 8 for
 * wider rows), the row kernel below that. */
typedef enum tk_kernel_kind {
    TK_KERNEL_ROWS = 0,         /* row_quant_kernel: register-prefetch row blocks, any width */
    TK_KERNEL_WARP_STREAM = 1,  /* warp_stream_kernel: a TMA ring per warp */
    TK_KERNEL_BLOCK_RING = 2    /* block_stream_kernel: one TMA ring per CTA, whole rows per slot */
} tk_kernel_kind;
tk_status tk_swiglu_quant_launch_info(tk_swiglu_quant_plan_t plan, int64_t num_tokens,
                                      int *grid, int *block, int *rows_per_cta, int *num_sms, int *kernel);

/* ------------------------------------------------------------------------
 * Host-buffer variant of the fused call
 *
 * For callers whose activations live in host memory: the rows are cut into
 * chunks of `chunk_rows`; chunk c is copied host->device, processed and its
 * codes and scales copied back, while the copy-in of the next chunk and the
 * copy-out of the previous one proceed on two further streams (three ring
 * slots of device workspace). A host pipe owns those internal streams and
 * events (host-side objects; no device memory) and serves one call at a time:
 * concurrent calls need one pipe each. The device workspace is the caller's.
 * ---------------------------------------------------------------------- */

typedef struct tk_swiglu_quant_host_pipe_s *tk_swiglu_quant_host_pipe_t;

/* Make a pipe for `plan` moving `chunk_rows` rows per chunk (>= 1). The
 * plan must outlive the pipe. Creates three streams and eleven events on the
 * plan's device (TK_ERR_CUDA if that fails). */
tk_status tk_swiglu_quant_host_pipe_create(tk_swiglu_quant_plan_t plan, int64_t chunk_rows,
                                           tk_swiglu_quant_host_pipe_t *pipe);

/* Release a pipe (NULL is accepted): waits for its streams, then destroys
 * them and its events. */
tk_status tk_swiglu_quant_host_pipe_destroy(tk_swiglu_quant_host_pipe_t pipe);

/* Bytes of device workspace run_host needs (three chunk slots of input,
 * weights, codes and scales, plus the clamp counter), at 256-byte alignment. */
tk_status tk_swiglu_quant_host_workspace_size(tk_swiglu_quant_host_pipe_t pipe, size_t *bytes);

/* Enqueue the fused op on host buffers, ordered after prior work on `stream`;
 * later work on `stream` is ordered after the last copy back. Returns without
 * synchronising: the host outputs are complete once `stream` has reached
 * this point (e.g. cudaStreamSynchronize).
 *   x_host, topk_weights_host    host inputs as in tk_swiglu_quant_run
 *   q_host, scales_host          host outputs as in tk_swiglu_quant_run; the
 *                                plan's scales must be row-major
 *   clamped_count_host           host int64[2], ADDED to like the device
 *                                counter (copied in, added to, copied back);
 *                                required iff count_clamped
 *   workspace                    device memory of at least
 *                                tk_swiglu_quant_host_workspace_size bytes,
 *                                256-byte aligned, not used by anything else
 *                                until `stream` passes this call
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to run asynchronously and overlap; pageable memory works but
 * the copies then serialise. The host buffers must stay valid and untouched
 * until `stream` passes this call. */
tk_status tk_swiglu_quant_run_host(tk_swiglu_quant_host_pipe_t pipe, int64_t num_tokens,
                                   const void *x_host, const float *topk_weights_host,
                                   void *q_host, void *scales_host, int64_t *clamped_count_host,
                                   void *workspace, size_t workspace_bytes, void *stream);

/* Size of the device array that tk_swiglu_quant_run_host_static uses as its
 * workspace: 32 MiB, held on every GPU that loads this library until the
 * process exits. */
#define TK_STATIC_SCRATCH_BYTES ((size_t)32 << 20)

/* The host-buffer call for callers that cannot allocate device memory.
 *
 * The pages describe no such entry point; it exists for integration. Some
 * callers are not allowed to call cudaMalloc or any allocating routine: a
 * plug-in running inside a host application whose allocator owns all device
 * memory (a serving runtime that has carved the whole HBM into its own pool),
 * code with a fixed memory budget that must not grow at run time, or a
 * process whose policy forbids new device allocations after start-up. Such a
 * caller still has its activations in host memory and wants the codes and
 * scales back in host memory.
 *
 * This call does exactly what tk_swiglu_quant_run_host does, with the same
 * arguments except the workspace: the three chunk slots and the clamp
 * counter live in one static device array of TK_STATIC_SCRATCH_BYTES inside
 * this library. The call allocates nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine); it only enqueues copies and kernels.
 *   - The pipe's workspace (tk_swiglu_quant_host_workspace_size) must fit in
 *     TK_STATIC_SCRATCH_BYTES; otherwise the call returns TK_ERR_UNSUPPORTED
 *     and enqueues nothing: make the pipe with fewer chunk_rows (1024 rows
 *     fit for hidden 2048; about 300 for hidden 7168).
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, once; make that first
 *     call before any stream capture. The address is kept per device ordinal
 *     for the rest of the process, so the call assumes the device's primary
 *     context (the runtime API's) throughout: not a driver-API context of the
 *     caller's own, and not across cudaDeviceReset.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents; nothing in it needs clearing, since each call writes
 *     every byte before reading it. Calls whose work overlaps on the GPU race
 *     on the array: issue them on one stream, or order them with events.
 * Statuses as tk_swiglu_quant_run_host. */
tk_status tk_swiglu_quant_run_host_static(tk_swiglu_quant_host_pipe_t pipe, int64_t num_tokens,
                                          const void *x_host, const float *topk_weights_host,
                                          void *q_host, void *scales_host,
                                          int64_t *clamped_count_host, void *stream);

/* Host buffers read and written in place by the kernel (no staging copies):
 * every buffer must be page-locked host memory that the device can address
 * (cudaHostAlloc / cudaMallocHost, or cudaHostRegister'ed), which this call
 * checks with cudaPointerGetAttributes (TK_ERR_INVALID_ARG otherwise). The
 * kernel loads x and stores the codes and scales across the host link
 * directly, so the link carries each byte once with no device copy in
 * between; the row-block kernel always runs (no TMA copies from host
 * memory). Arguments, layout and alignment as tk_swiglu_quant_run; the
 * clamp counters, if requested, are host memory too. Stream-ordered: the
 * outputs are complete when the stream is. */
tk_status tk_swiglu_quant_run_mapped(tk_swiglu_quant_plan_t plan, int64_t num_tokens, const void *x_host,
                                     const float *topk_weights_host, void *q_host, void *scales_host,
                                     int64_t *clamped_count_host, void *stream);

/* ------------------------------------------------------------------------
 * Standalone cast: x [T, H] (bf16 or fp32) -> codes + scales, per token, per
 * 1 x group_size block, or per channel ("TileLang + TileKernels：DeepSeek 的
 * GPU 内核开发新范式", zhichai.net/topic/177618740, section "3. Quantization",
 * format table: per-token, per-block and per-channel FP8 E4M3, FP4 E2M1,
 * UE8M0 scales), with the same scale and code rules as the fused call.
 * ---------------------------------------------------------------------- */

typedef enum tk_granularity {
    TK_GRAN_GROUPS = 0,       /* one scale per row (group_size 0) or per 1 x group_size block of a row */
    TK_GRAN_PER_CHANNEL = 1   /* one scale per column j: amax over all T rows of column j; scales [H] */
} tk_granularity;

typedef struct tk_quant_cast_desc {
    int64_t hidden;      /* H: 16 <= H <= 16384, H % 16 == 0 */
    int32_t group_size;  /* as in tk_swiglu_quant_desc; must be 0 with TK_GRAN_PER_CHANNEL */
    int32_t scale_fmt;   /* tk_scale_fmt */
    int32_t out_fmt;     /* tk_out_fmt */
    int32_t in_dtype;    /* tk_in_dtype */
    int32_t scale_layout;  /* tk_scale_layout; TK_SCALE_ROW_MAJOR with TK_GRAN_PER_CHANNEL */
    int32_t granularity;   /* tk_granularity */
} tk_quant_cast_desc;

typedef struct tk_quant_cast_plan_s *tk_quant_cast_plan_t;

tk_status tk_quant_cast_validate(const tk_quant_cast_desc *desc);
tk_status tk_quant_cast_plan(const tk_quant_cast_desc *desc, int device, tk_quant_cast_plan_t *plan);
tk_status tk_quant_cast_plan_destroy(tk_quant_cast_plan_t plan);

/* Bytes of the cast's outputs (host only): as tk_swiglu_quant_output_sizes
 * for per-token and per-block plans; per channel, q as there and scales
 * H * 4 (fp32) or H (UE8M0) bytes. */
tk_status tk_quant_cast_output_sizes(const tk_quant_cast_desc *desc, int64_t num_tokens,
                                     size_t *q_bytes, size_t *scale_bytes);

/* Enqueue a per-token or per-block cast. x [T, H] row-major, 32-byte
 * aligned; q, scales as in tk_swiglu_quant_run. num_tokens == 0 is a no-op.
 * A per-channel plan needs device workspace: it returns TK_ERR_INVALID_ARG
 * here; use tk_quant_cast_run_ws. */
tk_status tk_quant_cast_run(tk_quant_cast_plan_t plan, int64_t num_tokens, const void *x,
                            void *q, void *scales, void *stream);

/* Bytes of device workspace tk_quant_cast_run_ws needs for num_tokens rows
 * (host only): 0 for per-token and per-block plans; for a per-channel plan
 * one fp32 partial column maximum per row slab of the first pass and column,
 * at most ceil(4 * SMs / ceil(H / 512)) * H * 4 bytes (about 1.3 MB at
 * H = 7168 on 152 SMs, independent of T beyond a few thousand rows). */
tk_status tk_quant_cast_workspace_size(tk_quant_cast_plan_t plan, int64_t num_tokens, size_t *bytes);

/* Enqueue the cast with a caller-owned workspace (any granularity).
 *   x, q                as in tk_quant_cast_run
 *   scales              per token / per block: as tk_quant_cast_run; per
 *                       channel: [H] fp32 or UE8M0 bytes, 16-byte aligned
 *   workspace           device memory of at least tk_quant_cast_workspace_size
 *                       bytes for this num_tokens, 16-byte aligned, not used by
 *                       anything else until `stream` passes this call (NULL
 *                       when the size is 0). It need not be initialised and
 *                       is left holding intermediate values.
 * A per-channel column scale depends on every row, so the cast reads x
 * twice: one launch takes column maxima over row slabs into the workspace,
 * then either one launch reduces them per 512-column chunk and encodes
 * (outputs up to 96 MiB of codes) or two launches reduce them to the scales
 * and encode every row (larger outputs); stream-ordered. num_tokens == 0 is
 * a no-op (no scale is written). */
tk_status tk_quant_cast_run_ws(tk_quant_cast_plan_t plan, int64_t num_tokens, const void *x, void *q,
                               void *scales, void *workspace, size_t workspace_bytes, void *stream);

/* What a cast run of num_tokens rows enqueues (host only): *launches kernel
 * launches (0 when num_tokens == 0) and *form. Per token or per block, one
 * launch of the kernel the plan picks for that many rows: TK_CAST_ROWS (the
 * row-block kernel), TK_CAST_BLOCK_RING (the block-ring kernel, for inputs of
 * a middle size band) or TK_CAST_WARP_STREAM (the warp-stream kernel, only
 * when forced). Per channel: TK_CAST_CHANNEL_CHUNK (the amax pass, then the
 * quantize pass on the same grid, which reduces its own scales) or
 * TK_CAST_CHANNEL_SPLIT (the amax pass, the scale kernel, the row quantize
 * pass). Either output pointer may be NULL. */
typedef enum tk_cast_form {
    TK_CAST_ROWS = 0,
    TK_CAST_CHANNEL_CHUNK = 1,
    TK_CAST_CHANNEL_SPLIT = 2,
    TK_CAST_BLOCK_RING = 3,
    TK_CAST_WARP_STREAM = 4
} tk_cast_form;
tk_status tk_quant_cast_launch_info(tk_quant_cast_plan_t plan, int64_t num_tokens, int *launches, int *form);

/* ------------------------------------------------------------------------
 * Weighted top-k combine after the expert GEMMs
 *
 * "TileKernels从入门到精通" (zhichai.net/topic/177618752), chapter 3,
 * "结算中心的减法工程" and "动态寻址": the expert outputs of each token are
 * gathered through token_topk_to_pos and combined with the routing weights,
 * their quantization factors and a global scale in registers, reading every
 * expert row once and writing every output once:
 *
 *     out[t, :] = gs * sum_{k < K, pos[t,k] >= 0} w[t,k] * deq(y[pos[t,k], :])
 *
 * with deq(y) = y for bf16 rows, or decode(code) * y_scale[row, col / 128] for
 * E4M3 rows. The sum is accumulated in fp32 in k order and rounded once to
 * bf16 (round to nearest even).
 * ---------------------------------------------------------------------- */

typedef enum tk_reduce_in_fmt {
    TK_REDUCE_IN_BF16 = 0,   /* y [R, H] bf16 */
    TK_REDUCE_IN_E4M3 = 1    /* y [R, H] E4M3 codes with y_scale [R, H/128] fp32 */
} tk_reduce_in_fmt;

typedef struct tk_moe_reduce_desc {
    int64_t hidden;   /* H: 16 <= H <= 8192, H % 16 == 0 (H % 128 == 0 for E4M3 rows) */
    int32_t topk;     /* K: 1 <= K <= 64 slots per token */
    int32_t in_fmt;   /* tk_reduce_in_fmt */
} tk_moe_reduce_desc;

typedef struct tk_moe_reduce_plan_s *tk_moe_reduce_plan_t;

tk_status tk_moe_reduce_validate(const tk_moe_reduce_desc *desc);
tk_status tk_moe_reduce_plan(const tk_moe_reduce_desc *desc, int device, tk_moe_reduce_plan_t *plan);
tk_status tk_moe_reduce_plan_destroy(tk_moe_reduce_plan_t plan);

/* Enqueue the combine of num_tokens tokens.
 *   y                 [num_rows, H] expert rows, row-major: bf16 (32-byte aligned)
 *                     or E4M3 codes (16-byte aligned)
 *   y_scale           [num_rows, H/128] fp32 for E4M3 rows (4-byte aligned); else ignored
 *   token_topk_to_pos [T, K] int32, row-major: the row of y holding token t's
 *                     k-th expert output, or -1 for an empty slot. A value
 *                     outside [-1, num_rows) is not read through: the slot is
 *                     skipped and bit 1 of the device fault word is set.
 *   topk_weights      [T, K] fp32
 *   global_scale      gs
 *   out               [T, H] bf16, 16-byte aligned
 * num_tokens == 0 is a no-op. Stream-ordered and asynchronous. */
tk_status tk_moe_reduce_run(tk_moe_reduce_plan_t plan, int64_t num_tokens, const void *y,
                            const float *y_scale, int64_t num_rows, const int32_t *token_topk_to_pos,
                            const float *topk_weights, float global_scale, void *out, void *stream);

/* Which kernel and launch shape a run would use (host only). kernel: 1 for
 * the bulk-copy kernel (a producer warp per CTA gathers each token's K row
 * chunks into a shared-memory ring with TMA bulk copies), 0 for the register
 * kernel (any valid shape). The bulk kernel runs for E4M3 rows with K <= 32,
 * H % 512 == 0 and H >= 2048, and y and y_scale 16-byte aligned; bf16 rows
 * take the register kernel. Both give bit-identical outputs. grid and block
 * in CTAs and threads, smem_bytes the dynamic shared memory per CTA. */
tk_status tk_moe_reduce_launch_info(tk_moe_reduce_plan_t plan, int64_t num_tokens, const void *y,
                                    const float *y_scale, int *kernel, int *grid, int *block,
                                    int *smem_bytes);

/* ------------------------------------------------------------------------
 * SwiGLU backward, with the forward's FP8 codes optionally recomputed
 *
 * Not described on the pages, which give the forward only; this is the plain
 * derivation of the forward above. With g' = min(g, L) and u' = clamp(u, -L,
 * L) when clamping is on, s = sigmoid(g') and silu(g') = g' s:
 *
 *     dgate = dy * w * u' * s * (1 + g' * (1 - s))   (0 where g > L)
 *     dup   = dy * w * silu(g')                      (0 where |u| > L)
 *     dw    = sum over the row of dy * silu(g') * u'
 *
 * computed in fp32 and rounded to bf16 (dx) or kept in fp32 (dw, summed in a
 * fixed order, so runs repeat bit for bit). With recompute_quant the call
 * also writes the forward's codes and scales, recomputed from the same read
 * of x and bit-identical to tk_swiglu_quant_run's, for a following GEMM that
 * needs the quantized activation.
 * ---------------------------------------------------------------------- */

typedef struct tk_swiglu_backward_desc {
    int64_t hidden;            /* H: 16, 32, 64, 128, 256, or a multiple of 512 up to 8192 */
    int32_t has_topk_weights;  /* w: fp32 [T] (else weight 1) */
    int32_t use_clamp;
    float clamp_limit;         /* L > 0, as the forward */
    int32_t recompute_quant;   /* also write the forward's codes and scales */
    int32_t group_size;        /* recompute: 16 ... 512 (power of two, divides H); no per-token scale */
    int32_t scale_fmt;         /* recompute: tk_scale_fmt */
    int32_t out_fmt;           /* recompute: tk_out_fmt */
    int32_t scale_layout;      /* recompute: tk_scale_layout */
} tk_swiglu_backward_desc;

typedef struct tk_swiglu_backward_plan_s *tk_swiglu_backward_plan_t;

tk_status tk_swiglu_backward_validate(const tk_swiglu_backward_desc *desc);
tk_status tk_swiglu_backward_plan(const tk_swiglu_backward_desc *desc, int device,
                                  tk_swiglu_backward_plan_t *plan);
tk_status tk_swiglu_backward_plan_destroy(tk_swiglu_backward_plan_t plan);

/* Enqueue the backward of num_tokens rows.
 *   x             [T, 2H] bf16, the forward's input, 32-byte aligned
 *   topk_weights  [T] fp32, 4-byte aligned (required iff has_topk_weights)
 *   dy            [T, H] bf16, the gradient of the forward's output y, 32-byte aligned
 *   dx            [T, 2H] bf16: dgate in columns [0, H), dup in [H, 2H); 16-byte aligned
 *   dw            [T] fp32 or NULL; 4-byte aligned
 *   q, scales     recompute_quant only: as tk_swiglu_quant_run's outputs (else ignored)
 * num_tokens == 0 is a no-op. Stream-ordered and asynchronous; inputs and
 * outputs must not overlap. */
tk_status tk_swiglu_backward_run(tk_swiglu_backward_plan_t plan, int64_t num_tokens, const void *x,
                                 const float *topk_weights, const void *dy, void *dx, float *dw, void *q,
                                 void *scales, void *stream);

/* ------------------------------------------------------------------------
 * Diagnostics
 * ---------------------------------------------------------------------- */

/* Read, and if `clear` is non-zero reset, the fault word of `device`. Bit 0
 * is set by a kernel that gave up waiting for one of its own asynchronous
 * copies (a wait over a second long, which no correct run reaches) and
 * returned early, leaving that launch's outputs incomplete. Bit 1 is set by
 * the top-k combine when a position outside [-1, num_rows) was skipped. The word is
 * shared by every call on the device; the read is ordered after all work
 * already submitted to the device (it synchronises with it). */
tk_status tk_fault_word(int device, uint32_t *value, int clear);

/* Exercise the failure path of the kernels' bounded waits (not part of the
 * pages' method): one thread of one CTA waits on a shared-memory mbarrier that
 * nothing arrives at, gives up after `tries` (1 ... 2^22) tries of
 * mbarrier.try_wait exactly as the library's kernels do, sets bit 0 of the
 * fault word and returns, with nothing left in flight. Stream-ordered on
 * `stream`; `device` must be the current device (TK_ERR_DEVICE otherwise).
 * The library's kernels give up after 2^19 tries (about 1.8 s on GB300, where
 * an unanswered try takes 3.5 us). */
tk_status tk_diag_unanswered_wait(int device, uint32_t tries, void *stream);

/* Static name of a status ("TK_OK", ...). Never NULL. */
const char *tk_status_string(tk_status status);

/* Message of the last non-OK status returned on the calling thread ("" if
 * none). Valid until the next call into this library on the same thread. */
const char *tk_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* TK_SWIGLU_QUANT_H */
