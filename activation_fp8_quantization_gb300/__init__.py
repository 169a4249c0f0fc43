"""Fused SwiGLU + MoE top-k weight + FP8/FP4 activation cast for GB300 (sm_103a).

The computation runs in ``libtk_swiglu_quant.so`` (hand-written CUDA behind the
C ABI of ``include/tk_swiglu_quant.h``). This module only turns torch CUDA
tensors into device pointers and the current CUDA stream; PyTorch supplies
device memory and streams, nothing else.

    >>> op = SwigluQuant(hidden=2048, group_size=128, scale_fmt="fp32", out_fmt="e4m3")
    >>> q, scales = op(x, topk_weights)        # x: [T, 4096] bf16 on cuda

``q`` is uint8 ([T, H] E4M3 codes, or [T, H/2] packed E2M1 with value 2k in
the low nibble); ``scales`` is float32 or uint8 (UE8M0 exponent bytes),
[T, H / group_size] (one column when group_size == 0).
"""
from __future__ import annotations

import threading

from . import _abi
from ._abi import (GRANULARITIES, IN_DTYPES, OUT_FMTS, REDUCE_IN_FMTS, SCALE_FMTS, SCALE_LAYOUTS, MoeReduceDesc,
                   QuantCastDesc, SwigluBackwardDesc, SwigluQuantDesc, tk_swiglu_backward_plan,
                   tk_swiglu_backward_plan_destroy, tk_swiglu_backward_run, tk_swiglu_backward_validate, tk_moe_reduce_plan, tk_moe_reduce_plan_destroy,
                   tk_moe_reduce_launch_info, tk_moe_reduce_run, tk_moe_reduce_validate,
                   TkError, tk_diag_unanswered_wait, tk_fault_word, tk_last_error_message, tk_quant_cast_output_sizes,
                   tk_quant_cast_plan, tk_quant_cast_plan_destroy,
                   tk_quant_cast_launch_info, tk_quant_cast_run, tk_quant_cast_run_ws, tk_quant_cast_validate,
                   tk_quant_cast_workspace_size, tk_status_string,
                   tk_swiglu_quant_host_pipe_create, tk_swiglu_quant_host_pipe_destroy,
                   tk_swiglu_quant_host_workspace_size, tk_swiglu_quant_launch_info,
                   tk_swiglu_quant_output_sizes, tk_swiglu_quant_plan, tk_swiglu_quant_plan_destroy,
                   tk_swiglu_quant_run, tk_swiglu_quant_run_host, tk_swiglu_quant_run_host_static,
                   tk_swiglu_quant_run_mapped, tk_swiglu_quant_run_transposed, tk_swiglu_quant_transposed_size,
                   tk_swiglu_quant_validate)

__all__ = [
    "SwigluQuant", "HostPipe", "QuantCast", "MoeReduce", "SwigluBackward", "swiglu_quant", "quant_cast",
    "TkError", "SwigluBackwardDesc", "tk_swiglu_backward_validate", "tk_swiglu_backward_plan",
    "tk_swiglu_backward_plan_destroy", "tk_swiglu_backward_run",
    "MoeReduceDesc", "tk_moe_reduce_validate", "tk_moe_reduce_plan", "tk_moe_reduce_plan_destroy",
    "tk_moe_reduce_run", "tk_moe_reduce_launch_info",
    "tk_swiglu_quant_host_pipe_create", "tk_swiglu_quant_host_pipe_destroy",
    "tk_swiglu_quant_host_workspace_size", "tk_swiglu_quant_run_host",
    "tk_swiglu_quant_run_host_static",
    "SwigluQuantDesc", "QuantCastDesc", "tk_swiglu_quant_validate", "tk_swiglu_quant_plan",
    "tk_swiglu_quant_plan_destroy", "tk_swiglu_quant_output_sizes", "tk_swiglu_quant_run",
    "tk_swiglu_quant_launch_info", "tk_swiglu_quant_run_transposed", "tk_swiglu_quant_transposed_size",
    "tk_swiglu_quant_run_mapped",
    "tk_quant_cast_validate", "tk_quant_cast_plan",
    "tk_quant_cast_plan_destroy", "tk_quant_cast_output_sizes", "tk_quant_cast_run", "tk_quant_cast_run_ws",
    "tk_quant_cast_workspace_size", "tk_quant_cast_launch_info", "tk_status_string",
    "tk_last_error_message", "tk_fault_word", "tk_diag_unanswered_wait",
]


def _torch():
    import torch
    return torch


def _out_shapes(T: int, hidden: int, group_size: int, scale_fmt: str, out_fmt: str,
                scale_layout: str = "row"):
    """(codes shape, scales shape, scales dtype) for T rows. Column-major
    scales are [G, Tp] with Tp padded to 16 bytes of scale elements; packed
    UE8M0 scales are int32 words [G/4, Tp4], Tp4 = T padded to 4."""
    torch = _torch()
    G = 1 if group_size == 0 else hidden // group_size
    q_shape = (T, hidden if out_fmt == "e4m3" else hidden // 2)
    s_dtype = torch.float32 if scale_fmt == "fp32" else torch.uint8
    if scale_layout == "row":
        return q_shape, (T, G), s_dtype
    if scale_layout == "col":
        per16 = 4 if scale_fmt == "fp32" else 16
        return q_shape, (G, -(-T // per16) * per16), s_dtype
    return q_shape, (G // 4, -(-T // 4) * 4), torch.int32


def _check_cuda(t, name: str, dtype, shape=None):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))


class SwigluQuant:
    """A plan for the fused op on one device (see tk_swiglu_quant_plan)."""

    def __init__(self, hidden: int, group_size: int = 128, scale_fmt: str = "fp32",
                 out_fmt: str = "e4m3", topk_weights: bool = True,
                 clamp_limit: float | None = None, count_clamped: bool = False,
                 device: int | None = None, scale_layout: str = "row"):
        torch = _torch()
        self.hidden, self.group_size = int(hidden), int(group_size)
        self.scale_fmt, self.out_fmt, self.scale_layout = scale_fmt, out_fmt, scale_layout
        self.has_w = bool(topk_weights)
        self.clamp_limit = clamp_limit
        self.count_clamped = bool(count_clamped)
        self.desc = SwigluQuantDesc(self.hidden, self.group_size, SCALE_FMTS[scale_fmt],
                                    OUT_FMTS[out_fmt], int(self.has_w), int(clamp_limit is not None),
                                    float(clamp_limit or 0.0), int(self.count_clamped),
                                    SCALE_LAYOUTS[scale_layout])
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.plan = tk_swiglu_quant_plan(self.desc, self.device)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan:
            try:
                tk_swiglu_quant_plan_destroy(plan)
            except Exception:
                pass
            self.plan = None

    def output_shapes(self, T: int):
        return _out_shapes(T, self.hidden, self.group_size, self.scale_fmt, self.out_fmt,
                           self.scale_layout)

    def launch_info(self, T: int) -> dict:
        return tk_swiglu_quant_launch_info(self.plan, T)

    def __call__(self, x, topk_weights=None, *, q=None, scales=None, clamped_count=None,
                 stream=None):
        """Enqueue on ``stream`` (default: torch's current stream); returns (q, scales)."""
        torch = _torch()
        T = x.shape[0]
        _check_cuda(x, "x", torch.bfloat16, (T, 2 * self.hidden))
        if self.has_w:
            if topk_weights is None:
                raise ValueError("this op was planned with top-k weights")
            _check_cuda(topk_weights, "topk_weights", torch.float32, (T,))
        else:
            topk_weights = None
        if self.count_clamped:
            if clamped_count is None:
                raise ValueError("this op was planned with count_clamped; pass an int64[2] tensor")
            _check_cuda(clamped_count, "clamped_count", torch.int64, (2,))
        else:
            clamped_count = None
        q_shape, s_shape, s_dtype = self.output_shapes(T)
        if q is None:
            q = torch.empty(q_shape, dtype=torch.uint8, device=x.device)
        _check_cuda(q, "q", torch.uint8, q_shape)
        if scales is None:
            scales = torch.empty(s_shape, dtype=s_dtype, device=x.device)
        _check_cuda(scales, "scales", s_dtype, s_shape)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        with torch.cuda.device(x.device):
            tk_swiglu_quant_run(self.plan, T, x, topk_weights, q, scales, clamped_count,
                                stream.cuda_stream)
        return q, scales

    def mapped(self, x_host, topk_weights_host=None, *, q=None, scales=None, clamped_count=None,
               stream=None):
        """The op on page-locked host tensors, read and written in place by the
        kernel across the host link (tk_swiglu_quant_run_mapped). Outputs are
        page-locked host tensors; they are complete once ``stream`` is."""
        torch = _torch()
        T = x_host.shape[0]
        q_shape, s_shape, s_dtype = self.output_shapes(T)
        if q is None:
            q = torch.empty(q_shape, dtype=torch.uint8).pin_memory()
        if scales is None:
            scales = torch.empty(s_shape, dtype=s_dtype).pin_memory()
        for t, name, shape in ((x_host, "x", (T, 2 * self.hidden)), (q, "q", q_shape), (scales, "scales", s_shape)):
            if t.is_cuda or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
                raise ValueError("%s must be a contiguous host tensor of shape %s" % (name, shape))
        if stream is None:
            stream = torch.cuda.current_stream()
        tk_swiglu_quant_run_mapped(self.plan, T, x_host, topk_weights_host if self.has_w else None, q, scales,
                                   clamped_count if self.count_clamped else None, stream.cuda_stream)
        return q, scales

    def transposed(self, x, topk_weights=None, *, qt=None, scales=None, clamped_count=None,
                   stream=None):
        """The same op with the codes stored transposed (tk_swiglu_quant_run_transposed):
        returns (qt [H, ld] uint8 with ld = T rounded up to 32, scales)."""
        torch = _torch()
        T = x.shape[0]
        _check_cuda(x, "x", torch.bfloat16, (T, 2 * self.hidden))
        if self.has_w:
            if topk_weights is None:
                raise ValueError("this op was planned with top-k weights")
            _check_cuda(topk_weights, "topk_weights", torch.float32, (T,))
        else:
            topk_weights = None
        if self.count_clamped:
            if clamped_count is None:
                raise ValueError("this op was planned with count_clamped; pass an int64[2] tensor")
            _check_cuda(clamped_count, "clamped_count", torch.int64, (2,))
        else:
            clamped_count = None
        _, ld = tk_swiglu_quant_transposed_size(self.plan, T)
        _, s_shape, s_dtype = self.output_shapes(T)
        if qt is None:
            qt = torch.empty((self.hidden, ld), dtype=torch.uint8, device=x.device)
        _check_cuda(qt, "qt", torch.uint8, (self.hidden, ld))
        if scales is None:
            scales = torch.empty(s_shape, dtype=s_dtype, device=x.device)
        _check_cuda(scales, "scales", s_dtype, s_shape)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        with torch.cuda.device(x.device):
            tk_swiglu_quant_run_transposed(self.plan, T, x, topk_weights, qt, scales, clamped_count,
                                           stream.cuda_stream)
        return qt, scales


class HostPipe:
    """Host-buffer form of a SwigluQuant (tk_swiglu_quant_run_host): inputs
    and outputs are CPU tensors (pinned for overlap); a device workspace of
    three chunk slots is allocated once, here, through torch."""

    def __init__(self, op: SwigluQuant, chunk_rows: int = 1024):
        torch = _torch()
        self.op = op
        self.chunk_rows = int(chunk_rows)
        self.pipe = tk_swiglu_quant_host_pipe_create(op.plan, self.chunk_rows)
        self.ws_bytes = tk_swiglu_quant_host_workspace_size(self.pipe)
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda:%d" % op.device)

    def __del__(self):
        pipe = getattr(self, "pipe", None)
        if pipe:
            try:
                tk_swiglu_quant_host_pipe_destroy(pipe)
            except Exception:
                pass
            self.pipe = None

    def __call__(self, x, topk_weights=None, *, q=None, scales=None, clamped_count=None,
                 stream=None):
        """Enqueue; returns (q, scales) host tensors, complete once `stream`
        (default: torch's current stream) has passed this call."""
        torch = _torch()
        op = self.op
        T = x.shape[0]
        for t, name in ((x, "x"), (topk_weights, "topk_weights"), (q, "q"), (scales, "scales"),
                        (clamped_count, "clamped_count")):
            if t is not None and (t.is_cuda or not t.is_contiguous()):
                raise ValueError("%s must be a contiguous CPU tensor" % name)
        if x.dtype != torch.bfloat16 or tuple(x.shape) != (T, 2 * op.hidden):
            raise ValueError("x must be bf16 [T, %d]" % (2 * op.hidden))
        q_shape, s_shape, s_dtype = op.output_shapes(T)
        if q is None:
            q = torch.empty(q_shape, dtype=torch.uint8, pin_memory=True)
        if scales is None:
            scales = torch.empty(s_shape, dtype=s_dtype, pin_memory=True)
        if tuple(q.shape) != q_shape or tuple(scales.shape) != s_shape or scales.dtype != s_dtype:
            raise ValueError("q / scales have the wrong shape or dtype")
        if stream is None:
            stream = torch.cuda.current_stream(op.device)
        with torch.cuda.device(op.device):
            tk_swiglu_quant_run_host(self.pipe, T, x, topk_weights if op.has_w else None, q, scales,
                                     clamped_count if op.count_clamped else None, self.workspace,
                                     self.ws_bytes, stream.cuda_stream)
        return q, scales


class QuantCast:
    """A plan for the standalone cast (tk_quant_cast_plan): per token
    (group_size 0), per 1 x group_size block, or per channel
    (granularity="channel": one scale per column, scales [H])."""

    def __init__(self, hidden: int, group_size: int = 128, scale_fmt: str = "fp32",
                 out_fmt: str = "e4m3", in_dtype: str = "bf16", device: int | None = None,
                 scale_layout: str = "row", granularity: str = "groups"):
        torch = _torch()
        self.hidden, self.group_size = int(hidden), int(group_size)
        self.scale_fmt, self.out_fmt, self.in_dtype = scale_fmt, out_fmt, in_dtype
        self.scale_layout, self.granularity = scale_layout, granularity
        self.desc = QuantCastDesc(self.hidden, self.group_size, SCALE_FMTS[scale_fmt],
                                  OUT_FMTS[out_fmt], IN_DTYPES[in_dtype], SCALE_LAYOUTS[scale_layout],
                                  GRANULARITIES[granularity])
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.plan = tk_quant_cast_plan(self.desc, self.device)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan:
            try:
                tk_quant_cast_plan_destroy(plan)
            except Exception:
                pass
            self.plan = None

    def output_shapes(self, T: int):
        if self.granularity == "channel":
            torch = _torch()
            q_shape = (T, self.hidden if self.out_fmt == "e4m3" else self.hidden // 2)
            return q_shape, (self.hidden,), torch.float32 if self.scale_fmt == "fp32" else torch.uint8
        return _out_shapes(T, self.hidden, self.group_size, self.scale_fmt, self.out_fmt,
                           self.scale_layout)

    def workspace_bytes(self, T: int) -> int:
        return tk_quant_cast_workspace_size(self.plan, T)

    def launch_info(self, T: int) -> dict:
        """Launches and kernels a run of T rows enqueues (tk_quant_cast_launch_info)."""
        return tk_quant_cast_launch_info(self.plan, T)

    def __call__(self, x, *, q=None, scales=None, workspace=None, stream=None):
        torch = _torch()
        T = x.shape[0]
        dt = torch.bfloat16 if self.in_dtype == "bf16" else torch.float32
        _check_cuda(x, "x", dt, (T, self.hidden))
        q_shape, s_shape, s_dtype = self.output_shapes(T)
        if q is None:
            q = torch.empty(q_shape, dtype=torch.uint8, device=x.device)
        _check_cuda(q, "q", torch.uint8, q_shape)
        if scales is None:
            scales = torch.empty(s_shape, dtype=s_dtype, device=x.device)
        _check_cuda(scales, "scales", s_dtype, s_shape)
        nb = self.workspace_bytes(T)
        if nb and workspace is None:
            workspace = torch.empty(nb, dtype=torch.uint8, device=x.device)
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        with torch.cuda.device(x.device):
            tk_quant_cast_run_ws(self.plan, T, x, q, scales, workspace if nb else None,
                                 workspace.numel() if nb else 0, stream.cuda_stream)
        return q, scales


class SwigluBackward:
    """A plan for the SwiGLU backward (tk_swiglu_backward_plan). With
    ``recompute`` = dict(group_size=..., scale_fmt=..., out_fmt=..., scale_layout=...)
    it also writes the forward's codes and scales."""

    def __init__(self, hidden: int, topk_weights: bool = True, clamp_limit: float | None = None,
                 recompute: dict | None = None, device: int | None = None):
        torch = _torch()
        self.hidden = int(hidden)
        self.has_w = bool(topk_weights)
        self.clamp_limit = clamp_limit
        self.recompute = dict(recompute) if recompute else None
        r = self.recompute or {}
        self.group_size = int(r.get("group_size", 128)) if r else 0
        self.scale_fmt = r.get("scale_fmt", "fp32")
        self.out_fmt = r.get("out_fmt", "e4m3")
        self.scale_layout = r.get("scale_layout", "row")
        self.desc = SwigluBackwardDesc(self.hidden, int(self.has_w), int(clamp_limit is not None),
                                       float(clamp_limit or 0.0), int(bool(r)), self.group_size,
                                       SCALE_FMTS[self.scale_fmt], OUT_FMTS[self.out_fmt],
                                       SCALE_LAYOUTS[self.scale_layout])
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.plan = tk_swiglu_backward_plan(self.desc, self.device)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan:
            try:
                tk_swiglu_backward_plan_destroy(plan)
            except Exception:
                pass
            self.plan = None

    def __call__(self, x, dy, topk_weights=None, *, want_dw: bool = True, dx=None, dw=None, q=None,
                 scales=None, stream=None):
        """Returns (dx [T, 2H] bf16, dw [T] fp32 or None, q, scales) (q, scales
        None unless the plan recomputes the codes)."""
        torch = _torch()
        T = x.shape[0]
        _check_cuda(x, "x", torch.bfloat16, (T, 2 * self.hidden))
        _check_cuda(dy, "dy", torch.bfloat16, (T, self.hidden))
        if self.has_w:
            if topk_weights is None:
                raise ValueError("this op was planned with top-k weights")
            _check_cuda(topk_weights, "topk_weights", torch.float32, (T,))
        else:
            topk_weights = None
        if dx is None:
            dx = torch.empty((T, 2 * self.hidden), dtype=torch.bfloat16, device=x.device)
        _check_cuda(dx, "dx", torch.bfloat16, (T, 2 * self.hidden))
        if want_dw and dw is None:
            dw = torch.empty((T,), dtype=torch.float32, device=x.device)
        if dw is not None:
            _check_cuda(dw, "dw", torch.float32, (T,))
        if self.recompute:
            q_shape, s_shape, s_dtype = _out_shapes(T, self.hidden, self.group_size, self.scale_fmt,
                                                    self.out_fmt, self.scale_layout)
            if q is None:
                q = torch.empty(q_shape, dtype=torch.uint8, device=x.device)
            _check_cuda(q, "q", torch.uint8, q_shape)
            if scales is None:
                scales = torch.empty(s_shape, dtype=s_dtype, device=x.device)
            _check_cuda(scales, "scales", s_dtype, s_shape)
        else:
            q = scales = None
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        with torch.cuda.device(x.device):
            tk_swiglu_backward_run(self.plan, T, x, topk_weights, dy, dx, dw, q, scales, stream.cuda_stream)
        return dx, dw, q, scales


class MoeReduce:
    """A plan for the weighted top-k combine (tk_moe_reduce_plan)."""

    def __init__(self, hidden: int, topk: int, in_fmt: str = "bf16", device: int | None = None):
        torch = _torch()
        self.hidden, self.topk, self.in_fmt = int(hidden), int(topk), in_fmt
        self.desc = MoeReduceDesc(self.hidden, self.topk, REDUCE_IN_FMTS[in_fmt])
        self.device = torch.cuda.current_device() if device is None else int(device)
        self.plan = tk_moe_reduce_plan(self.desc, self.device)

    def __del__(self):
        plan = getattr(self, "plan", None)
        if plan:
            try:
                tk_moe_reduce_plan_destroy(plan)
            except Exception:
                pass
            self.plan = None

    def launch_info(self, num_tokens: int, y=None, y_scale=None) -> dict:
        """Kernel ("bulk" or "regs") and launch shape a run would use."""
        return tk_moe_reduce_launch_info(self.plan, num_tokens, y, y_scale)

    def __call__(self, y, token_topk_to_pos, topk_weights, global_scale: float = 1.0, *,
                 y_scale=None, out=None, stream=None):
        """y: [R, H] bf16 (or uint8 E4M3 codes with y_scale [R, H/128] fp32);
        token_topk_to_pos: [T, K] int32 (-1: empty); topk_weights: [T, K] fp32.
        Returns out [T, H] bf16."""
        torch = _torch()
        T = token_topk_to_pos.shape[0]
        R = y.shape[0]
        ydt = torch.bfloat16 if self.in_fmt == "bf16" else torch.uint8
        _check_cuda(y, "y", ydt, (R, self.hidden))
        if self.in_fmt == "e4m3":
            _check_cuda(y_scale, "y_scale", torch.float32, (R, self.hidden // 128))
        else:
            y_scale = None
        _check_cuda(token_topk_to_pos, "token_topk_to_pos", torch.int32, (T, self.topk))
        _check_cuda(topk_weights, "topk_weights", torch.float32, (T, self.topk))
        if out is None:
            out = torch.empty((T, self.hidden), dtype=torch.bfloat16, device=y.device)
        _check_cuda(out, "out", torch.bfloat16, (T, self.hidden))
        if stream is None:
            stream = torch.cuda.current_stream(y.device)
        with torch.cuda.device(y.device):
            tk_moe_reduce_run(self.plan, T, y, y_scale, R, token_topk_to_pos, topk_weights,
                              float(global_scale), out, stream.cuda_stream)
        return out


_plans: dict = {}
_plans_lock = threading.Lock()


def _cached(kind, key, make):
    with _plans_lock:
        p = _plans.get((kind, key))
        if p is None:
            p = _plans[(kind, key)] = make()
        return p


def swiglu_quant(x, topk_weights=None, *, group_size: int = 128, scale_fmt: str = "fp32",
                 out_fmt: str = "e4m3", clamp_limit: float | None = None, clamped_count=None):
    """Functional form: plans are cached per (shape, formats, device)."""
    hidden = x.shape[1] // 2
    key = (hidden, group_size, scale_fmt, out_fmt, topk_weights is not None, clamp_limit,
           clamped_count is not None, x.device.index)
    op = _cached("swiglu", key, lambda: SwigluQuant(
        hidden, group_size, scale_fmt, out_fmt, topk_weights is not None, clamp_limit,
        clamped_count is not None, x.device.index))
    return op(x, topk_weights, clamped_count=clamped_count)


def quant_cast(x, *, group_size: int = 128, scale_fmt: str = "fp32", out_fmt: str = "e4m3",
               granularity: str = "groups"):
    """Functional form of the standalone cast (bf16 or fp32 input); with
    granularity="channel" one scale per column (group_size is then 0)."""
    torch = _torch()
    in_dtype = "bf16" if x.dtype == torch.bfloat16 else "fp32"
    if granularity == "channel":
        group_size = 0
    key = (x.shape[1], group_size, scale_fmt, out_fmt, in_dtype, granularity, x.device.index)
    op = _cached("cast", key, lambda: QuantCast(x.shape[1], group_size, scale_fmt, out_fmt,
                                                in_dtype, x.device.index, granularity=granularity))
    return op(x)
