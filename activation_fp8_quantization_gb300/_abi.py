"""ctypes binding of include/tk_swiglu_quant.h: same names, argument
marshalling only. Every step of the computation runs in the CUDA library;
there is no CPU fallback. If the library is missing, loading raises."""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtk_swiglu_quant.so")

TK_OK = 0
STATUS_NAMES = {0: "TK_OK", 1: "TK_ERR_INVALID_ARG", 2: "TK_ERR_UNSUPPORTED",
                3: "TK_ERR_MISALIGNED", 4: "TK_ERR_CUDA", 5: "TK_ERR_DEVICE"}
SCALE_FMTS = {"fp32": 0, "ue8m0": 1}
OUT_FMTS = {"e4m3": 0, "e2m1": 1}
IN_DTYPES = {"bf16": 0, "fp32": 1}
SCALE_LAYOUTS = {"row": 0, "col": 1, "col_packed": 2}


class TkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(status, status), message))
        self.status = status


class SwigluQuantDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("group_size", ctypes.c_int32),
                ("scale_fmt", ctypes.c_int32), ("out_fmt", ctypes.c_int32),
                ("has_topk_weights", ctypes.c_int32), ("use_clamp", ctypes.c_int32),
                ("clamp_limit", ctypes.c_float), ("count_clamped", ctypes.c_int32),
                ("scale_layout", ctypes.c_int32)]


class QuantCastDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("group_size", ctypes.c_int32),
                ("scale_fmt", ctypes.c_int32), ("out_fmt", ctypes.c_int32),
                ("in_dtype", ctypes.c_int32), ("scale_layout", ctypes.c_int32),
                ("granularity", ctypes.c_int32)]


GRANULARITIES = {"groups": 0, "channel": 1}


class SwigluBackwardDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("has_topk_weights", ctypes.c_int32),
                ("use_clamp", ctypes.c_int32), ("clamp_limit", ctypes.c_float),
                ("recompute_quant", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("scale_fmt", ctypes.c_int32), ("out_fmt", ctypes.c_int32), ("scale_layout", ctypes.c_int32)]


class MoeReduceDesc(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int64), ("topk", ctypes.c_int32), ("in_fmt", ctypes.c_int32)]


REDUCE_IN_FMTS = {"bf16": 0, "e4m3": 1}

_VP = ctypes.c_void_p
_P64 = ctypes.POINTER(ctypes.c_int64)
_PINT = ctypes.POINTER(ctypes.c_int)
_PSZ = ctypes.POINTER(ctypes.c_size_t)

# name -> (restype, argtypes); mirrors the header one to one.
SIGNATURES = {
    "tk_swiglu_quant_validate": (ctypes.c_int, [ctypes.POINTER(SwigluQuantDesc)]),
    "tk_swiglu_quant_plan": (ctypes.c_int, [ctypes.POINTER(SwigluQuantDesc), ctypes.c_int,
                                            ctypes.POINTER(_VP)]),
    "tk_swiglu_quant_plan_destroy": (ctypes.c_int, [_VP]),
    "tk_swiglu_quant_output_sizes": (ctypes.c_int, [ctypes.POINTER(SwigluQuantDesc), ctypes.c_int64,
                                                    _PSZ, _PSZ]),
    "tk_swiglu_quant_run": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP]),
    "tk_swiglu_quant_launch_info": (ctypes.c_int, [_VP, ctypes.c_int64, _PINT, _PINT, _PINT, _PINT, _PINT]),
    "tk_swiglu_quant_run_mapped": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP]),
    "tk_swiglu_quant_transposed_size": (ctypes.c_int, [_VP, ctypes.c_int64, _PSZ,
                                                       ctypes.POINTER(ctypes.c_int64)]),
    "tk_swiglu_quant_run_transposed": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP]),
    "tk_swiglu_quant_host_pipe_create": (ctypes.c_int, [_VP, ctypes.c_int64, ctypes.POINTER(_VP)]),
    "tk_swiglu_quant_host_pipe_destroy": (ctypes.c_int, [_VP]),
    "tk_swiglu_quant_host_workspace_size": (ctypes.c_int, [_VP, _PSZ]),
    "tk_swiglu_quant_run_host": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP,
                                                ctypes.c_size_t, _VP]),
    "tk_swiglu_quant_run_host_static": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP,
                                                       _VP]),
    "tk_quant_cast_validate": (ctypes.c_int, [ctypes.POINTER(QuantCastDesc)]),
    "tk_quant_cast_plan": (ctypes.c_int, [ctypes.POINTER(QuantCastDesc), ctypes.c_int,
                                          ctypes.POINTER(_VP)]),
    "tk_quant_cast_plan_destroy": (ctypes.c_int, [_VP]),
    "tk_quant_cast_output_sizes": (ctypes.c_int, [ctypes.POINTER(QuantCastDesc), ctypes.c_int64,
                                                  _PSZ, _PSZ]),
    "tk_quant_cast_run": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP]),
    "tk_quant_cast_workspace_size": (ctypes.c_int, [_VP, ctypes.c_int64, _PSZ]),
    "tk_quant_cast_run_ws": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "tk_quant_cast_launch_info": (ctypes.c_int, [_VP, ctypes.c_int64, _PINT, _PINT]),
    "tk_moe_reduce_validate": (ctypes.c_int, [ctypes.POINTER(MoeReduceDesc)]),
    "tk_moe_reduce_plan": (ctypes.c_int, [ctypes.POINTER(MoeReduceDesc), ctypes.c_int, ctypes.POINTER(_VP)]),
    "tk_moe_reduce_plan_destroy": (ctypes.c_int, [_VP]),
    "tk_moe_reduce_run": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, ctypes.c_int64, _VP, _VP,
                                         ctypes.c_float, _VP, _VP]),
    "tk_moe_reduce_launch_info": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _PINT, _PINT, _PINT,
                                                 _PINT]),
    "tk_swiglu_backward_validate": (ctypes.c_int, [ctypes.POINTER(SwigluBackwardDesc)]),
    "tk_swiglu_backward_plan": (ctypes.c_int, [ctypes.POINTER(SwigluBackwardDesc), ctypes.c_int,
                                               ctypes.POINTER(_VP)]),
    "tk_swiglu_backward_plan_destroy": (ctypes.c_int, [_VP]),
    "tk_swiglu_backward_run": (ctypes.c_int, [_VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "tk_fault_word": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "tk_diag_unanswered_wait": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint32, _VP]),
    "tk_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tk_last_error_message": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library. Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "CUDA library %s is missing: build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
        return _lib


def check(status: int) -> None:
    if status != TK_OK:
        msg = lib().tk_last_error_message().decode(errors="replace")
        raise TkError(status, msg)


def _ptr(t) -> int | None:
    """Device address of a tensor (None stays NULL; ints pass through)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


# --------------------------------------------------------- same-name calls

def tk_swiglu_quant_validate(desc: SwigluQuantDesc) -> int:
    return lib().tk_swiglu_quant_validate(ctypes.byref(desc))


def tk_swiglu_quant_plan(desc: SwigluQuantDesc, device: int) -> int:
    h = _VP()
    check(lib().tk_swiglu_quant_plan(ctypes.byref(desc), device, ctypes.byref(h)))
    return h.value


def tk_swiglu_quant_plan_destroy(plan: int) -> None:
    check(lib().tk_swiglu_quant_plan_destroy(plan))


def tk_swiglu_quant_output_sizes(desc: SwigluQuantDesc, num_tokens: int) -> tuple[int, int]:
    qb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().tk_swiglu_quant_output_sizes(ctypes.byref(desc), num_tokens, ctypes.byref(qb),
                                             ctypes.byref(sb)))
    return qb.value, sb.value


def tk_swiglu_quant_run(plan: int, num_tokens: int, x, topk_weights, q, scales, clamped_count,
                        stream: int | None) -> None:
    check(lib().tk_swiglu_quant_run(plan, num_tokens, _ptr(x), _ptr(topk_weights), _ptr(q),
                                    _ptr(scales), _ptr(clamped_count), stream))


def tk_swiglu_quant_run_mapped(plan: int, num_tokens: int, x_host, topk_weights_host, q_host, scales_host,
                               clamped_count_host, stream: int | None) -> None:
    check(lib().tk_swiglu_quant_run_mapped(plan, num_tokens, _ptr(x_host), _ptr(topk_weights_host),
                                           _ptr(q_host), _ptr(scales_host), _ptr(clamped_count_host), stream))


def tk_swiglu_quant_transposed_size(plan: int, num_tokens: int) -> tuple[int, int]:
    """(bytes of qt, ld) for num_tokens rows."""
    n = ctypes.c_size_t()
    ld = ctypes.c_int64()
    check(lib().tk_swiglu_quant_transposed_size(plan, num_tokens, ctypes.byref(n), ctypes.byref(ld)))
    return n.value, ld.value


def tk_swiglu_quant_run_transposed(plan: int, num_tokens: int, x, topk_weights, qt, scales, clamped_count,
                                   stream: int | None) -> None:
    check(lib().tk_swiglu_quant_run_transposed(plan, num_tokens, _ptr(x), _ptr(topk_weights), _ptr(qt),
                                               _ptr(scales), _ptr(clamped_count), stream))


KERNEL_NAMES = {0: "row_quant_kernel", 1: "warp_stream_kernel", 2: "block_stream_kernel"}


def tk_swiglu_quant_launch_info(plan: int, num_tokens: int) -> dict:
    g, b, r, n, k = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    check(lib().tk_swiglu_quant_launch_info(plan, num_tokens, ctypes.byref(g), ctypes.byref(b),
                                            ctypes.byref(r), ctypes.byref(n), ctypes.byref(k)))
    return {"grid": g.value, "block": b.value, "rows_per_cta": r.value, "num_sms": n.value,
            "kernel": KERNEL_NAMES[k.value]}


def tk_swiglu_quant_host_pipe_create(plan: int, chunk_rows: int) -> int:
    h = _VP()
    check(lib().tk_swiglu_quant_host_pipe_create(plan, chunk_rows, ctypes.byref(h)))
    return h.value


def tk_swiglu_quant_host_pipe_destroy(pipe: int) -> None:
    check(lib().tk_swiglu_quant_host_pipe_destroy(pipe))


def tk_swiglu_quant_host_workspace_size(pipe: int) -> int:
    b = ctypes.c_size_t()
    check(lib().tk_swiglu_quant_host_workspace_size(pipe, ctypes.byref(b)))
    return b.value


def tk_swiglu_quant_run_host(pipe: int, num_tokens: int, x_host, topk_weights_host, q_host,
                             scales_host, clamped_count_host, workspace, workspace_bytes: int,
                             stream: int | None) -> None:
    check(lib().tk_swiglu_quant_run_host(pipe, num_tokens, _ptr(x_host), _ptr(topk_weights_host),
                                         _ptr(q_host), _ptr(scales_host), _ptr(clamped_count_host),
                                         _ptr(workspace), workspace_bytes, stream))


def tk_swiglu_quant_run_host_static(pipe: int, num_tokens: int, x_host, topk_weights_host, q_host,
                                    scales_host, clamped_count_host, stream: int | None) -> None:
    check(lib().tk_swiglu_quant_run_host_static(pipe, num_tokens, _ptr(x_host), _ptr(topk_weights_host),
                                                _ptr(q_host), _ptr(scales_host),
                                                _ptr(clamped_count_host), stream))


# TK_STATIC_SCRATCH_BYTES of the header
STATIC_SCRATCH_BYTES = 32 << 20


def tk_quant_cast_validate(desc: QuantCastDesc) -> int:
    return lib().tk_quant_cast_validate(ctypes.byref(desc))


def tk_quant_cast_plan(desc: QuantCastDesc, device: int) -> int:
    h = _VP()
    check(lib().tk_quant_cast_plan(ctypes.byref(desc), device, ctypes.byref(h)))
    return h.value


def tk_quant_cast_plan_destroy(plan: int) -> None:
    check(lib().tk_quant_cast_plan_destroy(plan))


def tk_quant_cast_output_sizes(desc: QuantCastDesc, num_tokens: int) -> tuple[int, int]:
    qb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    check(lib().tk_quant_cast_output_sizes(ctypes.byref(desc), num_tokens, ctypes.byref(qb),
                                           ctypes.byref(sb)))
    return qb.value, sb.value


def tk_quant_cast_run(plan: int, num_tokens: int, x, q, scales, stream: int | None) -> None:
    check(lib().tk_quant_cast_run(plan, num_tokens, _ptr(x), _ptr(q), _ptr(scales), stream))


def tk_quant_cast_workspace_size(plan: int, num_tokens: int) -> int:
    b = ctypes.c_size_t()
    check(lib().tk_quant_cast_workspace_size(plan, num_tokens, ctypes.byref(b)))
    return b.value


def tk_quant_cast_run_ws(plan: int, num_tokens: int, x, q, scales, workspace, workspace_bytes: int,
                         stream: int | None) -> None:
    check(lib().tk_quant_cast_run_ws(plan, num_tokens, _ptr(x), _ptr(q), _ptr(scales), _ptr(workspace),
                                     workspace_bytes, stream))


CAST_FORMS = {0: "row_quant_kernel", 1: "col_amax_kernel + col_chunk_quant_kernel",
              2: "col_amax_kernel + col_scale_kernel + col_quant_kernel", 3: "block_stream_kernel",
              4: "warp_stream_kernel"}


def tk_quant_cast_launch_info(plan: int, num_tokens: int) -> dict:
    n, f = ctypes.c_int(), ctypes.c_int()
    check(lib().tk_quant_cast_launch_info(plan, num_tokens, ctypes.byref(n), ctypes.byref(f)))
    return {"launches": n.value, "form": f.value, "kernels": CAST_FORMS[f.value]}


def tk_moe_reduce_validate(desc: MoeReduceDesc) -> int:
    return lib().tk_moe_reduce_validate(ctypes.byref(desc))


def tk_moe_reduce_plan(desc: MoeReduceDesc, device: int) -> int:
    h = _VP()
    check(lib().tk_moe_reduce_plan(ctypes.byref(desc), device, ctypes.byref(h)))
    return h.value


def tk_moe_reduce_plan_destroy(plan: int) -> None:
    check(lib().tk_moe_reduce_plan_destroy(plan))


def tk_moe_reduce_run(plan: int, num_tokens: int, y, y_scale, num_rows: int, token_topk_to_pos,
                      topk_weights, global_scale: float, out, stream: int | None) -> None:
    check(lib().tk_moe_reduce_run(plan, num_tokens, _ptr(y), _ptr(y_scale), num_rows,
                                  _ptr(token_topk_to_pos), _ptr(topk_weights), global_scale, _ptr(out),
                                  stream))


def tk_moe_reduce_launch_info(plan: int, num_tokens: int, y=None, y_scale=None) -> dict:
    v = [ctypes.c_int() for _ in range(4)]
    check(lib().tk_moe_reduce_launch_info(plan, num_tokens, _ptr(y), _ptr(y_scale),
                                          *[ctypes.byref(x) for x in v]))
    return {"kernel": ("regs", "bulk")[v[0].value], "grid": v[1].value, "block": v[2].value,
            "smem_bytes": v[3].value}


def tk_swiglu_backward_validate(desc: SwigluBackwardDesc) -> int:
    return lib().tk_swiglu_backward_validate(ctypes.byref(desc))


def tk_swiglu_backward_plan(desc: SwigluBackwardDesc, device: int) -> int:
    h = _VP()
    check(lib().tk_swiglu_backward_plan(ctypes.byref(desc), device, ctypes.byref(h)))
    return h.value


def tk_swiglu_backward_plan_destroy(plan: int) -> None:
    check(lib().tk_swiglu_backward_plan_destroy(plan))


def tk_swiglu_backward_run(plan: int, num_tokens: int, x, topk_weights, dy, dx, dw, q, scales,
                           stream: int | None) -> None:
    check(lib().tk_swiglu_backward_run(plan, num_tokens, _ptr(x), _ptr(topk_weights), _ptr(dy), _ptr(dx),
                                       _ptr(dw), _ptr(q), _ptr(scales), stream))


def tk_fault_word(device: int, clear: bool = False) -> int:
    v = ctypes.c_uint32()
    check(lib().tk_fault_word(device, ctypes.byref(v), int(clear)))
    return v.value


def tk_diag_unanswered_wait(device: int, tries: int, stream=None) -> None:
    check(lib().tk_diag_unanswered_wait(device, tries, stream))


def tk_status_string(status: int) -> str:
    return lib().tk_status_string(status).decode()


def tk_last_error_message() -> str:
    return lib().tk_last_error_message().decode(errors="replace")
