"""CPU oracle for fused SwiGLU + top-k weight + FP8/FP4 cast (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU legs
may import this package. The product path (the CUDA library and its binding)
never imports it, and it never imports the product path. The arithmetic lives
in ``tko_oracle.c``; this module only compiles it with gcc and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tko_oracle.c")
_LIB = os.path.join(_HERE, "libtko_oracle.so")

# -ffp-contract=off: no fused multiply-add contraction, so each C operation is
# the single IEEE operation written, identically on x86-64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

SCALE_FMTS = {"fp32": 0, "ue8m0": 1}
OUT_FMTS = {"e4m3": 0, "e2m1": 1}
SCALE_LAYOUTS = {"row": 0, "col": 1, "col_packed": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle into a shared library (gcc); returns its path."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) and declare the oracle's C functions."""
    global _lib
    if path is None:
        with _lock:
            if _lib is None:
                _lib = _declare(ctypes.CDLL(build()))
            return _lib
    return _declare(ctypes.CDLL(path))


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    c = ctypes
    lib.tko_e4m3_decode.argtypes = [c.c_uint8]
    lib.tko_e4m3_decode.restype = c.c_double
    lib.tko_e2m1_decode.argtypes = [c.c_uint8]
    lib.tko_e2m1_decode.restype = c.c_double
    lib.tko_e4m3_encode.argtypes = [c.c_float]
    lib.tko_e4m3_encode.restype = c.c_uint8
    lib.tko_e2m1_encode.argtypes = [c.c_float]
    lib.tko_e2m1_encode.restype = c.c_uint8
    lib.tko_ue8m0_byte.argtypes = [c.c_float, c.c_double]
    lib.tko_ue8m0_byte.restype = c.c_uint8
    lib.tko_ue8m0_value.argtypes = [c.c_uint8]
    lib.tko_ue8m0_value.restype = c.c_float
    lib.tko_fp32_scale.argtypes = [c.c_float, c.c_float]
    lib.tko_fp32_scale.restype = c.c_float
    lib.tko_quant_rows_f32.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64,
                                       c.c_int, c.c_int, c.c_void_p, c.c_void_p]
    lib.tko_quant_rows_f32.restype = c.c_int
    lib.tko_quant_cols_f32.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int, c.c_int, c.c_void_p,
                                       c.c_void_p]
    lib.tko_quant_cols_f32.restype = c.c_int
    lib.tko_swiglu_quant.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_void_p,
                                     c.c_int64, c.c_int, c.c_int, c.c_int, c.c_float,
                                     c.c_void_p, c.c_void_p, c.c_void_p, c.c_void_p]
    lib.tko_swiglu_quant.restype = c.c_int
    lib.tko_scale_ld.argtypes = [c.c_int, c.c_int, c.c_int64]
    lib.tko_scale_ld.restype = c.c_int64
    lib.tko_scales_to_layout.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int, c.c_int, c.c_void_p]
    lib.tko_scales_to_layout.restype = c.c_int
    lib.tko_swiglu_backward.argtypes = [c.c_void_p, c.c_void_p, c.c_int64, c.c_int64, c.c_void_p, c.c_int,
                                        c.c_float, c.c_void_p, c.c_void_p]
    lib.tko_swiglu_backward.restype = c.c_int
    lib.tko_codes_transposed.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int64, c.c_void_p]
    lib.tko_codes_transposed.restype = c.c_int
    lib.tko_moe_reduce.argtypes = [c.c_void_p, c.c_void_p, c.c_void_p, c.c_int64, c.c_int64,
                                   c.c_void_p, c.c_void_p, c.c_int64, c.c_int64, c.c_float, c.c_void_p]
    lib.tko_moe_reduce.restype = c.c_int
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def output_shapes(rows: int, hidden: int, group: int, scale_fmt: str, out_fmt: str):
    g = hidden if group == 0 else group
    q_shape = (rows, hidden if out_fmt == "e4m3" else hidden // 2)
    s_dtype = np.float32 if scale_fmt == "fp32" else np.uint8
    return q_shape, (rows, hidden // g), s_dtype


def swiglu_quant(x_bits: np.ndarray, w: np.ndarray | None, group: int, scale_fmt: str,
                 out_fmt: str, clamp: float | None = None, want_y: bool = False,
                 lib: ctypes.CDLL | None = None) -> dict:
    """Run the oracle on bf16 bit patterns x_bits [rows, 2H] (uint16).

    Returns a dict with ``q`` (uint8 codes), ``scales`` (float32 or uint8),
    ``counts`` (int64[2]: gate clamps, up clamps) and, if asked, ``y`` (the
    fp32 activation before quantization)."""
    lib = lib or load()
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, two_h = x_bits.shape
    hidden = two_h // 2
    q_shape, s_shape, s_dtype = output_shapes(rows, hidden, group, scale_fmt, out_fmt)
    q = np.zeros(q_shape, np.uint8)
    scales = np.zeros(s_shape, s_dtype)
    counts = np.zeros(2, np.int64)
    y = np.zeros((rows, hidden), np.float32) if want_y else None
    wa = None if w is None else np.ascontiguousarray(w, dtype=np.float32)
    rc = lib.tko_swiglu_quant(_ptr(x_bits), rows, hidden, _ptr(wa), group,
                              SCALE_FMTS[scale_fmt], OUT_FMTS[out_fmt],
                              int(clamp is not None), float(clamp or 0.0),
                              _ptr(q), _ptr(scales), _ptr(counts), _ptr(y))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    out = {"q": q, "scales": scales, "counts": counts}
    if want_y:
        out["y"] = y
    return out


def quant_rows_f32(y: np.ndarray, group: int, scale_fmt: str, out_fmt: str,
                   lib: ctypes.CDLL | None = None):
    """Quantize fp32 rows y [rows, H]; returns (codes, scales)."""
    lib = lib or load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    rows, hidden = y.shape
    q_shape, s_shape, s_dtype = output_shapes(rows, hidden, group, scale_fmt, out_fmt)
    q = np.zeros(q_shape, np.uint8)
    scales = np.zeros(s_shape, s_dtype)
    rc = lib.tko_quant_rows_f32(_ptr(y), rows, hidden, group, SCALE_FMTS[scale_fmt],
                                OUT_FMTS[out_fmt], _ptr(q), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return q, scales


def quant_cols_f32(y: np.ndarray, scale_fmt: str, out_fmt: str, lib: ctypes.CDLL | None = None):
    """Per-channel quantization of fp32 y [rows, H]: one scale per column;
    returns (codes [rows, H] or packed [rows, H/2], scales [H])."""
    lib = lib or load()
    y = np.ascontiguousarray(y, dtype=np.float32)
    rows, hidden = y.shape
    q = np.zeros((rows, hidden if out_fmt == "e4m3" else hidden // 2), np.uint8)
    scales = np.zeros(hidden, np.float32 if scale_fmt == "fp32" else np.uint8)
    rc = lib.tko_quant_cols_f32(_ptr(y), rows, hidden, SCALE_FMTS[scale_fmt], OUT_FMTS[out_fmt],
                                _ptr(q), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return q, scales


def e4m3_decode_table(lib: ctypes.CDLL | None = None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.tko_e4m3_decode(c) for c in range(256)], np.float64)


def e2m1_decode_table(lib: ctypes.CDLL | None = None) -> np.ndarray:
    lib = lib or load()
    return np.array([lib.tko_e2m1_decode(c) for c in range(16)], np.float64)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """Split packed bytes into nibbles: value 2k is the low nibble of byte k."""
    lo = packed & 0xF
    hi = packed >> 4
    return np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)


def scales_to_layout(scales: np.ndarray, scale_fmt: str, layout: str, fill=0,
                     lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Row-major scales [rows, G] -> a flat byte buffer in `layout`, padding
    left at `fill` (bytes)."""
    lib = lib or load()
    scales = np.ascontiguousarray(scales)
    rows, groups = scales.shape
    code = SCALE_LAYOUTS[layout]
    ld = lib.tko_scale_ld(code, SCALE_FMTS[scale_fmt], rows)
    esz = 4 if scale_fmt == "fp32" else 1
    if layout == "row":
        nbytes = rows * groups * esz
    elif layout == "col":
        nbytes = groups * ld * esz
    else:
        nbytes = (groups // 4) * ld * 4
    out = np.full(nbytes, fill, np.uint8)
    rc = lib.tko_scales_to_layout(_ptr(scales), rows, groups, SCALE_FMTS[scale_fmt], code, _ptr(out))
    if rc != 0:
        raise ValueError("no such scale layout for these scales")
    return out


def swiglu_backward(x_bits: np.ndarray, dy_bits: np.ndarray, w: np.ndarray | None,
                    clamp: float | None = None, lib: ctypes.CDLL | None = None):
    """SwiGLU backward on bf16 bit patterns x [rows, 2H] and dy [rows, H]
    (uint16); returns (dx bf16 bits [rows, 2H], dw float32 [rows])."""
    lib = lib or load()
    x_bits = np.ascontiguousarray(x_bits, np.uint16)
    dy_bits = np.ascontiguousarray(dy_bits, np.uint16)
    rows, two_h = x_bits.shape
    assert dy_bits.shape == (rows, two_h // 2)
    dx = np.zeros((rows, two_h), np.uint16)
    dw = np.zeros(rows, np.float32)
    wa = None if w is None else np.ascontiguousarray(w, np.float32)
    if lib.tko_swiglu_backward(_ptr(x_bits), _ptr(dy_bits), rows, two_h // 2, _ptr(wa), int(clamp is not None),
                               float(clamp or 0.0), _ptr(dx), _ptr(dw)) != 0:
        raise ValueError("oracle rejected the sizes")
    return dx, dw


def codes_transposed(q: np.ndarray, ld: int, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Row-major codes q [rows, H] -> qt [H, ld] with qt[i, t] = q[t, i] and
    zero padding for rows <= t < ld."""
    lib = lib or load()
    q = np.ascontiguousarray(q, np.uint8)
    rows, hidden = q.shape
    out = np.full((hidden, ld), 0xAB, np.uint8)   # every byte is written
    if lib.tko_codes_transposed(_ptr(q), rows, hidden, ld, _ptr(out)) != 0:
        raise ValueError("ld must be at least the number of rows")
    return out


def moe_reduce(y: np.ndarray, pos: np.ndarray, w: np.ndarray, gs: float, y_scale=None,
               lib: ctypes.CDLL | None = None) -> np.ndarray:
    """The weighted top-k combine. y: bf16 bits [R, H] (uint16) or E4M3 codes
    [R, H] (uint8, with y_scale fp32 [R, H/128]); pos int32 [T, K] (-1 empty);
    w fp32 [T, K]. Returns bf16 bits [T, H] (uint16)."""
    lib = lib or load()
    pos = np.ascontiguousarray(pos, np.int32)
    w = np.ascontiguousarray(w, np.float32)
    T, K = pos.shape
    R, H = y.shape
    out = np.zeros((T, H), np.uint16)
    if y.dtype == np.uint16:
        yb, yf, ys = np.ascontiguousarray(y), None, None
    else:
        yb, yf = None, np.ascontiguousarray(y, np.uint8)
        ys = np.ascontiguousarray(y_scale, np.float32)
    rc = lib.tko_moe_reduce(_ptr(yb), _ptr(yf), _ptr(ys), R, H, _ptr(pos), _ptr(w), T, K, float(gs),
                            _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out