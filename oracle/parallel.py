"""The oracle over many host cores (test infrastructure, like the rest of
this package: only the tests, the smoke check and the benchmark's CPU legs
use it).

The oracle computes each row of the fused op (and each column of the
per-channel cast) independently, so a large case is cut into contiguous row
(column) ranges and each range runs the single-threaded C oracle in its own
process. The processes are started with ``spawn``, never forked, so the
caller may already hold a CUDA context. Inputs and outputs travel through
shared memory; every worker writes only its own range of the outputs. The
result is the same bytes as one call over the whole input.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from multiprocessing import shared_memory

import numpy as np

from . import OUT_FMTS, SCALE_FMTS, _ptr, load, output_shapes


def _cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


class _Shared:
    """numpy arrays in named shared-memory blocks (owned by the parent)."""

    def __init__(self):
        self.blocks = []

    def put(self, a: np.ndarray):
        shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
        self.blocks.append(shm)
        view = np.ndarray(a.shape, a.dtype, buffer=shm.buf)
        view[...] = a
        return (shm.name, a.shape, a.dtype.str), view

    def empty(self, shape, dtype):
        dtype = np.dtype(dtype)
        n = int(np.prod(shape)) * dtype.itemsize
        shm = shared_memory.SharedMemory(create=True, size=max(1, n))
        self.blocks.append(shm)
        return (shm.name, tuple(shape), dtype.str), np.ndarray(shape, dtype, buffer=shm.buf)

    def close(self):
        for shm in self.blocks:
            shm.close()
            shm.unlink()
        self.blocks = []


def _attach(desc):
    name, shape, dtype = desc
    shm = shared_memory.SharedMemory(name=name)
    return shm, np.ndarray(shape, np.dtype(dtype), buffer=shm.buf)


def _swiglu_worker(job):
    (xd, wd, qd, sd, yd, cd), (r0, r1), (group, scale_fmt, out_fmt, clamp) = job
    lib = load()
    handles = []
    arrays = []
    for d in (xd, wd, qd, sd, yd, cd):
        if d is None:
            arrays.append(None)
            continue
        h, a = _attach(d)
        handles.append(h)
        arrays.append(a)
    x, w, q, s, y, counts = arrays
    n = r1 - r0
    hidden = x.shape[1] // 2
    cnt = np.zeros(2, np.int64)
    rc = lib.tko_swiglu_quant(_ptr(x[r0:r1]), n, hidden, None if w is None else _ptr(w[r0:r1]), group,
                              SCALE_FMTS[scale_fmt], OUT_FMTS[out_fmt], int(clamp is not None),
                              float(clamp or 0.0), _ptr(q[r0:r1]), _ptr(s[r0:r1]), _ptr(cnt),
                              None if y is None else _ptr(y[r0:r1]))
    del x, w, q, s, y, arrays
    for h in handles:
        h.close()
    if rc != 0:
        raise ValueError("oracle rejected the sizes")
    return cnt


def swiglu_quant(x_bits: np.ndarray, w: np.ndarray | None, group: int, scale_fmt: str, out_fmt: str,
                 clamp: float | None = None, want_y: bool = False, procs: int | None = None) -> dict:
    """As ``oracle.swiglu_quant``, with the rows split over `procs`
    processes (default: every core)."""
    x_bits = np.ascontiguousarray(x_bits, np.uint16)
    rows, two_h = x_bits.shape
    hidden = two_h // 2
    procs = max(1, min(procs or _cores(), rows))
    q_shape, s_shape, s_dtype = output_shapes(rows, hidden, group, scale_fmt, out_fmt)
    sh = _Shared()
    try:
        xd, _ = sh.put(x_bits)
        wd = None if w is None else sh.put(np.ascontiguousarray(w, np.float32))[0]
        qd, q = sh.empty(q_shape, np.uint8)
        sd, s = sh.empty(s_shape, s_dtype)
        yd, y = sh.empty((rows, hidden), np.float32) if want_y else (None, None)
        bounds = np.linspace(0, rows, procs + 1).astype(np.int64)
        jobs = [((xd, wd, qd, sd, yd, None), (int(bounds[i]), int(bounds[i + 1])),
                 (group, scale_fmt, out_fmt, clamp)) for i in range(procs) if bounds[i + 1] > bounds[i]]
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            counts = pool.map(_swiglu_worker, jobs)
        out = {"q": q.copy(), "scales": s.copy(), "counts": np.sum(counts, axis=0).astype(np.int64)}
        if want_y:
            out["y"] = y.copy()
        del q, s, y
        return out
    finally:
        sh.close()


def _cols_worker(job):
    yd, (c0, c1), (scale_fmt, out_fmt) = job
    from . import quant_cols_f32
    h, y = _attach(yd)
    part = np.ascontiguousarray(y[:, c0:c1])
    del y
    h.close()
    return c0, quant_cols_f32(part, scale_fmt, out_fmt)


def quant_cols_f32(y: np.ndarray, scale_fmt: str, out_fmt: str, procs: int | None = None):
    """As ``oracle.quant_cols_f32``, with the columns split over `procs`
    processes (ranges of an even number of columns, so E2M1 bytes never
    straddle two ranges)."""
    y = np.ascontiguousarray(y, np.float32)
    rows, hidden = y.shape
    procs = max(1, min(procs or _cores(), hidden // 2 if hidden >= 2 else 1))
    bounds = (np.linspace(0, hidden // 2, procs + 1).astype(np.int64) * 2).tolist()
    bounds[-1] = hidden
    sh = _Shared()
    try:
        yd, _ = sh.put(y)
        jobs = [(yd, (bounds[i], bounds[i + 1]), (scale_fmt, out_fmt)) for i in range(procs)
                if bounds[i + 1] > bounds[i]]
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            parts = pool.map(_cols_worker, jobs)
    finally:
        sh.close()
    q = np.zeros((rows, hidden if out_fmt == "e4m3" else hidden // 2), np.uint8)
    scales = np.zeros(hidden, np.float32 if scale_fmt == "fp32" else np.uint8)
    for c0, (qp, sp) in parts:
        c1 = c0 + sp.shape[0]
        scales[c0:c1] = sp
        if out_fmt == "e4m3":
            q[:, c0:c1] = qp
        else:
            q[:, c0 // 2:c1 // 2] = qp
    return q, scales
