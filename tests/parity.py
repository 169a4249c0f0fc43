"""Comparison of the CUDA path's outputs with the oracle's.

Acceptance (per output tensor):
  * fp32 scales within 1e-6 relative of the oracle's (or within 2^-147,
    four subnormal ulps, where the scale is below the fp32 normal range);
  * UE8M0 scale bytes identical, except groups whose oracle amax lies within
    4 fp32 ulp of a power-of-two boundary Qmax * 2^k, where the kernel's fp32
    activation (a few ulp from the oracle's) may land on the other side; those
    are counted, either exponent is accepted, and the group's oracle codes are
    recomputed with the kernel's scale and must then equal the kernel's codes
    exactly;
  * at least 99.9% of codes identical and every code within one step of the
    oracle's (signed ordinal distance <= 1, +0 and -0 both ordinal 0).
Integer outputs (clamp counters) must match exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

import oracle

QMAX = {"e4m3": 448.0, "e2m1": 6.0}


def ordinal(codes: np.ndarray, out_fmt: str) -> np.ndarray:
    c = codes.astype(np.int32)
    if out_fmt == "e4m3":
        mag, neg = c & 0x7F, (c & 0x80) != 0
    else:
        mag, neg = c & 0x7, (c & 0x8) != 0
    return np.where(neg, -mag, mag)


def unpack(q: np.ndarray, out_fmt: str) -> np.ndarray:
    return q if out_fmt == "e4m3" else oracle.unpack_e2m1(q)


@dataclass
class Report:
    n_codes: int = 0
    n_code_mismatch: int = 0
    max_step: int = 0
    n_groups: int = 0
    n_boundary_groups: int = 0
    n_boundary_flips: int = 0
    n_flip_code_mismatch: int = 0
    max_scale_rel: float = 0.0
    notes: list = field(default_factory=list)

    @property
    def identical_frac(self) -> float:
        return 1.0 - self.n_code_mismatch / max(1, self.n_codes)

    def check(self, what: str = ""):
        assert self.max_step <= 1, "%s: a code is %d steps from the oracle's" % (what, self.max_step)
        assert self.identical_frac >= 0.999, "%s: only %.5f%% codes identical (%d of %d differ)" % (
            what, 100 * self.identical_frac, self.n_code_mismatch, self.n_codes)
        assert self.max_scale_rel <= 1e-6, "%s: fp32 scale off by %.3g relative" % (what, self.max_scale_rel)
        assert self.n_flip_code_mismatch == 0, "%s: %d codes of boundary groups differ from the oracle's " \
            "recomputed with the kernel's scale" % (what, self.n_flip_code_mismatch)
        assert not self.notes, "%s: %s" % (what, "; ".join(self.notes[:5]))


def _near_boundary(amax: np.ndarray, qmax: float) -> np.ndarray:
    """amax within 4 fp32 ulp of qmax * 2^k for some integer k."""
    a = amax.astype(np.float64)
    out = np.zeros(a.shape, bool)
    pos = a > 0
    k = np.round(np.log2(np.where(pos, a, 1.0) / qmax))
    b = qmax * 2.0 ** k
    ulp = np.spacing(b.astype(np.float32)).astype(np.float64)
    out[pos] = np.abs(a[pos] - b[pos]) <= 4 * ulp[pos]
    return out


def compare(gpu_q: np.ndarray, gpu_s: np.ndarray, ref: dict, group: int, scale_fmt: str,
            out_fmt: str, lib=None) -> Report:
    """ref: oracle.swiglu_quant(..., want_y=True) output for the same rows."""
    lib = lib or oracle.load()
    rep = Report()
    y = ref["y"]
    rows, H = y.shape
    g = H if group == 0 else group
    G = H // g
    gq = unpack(gpu_q, out_fmt).reshape(rows, G, g).astype(np.int32)
    oq = unpack(ref["q"], out_fmt).reshape(rows, G, g).astype(np.int32)
    rep.n_groups = rows * G
    if scale_fmt == "fp32":
        gs, os_ = gpu_s.astype(np.float64), ref["scales"].astype(np.float64)
        # Below the fp32 normal range a scale carries fewer than 24 bits, so
        # the relative bound gets a floor of 4 subnormal ulps (2^-147).
        err = np.abs(gs - os_)
        rel = np.where(err <= 2.0 ** -147, 0.0, err / np.maximum(np.abs(os_), 1e-300))
        rep.max_scale_rel = float(rel.max()) if rel.size else 0.0
    else:
        gs, os_ = gpu_s.astype(np.int32), ref["scales"].astype(np.int32)
        diff = gs != os_
        amax = np.abs(y.reshape(rows, G, g)).max(axis=2)
        nb = _near_boundary(amax, QMAX[out_fmt])
        rep.n_boundary_groups = int(nb.sum())
        if diff.any():
            bad = diff & ~(nb & (np.abs(gs - os_) == 1))
            if bad.any():
                r, j = np.argwhere(bad)[0]
                rep.notes.append("UE8M0 byte %d vs oracle %d at row %d group %d" % (gs[r, j], os_[r, j], r, j))
            flips = np.argwhere(diff & ~bad)
            rep.n_boundary_flips = len(flips)
            enc = lib.tko_e4m3_encode if out_fmt == "e4m3" else lib.tko_e2m1_encode
            for r, j in flips:
                s = np.float32(2.0 ** (int(gs[r, j]) - 127))
                yy = y[r, j * g:(j + 1) * g]
                oq[r, j] = [enc(float(np.float32(v) / s)) for v in yy]
                rep.n_flip_code_mismatch += int((gq[r, j] != oq[r, j]).sum())
    go, oo = ordinal(gq, out_fmt), ordinal(oq, out_fmt)
    rep.n_codes = go.size
    rep.n_code_mismatch = int((gq != oq).sum())
    rep.max_step = int(np.abs(go - oo).max()) if go.size else 0
    return rep


def compare_chunked(gpu_q: np.ndarray, gpu_s: np.ndarray, ref: dict, group: int, scale_fmt: str,
                    out_fmt: str, chunk_rows: int = 8192, lib=None) -> Report:
    """compare() over consecutive row chunks (bounded memory for outputs of
    hundreds of millions of codes), merged into one Report; row-major scales."""
    total = Report()
    rows = ref["y"].shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        part = {"y": ref["y"][r0:r1], "q": ref["q"][r0:r1], "scales": ref["scales"][r0:r1]}
        rep = compare(gpu_q[r0:r1], gpu_s[r0:r1], part, group, scale_fmt, out_fmt, lib=lib)
        total.n_codes += rep.n_codes
        total.n_code_mismatch += rep.n_code_mismatch
        total.max_step = max(total.max_step, rep.max_step)
        total.n_groups += rep.n_groups
        total.n_boundary_groups += rep.n_boundary_groups
        total.n_boundary_flips += rep.n_boundary_flips
        total.n_flip_code_mismatch += rep.n_flip_code_mismatch
        total.max_scale_rel = max(total.max_scale_rel, rep.max_scale_rel)
        total.notes += ["rows %d..%d: %s" % (r0, r1, n) for n in rep.notes]
    return total
