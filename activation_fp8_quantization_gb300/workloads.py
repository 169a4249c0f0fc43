"""Seeded synthetic inputs shaped like expanded-token MoE activations.

This module only draws random numbers: it holds none of the SwiGLU or
quantization arithmetic, so both the CUDA path's tests and the CPU oracle can
take their inputs from here without sharing any of the method.

The workloads follow the MoE setting of "TileKernels从入门到精通" (zhichai.net/
topic/177618752), ch.2: each row of ``x [T, 2H]`` is one (token, expert) pair
after top-k expansion, gate half first, with one top-k routing weight per row.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                      # expanded-token rows
    H: int                      # output width; x has 2H columns
    group: int                  # 0 = one scale per row, else columns per scale
    scale_fmt: str              # "fp32" | "ue8m0"
    out_fmt: str                # "e4m3" | "e2m1"
    x_dist: str                 # "normal" | "row_lognormal" | "col_lognormal" | "outliers"
    x_sigma: float = 1.0
    w_dist: str | None = None   # None | "topk8_norm" | "uniform"
    clamp: float | None = None
    seed: int = 0
    op: str = "swiglu"          # "swiglu": x is [T, 2H] bf16; "cast": x is [T, H]; "reduce"
    in_dtype: str = "bf16"      # cast input: "bf16" | "fp32"; reduce rows: "bf16" | "e4m3"
    topk: int = 8               # reduce: slots per token (T tokens, T * topk expert rows)
    empty_frac: float = 0.0     # reduce: share of empty slots
    gran: str = "groups"        # cast: "groups" (per token / per block) | "channel" (one scale per column)

    @property
    def groups_per_row(self) -> int:
        return 1 if self.group == 0 else self.H // self.group

    @property
    def channel(self) -> bool:
        return self.gran == "channel"

    @property
    def x_cols(self) -> int:
        return 2 * self.H if self.op == "swiglu" else self.H

    def algo_bytes(self, rows: int | None = None) -> int:
        """Minimum HBM bytes one pass moves: input, codes, scales, weights."""
        T = self.T if rows is None else rows
        if self.op == "reduce":
            # every expert row read once (bf16, or E4M3 + 1x128 fp32 scales),
            # positions and weights, one bf16 output row per token
            row = 2 * self.H if self.in_dtype == "bf16" else self.H + 4 * (self.H // 128)
            used = round(T * self.topk * (1.0 - self.empty_frac))
            return used * row + 8 * T * self.topk + 2 * T * self.H
        if self.op == "backward":
            # x and dy read, dx and dw written, the recomputed codes and scales written
            q = T * self.H if self.out_fmt == "e4m3" else T * self.H // 2
            s = T * self.groups_per_row * (4 if self.scale_fmt == "fp32" else 1)
            return T * (4 * self.H + 2 * self.H + 4 * self.H + 4 + (4 if self.w_dist else 0)) + q + s
        x = T * self.x_cols * (4 if self.in_dtype == "fp32" else 2)
        q = T * self.H if self.out_fmt == "e4m3" else T * self.H // 2
        if self.channel:
            # a column's scale needs every row, so x is read twice (one pass
            # for the column maxima, one to encode); one scale per column
            return 2 * x + q + self.H * (4 if self.scale_fmt == "fp32" else 1)
        s = T * self.groups_per_row * (4 if self.scale_fmt == "fp32" else 1)
        w = 4 * T if self.w_dist else 0
        return x + q + s + w

    def with_rows(self, T: int) -> "Workload":
        return Workload(**{**self.__dict__, "T": T})


# The five configurations, smallest first. Distributions: "normal" is
# N(0, sigma^2); "row_lognormal" multiplies each whole row (both halves) by one
# LogNormal(0, 1) factor; "outliers" multiplies 0.1% of elements, at uniform
# positions, by 50. "topk8_norm" weights are U(0,1) normalised to sum 1 over
# each consecutive run of 8 rows (one token's top-8 experts).
WORKLOADS = {
    "per_token_T256_H512": Workload("per_token_T256_H512", 256, 512, 0, "fp32", "e4m3",
                                    "normal", seed=1001),
    "moe_T8192_H2048_g128": Workload("moe_T8192_H2048_g128", 8192, 2048, 128, "fp32", "e4m3",
                                     "row_lognormal", w_dist="topk8_norm", seed=1002),
    "moe_T32768_H2048_g128_ue8m0_clamp7": Workload(
        "moe_T32768_H2048_g128_ue8m0_clamp7", 32768, 2048, 128, "ue8m0", "e4m3",
        "outliers", w_dist="topk8_norm", clamp=7.0, seed=1003),
    "ragged_T100003_H3072_g128": Workload("ragged_T100003_H3072_g128", 100003, 3072, 128,
                                          "fp32", "e4m3", "normal", x_sigma=0.5,
                                          w_dist="uniform", seed=1004),
    "fp4_T65536_H2048_g32_ue8m0_clamp7": Workload(
        "fp4_T65536_H2048_g32_ue8m0_clamp7", 65536, 2048, 32, "ue8m0", "e2m1",
        "row_lognormal", w_dist="topk8_norm", clamp=7.0, seed=1005),
}

ORDER = list(WORKLOADS)

# Inputs of the standalone per-token / per-block cast (no SwiGLU): an
# activation that is already computed, [T, H].
CAST_WORKLOADS = {
    "cast_T8192_H4096_g128_bf16": Workload("cast_T8192_H4096_g128_bf16", 8192, 4096, 128, "fp32",
                                           "e4m3", "row_lognormal", seed=2001, op="cast"),
    "cast_T16384_H7168_g128_ue8m0_bf16": Workload("cast_T16384_H7168_g128_ue8m0_bf16", 16384, 7168, 128,
                                                  "ue8m0", "e4m3", "normal", seed=2002, op="cast"),
    "cast_T8192_H4096_token_fp32": Workload("cast_T8192_H4096_token_fp32", 8192, 4096, 0, "fp32", "e4m3",
                                            "row_lognormal", seed=2003, op="cast", in_dtype="fp32"),
    # per channel: one scale per column; "col_lognormal" gives every column
    # its own LogNormal(0, 1) magnitude (outlier channels)
    "cast_T8192_H4096_channel_bf16": Workload("cast_T8192_H4096_channel_bf16", 8192, 4096, 0, "fp32", "e4m3",
                                              "col_lognormal", seed=2004, op="cast", gran="channel"),
    "cast_T16384_H7168_channel_ue8m0_bf16": Workload("cast_T16384_H7168_channel_ue8m0_bf16", 16384, 7168, 0,
                                                     "ue8m0", "e4m3", "col_lognormal", seed=2005, op="cast",
                                                     gran="channel"),
    "cast_T32768_H4096_channel_ue8m0_e2m1_bf16": Workload("cast_T32768_H4096_channel_ue8m0_e2m1_bf16", 32768,
                                                          4096, 0, "ue8m0", "e2m1", "col_lognormal", seed=2006,
                                                          op="cast", gran="channel"),
    "cast_T8192_H4096_channel_fp32": Workload("cast_T8192_H4096_channel_fp32", 8192, 4096, 0, "fp32", "e4m3",
                                              "col_lognormal", seed=2007, op="cast", in_dtype="fp32",
                                              gran="channel"),
}
# The weighted top-k combine after the expert GEMMs: T tokens, each gathering
# `topk` expert rows (a random permutation of the T * topk rows, as after a
# dispatch, with a share of empty slots), weights normalised per token.
REDUCE_WORKLOADS = {
    "reduce_T4096_K8_H2048_bf16": Workload("reduce_T4096_K8_H2048_bf16", 4096, 2048, 0, "fp32", "e4m3",
                                           "normal", seed=3001, op="reduce", topk=8, empty_frac=0.01),
    "reduce_T4096_K8_H7168_e4m3": Workload("reduce_T4096_K8_H7168_e4m3", 4096, 7168, 0, "fp32", "e4m3",
                                           "normal", seed=3002, op="reduce", in_dtype="e4m3", topk=8,
                                           empty_frac=0.01),
}
# The SwiGLU backward with the forward's codes recomputed: x and w as the
# fused workloads of the same shape, dy ~ N(0, 1) in bf16.
BACKWARD_WORKLOADS = {
    "bwd_T8192_H2048_g128": Workload("bwd_T8192_H2048_g128", 8192, 2048, 128, "fp32", "e4m3", "row_lognormal",
                                     w_dist="topk8_norm", seed=4001, op="backward"),
    "bwd_T32768_H2048_g128_ue8m0_clamp7": Workload("bwd_T32768_H2048_g128_ue8m0_clamp7", 32768, 2048, 128,
                                                   "ue8m0", "e4m3", "outliers", w_dist="topk8_norm", clamp=7.0,
                                                   seed=4002, op="backward"),
}

ALL_WORKLOADS = {**WORKLOADS, **CAST_WORKLOADS, **REDUCE_WORKLOADS, **BACKWARD_WORKLOADS}

_CHUNK_ROWS = 4096


def make_inputs(wl: Workload, device: str | torch.device = "cpu"):
    """Return (x [T, 2H] bf16, or [T, H] for a cast workload; w fp32 [T] or
    None) for a workload, drawn from
    one torch.Generator seeded with wl.seed on ``device``. Rows are drawn in
    chunks of 4096 so that peak memory stays bounded at large T."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    T, C = wl.T, wl.x_cols
    xdt = torch.float32 if wl.in_dtype == "fp32" else torch.bfloat16
    x = torch.empty((T, C), dtype=xdt, device=device)
    col = None
    if wl.x_dist == "col_lognormal":
        col = torch.randn((1, C), generator=gen, device=device).exp_()
    for r0 in range(0, T, _CHUNK_ROWS):
        r1 = min(T, r0 + _CHUNK_ROWS)
        n = r1 - r0
        v = torch.randn((n, C), generator=gen, device=device, dtype=torch.float32)
        if wl.x_sigma != 1.0:
            v.mul_(wl.x_sigma)
        if wl.x_dist == "row_lognormal":
            v.mul_(torch.randn((n, 1), generator=gen, device=device).exp_())
        elif wl.x_dist == "col_lognormal":
            v.mul_(col)
        elif wl.x_dist == "outliers":
            hit = torch.rand((n, C), generator=gen, device=device) < 1e-3
            v = torch.where(hit, v * 50.0, v)
        elif wl.x_dist != "normal":
            raise ValueError(wl.x_dist)
        x[r0:r1] = v.to(xdt)
    w = None
    if wl.w_dist is not None:
        w = torch.rand((T,), generator=gen, device=device, dtype=torch.float32)
        if wl.w_dist == "topk8_norm":
            full = (T // 8) * 8
            if full:
                blk = w[:full].view(-1, 8)
                w[:full] = (blk / blk.sum(dim=1, keepdim=True)).reshape(-1)
            if full < T:
                w[full:] = w[full:] / w[full:].sum()
        elif wl.w_dist != "uniform":
            raise ValueError(wl.w_dist)
    return x, w


def bf16_bits(x: torch.Tensor):
    """View a bf16 tensor's bit patterns as a numpy uint16 array (host copy)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def make_backward_inputs(wl: Workload, device: str | torch.device = "cpu"):
    """(x, w, dy) of a backward workload: x and w as make_inputs draws them for
    the same shape and seed, dy [T, H] bf16 N(0, 1) from seed + 1."""
    x, w = make_inputs(Workload(**{**wl.__dict__, "op": "swiglu"}), device)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed + 1)
    dy = torch.empty((wl.T, wl.H), dtype=torch.bfloat16, device=device)
    for r0 in range(0, wl.T, _CHUNK_ROWS):
        r1 = min(wl.T, r0 + _CHUNK_ROWS)
        dy[r0:r1] = torch.randn((r1 - r0, wl.H), generator=gen, device=device).to(torch.bfloat16)
    return x, w, dy


def make_reduce_inputs(wl: Workload, device: str | torch.device = "cpu") -> dict:
    """Inputs of a combine workload: y (bf16 [R, H], or E4M3 codes uint8 [R, H]
    drawn as random non-NaN bytes with fp32 y_scale [R, H/128] in [2^-4, 2^4)),
    token_topk_to_pos int32 [T, K] (a permutation of the R = T * K rows, a
    share of slots emptied to -1), topk_weights fp32 [T, K] (U(0,1),
    normalised per token) and the global scale gs."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    T, K, H = wl.T, wl.topk, wl.H
    R = T * K
    if wl.in_dtype == "bf16":
        y = torch.empty((R, H), dtype=torch.bfloat16, device=device)
        for r0 in range(0, R, _CHUNK_ROWS):
            r1 = min(R, r0 + _CHUNK_ROWS)
            y[r0:r1] = torch.randn((r1 - r0, H), generator=gen, device=device).to(torch.bfloat16)
        y_scale = None
    else:
        y = torch.randint(0, 256, (R, H), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
        y[(y & 0x7F) == 0x7F] = 0          # no NaN codes
        y_scale = torch.exp2(torch.rand((R, H // 128), generator=gen, device=device) * 8 - 4)
    perm = torch.randperm(R, generator=gen, device=device).to(torch.int32).view(T, K)
    empty = torch.rand((T, K), generator=gen, device=device) < wl.empty_frac
    pos = torch.where(empty, torch.full_like(perm, -1), perm)
    w = torch.rand((T, K), generator=gen, device=device)
    w = w / w.sum(dim=1, keepdim=True)
    return {"y": y, "y_scale": y_scale, "pos": pos.contiguous(), "w": w.contiguous(), "gs": 2.5}