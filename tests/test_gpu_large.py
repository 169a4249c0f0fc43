"""Operands larger than 2^32 bytes: every offset the kernels form must be
64-bit. Rows just below and above the 2^31- and 2^32-byte marks (and the
first and last rows) are checked against the oracle, or, where the output is
a permutation of another kernel's, against that kernel bit for bit. These
tests hold up to ~25 GB of device memory at a time."""
import numpy as np
import pytest
import torch

import oracle
from parity import compare
from test_gpu_reduce import check_close

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _rows_near(row_bytes, T):
    """Rows whose start lies just below or just past 2^31 and 2^32 bytes, plus the ends."""
    rows = {0, 1, T - 2, T - 1}
    for mark in (1 << 31, 1 << 32):
        r = mark // row_bytes
        rows.update(x for x in (r - 2, r - 1, r, r + 1) if 0 <= x < T)
    return np.array(sorted(rows))


@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
def test_fused_op_past_4_gib(kernel, monkeypatch):
    monkeypatch.setenv("TK_KERNEL", kernel)
    wl = wls.WORKLOADS["moe_T8192_H2048_g128"].with_rows(540_000)   # x: 4.42 GB
    x, w = wls.make_inputs(wl, "cuda")
    op = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, True)
    q, s = op(x, w)
    torch.cuda.synchronize()
    idx = _rows_near(4 * wl.H, wl.T)
    xi = x[idx].cpu()
    ref = oracle.swiglu_quant(wls.bf16_bits(xi), w[idx].cpu().numpy(), wl.group, wl.scale_fmt, wl.out_fmt,
                              want_y=True)
    rep = compare(q[idx].cpu().numpy(), s[idx].cpu().numpy(), ref, wl.group, wl.scale_fmt, wl.out_fmt)
    rep.check("past 4 GiB, %s kernel" % kernel)
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0
    del x, w, q, s
    torch.cuda.empty_cache()


@pytest.mark.parametrize("kernel", ["regs", "bulk"])
@pytest.mark.parametrize("in_fmt,H,R", [("bf16", 8192, 300_000), ("e4m3", 7168, 300_000)])
def test_combine_rows_past_4_gib(in_fmt, H, R, kernel, monkeypatch):
    """Positions into the top of y (bf16: 4.9 GB; E4M3: 2.2 GB of codes)."""
    g = torch.Generator(device="cuda").manual_seed(R + H)
    if in_fmt == "bf16":
        y = torch.empty((R, H), dtype=torch.bfloat16, device="cuda")
        for r0 in range(0, R, 16384):
            y[r0:r0 + 16384] = torch.randn((min(16384, R - r0), H), generator=g, device="cuda").to(torch.bfloat16)
        ys = None
    else:
        y = torch.randint(0, 126, (R, H), generator=g, device="cuda", dtype=torch.int32).to(torch.uint8)
        ys = torch.exp2(torch.rand((R, H // 128), generator=g, device="cuda") * 4 - 2)
    T, K = 512, 4
    top = torch.randint(R - 4096, R, (T, K), generator=g, device="cuda", dtype=torch.int32)
    low = torch.randint(0, 4096, (T, K), generator=g, device="cuda", dtype=torch.int32)
    pos = torch.where(torch.rand((T, K), generator=g, device="cuda") < 0.5, top, low)
    w = torch.rand((T, K), generator=g, device="cuda")
    monkeypatch.setenv("TK_REDUCE_KERNEL", kernel)
    op = tk.MoeReduce(H, K, in_fmt)
    monkeypatch.delenv("TK_REDUCE_KERNEL")
    out = op(y, pos, w, 1.5, y_scale=ys)
    torch.cuda.synchronize()
    used = torch.unique(pos.flatten()).long()
    remap = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    remap[used] = torch.arange(used.numel(), dtype=torch.int32, device="cuda")
    pos_small = remap[pos.long()].cpu().numpy()
    if ys is None:
        want = oracle.moe_reduce(y[used].cpu().view(torch.int16).numpy().view(np.uint16), pos_small,
                                 w.cpu().numpy(), 1.5)
    else:
        want = oracle.moe_reduce(y[used].cpu().numpy(), pos_small, w.cpu().numpy(), 1.5, y_scale=ys[used].cpu().numpy())
    got = out.cpu().view(torch.int16).numpy().view(np.uint16)
    small = {"y": y[used], "y_scale": None if ys is None else ys[used], "pos": torch.from_numpy(pos_small),
             "w": w, "gs": 1.5}
    check_close(got, want, small, what="%s %s past 4 GiB" % (in_fmt, kernel))
    del y, ys
    torch.cuda.empty_cache()


def test_backward_past_4_gib():
    wl = wls.BACKWARD_WORKLOADS["bwd_T8192_H2048_g128"].with_rows(540_000)   # x 4.42 GB, dx 4.42 GB
    x, w, dy = wls.make_backward_inputs(wl, "cuda")
    op = tk.SwigluBackward(wl.H, True)
    dx, dw, _, _ = op(x, dy, w)
    torch.cuda.synchronize()
    idx = _rows_near(4 * wl.H, wl.T)
    dx_want, dw_want = oracle.swiglu_backward(wls.bf16_bits(x[idx].cpu()), wls.bf16_bits(dy[idx].cpu()),
                                              w[idx].cpu().numpy())
    got = dx[idx].cpu().view(torch.int16).numpy().view(np.uint16)
    assert (got == dx_want).mean() >= 0.999
    rel = np.abs(dw[idx].cpu().numpy() - dw_want) / np.maximum(np.abs(dw_want), 1e-3)
    assert rel.max() < 1e-3
    del x, w, dy, dx, dw
    torch.cuda.empty_cache()


def test_transposed_codes_past_4_gib():
    """qT of 8192 x 530,000 bytes (4.3 GB): its columns are the row-major kernel's rows."""
    wl = wls.WORKLOADS["moe_T8192_H2048_g128"].with_rows(530_000)
    wl = wls.Workload(**{**wl.__dict__, "H": 8192})
    x, w = wls.make_inputs(wl, "cuda")
    op = tk.SwigluQuant(wl.H, 128, "fp32", "e4m3", True)
    qt, st = op.transposed(x, w)
    torch.cuda.synchronize()
    idx = torch.tensor(_rows_near(4 * wl.H, wl.T), device="cuda")
    q_rows, s_rows = op(x[idx], w[idx])
    torch.cuda.synchronize()
    assert torch.equal(qt[:, idx].t(), q_rows) and torch.equal(st[idx], s_rows)
    cols = torch.tensor([0, 1, 4095, 4096, 8190, 8191], device="cuda")
    assert not qt[cols][:, wl.T:].any()
    del x, w, qt, st
    torch.cuda.empty_cache()


@pytest.mark.parametrize("scale_fmt,out_fmt", [("fp32", "e4m3"), ("ue8m0", "e2m1")])
def test_channel_cast_past_4_gib(scale_fmt, out_fmt):
    """The per-channel cast on a 4.9 GB bf16 input (300000 x 8192): a column's
    result depends on that column only, so the oracle takes a slice of
    columns over every row (the first and last chunks and chunks in
    between), which must match bit for bit, codes of every row included."""
    from oracle import parallel
    T, H = 300_000, 8192
    wl = wls.Workload("c", T, H, 0, scale_fmt, out_fmt, "col_lognormal", seed=77, op="cast", gran="channel")
    x, _ = wls.make_inputs(wl, "cuda")
    op = tk.QuantCast(H, 0, scale_fmt, out_fmt, "bf16", granularity="channel")
    q, s = op(x)
    torch.cuda.synchronize()
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0
    for c0 in (0, 4096, H - 32):
        xc = x[:, c0:c0 + 32].float().cpu().numpy()
        rq, rs = parallel.quant_cols_f32(xc, scale_fmt, out_fmt)
        gs = s[c0:c0 + 32].cpu().numpy()
        if scale_fmt == "fp32":
            assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32)), c0
        else:
            assert np.array_equal(gs, rs), c0
        gq = q[:, c0:c0 + 32].cpu().numpy() if out_fmt == "e4m3" else q[:, c0 // 2:c0 // 2 + 16].cpu().numpy()
        assert np.array_equal(gq, rq), c0
    del x, q, s
    torch.cuda.empty_cache()
