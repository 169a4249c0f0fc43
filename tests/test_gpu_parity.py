"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Small cases take each workload's shape, formats and value distribution at a
row count that makes every CTA of the persistent grid walk two row blocks and
leaves a ragged tail; the oracle computes every row. Full-size cases run the
exact launch the benchmark times and compare sampled rows (first, last and
random ones) with the oracle, plus properties checked on every row.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import compare, unpack

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _op(wl, count=False):
    return tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, wl.w_dist is not None,
                          wl.clamp, count and wl.clamp is not None)


def _run(op, x, w, counts=None):
    q, s = op(x, w, clamped_count=counts)
    torch.cuda.synchronize()
    return q, s


def _oracle(wl, x_cpu, w_cpu):
    return oracle.swiglu_quant(wls.bf16_bits(x_cpu), None if w_cpu is None else w_cpu.numpy(),
                               wl.group, wl.scale_fmt, wl.out_fmt, clamp=wl.clamp, want_y=True)


def _rows_for_two_passes(op):
    """Rows that make every CTA (row kernel: rows per iteration; block-ring
    kernel: rows per ring slot) or every warp (warp-stream kernel) of the full
    grid take two steps, plus a ragged tail."""
    info = op.launch_info(1 << 30)
    if info["rows_per_cta"]:
        return 2 * info["grid"] * info["rows_per_cta"] + 37
    wpr = op.hidden // 512
    return 2 * info["grid"] * (info["block"] // 32) // wpr + 37


@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
@pytest.mark.parametrize("name", wls.ORDER)
def test_workload_small_parity(name, kernel, monkeypatch):
    monkeypatch.setenv("TK_KERNEL", kernel)
    wl = wls.WORKLOADS[name]
    op = _op(wl, count=True)
    rows = _rows_for_two_passes(op)
    wl_s = wl.with_rows(rows)
    x, w = wls.make_inputs(wl_s, "cpu")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    q, s = _run(op, x.cuda(), None if w is None else w.cuda(), counts if op.count_clamped else None)
    ref = _oracle(wl, x, w)
    rep = compare(q.cpu().numpy(), s.cpu().numpy(), ref, wl.group, wl.scale_fmt, wl.out_fmt)
    rep.check(name)
    if op.count_clamped:
        assert counts.cpu().tolist() == ref["counts"].tolist()
    print(name, kernel, rows, "rows: identical %.6f, boundary groups %d, flips %d" % (
        rep.identical_frac, rep.n_boundary_groups, rep.n_boundary_flips))


def _torch_counts(x, H, L):
    g = x[:, :H].float()
    u = x[:, H:].float()
    return [int((g > L).sum().item()), int((u.abs() > L).sum().item())]


@pytest.mark.parametrize("name", wls.ORDER)
def test_workload_full_size(name):
    wl = wls.WORKLOADS[name]
    op = _op(wl, count=True)
    x, w = wls.make_inputs(wl, "cuda")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    q, s = _run(op, x, w, counts if op.count_clamped else None)
    T, H = wl.T, wl.H
    # properties of every row
    qc = q.to(torch.int32)
    if wl.out_fmt == "e4m3":
        assert not ((qc & 0x7F) == 0x7F).any(), "NaN code written"
    if wl.scale_fmt == "fp32":
        assert bool((s > 0).all())
        if wl.out_fmt == "e4m3":
            g = H if wl.group == 0 else wl.group
            top = ((qc & 0x7F) == 0x7E).view(T, H // g, g).any(dim=2)
            assert bool(top.all()), "a group has no element at +-448"
    else:
        assert int(s.max()) <= 254
    if op.count_clamped:
        assert counts.cpu().tolist() == _torch_counts(x, H, wl.clamp)
    # sampled rows against the oracle
    gen = np.random.default_rng(wl.seed)
    idx = np.unique(np.concatenate([np.arange(64), np.arange(T - 64, T),
                                    gen.choice(T, size=min(T, 768), replace=False)]))
    it = torch.from_numpy(idx).cuda()
    xs = x.index_select(0, it).cpu()
    ws = None if w is None else w.index_select(0, it).cpu()
    ref = _oracle(wl, xs, ws)
    rep = compare(q.index_select(0, it).cpu().numpy(), s.index_select(0, it).cpu().numpy(), ref,
                  wl.group, wl.scale_fmt, wl.out_fmt)
    rep.check(name + " full")
    print(name, "full: %d sampled rows, identical %.6f" % (len(idx), rep.identical_frac))


LARGE = ["moe_T32768_H2048_g128_ue8m0_clamp7", "ragged_T100003_H3072_g128", "fp4_T65536_H2048_g32_ue8m0_clamp7"]


@pytest.mark.parametrize("name", LARGE)
def test_workload_full_output(name):
    """The three largest workloads at full size in the benchmark's launch
    configuration, every row compared with the oracle (run over all host
    cores): at least 99.9% of the codes identical, none more than one step
    away, UE8M0 scales exact up to counted boundary groups (whose codes must
    then follow the kernel's scale exactly), fp32 scales within 1e-6, and the
    clamp counters exact."""
    from oracle import parallel
    from parity import compare_chunked
    wl = wls.WORKLOADS[name]
    op = _op(wl, count=True)
    x_cpu, w_cpu = wls.make_inputs(wl, "cpu")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    q, s = _run(op, x_cpu.cuda(), None if w_cpu is None else w_cpu.cuda(),
                counts if op.count_clamped else None)
    kernel = op.launch_info(wl.T)["kernel"]
    gq, gs = q.cpu().numpy(), s.cpu().numpy()
    del q, s
    ref = parallel.swiglu_quant(wls.bf16_bits(x_cpu), None if w_cpu is None else w_cpu.numpy(), wl.group,
                                wl.scale_fmt, wl.out_fmt, clamp=wl.clamp, want_y=True)
    rep = compare_chunked(gq, gs, ref, wl.group, wl.scale_fmt, wl.out_fmt)
    print(name, kernel, "every row: %d codes, identical %.7f, max step %d, %d groups, boundary groups %d, "
          "flips %d, max fp32 scale rel %.3g" % (rep.n_codes, rep.identical_frac, rep.max_step, rep.n_groups,
                                                rep.n_boundary_groups, rep.n_boundary_flips, rep.max_scale_rel))
    rep.check(name + " every row")
    assert rep.n_codes == wl.T * wl.H
    if op.count_clamped:
        assert counts.cpu().tolist() == ref["counts"].tolist()


# ------------------------------------------------------------- edge cases

GEOMS = [  # (H, group) incl. the CTA-reduction path (one scale per row, wide or odd rows)
    (16, 16), (16, 0), (48, 16), (48, 0), (80, 16), (512, 0), (512, 512), (1040, 16),
    (2048, 64), (2048, 256), (4096, 0), (7168, 128), (7168, 0), (16384, 512), (16384, 0),
]


@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
@pytest.mark.parametrize("H,group", GEOMS)
@pytest.mark.parametrize("scale_fmt,out_fmt", [("fp32", "e4m3"), ("ue8m0", "e4m3"),
                                               ("ue8m0", "e2m1"), ("fp32", "e2m1")])
def test_geometry_sweep(H, group, scale_fmt, out_fmt, kernel, monkeypatch):
    """Forcing the stream kernel on a shape it does not apply to leaves the
    row kernel in place, so those cases run the row kernel twice."""
    monkeypatch.setenv("TK_KERNEL", kernel)
    rng = np.random.default_rng(H * 7 + group)
    T = 29
    x = torch.from_numpy(rng.standard_normal((T, 2 * H)).astype(np.float32) * 2).to(torch.bfloat16)
    w = torch.from_numpy(rng.uniform(0.0, 1.0, T).astype(np.float32))
    op = tk.SwigluQuant(H, group, scale_fmt, out_fmt, True, 3.0, True)
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    q, s = _run(op, x.cuda(), w.cuda(), counts)
    ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), group, scale_fmt, out_fmt, clamp=3.0,
                              want_y=True)
    compare(q.cpu().numpy(), s.cpu().numpy(), ref, group, scale_fmt, out_fmt).check((H, group))
    assert counts.cpu().tolist() == ref["counts"].tolist()


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def _bf16_neighbours(v):
    """The bf16 values just below, at (if representable) and just above v."""
    b = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item() & 0xFFFF
    near = sorted({(b - 1) & 0xFFFF, b, (b + 1) & 0xFFFF})
    return torch.tensor(near, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().tolist()


@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
@pytest.mark.parametrize("limit", [3.0, 2.7182817, 0.1])
@pytest.mark.parametrize("H,group,scale_fmt,out_fmt", [(2048, 128, "ue8m0", "e4m3"), (512, 32, "ue8m0", "e2m1"),
                                                       (1024, 0, "fp32", "e4m3")])
def test_clamp_limits_bf16_and_not(H, group, scale_fmt, out_fmt, limit, kernel, monkeypatch):
    """A limit that is a bf16 value is applied on the bf16 pairs, any other in
    fp32; both give the oracle's codes, scales and counts. Values at the
    limit's bf16 neighbours, at +-limit and past it in both halves, and rows
    with no value near the limit (the test that skips clamping)."""
    monkeypatch.setenv("TK_KERNEL", kernel)
    rng = np.random.default_rng(int(limit * 1000) + H + group)
    T = 67
    v = rng.standard_normal((T, 2 * H)).astype(np.float32) * 0.5 * limit
    near = _bf16_neighbours(limit)
    cand = np.array(near + [-x for x in near] + [4 * limit, -4 * limit, limit, -limit], np.float32)
    for r in range(0, T, 3):   # every third row holds planted values in both halves
        cols = rng.choice(2 * H, size=24, replace=False)
        v[r, cols] = rng.choice(cand, size=24)
    x = _bf16(v)
    w = torch.from_numpy(rng.uniform(0.0, 1.0, T).astype(np.float32))
    op = tk.SwigluQuant(H, group, scale_fmt, out_fmt, True, limit, True)
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    q, s = _run(op, x.cuda(), w.cuda(), counts)
    ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), group, scale_fmt, out_fmt, clamp=limit, want_y=True)
    compare(q.cpu().numpy(), s.cpu().numpy(), ref, group, scale_fmt, out_fmt).check((H, group, limit))
    assert counts.cpu().tolist() == ref["counts"].tolist()
    assert min(ref["counts"].tolist()) > 0


@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
def test_special_rows(kernel, monkeypatch):
    monkeypatch.setenv("TK_KERNEL", kernel)
    H, g = 512, 128
    rows = []
    rows.append(np.zeros(2 * H))                                            # all zero
    rows.append(np.concatenate([np.full(H, -95.0), np.full(H, 3.0)]))      # silu underflows to subnormals
    rows.append(np.concatenate([np.full(H, 1e-20), np.full(H, 1e-20)]))    # y ~ 1e-40: subnormal amax
    rows.append(np.concatenate([np.full(H, 2.0), np.full(H, -2.0)]))       # equal magnitudes
    one_hot = np.zeros(2 * H)
    one_hot[5], one_hot[H + 5] = 3.0, 1.0
    rows.append(one_hot)
    big = np.concatenate([np.full(H, 1e18), np.linspace(-1e18, 1e18, H)])
    rows.append(big)
    rng = np.random.default_rng(0)
    rows.append(rng.standard_normal(2 * H) * 1e-3)
    x = _bf16(np.stack(rows))
    for scale_fmt in ("fp32", "ue8m0"):
        for out_fmt in ("e4m3", "e2m1"):
            op = tk.SwigluQuant(H, g, scale_fmt, out_fmt, False)
            q, s = _run(op, x.cuda(), None)
            ref = oracle.swiglu_quant(wls.bf16_bits(x), None, g, scale_fmt, out_fmt, want_y=True)
            compare(q.cpu().numpy(), s.cpu().numpy(), ref, g, scale_fmt, out_fmt).check(
                "special %s %s" % (scale_fmt, out_fmt))


def test_zero_rows_is_noop_and_tails():
    H = 512
    op = tk.SwigluQuant(H, 128, "fp32", "e4m3", True)
    x = torch.zeros(0, 2 * H, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(0, dtype=torch.float32, device="cuda")
    q, s = _run(op, x, w)
    assert q.shape == (0, H) and s.shape == (0, 4)
    for T in (1, 2, 3, 5, 17):
        xr = _bf16(np.random.default_rng(T).standard_normal((T, 2 * H)))
        wr = torch.rand(T)
        q, s = _run(op, xr.cuda(), wr.cuda())
        ref = oracle.swiglu_quant(wls.bf16_bits(xr), wr.numpy(), 128, "fp32", "e4m3", want_y=True)
        compare(q.cpu().numpy(), s.cpu().numpy(), ref, 128, "fp32", "e4m3").check("T=%d" % T)


@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
def test_guard_bands_untouched(kernel, monkeypatch):
    """Outputs live inside larger buffers filled with a sentinel; only the
    output bytes may change."""
    monkeypatch.setenv("TK_KERNEL", kernel)
    H, T, g = 1024, 301, 32
    for scale_fmt, out_fmt in (("fp32", "e4m3"), ("ue8m0", "e2m1")):
        op = tk.SwigluQuant(H, g, scale_fmt, out_fmt, True, 7.0, False)
        q_shape, s_shape, s_dtype = op.output_shapes(T)
        pad = 256
        qn = q_shape[0] * q_shape[1]
        qbuf = torch.full((qn + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda")
        q = qbuf[pad:pad + qn].view(q_shape)
        sn = s_shape[0] * s_shape[1]
        sbuf = torch.full((sn + 2 * pad,), -7.0 if s_dtype == torch.float32 else 0x5A,
                          dtype=s_dtype, device="cuda")
        s = sbuf[pad:pad + sn].view(s_shape)
        x = _bf16(np.random.default_rng(1).standard_normal((T, 2 * H)) * 4).cuda()
        w = torch.rand(T, device="cuda")
        op(x, w, q=q, scales=s)
        torch.cuda.synchronize()
        assert bool((qbuf[:pad] == 0xA5).all()) and bool((qbuf[pad + qn:] == 0xA5).all())
        fill = -7.0 if s_dtype == torch.float32 else 0x5A
        assert bool((sbuf[:pad] == fill).all()) and bool((sbuf[pad + sn:] == fill).all())


def test_clamp_counter_accumulates_and_streams():
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(4096)
    x, w = wls.make_inputs(wl, "cuda")
    op = _op(wl, count=True)
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for st in streams:
        with torch.cuda.stream(st):
            outs.append(op(x, w, clamped_count=counts, stream=st))
    torch.cuda.synchronize()
    one = _torch_counts(x, wl.H, wl.clamp)
    assert counts.cpu().tolist() == [2 * one[0], 2 * one[1]]
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_host_side_errors():
    H = 256
    op = tk.SwigluQuant(H, 128, "fp32", "e4m3", True, 7.0, True)
    x = torch.zeros(8, 2 * H + 16, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(8, device="cuda")
    q = torch.empty(8, H, dtype=torch.uint8, device="cuda")
    s = torch.empty(8, 2, device="cuda")
    c = torch.zeros(2, dtype=torch.int64, device="cuda")
    base = x.data_ptr()
    with pytest.raises(tk.TkError) as e:   # x not 32-byte aligned
        tk.tk_swiglu_quant_run(op.plan, 8, base + 2, w, q, s, c, None)
    assert e.value.status == 3
    with pytest.raises(tk.TkError) as e:   # q not 16-byte aligned
        tk.tk_swiglu_quant_run(op.plan, 8, base, w, q.data_ptr() + 1, s, c, None)
    assert e.value.status == 3
    with pytest.raises(tk.TkError) as e:   # weights expected
        tk.tk_swiglu_quant_run(op.plan, 8, base, None, q, s, c, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:   # counter expected
        tk.tk_swiglu_quant_run(op.plan, 8, base, w, q, s, None, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:
        tk.tk_swiglu_quant_run(op.plan, -1, base, w, q, s, c, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:
        tk.tk_swiglu_quant_plan(tk.SwigluQuantDesc(H, 128, 0, 0, 1, 0, 0.0, 0, 0), 4096)
    assert e.value.status == 1
    torch.cuda.synchronize()


# ----------------------------------------------------- standalone cast

@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
@pytest.mark.parametrize("in_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("H,group", [(2048, 128), (512, 0), (7168, 0), (1024, 32), (48, 16)])
@pytest.mark.parametrize("scale_fmt,out_fmt", [("fp32", "e4m3"), ("ue8m0", "e4m3"),
                                               ("ue8m0", "e2m1"), ("fp32", "e2m1")])
def test_cast_bit_exact(in_dtype, H, group, scale_fmt, out_fmt, kernel, monkeypatch):
    monkeypatch.setenv("TK_KERNEL", kernel)
    """With the activation given as input there is nothing approximate left:
    scales and codes must equal the oracle's bit for bit."""
    rng = np.random.default_rng(H + group)
    T = 211
    v = rng.standard_normal((T, H)) * np.exp2(rng.integers(-40, 40, (T, 1)))
    v[3] = 0.0
    v[4, : H // 2] = 2.0 ** -140                    # fp32 subnormals
    v[5] = np.where(np.arange(H) % 3 == 0, 448.0, -0.0)
    v[6] = rng.standard_normal(H) * 1e-30
    y = torch.from_numpy(v.astype(np.float32))
    if in_dtype == "bf16":
        y = y.to(torch.bfloat16)
    op = tk.QuantCast(H, group, scale_fmt, out_fmt, in_dtype)
    q, s = op(y.cuda())
    torch.cuda.synchronize()
    yf = y.float().numpy()
    rq, rs = oracle.quant_rows_f32(yf, group, scale_fmt, out_fmt)
    gq, gs = q.cpu().numpy(), s.cpu().numpy()
    if scale_fmt == "fp32":
        assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32)), "scales differ"
    else:
        assert np.array_equal(gs, rs), "scale bytes differ"
    bad = np.argwhere(unpack(gq, out_fmt) != unpack(rq, out_fmt))
    assert bad.size == 0, "codes differ at %s" % (bad[:5].tolist(),)


@pytest.mark.parametrize("name", [n for n, w in wls.CAST_WORKLOADS.items() if not w.channel])
def test_cast_workload_full_size(name):
    """The standalone cast on its benchmark workloads, full size, in the
    benchmark's launch configuration; sampled rows bit for bit."""
    wl = wls.CAST_WORKLOADS[name]
    x, _ = wls.make_inputs(wl, "cuda")
    op = tk.QuantCast(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, wl.in_dtype)
    q, s = op(x)
    torch.cuda.synchronize()
    gen = np.random.default_rng(wl.seed)
    idx = np.unique(np.concatenate([np.arange(32), np.arange(wl.T - 32, wl.T),
                                    gen.choice(wl.T, size=256, replace=False)]))
    it = torch.from_numpy(idx).cuda()
    y = x.index_select(0, it).float().cpu().numpy()
    rq, rs = oracle.quant_rows_f32(y, wl.group, wl.scale_fmt, wl.out_fmt)
    gq, gs = q.index_select(0, it).cpu().numpy(), s.index_select(0, it).cpu().numpy()
    assert np.array_equal(gq, rq)
    if wl.scale_fmt == "fp32":
        assert np.array_equal(gs.view(np.uint32), rs.view(np.uint32))
    else:
        assert np.array_equal(gs, rs)


# ------------------------------------------------------ host-buffer pipe

@pytest.mark.parametrize("kernel", ["auto", "block"])
@pytest.mark.parametrize("chunk_rows", [1, 7, 1000, 4096, 100000])
def test_host_pipe_matches_device_call(chunk_rows, kernel, monkeypatch):
    """The pipe's chunks run the plan's kernel for their size (the block-ring
    kernel too when forced) and must give the device call's bytes."""
    if kernel == "block":
        monkeypatch.setenv("TK_KERNEL", "block")
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(3001)
    x, w = wls.make_inputs(wl, "cpu")
    op = _op(wl, count=True)
    counts_d = torch.zeros(2, dtype=torch.int64, device="cuda")
    qd, sd = _run(op, x.cuda(), w.cuda(), counts_d)
    pipe = tk.HostPipe(op, chunk_rows)
    xh, wh = x.pin_memory(), w.pin_memory()
    counts_h = torch.tensor([5, 7], dtype=torch.int64).pin_memory()
    for _ in range(2):   # the pipe and its workspace are reusable
        qh, sh = pipe(xh, wh, clamped_count=counts_h)
        torch.cuda.synchronize()
        assert torch.equal(qh, qd.cpu()) and torch.equal(sh, sd.cpu())
    c = counts_d.cpu()
    assert counts_h.tolist() == [5 + 2 * int(c[0]), 7 + 2 * int(c[1])]


def test_host_pipe_pageable_and_fp32_scales():
    wl = wls.WORKLOADS["ragged_T100003_H3072_g128"].with_rows(777)
    x, w = wls.make_inputs(wl, "cpu")
    op = _op(wl)
    qd, sd = _run(op, x.cuda(), w.cuda())
    pipe = tk.HostPipe(op, 100)
    q = torch.empty(op.output_shapes(777)[0], dtype=torch.uint8)          # pageable
    s = torch.empty(op.output_shapes(777)[1], dtype=torch.float32)
    pipe(x, w, q=q, scales=s)
    torch.cuda.synchronize()
    assert torch.equal(q, qd.cpu()) and torch.equal(s, sd.cpu())


def test_host_pipe_errors():
    op = tk.SwigluQuant(256, 128, "fp32", "e4m3", True)
    pipe = tk.HostPipe(op, 64)
    x = torch.zeros(8, 512, dtype=torch.bfloat16)
    w = torch.ones(8)
    q = torch.empty(8, 256, dtype=torch.uint8)
    s = torch.empty(8, 2)
    with pytest.raises(tk.TkError) as e:   # workspace too small
        tk.tk_swiglu_quant_run_host(pipe.pipe, 8, x, w, q, s, None, pipe.workspace, 16, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:   # misaligned workspace
        tk.tk_swiglu_quant_run_host(pipe.pipe, 8, x, w, q, s, None, pipe.workspace.data_ptr() + 8,
                                    pipe.ws_bytes, None)
    assert e.value.status == 3
    with pytest.raises(tk.TkError) as e:   # weights expected
        tk.tk_swiglu_quant_run_host(pipe.pipe, 8, x, None, q, s, None, pipe.workspace, pipe.ws_bytes, None)
    assert e.value.status == 1


# ------------------------------------------- both kernels on the same shapes

def test_cast_plan_picks_the_kernel_by_input_size(monkeypatch):
    """The per-token / per-block cast runs the block ring for inputs of 48 to
    288 MiB (bf16) or 160 to 640 MiB (fp32) and the row kernel otherwise;
    per-token scales at widths a warp group cannot cover have only the row
    kernel; TK_KERNEL forces one."""
    op = tk.QuantCast(4096, 128, "fp32", "e4m3", "bf16")
    assert op.launch_info(1024)["kernels"] == "row_quant_kernel"
    assert op.launch_info(6143)["kernels"] == "row_quant_kernel"      # just under 48 MiB
    assert op.launch_info(6144)["kernels"] == "block_stream_kernel"   # 48 MiB
    assert op.launch_info(8192)["form"] == 3 and op.launch_info(8192)["launches"] == 1
    assert op.launch_info(36864)["kernels"] == "block_stream_kernel"  # 288 MiB
    assert op.launch_info(36865)["kernels"] == "row_quant_kernel"
    assert op.launch_info(65536)["kernels"] == "row_quant_kernel"
    f32 = tk.QuantCast(4096, 128, "fp32", "e4m3", "fp32")
    assert f32.launch_info(8192)["form"] == 0 and f32.launch_info(16384)["form"] == 3
    assert f32.launch_info(65536)["form"] == 0
    assert tk.QuantCast(4096, 0, "fp32", "e4m3", "bf16").launch_info(16384)["form"] == 0
    assert tk.QuantCast(1040, 16, "fp32", "e4m3", "bf16").launch_info(1 << 16)["form"] == 0
    monkeypatch.setenv("TK_KERNEL", "block")
    assert tk.QuantCast(4096, 128, "fp32", "e4m3", "bf16").launch_info(100)["form"] == 3
    monkeypatch.setenv("TK_KERNEL", "stream")
    assert tk.QuantCast(4096, 128, "fp32", "e4m3", "bf16").launch_info(8192)["kernels"] == "warp_stream_kernel"
    monkeypatch.setenv("TK_KERNEL", "rows")
    assert tk.QuantCast(4096, 128, "fp32", "e4m3", "bf16").launch_info(8192)["form"] == 0


def test_plan_picks_the_kernel_by_batch_size(monkeypatch):
    # The block-ring kernel applies to widths that are multiples of 512 whose
    # scale groups fit in 512 columns, and runs once every resident CTA has
    # enough row blocks to stream (at width 2048: 32, or 16 with the clamp;
    # 8 at width 3072); the row kernel runs everything else.
    op = tk.SwigluQuant(2048, 128)
    small, big = op.launch_info(1024), op.launch_info(65536)
    assert op.launch_info(32768)["kernel"] == "row_quant_kernel"
    clamped = tk.SwigluQuant(2048, 128, "ue8m0", "e4m3", True, 7.0)
    assert clamped.launch_info(32768)["kernel"] == "block_stream_kernel"
    assert clamped.launch_info(16384)["kernel"] == "row_quant_kernel"
    assert tk.SwigluQuant(3072, 128).launch_info(25000)["kernel"] == "block_stream_kernel"
    assert small["kernel"] == "row_quant_kernel" and small["rows_per_cta"] > 0
    assert big["kernel"] == "block_stream_kernel" and big["block"] == 288
    assert big["rows_per_cta"] * 4 >= 8          # at least one slice per consumer warp in a block
    assert big["grid"] % big["num_sms"] == 0
    assert tk.SwigluQuant(512, 0).launch_info(1 << 20)["kernel"] == "block_stream_kernel"
    info = tk.SwigluQuant(4096, 0).launch_info(1 << 20)    # per-token scales: a CTA-wide reduction
    assert info["kernel"] == "row_quant_kernel" and info["rows_per_cta"] == 1
    assert tk.SwigluQuant(1040, 16).launch_info(1 << 20)["kernel"] == "row_quant_kernel"
    # forcing a kernel (read when the plan is made)
    monkeypatch.setenv("TK_KERNEL", "stream")
    info = tk.SwigluQuant(2048, 128).launch_info(1024)
    assert info["kernel"] == "warp_stream_kernel" and info["rows_per_cta"] == 0
    monkeypatch.setenv("TK_KERNEL", "block")
    assert tk.SwigluQuant(2048, 128).launch_info(1024)["kernel"] == "block_stream_kernel"
    assert tk.SwigluQuant(1040, 16).launch_info(1024)["kernel"] == "row_quant_kernel"   # does not apply


def test_back_to_back_launches_see_the_previous_output():
    """Launches may be scheduled while the previous kernel of the stream
    drains; each waits for it before reading. Chain the fused kernel into a
    cast that reads the fused kernel's fp32 scales as its input, on one stream
    with no synchronisation in between, and compare with a synchronised run."""
    wl = wls.WORKLOADS["moe_T8192_H2048_g128"]
    x, w = wls.make_inputs(wl, "cuda")
    op = _op(wl)
    cast = tk.QuantCast(16, 16, "fp32", "e4m3", "fp32")
    ref_s = None
    for chained in (False, True):
        s = torch.full((wl.T, 16), -1.0, device="cuda")
        q = torch.empty((wl.T, wl.H), dtype=torch.uint8, device="cuda")
        for _ in range(3):
            s.fill_(-1.0)
            op(x, w, q=q, scales=s)
            if not chained:
                torch.cuda.synchronize()
            q2, s2 = cast(s)
        torch.cuda.synchronize()
        if ref_s is None:
            ref_s = (s.clone(), q2.clone(), s2.clone())
        else:
            assert torch.equal(s, ref_s[0]) and torch.equal(q2, ref_s[1]) and torch.equal(s2, ref_s[2])
    assert bool((ref_s[0] > 0).all())


@pytest.mark.parametrize("stages", [2, 3, 5, 8])
def test_stream_ring_depths(stages, monkeypatch):
    monkeypatch.setenv("TK_PIPELINE_STAGES", str(stages))
    monkeypatch.setenv("TK_KERNEL", "stream")
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(5000)
    op = _op(wl, count=True)
    x, w = wls.make_inputs(wl, "cpu")
    counts = torch.zeros(2, dtype=torch.int64, device="cuda")
    q, s = _run(op, x.cuda(), w.cuda(), counts)
    ref = _oracle(wl, x, w)
    compare(q.cpu().numpy(), s.cpu().numpy(), ref, wl.group, wl.scale_fmt, wl.out_fmt).check(str(stages))
    assert counts.cpu().tolist() == ref["counts"].tolist()


def test_fault_word_clear_after_runs():
    torch.cuda.synchronize()
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0


# ------------------------------------------------------------ scale layouts

@pytest.mark.parametrize("kernel", ["rows", "stream", "block"])
@pytest.mark.parametrize("layout,scale_fmt,group,out_fmt", [
    ("col", "fp32", 128, "e4m3"), ("col", "ue8m0", 128, "e4m3"), ("col_packed", "ue8m0", 128, "e4m3"),
    ("col_packed", "ue8m0", 32, "e2m1"), ("col", "fp32", 0, "e4m3")])
@pytest.mark.parametrize("T", [1, 29, 1001])
def test_scale_layouts(kernel, layout, scale_fmt, group, out_fmt, T, monkeypatch):
    """Scales written column-major (padded to 16 bytes per column) or as
    packed UE8M0 words match the oracle's row-major scales moved by the
    oracle's layout function; padding is left untouched and the codes are
    those of the row-major run."""
    monkeypatch.setenv("TK_KERNEL", kernel)
    H = 2048
    wl = wls.WORKLOADS["moe_T32768_H2048_g128_ue8m0_clamp7"].with_rows(T)
    x, w = wls.make_inputs(wl, "cpu")
    fused = tk.SwigluQuant(H, group, scale_fmt, out_fmt, True, 7.0, False, scale_layout=layout)
    flat = tk.SwigluQuant(H, group, scale_fmt, out_fmt, True, 7.0, False)
    q_ref, s_ref = _run(flat, x.cuda(), w.cuda())
    q_shape, s_shape, s_dtype = fused.output_shapes(T)
    sentinel = 0xA7
    s_buf = torch.full(s_shape, 0, dtype=s_dtype, device="cuda")
    s_buf.view(torch.uint8).fill_(sentinel)
    q, s = fused(x.cuda(), w.cuda(), scales=s_buf)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref)
    want = oracle.scales_to_layout(s_ref.cpu().numpy(), scale_fmt, layout, fill=sentinel)
    got = s.cpu().contiguous().view(torch.uint8).numpy().reshape(-1)
    assert np.array_equal(got, want)
    # and the same layouts from the standalone cast (fp32 input, bit-exact)
    y = torch.randn(T, H) * 3
    cast = tk.QuantCast(H, group, scale_fmt, out_fmt, "fp32", scale_layout=layout)
    cs_buf = torch.full(s_shape, 0, dtype=s_dtype, device="cuda")
    cs_buf.view(torch.uint8).fill_(sentinel)
    cq, cs = cast(y.cuda(), scales=cs_buf)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_rows_f32(y.numpy(), group, scale_fmt, out_fmt)
    assert np.array_equal(cq.cpu().numpy(), rq)
    want = oracle.scales_to_layout(rs, scale_fmt, layout, fill=sentinel)
    got = cs.cpu().contiguous().view(torch.uint8).numpy().reshape(-1)
    assert np.array_equal(got, want)


def test_host_pipe_refuses_column_major_scales():
    op = tk.SwigluQuant(2048, 128, "fp32", "e4m3", True, scale_layout="col")
    with pytest.raises(tk.TkError) as e:
        pipe = tk.HostPipe(op, 64)
        pipe(torch.zeros(8, 4096, dtype=torch.bfloat16), torch.ones(8),
             q=torch.empty(8, 2048, dtype=torch.uint8), scales=torch.empty(op.output_shapes(8)[1]))
    assert e.value.status == 2


@pytest.mark.parametrize("H,group,scale_fmt,out_fmt,clamp", [
    (512, 128, "fp32", "e4m3", None), (2048, 128, "ue8m0", "e4m3", 7.0), (3072, 128, "fp32", "e4m3", None),
    (2048, 32, "ue8m0", "e2m1", 7.0), (7168, 128, "ue8m0", "e4m3", None)])
def test_block_ring_equals_row_kernel_at_block_boundaries(H, group, scale_fmt, out_fmt, clamp, monkeypatch):
    """The block-ring kernel runs the row kernel's arithmetic, so codes, scales
    and clamp counters agree bit for bit; row counts around whole blocks and
    around one block per CTA exercise ragged last blocks and grids smaller
    than the resident maximum."""
    ops = {}
    for kernel in ("rows", "block"):
        monkeypatch.setenv("TK_KERNEL", kernel)
        ops[kernel] = tk.SwigluQuant(H, group, scale_fmt, out_fmt, True, clamp, clamp is not None)
    info = ops["block"].launch_info(1 << 30)
    assert info["kernel"] == "block_stream_kernel"
    rb, grid = info["rows_per_cta"], info["grid"]
    rng = np.random.default_rng(H + group)
    for T in sorted({1, rb - 1, rb, rb + 1, grid * rb - 1, grid * rb, grid * rb + 1, 2 * grid * rb + 3} - {0}):
        x = torch.from_numpy(rng.standard_normal((T, 2 * H)).astype(np.float32) * 3).to(torch.bfloat16).cuda()
        w = torch.from_numpy(rng.uniform(0.0, 1.0, T).astype(np.float32)).cuda()
        out = {}
        for kernel, op in ops.items():
            counts = torch.zeros(2, dtype=torch.int64, device="cuda") if clamp is not None else None
            q, s = _run(op, x, w, counts)
            out[kernel] = (q, s, counts)
        torch.cuda.synchronize()
        (q0, s0, c0), (q1, s1, c1) = out["rows"], out["block"]
        assert torch.equal(q0, q1) and torch.equal(s0.view(torch.uint8), s1.view(torch.uint8)), (H, T)
        if clamp is not None:
            assert torch.equal(c0, c1), (H, T)
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0


@pytest.mark.parametrize("kernel", ["rows", "block"])
def test_every_row_count_up_to_257(kernel, monkeypatch):
    """Every batch size from 1 to 257 rows against the oracle, clamp counters
    included: every ragged tail of the row blocks and of the block ring's
    slots (16 rows at this width)."""
    monkeypatch.setenv("TK_KERNEL", kernel)
    H, g, L = 512, 128, 7.0
    op = tk.SwigluQuant(H, g, "ue8m0", "e4m3", True, L, True)
    rng = np.random.default_rng(257)
    xr = _bf16(rng.standard_normal((257, 2 * H)) * 3)
    wr = torch.from_numpy(rng.uniform(0.0, 1.0, 257).astype(np.float32))
    xc, wc = xr.cuda(), wr.cuda()
    for T in range(1, 258):
        counts = torch.zeros(2, dtype=torch.int64, device="cuda")
        q, s = _run(op, xc[:T], wc[:T], counts)
        ref = oracle.swiglu_quant(wls.bf16_bits(xr[:T]), wr[:T].numpy(), g, "ue8m0", "e4m3", clamp=L, want_y=True)
        compare(q.cpu().numpy(), s.cpu().numpy(), ref, g, "ue8m0", "e4m3").check("%s T=%d" % (kernel, T))
        assert counts.cpu().tolist() == ref["counts"].tolist(), T
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0
