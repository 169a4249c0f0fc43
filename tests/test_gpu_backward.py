"""Parity of the SwiGLU backward (tk_swiglu_backward_run) with the CPU oracle,
through the C ABI.

The oracle evaluates the gradients in double and rounds once (bf16 dx, fp32
dw). The kernel evaluates them in fp32 from the forward's t = e^{-|g'|}
(hardware exp2, squared) and r = 1/(1 + t) (hardware reciprocal), each a
few fp32 ulps off, so an output may differ from the oracle by one bf16 ulp
plus a small multiple of the magnitudes that build it:
  dgate: 2^-17 * |dy w u'| * (p + |silu| q) * r   (silu' = (silu q + p) r, p q = t,
                                                   p + q = 1 + t; it cancels near
                                                   its zero at g' = -1.28)
  dup:   2^-17 * |dy w silu|
  dw:    (H + 64) * 2^-24 * S + 2^-17 * S,  S = sum |dy silu u'|   (fp32 row sum)
2^-17 is 128 fp32 ulps, far below one bf16 step (2^-8): a wrong term would
show as an O(1) relative error. At least 99.9% of dx must also be identical.
The recomputed codes and scales must equal the forward kernel's bit for bit;
clamped elements' gradients are exactly +0 on both sides.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle

import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def check_backward(xb, db, w, L, dx_got, dw_got, what):
    """Compare the kernel's dx (bf16 bits) and dw with the oracle under the bounds above."""
    dx_want, dw_want = oracle.swiglu_backward(xb, db, w, clamp=L)
    T, H = db.shape
    xv, d = _f64(xb), _f64(db)
    g, u = xv[:, :H], xv[:, H:]
    if L is not None:
        g, u = np.minimum(g, L), np.clip(u, -L, L)
    wv = np.ones((T, 1)) if w is None else w.astype(np.float64)[:, None]
    sig = expit(g)
    silu = g * sig
    t = np.exp(-np.abs(g))
    r = 1.0 / (1.0 + t)
    p = np.where(g >= 0, 1.0, t)
    q = np.where(g >= 0, t, 1.0)
    bound = np.concatenate([np.abs(d * wv * u) * (p + np.abs(silu) * q) * r, np.abs(d * wv * silu)], axis=1)
    got, want = _f64(dx_got), _f64(dx_want)
    m = np.maximum(np.abs(got), np.abs(want))
    ulp = np.exp2(np.floor(np.log2(np.maximum(m, 2.0 ** -126))) - 7)
    excess = np.abs(got - want) - (ulp + 2.0 ** -17 * bound)
    if excess.size:
        i = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess.max() <= 0, "%s: dx%s = %g, oracle %g, bound %g" % (what, i, got[i], want[i], bound[i])
    same = float((dx_got == dx_want).mean()) if dx_got.size else 1.0
    assert same >= 0.999, "%s: only %.5f of dx identical" % (what, same)
    if dw_got is not None:
        S = np.abs(d * silu * u).sum(axis=1)
        dwg = dw_got.astype(np.float64)
        dww = dw_want.astype(np.float64)
        ulp32 = np.exp2(np.floor(np.log2(np.maximum(np.abs(dww), 2.0 ** -126))) - 23)
        tol = ulp32 + (H + 64) * 2.0 ** -24 * S + 2.0 ** -17 * S
        err = np.abs(dwg - dww)
        assert (err <= tol).all(), "%s: dw off by %g (bound %g)" % (what, err.max(), tol[np.argmax(err - tol)])
    return same


def _case(T, H, seed, dist="row_lognormal", clamp=None):
    wl = wls.Workload("b", T, H, 128 if H % 128 == 0 else 16, "fp32", "e4m3", dist, w_dist="topk8_norm",
                      clamp=clamp, seed=seed, op="backward")
    return wls.make_backward_inputs(wl, "cpu")


def _run(op, x, dy, w, want_dw=True):
    dx, dw, q, s = op(x.cuda(), dy.cuda(), None if w is None else w.cuda(), want_dw=want_dw)
    torch.cuda.synchronize()
    return dx, dw, q, s


@pytest.mark.parametrize("name", list(wls.BACKWARD_WORKLOADS))
def test_backward_small_parity(name):
    """Enough rows for every CTA of the grid to take two row blocks, plus a tail."""
    wl = wls.BACKWARD_WORKLOADS[name]
    op = tk.SwigluBackward(wl.H, True, wl.clamp)
    rows = 2 * 152 * 4 * 2 + 37
    x, w, dy = wls.make_backward_inputs(wl.with_rows(rows), "cpu")
    dx, dw, _, _ = _run(op, x, dy, w)
    same = check_backward(wls.bf16_bits(x), wls.bf16_bits(dy), w.numpy(), wl.clamp, _bits(dx),
                          dw.cpu().numpy(), name)
    print(name, rows, "rows: dx identical %.6f" % same)


@pytest.mark.parametrize("clamp", [None, 1.5, 1.3])   # 1.5 is a bf16 value (bf16-pair clamp), 1.3 is not (fp32)
@pytest.mark.parametrize("weights", [True, False])
@pytest.mark.parametrize("H", [16, 32, 64, 128, 256, 512, 1536, 3072, 7168, 8192])
def test_backward_shapes(H, weights, clamp):
    T = 301
    x, w, dy = _case(T, H, seed=H + 3 * int(weights) + (5 if clamp else 0), clamp=clamp)
    op = tk.SwigluBackward(H, weights, clamp)
    wv = w if weights else None
    dx, dw, _, _ = _run(op, x, dy, wv)
    check_backward(wls.bf16_bits(x), wls.bf16_bits(dy), None if wv is None else wv.numpy(), clamp, _bits(dx),
                   dw.cpu().numpy(), "H=%d w=%s L=%s" % (H, weights, clamp))


@pytest.mark.parametrize("layout", ["row", "col", "col_packed"])
@pytest.mark.parametrize("fmt", [("fp32", "e4m3", 128), ("ue8m0", "e4m3", 128), ("ue8m0", "e2m1", 32),
                                 ("fp32", "e4m3", 512)])
@pytest.mark.parametrize("clamp", [None, 7.0])
def test_backward_recompute_equals_forward(fmt, layout, clamp):
    scale_fmt, out_fmt, group = fmt
    if layout == "col_packed" and scale_fmt != "ue8m0":
        pytest.skip("the packed layout holds UE8M0 exponents")
    H, T = 2048, 1000
    x, w, dy = _case(T, H, seed=group + len(layout), dist="outliers", clamp=clamp)
    fwd = tk.SwigluQuant(H, group, scale_fmt, out_fmt, True, clamp, scale_layout=layout)
    bwd = tk.SwigluBackward(H, True, clamp, recompute=dict(group_size=group, scale_fmt=scale_fmt, out_fmt=out_fmt,
                                                         scale_layout=layout))
    xc, wc, dc = x.cuda(), w.cuda(), dy.cuda()
    q0, s0 = fwd(xc, wc)
    dx, dw, q1, s1 = bwd(xc, dc, wc)
    dx2, dw2, _, _ = tk.SwigluBackward(H, True, clamp)(xc, dc, wc)
    torch.cuda.synchronize()
    if layout == "row":
        assert torch.equal(q0, q1) and torch.equal(s0, s1)
    else:   # padding entries of the column layouts are not written: compare the codes and written scales
        assert torch.equal(q0, q1)
        ref = oracle.swiglu_quant(wls.bf16_bits(x), w.numpy(), group, scale_fmt, out_fmt, clamp=clamp)
        mask = oracle.scales_to_layout(np.ones_like(ref["scales"]), scale_fmt, layout, fill=0) != 0
        b0 = s0.cpu().numpy().view(np.uint8).reshape(-1)
        b1 = s1.cpu().numpy().view(np.uint8).reshape(-1)
        assert np.array_equal(b0[mask], b1[mask])
    # the gradients do not depend on the recompute
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2)


@pytest.mark.parametrize("name", list(wls.BACKWARD_WORKLOADS))
def test_backward_full_size_and_deterministic(name):
    """The workloads the benchmark times, at full size and in its launch
    configuration (the plan's prefetch form): runs repeat bit for bit, the
    recomputed codes equal the forward kernel's, sampled rows match the
    oracle."""
    wl = wls.BACKWARD_WORKLOADS[name]
    x, w, dy = wls.make_backward_inputs(wl, "cuda")
    op = tk.SwigluBackward(wl.H, True, wl.clamp, recompute=dict(group_size=wl.group, scale_fmt=wl.scale_fmt,
                                                                out_fmt=wl.out_fmt))
    dx, dw, q, s = op(x, dy, w)
    dx2, dw2, q2, s2 = op(x, dy, w)
    q0, s0 = tk.SwigluQuant(wl.H, wl.group, wl.scale_fmt, wl.out_fmt, True, wl.clamp)(x, w)
    torch.cuda.synchronize()
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2)          # fixed-order sums: runs repeat
    assert torch.equal(q, q0) and torch.equal(s, s0)
    rng = np.random.default_rng(wl.seed)
    idx = np.unique(np.concatenate([np.arange(8), np.arange(wl.T - 8, wl.T), rng.choice(wl.T, 112, replace=False)]))
    xi, di = x[idx].cpu(), dy[idx].cpu()
    check_backward(wls.bf16_bits(xi), wls.bf16_bits(di), w[idx].cpu().numpy(), wl.clamp, _bits(dx[idx]),
                   dw[idx].cpu().numpy(), "full")
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0


def test_backward_without_dw_and_zero_rows():
    H, T = 512, 50
    x, w, dy = _case(T, H, seed=77)
    op = tk.SwigluBackward(H, True)
    dx_a, dw_a, _, _ = _run(op, x, dy, w)
    dx_b, dw_b, _, _ = _run(op, x, dy, w, want_dw=False)
    assert dw_b is None and torch.equal(dx_a, dx_b)
    # zero rows: nothing happens
    op(torch.empty((0, 2 * H), dtype=torch.bfloat16, device="cuda"),
       torch.empty((0, H), dtype=torch.bfloat16, device="cuda"), torch.empty((0,), device="cuda"))
    torch.cuda.synchronize()


def test_backward_host_side_errors():
    H, T = 256, 8
    op = tk.SwigluBackward(H, True)
    x = torch.zeros((T, 2 * H + 16), dtype=torch.bfloat16, device="cuda")
    dy = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((T, 2 * H), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(T, device="cuda")
    run = tk.tk_swiglu_backward_run
    with pytest.raises(tk.TkError) as e:   # x not 32-byte aligned
        run(op.plan, T, x.data_ptr() + 16, w, dy, dx, None, None, None, None)
    assert e.value.status == 3
    with pytest.raises(tk.TkError) as e:   # the plan expects weights
        run(op.plan, T, x, None, dy, dx, None, None, None, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:   # dy missing
        run(op.plan, T, x, w, None, dx, None, None, None, None)
    assert e.value.status == 1
    rec = tk.SwigluBackward(H, True, recompute=dict(group_size=128))
    with pytest.raises(tk.TkError) as e:   # the recompute needs q and scales
        run(rec.plan, T, x, w, dy, dx, None, None, None, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:
        tk.SwigluBackward(96, True)
    assert e.value.status == 2


def test_backward_guard_bands_untouched():
    """dx, dw, the codes and the scales live inside larger buffers filled with
    a sentinel; only their bytes may change."""
    H, T, pad = 2048, 97, 512
    x, w, dy = _case(T, H, seed=5, clamp=7.0)
    op = tk.SwigluBackward(H, True, 7.0, recompute=dict(group_size=128, scale_fmt="ue8m0", out_fmt="e4m3"))
    bufs = {
        "dx": torch.full((T * 2 * H + 2 * pad,), 0x5A5A, dtype=torch.int16, device="cuda"),
        "dw": torch.full((T + 2 * pad,), -3.0, dtype=torch.float32, device="cuda"),
        "q": torch.full((T * H + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda"),
        "s": torch.full((T * (H // 128) + 2 * pad,), 0xA5, dtype=torch.uint8, device="cuda"),
    }
    dx = bufs["dx"][pad:pad + T * 2 * H].view(torch.bfloat16).view(T, 2 * H)
    dw = bufs["dw"][pad:pad + T]
    q = bufs["q"][pad:pad + T * H].view(T, H)
    s = bufs["s"][pad:pad + T * (H // 128)].view(T, H // 128)
    op(x.cuda(), dy.cuda(), w.cuda(), dx=dx, dw=dw, q=q, scales=s)
    torch.cuda.synchronize()
    for name, b in bufs.items():
        fill = b[0].item()
        n = b.numel() - 2 * pad
        assert bool((b[:pad] == fill).all()) and bool((b[pad + n:] == fill).all()), name
