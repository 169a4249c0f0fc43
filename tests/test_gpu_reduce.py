"""Parity of the weighted top-k combine (tk_moe_reduce) with the CPU oracle,
through the C ABI.

The oracle sums in double and rounds once to bf16. The kernel accumulates in
fp32 with one FMA per slot in k order (E4M3 rows first form fl(w * s)), scales
by gs and rounds once to bf16. With u = 2^-24 and S = sum_k |w_k deq(y_k)|,
the fp32 value before the last rounding lies within (K + 2) u |gs| S of the
exact gs * sum (recursive summation with one rounding per step, plus the
w * s product and the final multiply by gs). Two round-to-nearest results of
values that close differ by at most that much plus one bf16 ulp at the larger
magnitude. That is the per-element bound every test here checks. Where the
terms cancel, one bf16 step of the small result is less than the fp32 error,
so no fixed step count would hold. A bound is no proof of rounding parity, so
the tests also require at least 99.9% of the outputs to be identical; an fp32
emulation of this order matches the oracle on about 99.995%. One slot with
weight 1 (an exact copy) and no slots (zeros) must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import activation_fp8_quantization_gb300 as tk
from activation_fp8_quantization_gb300 import workloads as wls

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16_value(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _abs_terms(d: dict, tokens: np.ndarray) -> np.ndarray:
    """S[t, :] = sum over valid slots of |w[t,k] * deq(y[pos[t,k], :])|, in float64."""
    pos = d["pos"].cpu().numpy()[tokens]
    w = d["w"].cpu().numpy()[tokens].astype(np.float64)
    y = d["y"].cpu()
    if d["y_scale"] is None:
        yv = y.float().numpy().astype(np.float64)
        ys = None
    else:
        yv = oracle.e4m3_decode_table()[y.numpy()]
        ys = d["y_scale"].cpu().numpy().astype(np.float64)
    S = np.zeros((len(tokens), yv.shape[1]))
    for k in range(pos.shape[1]):
        r = pos[:, k]
        ok = (r >= 0) & (r < yv.shape[0])
        rr = np.where(ok, r, 0)
        term = np.abs(yv[rr]) * np.abs(w[:, k])[:, None]
        if ys is not None:
            term *= np.repeat(ys[rr], 128, axis=1)
        S += np.where(ok[:, None], term, 0.0)
    return S


def check_close(got: np.ndarray, want: np.ndarray, d: dict, tokens=None, what=""):
    """Element-wise bound (module docstring) plus an identical-fraction floor."""
    if tokens is None:
        tokens = np.arange(got.shape[0])
    K = d["pos"].shape[1]
    gv, wv = _bf16_value(got), _bf16_value(want)
    m = np.maximum(np.abs(gv), np.abs(wv))
    ulp = np.exp2(np.floor(np.log2(np.maximum(m, 2.0 ** -126))) - 7)
    u = 2.0 ** -24
    tol = ulp + abs(d["gs"]) * (K + 2) * u / (1 - (K + 2) * u) * _abs_terms(d, tokens)
    excess = np.abs(gv - wv) - tol
    worst = np.unravel_index(np.argmax(excess), excess.shape) if excess.size else None
    assert excess.size == 0 or excess.max() <= 0, (
        "%s: output %s is %g from the oracle's %g (bound %g)" % (
            what, worst, gv[worst], wv[worst], tol[worst]))
    same = float((got == want).mean()) if got.size else 1.0
    assert same >= 0.999, "%s: only %.5f identical" % (what, same)
    return same


def _oracle(d: dict, pos_rows=None):
    pos = d["pos"].cpu().numpy()
    w = d["w"].cpu().numpy()
    if pos_rows is not None:
        pos, w = pos[pos_rows], w[pos_rows]
    if d["y_scale"] is None:
        return oracle.moe_reduce(_bits(d["y"]), pos, w, d["gs"])
    return oracle.moe_reduce(d["y"].cpu().numpy(), pos, w, d["gs"], y_scale=d["y_scale"].cpu().numpy())


def _run(op, d):
    out = op(d["y"], d["pos"], d["w"], d["gs"], y_scale=d["y_scale"])
    torch.cuda.synchronize()
    return out


KERNELS = ["regs", "bulk"]


def _plan(monkeypatch, kernel, H, K, in_fmt="bf16"):
    """A plan made with the kernel choice forced (read when the plan is made)."""
    monkeypatch.setenv("TK_REDUCE_KERNEL", kernel)
    op = tk.MoeReduce(H, K, in_fmt)
    monkeypatch.delenv("TK_REDUCE_KERNEL")
    return op


def _expect_kernel(op, d, kernel):
    info = op.launch_info(d["pos"].shape[0], d["y"], d["y_scale"])
    bulk_ok = op.topk <= 32 and op.hidden * (2 if op.in_fmt == "bf16" else 1) >= 2048 and (
        op.in_fmt == "bf16" or op.hidden % 512 == 0)
    assert info["kernel"] == ("bulk" if kernel == "bulk" and bulk_ok else "regs"), info
    return info


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", list(wls.REDUCE_WORKLOADS))
def test_reduce_small_parity(name, kernel, monkeypatch):
    wl = wls.REDUCE_WORKLOADS[name].with_rows(3001)
    d = wls.make_reduce_inputs(wl, "cuda")
    op = _plan(monkeypatch, kernel, wl.H, wl.topk, wl.in_dtype)
    _expect_kernel(op, d, kernel)
    got = _bits(_run(op, d))
    same = check_close(got, _oracle(d), d, what=name)
    print(name, kernel, "identical %.6f" % same)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", list(wls.REDUCE_WORKLOADS))
def test_reduce_full_size(name, kernel, monkeypatch):
    wl = wls.REDUCE_WORKLOADS[name]
    d = wls.make_reduce_inputs(wl, "cuda")
    op = _plan(monkeypatch, kernel, wl.H, wl.topk, wl.in_dtype)
    _expect_kernel(op, d, kernel)
    tk.tk_fault_word(torch.cuda.current_device(), clear=True)
    out = _run(op, d)
    rng = np.random.default_rng(wl.seed)
    idx = np.unique(np.concatenate([np.arange(16), np.arange(wl.T - 16, wl.T),
                                    rng.choice(wl.T, 192, replace=False)]))
    got = _bits(out)[idx]
    check_close(got, _oracle(d, idx), d, idx, name + " full")
    assert tk.tk_fault_word(torch.cuda.current_device()) == 0


def _random_case(H, K, in_fmt, T, seed):
    R = 3 * T + 1
    g = torch.Generator().manual_seed(seed)
    if in_fmt == "bf16":
        y = torch.randn((R, H), generator=g).to(torch.bfloat16)
        ys = None
    else:
        y = torch.randint(0, 256, (R, H), generator=g, dtype=torch.int32).to(torch.uint8)
        y[(y & 0x7F) == 0x7F] = 1
        ys = torch.exp2(torch.rand((R, H // 128), generator=g) * 6 - 3)
    # positions may repeat (rows shared by tokens) and include empty slots
    pos = torch.randint(-1, R, (T, K), generator=g, dtype=torch.int32)
    w = torch.rand((T, K), generator=g)
    return {"y": y.cuda(), "y_scale": None if ys is None else ys.cuda(), "pos": pos.cuda(), "w": w.cuda(),
            "gs": 0.5}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("in_fmt", ["bf16", "e4m3"])
@pytest.mark.parametrize("H,K", [(16, 1), (48, 3), (128, 17), (1024, 5), (2048, 8), (4096, 32),
                                 (7168, 8), (8192, 2), (8192, 33)])
def test_reduce_shapes(H, K, in_fmt, kernel, monkeypatch):
    if in_fmt == "e4m3" and H % 128:
        pytest.skip("E4M3 rows need 1x128 scale groups")
    d = _random_case(H, K, in_fmt, 77, H * 31 + K)
    op = _plan(monkeypatch, kernel, H, K, in_fmt)
    _expect_kernel(op, d, kernel)
    got = _bits(_run(op, d))
    check_close(got, _oracle(d), d, what="H=%d K=%d %s %s" % (H, K, in_fmt, kernel))


@pytest.mark.parametrize("in_fmt", ["bf16", "e4m3"])
@pytest.mark.parametrize("H,K,T", [(1024, 1, 1), (2048, 8, 5), (2048, 3, 151), (4096, 17, 153),
                                   (7168, 8, 300), (7168, 32, 64), (8192, 8, 1000), (3584, 6, 77)])
def test_reduce_kernels_agree_bit_for_bit(H, K, T, in_fmt, monkeypatch):
    """Both kernels take the same arithmetic in the same order: identical bits,
    including where tokens are fewer than CTAs and where a token spans chunks."""
    if in_fmt == "e4m3" and H % 128:
        pytest.skip("E4M3 rows need 1x128 scale groups")
    d = _random_case(H, K, in_fmt, T, H + 7 * K + T)
    outs = {}
    for kernel in KERNELS:
        op = _plan(monkeypatch, kernel, H, K, in_fmt)
        _expect_kernel(op, d, kernel)
        outs[kernel] = _bits(_run(op, d))
    assert np.array_equal(outs["regs"], outs["bulk"])
    check_close(outs["bulk"], _oracle(d), d, what="H=%d K=%d T=%d %s" % (H, K, T, in_fmt))


def test_reduce_unaligned_scales_take_the_register_kernel():
    H, K, T = 2048, 8, 50
    d = _random_case(H, K, "e4m3", T, 5)
    R = d["y"].shape[0]
    buf = torch.empty(R * (H // 128) + 1, dtype=torch.float32, device="cuda")
    ys = buf[1:].view(R, H // 128)          # 4-byte but not 16-byte aligned
    ys.copy_(d["y_scale"])
    op = tk.MoeReduce(H, K, "e4m3")
    assert op.launch_info(T, d["y"], d["y_scale"])["kernel"] == "bulk"
    assert op.launch_info(T, d["y"], ys)["kernel"] == "regs"
    a = _bits(_run(op, d))
    b = _bits(_run(op, dict(d, y_scale=ys)))
    assert np.array_equal(a, b)


def test_reduce_exact_cases():
    H, T, R = 1024, 64, 200
    y = torch.randn((R, H)).to(torch.bfloat16).cuda()
    # one slot, weight 1, scale 1: a bit-exact gather
    perm = torch.randperm(R)[:T].to(torch.int32).view(T, 1).cuda()
    out = tk.MoeReduce(H, 1)(y, perm, torch.ones((T, 1)).cuda(), 1.0)
    torch.cuda.synchronize()
    assert torch.equal(out, y[perm.view(-1).long()])
    # no slots in use: zeros
    op = tk.MoeReduce(H, 4)
    out = op(y, torch.full((T, 4), -1, dtype=torch.int32).cuda(), torch.ones((T, 4)).cuda(), 3.0)
    torch.cuda.synchronize()
    assert not out.float().abs().max().item()
    # zero tokens: nothing happens
    op(y, torch.empty((0, 4), dtype=torch.int32).cuda(), torch.empty((0, 4)).cuda(), 1.0)


@pytest.mark.parametrize("H", [256, 2048])
def test_reduce_invalid_positions_are_skipped_and_flagged(H):
    """Also run through the bulk kernel below (E4M3 rows take it by default)."""
    T, R, K = 32, 50, 2
    dev = torch.cuda.current_device()
    tk.tk_fault_word(dev, clear=True)
    y = torch.randn((R, H)).to(torch.bfloat16).cuda()
    pos = torch.tensor([[0, R]] * (T // 2) + [[1, -7]] * (T // 2), dtype=torch.int32).cuda()
    w = torch.ones((T, K)).cuda()
    op = tk.MoeReduce(H, K)
    assert op.launch_info(T, y)["kernel"] == "regs"       # bf16 rows: the register kernel by default
    out = op(y, pos, w, 1.0)
    torch.cuda.synchronize()
    assert tk.tk_fault_word(dev, clear=True) & 2
    # the bad slot contributed nothing
    assert torch.equal(out[: T // 2], y[0].expand(T // 2, H))
    assert torch.equal(out[T // 2:], y[1].expand(T // 2, H))
    assert tk.tk_fault_word(dev) == 0


def test_reduce_invalid_positions_bulk_kernel():
    H, T, R, K = 2048, 32, 50, 2
    dev = torch.cuda.current_device()
    tk.tk_fault_word(dev, clear=True)
    y = torch.randint(0, 0x7E, (R, H), dtype=torch.int32).to(torch.uint8).cuda()
    ys = torch.full((R, H // 128), 0.5).cuda()
    pos = torch.tensor([[0, R]] * (T // 2) + [[1, -7]] * (T // 2), dtype=torch.int32).cuda()
    w = torch.ones((T, K)).cuda()
    op = tk.MoeReduce(H, K, "e4m3")
    assert op.launch_info(T, y, ys)["kernel"] == "bulk"
    out = op(y, pos, w, 1.0, y_scale=ys)
    torch.cuda.synchronize()
    assert tk.tk_fault_word(dev, clear=True) & 2
    one = tk.MoeReduce(H, 1, "e4m3")   # the valid slot alone, through the same kernel
    want0 = one(y, torch.zeros((T // 2, 1), dtype=torch.int32).cuda(), torch.ones((T // 2, 1)).cuda(), 1.0,
                y_scale=ys)
    want1 = one(y, torch.ones((T // 2, 1), dtype=torch.int32).cuda(), torch.ones((T // 2, 1)).cuda(), 1.0,
                y_scale=ys)
    torch.cuda.synchronize()
    assert torch.equal(out[: T // 2], want0)
    assert torch.equal(out[T // 2:], want1)
    assert tk.tk_fault_word(dev) == 0


def test_reduce_host_side_errors():
    op = tk.MoeReduce(256, 2)
    y = torch.zeros((10, 256 + 16), dtype=torch.bfloat16).cuda()
    pos = torch.zeros((4, 2), dtype=torch.int32).cuda()
    w = torch.ones((4, 2)).cuda()
    out = torch.empty((4, 256), dtype=torch.bfloat16).cuda()
    with pytest.raises(tk.TkError) as e:   # rows not 32-byte aligned
        tk.tk_moe_reduce_run(op.plan, 4, y.data_ptr() + 2, None, 10, pos, w, 1.0, out, None)
    assert e.value.status == 3
    with pytest.raises(tk.TkError) as e:
        tk.tk_moe_reduce_run(op.plan, 4, y, None, 10, None, w, 1.0, out, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:
        tk.tk_moe_reduce_run(op.plan, 4, y, None, 10, pos, w, float("nan"), out, None)
    assert e.value.status == 1
    with pytest.raises(tk.TkError) as e:     # a width that is not a multiple of 16
        tk.tk_moe_reduce_plan(tk.MoeReduceDesc(200, 2, 0), 0)
    assert e.value.status == 2


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", list(wls.REDUCE_WORKLOADS))
def test_reduce_guard_bands_untouched(name, kernel, monkeypatch):
    """The output lives inside a larger buffer filled with a sentinel; only
    its bytes may change."""
    rw = wls.REDUCE_WORKLOADS[name].with_rows(97)
    d = wls.make_reduce_inputs(rw, "cuda")
    monkeypatch.setenv("TK_REDUCE_KERNEL", kernel)
    op = tk.MoeReduce(rw.H, rw.topk, rw.in_dtype)
    pad, n = 512, rw.T * rw.H
    buf = torch.full((n + 2 * pad,), 0x5A5A, dtype=torch.int16, device="cuda")
    out = buf[pad:pad + n].view(torch.bfloat16).view(rw.T, rw.H)
    op(d["y"], d["pos"], d["w"], d["gs"], y_scale=d["y_scale"], out=out)
    torch.cuda.synchronize()
    assert bool((buf[:pad] == 0x5A5A).all()) and bool((buf[pad + n:] == 0x5A5A).all())
    assert not bool((buf[pad:pad + n] == 0x5A5A).all())
